"""GPU parity: syncbn_merge_apply against the fp64 oracle.

Tolerances (the computation is not bit-reproducible against fp64 by design:
fp32 partial sums, float-float merge, fp32 apply):
  mean               |gpu − oracle| <= 1e-5 · |oracle| + 1e-7 · σ_c
  invstd             |gpu − oracle| <= 1e-5 · |oracle|
  y (fp32 output)    |gpu − oracle| <= 1e-5 · |oracle| + 1e-6
  y (bf16 output)    within one bf16 ulp of the oracle's fp64 value rounded to
                     bf16, plus the fp32 allowance above (the fp32 result
                     may sit on the other side of a bf16 rounding boundary)
σ_c = 1/invstd_c is the channel's standard deviation.  The GPU sums x − K_c
in fp32, so its mean carries an absolute error of the order of the fp32
unit roundoff (6e-8) times the spread of the summed values, whatever the
mean: no relative bound can hold for a channel whose mean is near zero
(some test channels have means of 0.002 with σ_c = 2).  1e-7 · σ_c is
stricter than y needs: an error δ in the mean moves y by δ · invstd, and
y's absolute allowance of 1e-6 admits δ up to 1e-6 · σ_c.
The 1e-6 absolute term of y covers outputs near zero (x near the mean),
where a relative bound means nothing: there y's error is the fp32 rounding
of the shift β − m_lo·scale plus the mean's error times invstd·γ, both far
below 1e-6 for the inputs here (means of 0.5 or 1000 and standard
deviations of 2 or 0.1 computed to about 1e-7 relative).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_common import dev_bf16, dev_f32, load_library, sync

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    return load_library()


def _bf16_ulp(v):
    v = np.abs(np.asarray(v, np.float64))
    e = np.floor(np.log2(np.maximum(v, 2.0 ** -126)))
    return 2.0 ** (e - 7)


def _check_stats(mean, invstd, m_w, s_w, what):
    m = mean.cpu().numpy().astype(np.float64)
    s = invstd.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(m - m_w) <= 1e-5 * np.abs(m_w) + 1e-7 / s_w), what
    assert np.all(np.abs(s - s_w) <= 1e-5 * np.abs(s_w)), what


def _check_y(y_t, y_w, what):
    y_w = np.asarray(y_w, np.float64)
    if y_t.dtype == torch.bfloat16:
        got = y_t.float().cpu().numpy().astype(np.float64)
        want = oracle.f64_to_bf16_rne(y_w)
        tol = _bf16_ulp(want) * 1.0001 + 1e-5 * np.abs(y_w) + 1e-6
    else:
        got = y_t.cpu().numpy().astype(np.float64)
        want = y_w
        tol = 1e-5 * np.abs(y_w) + 1e-6
    err = np.abs(got - want)
    if not np.all(err <= tol):
        i = int(np.argmax(err - tol))
        raise AssertionError(f"{what}: {int((err > tol).sum())} of {err.size} outside tolerance; worst at flat "
                             f"{i}: gpu {got.reshape(-1)[i]!r} oracle {want.reshape(-1)[i]!r} "
                             f"(fp64 {y_w.reshape(-1)[i]!r}) tol {tol.reshape(-1)[i]!r}")


def _run(g, xs_dev, ys_dev, C, eps=1e-5, gamma=None, beta=None):
    n = len(xs_dev)
    B, _, H, W = xs_dev[0].shape
    ws = torch.empty(g.syncbn_workspace_bytes(n, B, C, H, W), dtype=torch.uint8, device="cuda")
    mean = torch.empty(C, device="cuda")
    invstd = torch.empty(C, device="cuda")
    g.syncbn_merge_apply(xs_dev, ys_dev, mean, invstd, ws, eps, gamma, beta)
    sync()
    return mean, invstd


@pytest.mark.parametrize("shape", [(2, 2, 3, 5, 7), (3, 4, 16, 8, 8), (8, 2, 5, 1, 1), (4, 3, 7, 7, 7),
                                   (1, 1, 1, 1, 1), (16, 1, 9, 4, 6), (2, 1, 7, 13, 17), (3, 5, 1000, 3, 3),
                                   (1, 1, 3, 111, 111), (2, 3, 5, 64, 64), (8, 32, 2048, 7, 7),
                                   (2, 2, 70, 3, 7), (2, 2, 300, 1, 5), (3, 2, 260, 1, 7),
                                   (2, 3, 4, 67, 8), (5, 3, 24, 7, 7), (2, 3, 12, 14, 14), (6, 5, 32, 5, 5),
                                   (3, 7, 40, 28, 28), (16, 2, 8, 56, 56), (2, 2, 40000, 2, 4),
                                   (2, 2, 512, 14, 14), (2, 1, 2048, 7, 7), (2, 3, 300, 4, 4), (2, 3, 200, 4, 8),
                                   (3, 2, 100, 8, 8)])
@pytest.mark.parametrize("io", [("bf16", "bf16"), ("bf16", "f32"), ("f32", "f32"), ("f32", "bf16")])
def test_small_shapes(g, shape, io):
    n, B, C, H, W = shape
    if shape == (8, 32, 2048, 7, 7) and io != ("bf16", "bf16"):
        pytest.skip("full-size shape checked once, bf16 in/out")
    xs = workloads.syncbn_input(4, n, B, C, H, W)
    gen = np.random.Generator(np.random.PCG64(C * H + W))
    gamma = gen.standard_normal(C).astype(np.float32)
    beta = gen.standard_normal(C).astype(np.float32)
    if io[0] == "f32":
        xs_f = [oracle.bf16_bits_to_f32(x) + np.float32(1e-3) * gen.standard_normal(x.shape).astype(np.float32)
                for x in xs]
        xs_dev = [dev_f32(x) for x in xs_f]
        m_w, s_w, y_w = oracle.syncbn(xs_f, 1e-5, gamma, beta, dtype="f32")
    else:
        xs_dev = [dev_bf16(x) for x in xs]
        m_w, s_w, y_w = oracle.syncbn(xs, 1e-5, gamma, beta)
    odt = torch.bfloat16 if io[1] == "bf16" else torch.float32
    ys = [torch.empty((B, C, H, W), dtype=odt, device="cuda") for _ in range(n)]
    mean, invstd = _run(g, xs_dev, ys, C, 1e-5, dev_f32(gamma), dev_f32(beta))
    _check_stats(mean, invstd, m_w, s_w, f"{shape} {io}")
    for r in range(n):
        _check_y(ys[r], y_w[r], f"{shape} {io} y[{r}]")


@pytest.mark.parametrize("shape", [(4, 2, 6, 5, 5), (4, 3, 6, 8, 16), (2, 4, 3, 28, 28)])
def test_in_place_and_defaults(g, shape):
    """y written over x, for unaligned (5x5) and aligned (8x16, 28x28)
    planes: the apply reads x through the coherent path when they alias."""
    n, B, C, H, W = shape
    xs = workloads.syncbn_input(4, n, B, C, H, W)
    xs_dev = [dev_bf16(x) for x in xs]
    mean, invstd = _run(g, xs_dev, xs_dev, C)
    m_w, s_w, y_w = oracle.syncbn(xs, 1e-5)
    _check_stats(mean, invstd, m_w, s_w, f"in place {shape}")
    for r in range(n):
        _check_y(xs_dev[r], y_w[r], f"in place {shape} y[{r}]")


def test_constant_channel(g):
    n, B, C, H, W = 2, 3, 4, 4, 4
    xs = workloads.syncbn_input(4, n, B, C, H, W)
    for x in xs:
        x[:, 2] = 0x4040   # 3.0
    xs_dev = [dev_bf16(x) for x in xs]
    ys = [torch.empty((B, C, H, W), device="cuda") for _ in range(n)]
    mean, invstd = _run(g, xs_dev, ys, C)
    assert mean[2].item() == 3.0
    assert abs(invstd[2].item() - 1 / np.sqrt(1e-5)) <= 1e-5 / np.sqrt(1e-5)
    assert all(float(y[:, 2].abs().max()) == 0.0 for y in ys)


@pytest.mark.parametrize("C,H,W", workloads.SYNCBN_SHAPES)
def test_full_size_shapes(g, C, H, W):
    """N = 8 replicas x [32, C, H, W] bf16 drawn N(0.5, 2) on the device, in
    the launch configuration the benchmark times.  Checked: mean and invstd
    of every channel against the fp64 oracle over every element, and y at
    2^16 random positions of every replica (all channels)."""
    n, B = 8, workloads.SYNCBN_BATCH
    xs = [workloads.device_normal((B, C, H, W), 0.5, 2.0, workloads.seed_for(4, r), dtype=torch.bfloat16)
          for r in range(n)]
    ys = [torch.empty_like(x) for x in xs]
    mean, invstd = _run(g, xs, ys, C)
    xh = [x.view(torch.int16).cpu().numpy().view(np.uint16) for x in xs]
    m_w, s_w = oracle.syncbn_stats(xh, 1e-5)
    _check_stats(mean, invstd, m_w, s_w, f"C={C} H={H} W={W}")
    gen = np.random.Generator(np.random.PCG64(C))
    E = B * C * H * W
    for r in range(n):
        pos = gen.integers(0, E, 1 << 16)
        c = (pos // (H * W)) % C
        xv = oracle.bf16_bits_to_f32(xh[r].reshape(-1)[pos]).astype(np.float64)
        y_w = (xv - m_w[c]) * s_w[c]
        got = ys[r].reshape(-1)[torch.from_numpy(pos).cuda()]
        _check_y(got, y_w, f"C={C} H={H} W={W} r={r}")


def test_large_mean_small_std(g):
    """|mean| >> std: fp32 activations N(1000, 0.1).  Q/M − mean² would
    cancel 8 decimal digits; the shifted sums keep invstd within tolerance."""
    n, B, C, H, W = 4, 8, 3, 16, 16
    gen = np.random.Generator(np.random.PCG64(1000))
    xs = [(gen.standard_normal((B, C, H, W)) * 0.1 + 1000.0).astype(np.float32) for _ in range(n)]
    ys = [torch.empty((B, C, H, W), device="cuda") for _ in range(n)]
    mean, invstd = _run(g, [dev_f32(x) for x in xs], ys, C)
    m_w, s_w, y_w = oracle.syncbn(xs, 1e-5, dtype="f32")
    _check_stats(mean, invstd, m_w, s_w, "large mean")
    # x − m_hi is exact (both within a factor of two of 1000) and the mean's low part goes into the
    # shift, so y keeps the ordinary fp32 tolerance although invstd ≈ 10 magnifies any error in the mean
    for r in range(n):
        _check_y(ys[r], y_w[r], f"large mean y[{r}]")


@pytest.mark.parametrize("shape,in_place", [((8, 32, 128, 28, 28), False), ((8, 32, 256, 14, 14), False),
                                            ((8, 32, 128, 28, 28), True), ((8, 32, 256, 14, 14), True),
                                            ((8, 32, 2048, 7, 7), True), ((8, 32, 256, 28, 28), False),
                                            ((8, 32, 256, 28, 28), True)])
def test_chained_layers_equal_separate_calls(g, shape, in_place):
    """Three SyncBN calls back to back on one stream, each reading the
    previous call's output: a call's apply reads its first vectors of x
    before waiting for its merge, so it must not start before the previous
    call's apply has written that x.  The chained result equals, bit for
    bit, the same three calls each followed by a device synchronisation
    (the kernels' reduction orders are fixed, so equal inputs give equal
    bits).  Aligned 28x28 planes (plane statistics; with 256 channels the
    call runs as two channel halves on two streams) and unaligned 14x14 and
    7x7 planes (bulk-staged statistics), out of place and in place."""
    n, B, C, H, W = shape
    xs = [dev_bf16(x) for x in workloads.syncbn_input(4, n, B, C, H, W)]
    ws = torch.empty(g.syncbn_workspace_bytes(n, B, C, H, W), dtype=torch.uint8, device="cuda")
    mean, invstd = torch.empty(C, device="cuda"), torch.empty(C, device="cuda")

    def three_layers(sync_each):
        cur = [x.clone() for x in xs]
        for _ in range(3):
            nxt = cur if in_place else [torch.empty_like(x) for x in cur]
            g.syncbn_merge_apply(cur, nxt, mean, invstd, ws)
            if sync_each:
                sync()
            cur = nxt
        sync()
        return [c.clone() for c in cur], mean.clone(), invstd.clone()

    sep, m_sep, s_sep = three_layers(True)
    for _ in range(3):
        got, m_got, s_got = three_layers(False)
        assert torch.equal(m_got.view(torch.int32), m_sep.view(torch.int32))
        assert torch.equal(s_got.view(torch.int32), s_sep.view(torch.int32))
        for r in range(n):
            assert torch.equal(got[r].view(torch.int16), sep[r].view(torch.int16)), f"replica {r}"


@pytest.mark.parametrize("shape", [(4, 2, 6, 8, 8), (4, 2, 6, 7, 7), (4, 2, 6, 16, 32)])
def test_non_finite_channel_stays_in_its_channel(g, shape):
    """A NaN in channel 1 and an infinity in channel 4 of one replica: those
    channels' statistics are not finite (the oracle's are not either), and
    every other channel's mean, invstd and output match the oracle, so a
    non-finite activation reaches no other channel (aligned 8x8 and
    unaligned 7x7 planes: bulk-staged statistics; aligned 16x32 planes:
    plane statistics)."""
    n, B, C, H, W = shape
    xs = workloads.syncbn_input(4, n, B, C, H, W)
    xs[2][1, 1, 3, 2] = 0x7FC0          # NaN
    xs[1][0, 4, 5, 5] = 0x7F80          # +inf
    xs_dev = [dev_bf16(x) for x in xs]
    ys = [torch.empty((B, C, H, W), device="cuda") for _ in range(n)]
    mean, invstd = _run(g, xs_dev, ys, C)
    with np.errstate(invalid="ignore"):
        m_w, s_w, y_w = oracle.syncbn(xs, 1e-5)
    m, s = mean.cpu().numpy().astype(np.float64), invstd.cpu().numpy().astype(np.float64)
    bad = [1, 4]
    for c in bad:
        assert not (np.isfinite(m_w[c]) and np.isfinite(s_w[c]))
        assert not (np.isfinite(m[c]) and np.isfinite(s[c])), (c, m[c], s[c])
    good = [c for c in range(C) if c not in bad]
    assert np.all(np.abs(m[good] - m_w[good]) <= 1e-5 * np.abs(m_w[good]) + 1e-7 / s_w[good])
    assert np.all(np.abs(s[good] - s_w[good]) <= 1e-5 * np.abs(s_w[good]))
    for r in range(n):
        _check_y(ys[r][:, good], np.asarray(y_w[r])[:, good], f"{shape} y[{r}] finite channels")
