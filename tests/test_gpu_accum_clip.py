"""GPU parity: accumulation, average with norm side output, norm finalize and
the SGD step with a clip factor, against the oracle.

Tolerances: accumulation, the average and the SGD step given the same clip
factor are bit-exact (fp32, separately rounded operations).  The norm is a
sum of squares over millions of elements (fp32 per thread, float-float per
CTA and across CTAs) compared with the oracle's fp64 sum: 2e-6 relative; the
clip factor derived from it likewise.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_common import assert_bit_exact, dev_bf16, dev_f32, load_library, sync

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    return load_library()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_accumulate_three_micro_steps(g, dtype):
    for n in (1, 3, 8):
        for numel in (1, 7, 4099, 300_003):
            gen = np.random.Generator(np.random.PCG64(n * 7 + numel))
            accs = [(gen.standard_normal(numel) * 0.01).astype(np.float32) for _ in range(n)]
            acc_d = [dev_f32(a) for a in accs]
            for step in range(3):
                micro = [(gen.standard_normal(numel) * 0.01).astype(np.float32) for _ in range(n)]
                if dtype == "bf16":
                    micro = [workloads.f32_to_bf16_bits(m) for m in micro]
                md = [dev_f32(m) if dtype == "f32" else dev_bf16(m) for m in micro]
                g.ddp_bucket_accumulate(md, acc_d)
                accs = [oracle.accumulate(a, m, dtype) for a, m in zip(accs, micro)]
            sync()
            for r in range(n):
                assert_bit_exact(acc_d[r], accs[r], f"acc {dtype} N={n} numel={numel} r={r}")


def _flow(g, bucket_sizes, n, seed, max_norm, dtype="f32", poison=None):
    """Average each bucket with the norm side output, finalize, SGD with the
    clip factor; return GPU results and the inputs."""
    gen = np.random.Generator(np.random.PCG64(seed))
    reps = [[(gen.standard_normal(sz) * 0.05).astype(np.float32) for _ in range(n)] for sz in bucket_sizes]
    if poison is not None:
        b, r, i, val = poison
        reps[b][r][i] = val
    ws = torch.empty(g.ddp_norm_workspace_bytes(len(bucket_sizes)), dtype=torch.uint8, device="cuda")
    outs = [torch.empty(sz, device="cuda") for sz in bucket_sizes]
    for b, sz in enumerate(bucket_sizes):
        g.ddp_bucket_allreduce_mean_norm([dev_f32(x) for x in reps[b]], outs[b], ws, b)
    norm = torch.empty(1, device="cuda")
    coef = torch.empty(1, device="cuda")
    nf = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    g.ddp_grad_norm_finalize(ws, len(bucket_sizes), max_norm, norm, coef, nf)
    sync()
    return reps, outs, norm.item(), coef, nf.item()


def test_mean_norm_finalize(g):
    sizes = [4099, 1, 300_001, 2_000_003]
    for n in (1, 3, 8):
        for max_norm in (0.0, 1.0, 1e9):
            reps, outs, norm, coef, nf = _flow(g, sizes, n, 100 + n, max_norm)
            means = [oracle.grad_mean(r) for r in reps]
            for b in range(len(sizes)):
                assert_bit_exact(outs[b], means[b], f"mean bucket {b}")
            want = oracle.grad_global_norm(means)
            assert abs(norm - want) <= 2e-6 * want, (norm, want)
            c_want = oracle.clip_coefficient(want, max_norm)
            assert abs(coef.item() - c_want) <= 2e-6 * c_want, (coef.item(), c_want)
            assert nf == 0


def test_nonfinite_flag(g):
    for val in (float("nan"), float("inf"), float("-inf")):
        _, _, norm, _, nf = _flow(g, [1000, 5000], 4, 7, 1.0, poison=(1, 2, 4321, val))
        assert nf == 1
        assert not np.isfinite(norm)


def test_empty_bucket_contributes_nothing(g):
    sizes = [0, 5000, 0]
    reps, outs, norm, coef, nf = _flow(g, sizes, 2, 3, 1.0)
    want = oracle.grad_global_norm([oracle.grad_mean(reps[1])])
    assert abs(norm - want) <= 2e-6 * want and nf == 0


def test_sgd_with_scale(g):
    """ddp_bucket_sgd multiplies the averaged gradient by a device scalar
    before the step: bit-exact with the oracle for the same scale value
    (chosen here on the host, copied to the device)."""
    gen = np.random.Generator(np.random.PCG64(56))
    for numel in (1, 4099, 300_001):
        g_avg = (gen.standard_normal(numel) * 0.05).astype(np.float32)
        for scale in (0.3125, float(np.float32(0.8137)), 1.0):
            th = (gen.standard_normal(numel) * 0.02).astype(np.float32)
            buf = (gen.standard_normal(numel) * 0.001).astype(np.float32)
            th_d, b_d = dev_f32(th), dev_f32(buf)
            sc = torch.tensor([scale], dtype=torch.float32, device="cuda")
            g.ddp_bucket_sgd(dev_f32(g_avg), th_d, b_d, 0.1, 0.9, 1e-4, grad_scale=sc)
            sync()
            th_w, b_w = oracle.sgd_from_grad(g_avg, th, buf, 0.1, 0.9, 1e-4, scale=np.float32(scale))
            assert_bit_exact(th_d, th_w, f"theta numel={numel} scale={scale}")
            assert_bit_exact(b_d, b_w, f"buf numel={numel} scale={scale}")
    th = gen.standard_normal(4099).astype(np.float32)
    g_avg = gen.standard_normal(4099).astype(np.float32)
    th_d = dev_f32(th)
    g.ddp_bucket_sgd(dev_f32(g_avg), th_d, None, 0.25, 0.0, 0.0)
    sync()
    assert_bit_exact(th_d, oracle.sgd_from_grad(g_avg, th, None, 0.25, 0.0, 0.0)[0], "plain")


def test_gpt2_accumulate_then_clipped_step(g):
    """GPT-2 small layout, 8 replicas: two bf16 micro-steps accumulated into
    fp32 gradients, the DEEP/FIRST buckets averaged with the norm side
    output, clip to max_norm 1.0, and the SGD step (momentum 0.9, wd 1e-4)
    with the clip factor.  The oracle redoes accumulate -> average -> fp64
    norm -> clip factor over every element (in chunks, from the same input
    bits); the averaged gradient is compared bit for bit on 2^18 sampled
    positions, the norm and factor within 2e-6, and θ / the buffer there
    within what a 2e-6 difference of the factor allows."""
    layout, first = workloads.gpt2_small_layout()
    plan = g.ddp_plan_buckets(workloads.numels(layout), 4, 0, g.PLAN_DEEP_FIRST, first)
    total, n = plan["total_elems"], 8
    acc = [torch.zeros(total, device="cuda") for _ in range(n)]
    micro = [[workloads.device_normal((total,), 0.0, 0.01, 7000 + 100 * step + r, dtype=torch.bfloat16)
              for r in range(n)] for step in range(2)]
    for step in range(2):
        g.ddp_bucket_accumulate(micro[step], acc)
    ws = torch.empty(g.ddp_norm_workspace_bytes(2), dtype=torch.uint8, device="cuda")
    gavg = torch.empty(total, device="cuda")
    for b, (off, numel, _, _) in enumerate(plan["buckets"]):
        g.ddp_bucket_allreduce_mean_norm([x[off:off + numel] for x in acc], gavg[off:off + numel], ws, b)
    norm, coef = torch.empty(1, device="cuda"), torch.empty(1, device="cuda")
    g.ddp_grad_norm_finalize(ws, 2, 1.0, norm, coef, None)
    theta = workloads.device_normal((total,), 0.0, 0.02, 7999)
    gen = np.random.Generator(np.random.PCG64(8))
    in_bucket = np.zeros(total, bool)
    for off, numel, _, _ in plan["buckets"]:
        in_bucket[off:off + numel] = True
    idx = np.unique(gen.integers(0, total, 1 << 18))
    idx = idx[in_bucket[idx]]                          # positions inside buckets only
    idx_d = torch.from_numpy(idx).cuda()
    th0 = theta[idx_d].cpu().numpy()
    buf = torch.zeros(total, device="cuda")
    for off, numel, _, _ in plan["buckets"]:
        g.ddp_bucket_sgd(gavg[off:off + numel], theta[off:off + numel], buf[off:off + numel], 0.1, 0.9, 1e-4,
                         grad_scale=coef)
    sync()

    def bits(t):
        return t.view(torch.int16).cpu().numpy().view(np.uint16)

    # oracle over every element, in chunks of the flat buffer; only bucket elements enter the norm
    sq = 0.0
    g_sample = np.empty(idx.size, np.float32)
    chunk = 1 << 23
    for s0 in range(0, total, chunk):
        s1 = min(total, s0 + chunk)
        accs = [np.zeros(s1 - s0, np.float32) for _ in range(n)]
        for step in range(2):
            for r in range(n):
                accs[r] = oracle.accumulate(accs[r], bits(micro[step][r][s0:s1]), "bf16")
        gm = oracle.grad_mean(accs)
        inside = np.zeros(s1 - s0, bool)
        for off, numel, _, _ in plan["buckets"]:
            lo, hi = max(off, s0), min(off + numel, s1)
            if lo < hi:
                inside[lo - s0:hi - s0] = True
        sq += oracle.grad_global_norm([gm[inside]]) ** 2
        sel = (idx >= s0) & (idx < s1)
        g_sample[sel] = gm[idx[sel] - s0]
    want_norm = sq ** 0.5
    want_coef = oracle.clip_coefficient(want_norm, 1.0)
    assert_bit_exact(gavg[idx_d], g_sample, "averaged gradient (sampled)")
    assert abs(norm.item() - want_norm) <= 2e-6 * want_norm, (norm.item(), want_norm)
    assert abs(coef.item() - want_coef) <= 2e-6 * want_coef, (coef.item(), want_coef)
    th_w, b_w = oracle.sgd_from_grad(g_sample, th0, np.zeros(idx.size, np.float32), 0.1, 0.9, 1e-4,
                                     scale=np.float32(want_coef))
    np.testing.assert_allclose(buf[idx_d].cpu().numpy(), b_w, rtol=3e-6, atol=1e-12)
    np.testing.assert_allclose(theta[idx_d].cpu().numpy(), th_w, rtol=1e-6, atol=1e-9)
