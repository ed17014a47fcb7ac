"""SyncBN calls that run as two channel halves on two streams.

Calls on aligned planes that take the plane statistics kernel (H*W a
multiple of 8; an even C of at least 32 and at least 16 MiB of input over
all replicas), and calls on unaligned planes that take the per-warp
bulk-staged statistics (halves of whole channel groups, 32 MiB), run the
statistics, merge and apply of channels [0, C/2) on the caller's stream and
those of [C/2, C) on a side stream that the library keeps per host thread
and device, joined back before the call returns.  Both halves use one slice count, so the split call and the call
run as one sequence give the same bits: a thread's first call made inside a
stream capture, which finds no side stream yet, runs as one sequence, and
its replay must equal the split call bit for bit.  The statistics are
checked against the oracle on every channel by the full-size tests of the
SyncBN parity file; here: the split call against the oracle on a few
channels for every input and output dtype, in a graph, from a capture that
runs unsplit, and from several threads at once (chained in place: the
SyncBN parity file).
"""
import threading

import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_common import load_library, sync

pytestmark = pytest.mark.gpu

SHAPE = (8, 32, 64, 56, 56)           # n, batch, C, H, W: 103 MB of bf16 input, split


@pytest.fixture(scope="module")
def g():
    return load_library()


def _inputs(shape, seed):
    n, B, C, H, W = shape
    return [workloads.device_normal((B, C, H, W), 0.5, 2.0, seed + r, dtype=torch.bfloat16) for r in range(n)]


def _outputs(xs, C):
    return [torch.full_like(x, float("nan")) for x in xs], torch.full((C,), float("nan"), device="cuda"), \
        torch.full((C,), float("nan"), device="cuda")


def _same(a, b):
    if a.dtype == torch.float32:
        return torch.equal(a.view(torch.int32), b.view(torch.int32))
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


def _bf16_ulp(v):
    v = np.abs(np.asarray(v, np.float64))
    return 2.0 ** (np.floor(np.log2(np.maximum(v, 2.0 ** -126))) - 7)


def _check_channels(xs, ys, m, s, gamma, beta, chans, what):
    """fp64 oracle on channels `chans`: mean within 1e-5 relative + 1e-7
    standard deviations, invstd within 1e-5 relative; y within 1e-5 relative
    + 1e-6 of the fp64 value (fp32 output), or within one bf16 ulp of that
    value rounded to bf16 plus the same allowance (bf16 output)."""
    m_all, s_all = m.cpu().numpy().astype(np.float64), s.cpu().numpy().astype(np.float64)
    g_h = gamma.cpu().numpy().astype(np.float64) if gamma is not None else None
    b_h = beta.cpu().numpy().astype(np.float64) if beta is not None else None
    f32_in = xs[0].dtype == torch.float32
    for c in chans:
        if f32_in:
            xc = [x[:, c].contiguous().cpu().numpy().reshape(-1, 1) for x in xs]
            m_w, s_w = oracle.syncbn_stats_at(xc, 0, 1e-5, dtype="f32")
        else:
            xc = [x[:, c].contiguous().view(torch.int16).cpu().numpy().view(np.uint16).reshape(-1, 1) for x in xs]
            m_w, s_w = oracle.syncbn_stats_at(xc, 0, 1e-5)
        assert abs(m_all[c] - m_w) <= 1e-5 * abs(m_w) + 1e-7 / s_w, (what, c, m_all[c], m_w)
        assert abs(s_all[c] - s_w) <= 1e-5 * s_w, (what, c, s_all[c], s_w)
        gc = g_h[c] if g_h is not None else 1.0
        bc = b_h[c] if b_h is not None else 0.0
        for r in range(len(xs)):
            xv = (xc[r][:, 0] if f32_in else oracle.bf16_bits_to_f32(xc[r][:, 0])).astype(np.float64)
            y_w = (xv - m_w) * s_w * gc + bc
            got = ys[r][:, c].float().cpu().numpy().reshape(-1).astype(np.float64)
            if ys[r].dtype == torch.bfloat16:
                want = oracle.f64_to_bf16_rne(y_w)
                tol = _bf16_ulp(want) * 1.0001 + 1e-5 * np.abs(y_w) + 1e-6
            else:
                want = y_w
                tol = 1e-5 * np.abs(y_w) + 1e-6
            assert np.all(np.abs(got - want) <= tol), (what, c, r)


@pytest.mark.parametrize("io", [("bf16", "bf16"), ("bf16", "f32"), ("f32", "f32"), ("f32", "bf16")])
def test_split_call_matches_oracle(g, io):
    n, B, C, H, W = SHAPE
    if io[0] == "f32":
        B = B // 2                       # fp32: the same 103 MB of input
        xs = [workloads.device_normal((B, C, H, W), 0.5, 2.0, 1000 + r) for r in range(n)]
    else:
        xs = _inputs(SHAPE, 1000)
    assert g.syncbn_channel_parts(n, g.F32 if io[0] == "f32" else g.BF16, B, C, H, W) == 2
    gamma = workloads.device_normal((C,), 1.0, 0.1, 1100)
    beta = workloads.device_normal((C,), 0.0, 0.1, 1101)
    odt = torch.float32 if io[1] == "f32" else torch.bfloat16
    ys = [torch.full(x.shape, float("nan"), dtype=odt, device="cuda") for x in xs]
    m, s = torch.full((C,), float("nan"), device="cuda"), torch.full((C,), float("nan"), device="cuda")
    ws = torch.empty(g.syncbn_workspace_bytes(n, B, C, H, W), dtype=torch.uint8, device="cuda")
    g.syncbn_merge_apply(xs, ys, m, s, ws, 1e-5, gamma, beta)
    sync()
    # both halves' first and last channels and one inside each
    _check_channels(xs, ys, m, s, gamma, beta, [0, 13, C // 2 - 1, C // 2, C // 2 + 17, C - 1], f"split call {io}")


def test_split_call_in_graph_matches_eager(g):
    """The fork and join become graph edges; the replay equals the eager call."""
    n, B, C, H, W = SHAPE
    xs = _inputs(SHAPE, 1200)
    ws = torch.empty(g.syncbn_workspace_bytes(n, B, C, H, W), dtype=torch.uint8, device="cuda")
    ys_e, m_e, s_e = _outputs(xs, C)
    g.syncbn_merge_apply(xs, ys_e, m_e, s_e, ws)
    sync()
    ys, m, s = _outputs(xs, C)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        g.syncbn_merge_apply(xs, ys, m, s, ws)
    for _ in range(2):
        graph.replay()
    sync()
    assert _same(m, m_e) and _same(s, s_e)
    for r in range(n):
        assert _same(ys[r], ys_e[r]), f"replica {r}"


def test_first_call_of_a_thread_inside_capture_runs_unsplit_with_the_same_bits(g):
    """A new host thread has no side stream; its first call is captured, so
    it runs as one sequence on the capturing stream.  Its replay equals the
    split call of the main thread bit for bit."""
    n, B, C, H, W = SHAPE
    xs = _inputs(SHAPE, 1300)
    ws = torch.empty(g.syncbn_workspace_bytes(n, B, C, H, W), dtype=torch.uint8, device="cuda")
    ys_e, m_e, s_e = _outputs(xs, C)
    g.syncbn_merge_apply(xs, ys_e, m_e, s_e, ws)
    sync()
    ys, m, s = _outputs(xs, C)
    ws2 = torch.empty_like(ws)
    errors = []

    def worker():
        try:
            torch.cuda.set_device(0)
            side = torch.cuda.Stream()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=side):
                g.syncbn_merge_apply(xs, ys, m, s, ws2)
            graph.replay()
            torch.cuda.synchronize()
        except Exception as e:         # reported by the main thread
            errors.append(repr(e))

    t = threading.Thread(target=worker)
    t.start()
    t.join(timeout=300)
    assert not errors, errors
    assert _same(m, m_e) and _same(s, s_e)
    for r in range(n):
        assert _same(ys[r], ys_e[r]), f"replica {r}"


def test_split_calls_from_three_threads(g):
    """Three host threads, each with its own stream, workspace and side
    stream, run split calls at the same time; each result equals the same
    call made alone."""
    n, B, C, H, W = SHAPE
    inputs = [_inputs(SHAPE, 1400 + 20 * k) for k in range(3)]
    alone = []
    for xs in inputs:
        ws = torch.empty(g.syncbn_workspace_bytes(n, B, C, H, W), dtype=torch.uint8, device="cuda")
        ys, m, s = _outputs(xs, C)
        g.syncbn_merge_apply(xs, ys, m, s, ws)
        sync()
        alone.append((ys, m, s))
    got, errors = {}, []

    def worker(k):
        try:
            torch.cuda.set_device(0)
            st = torch.cuda.Stream()
            with torch.cuda.stream(st):
                ws = torch.empty(g.syncbn_workspace_bytes(n, B, C, H, W), dtype=torch.uint8, device="cuda")
                ys, m, s = _outputs(inputs[k], C)
                for _ in range(5):
                    g.syncbn_merge_apply(inputs[k], ys, m, s, ws, stream=st)
            st.synchronize()
            got[k] = (ys, m, s)
        except Exception as e:         # reported by the main thread
            errors.append((k, repr(e)))

    ths = [threading.Thread(target=worker, args=(k,)) for k in range(3)]
    for t in ths:
        t.start()
    for t in ths:
        t.join(timeout=300)
    assert not errors, errors
    for k in range(3):
        ys, m, s = got[k]
        ys_a, m_a, s_a = alone[k]
        assert _same(m, m_a) and _same(s, s_a), f"thread {k}"
        for r in range(n):
            assert _same(ys[r], ys_a[r]), f"thread {k} replica {r}"


@pytest.mark.parametrize("shape", [(8, 16, 96, 28, 28), (8, 32, 34, 56, 56)])
def test_split_halves_not_a_multiple_of_the_merge_width(g, shape):
    """Halves of 48 and 17 channels: the merge's last CTA of each half is
    part-full, and the second half starts inside a 32-channel group of the
    whole call.  Every channel's statistics against the oracle, and the
    outputs of the channels on both sides of the split."""
    n, B, C, H, W = shape
    assert g.syncbn_channel_parts(n, g.BF16, B, C, H, W) == 2
    xs = _inputs(shape, 1500 + C)
    ys, m, s = _outputs(xs, C)
    ws = torch.empty(g.syncbn_workspace_bytes(n, B, C, H, W), dtype=torch.uint8, device="cuda")
    g.syncbn_merge_apply(xs, ys, m, s, ws)
    sync()
    host = [x.view(torch.int16).cpu().numpy().view(np.uint16) for x in xs]
    m_w, s_w = oracle.syncbn_stats(host, 1e-5)
    m_all, s_all = m.cpu().numpy().astype(np.float64), s.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(m_all - m_w) <= 1e-5 * np.abs(m_w) + 1e-7 / s_w)
    assert np.all(np.abs(s_all - s_w) <= 1e-5 * s_w)
    _check_channels(xs, ys, m, s, None, None, [0, C // 2 - 1, C // 2, C - 1], f"split {shape}")


@pytest.mark.parametrize("shape,out_dtype", [((8, 32, 2048, 7, 7), torch.bfloat16), ((8, 32, 2048, 7, 7), torch.float32),
                                             ((8, 16, 1024, 14, 14), torch.bfloat16),
                                             ((8, 16, 1024, 17, 17), torch.bfloat16)])
def test_bulk_statistics_split_matches_oracle(g, shape, out_dtype):
    """Calls whose statistics take the per-warp bulk-staged kernel split into
    halves of whole channel groups (unaligned 7x7, 14x14 and 17x17 planes;
    the apply's mode 5, with bf16 and fp32 outputs).  Every channel's
    statistics against the oracle, and the outputs on both sides of the
    split."""
    n, B, C, H, W = shape
    assert g.syncbn_channel_parts(n, g.BF16, B, C, H, W) == 2
    xs = _inputs(shape, 1600 + H)
    gamma = workloads.device_normal((C,), 1.0, 0.1, 1700)
    beta = workloads.device_normal((C,), 0.0, 0.1, 1701)
    ys = [torch.full(x.shape, float("nan"), dtype=out_dtype, device="cuda") for x in xs]
    m, s = torch.full((C,), float("nan"), device="cuda"), torch.full((C,), float("nan"), device="cuda")
    ws = torch.empty(g.syncbn_workspace_bytes(n, B, C, H, W), dtype=torch.uint8, device="cuda")
    g.syncbn_merge_apply(xs, ys, m, s, ws, 1e-5, gamma, beta)
    sync()
    host = [x.view(torch.int16).cpu().numpy().view(np.uint16) for x in xs]
    m_w, s_w = oracle.syncbn_stats(host, 1e-5)
    m_all, s_all = m.cpu().numpy().astype(np.float64), s.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(m_all - m_w) <= 1e-5 * np.abs(m_w) + 1e-7 / s_w)
    assert np.all(np.abs(s_all - s_w) <= 1e-5 * s_w)
    _check_channels(xs, ys, m, s, gamma, beta, [0, 1, C // 2 - 1, C // 2, C // 2 + 1, C - 1], f"bulk split {shape}")


def test_bulk_split_in_graph_and_unsplit_capture_give_the_same_bits(g):
    """7x7 planes: the eager split call, its graph replay, and a new thread's
    first call made inside a capture (one sequence on the capturing stream)
    agree bit for bit."""
    shape = (8, 32, 2048, 7, 7)
    n, B, C, H, W = shape
    xs = _inputs(shape, 1800)
    ws = torch.empty(g.syncbn_workspace_bytes(n, B, C, H, W), dtype=torch.uint8, device="cuda")
    ys_e, m_e, s_e = _outputs(xs, C)
    g.syncbn_merge_apply(xs, ys_e, m_e, s_e, ws)
    sync()
    ys_g, m_g, s_g = _outputs(xs, C)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        g.syncbn_merge_apply(xs, ys_g, m_g, s_g, ws)
    graph.replay()
    sync()
    ys_t, m_t, s_t = _outputs(xs, C)
    ws2 = torch.empty_like(ws)
    errors = []

    def worker():
        try:
            torch.cuda.set_device(0)
            st = torch.cuda.Stream()
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=st):
                g.syncbn_merge_apply(xs, ys_t, m_t, s_t, ws2)
            gr.replay()
            torch.cuda.synchronize()
        except Exception as e:         # reported by the main thread
            errors.append(repr(e))

    t = threading.Thread(target=worker)
    t.start()
    t.join(timeout=300)
    assert not errors, errors
    for m, s, ys, what in ((m_g, s_g, ys_g, "graph"), (m_t, s_t, ys_t, "unsplit capture")):
        assert _same(m, m_e) and _same(s, s_e), what
        for r in range(n):
            assert _same(ys[r], ys_e[r]), f"{what} replica {r}"
