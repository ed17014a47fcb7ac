"""syncbn_merge_apply_noalloc, called through the C ABI, against syncbn_merge_apply.

The no-allocation entry point serves callers that cannot allocate device
memory (a host framework that owns the device's memory pool, a memory budget
fixed up front, loops that cannot afford cudaMalloc's implicit
synchronisation): its scratch is a fixed array inside the library.

Three calls in a row on different shapes, each checked twice:
  * bit for bit against the workspace entry point on the same inputs (both
    run the same kernels with fixed reduction orders, so a stale partial or
    a wrong offset in the fixed array would show as a changed bit);
  * against the fp64 oracle on a few channels, with the tolerances of the
    SyncBN parity tests.
The shapes go from a small footprint (64 channels of 14x14: bulk-staged
statistics) to a large one (16000 channels of 16x32 planes: the plane
statistics kernel, the call run as two channel halves on two streams) and
back to a smaller one (2048 channels of 7x7: bulk-staged statistics), so
leftover contents of the array are exercised in both directions, through
two different statistics kernels.

This file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_common import load_library, sync

pytestmark = pytest.mark.gpu

ARGTYPES = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
            ctypes.c_int32, ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]


def _ptrs(ts):
    return (ctypes.c_void_p * len(ts))(*[t.data_ptr() for t in ts])


def _bf16_ulp(v):
    v = np.abs(np.asarray(v, np.float64))
    return 2.0 ** (np.floor(np.log2(np.maximum(v, 2.0 ** -126))) - 7)


def _entry(g):
    f = g.lib_handle().syncbn_merge_apply_noalloc
    f.restype = ctypes.c_int
    f.argtypes = ARGTYPES
    return f


def _same_bits(a, b):
    if a.dtype == torch.float32:
        return torch.equal(a.view(torch.int32), b.view(torch.int32))
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


def _check_oracle_channels(xs, y, m, s, gamma, beta, chans, what):
    """fp64 oracle on channels `chans`, with the SyncBN parity tolerances:
    mean within 1e-5 relative + 1e-7 standard deviations, invstd within
    1e-5 relative, y within one bf16 ulp of the oracle's value rounded to
    bf16 plus 1e-5 relative + 1e-6."""
    m_all, s_all = m.cpu().numpy().astype(np.float64), s.cpu().numpy().astype(np.float64)
    g_h, b_h = gamma.cpu().numpy().astype(np.float64), beta.cpu().numpy().astype(np.float64)
    for c in chans:
        xc = [x[:, c].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)[:, None] for x in xs]
        m_w, s_w = oracle.syncbn_stats_at(xc, 0, 1e-5)
        assert abs(m_all[c] - m_w) <= 1e-5 * abs(m_w) + 1e-7 / s_w, (what, c, m_all[c], m_w)
        assert abs(s_all[c] - s_w) <= 1e-5 * s_w, (what, c, s_all[c], s_w)
        for r in range(len(xs)):
            xv = oracle.bf16_bits_to_f32(xc[r][:, 0]).astype(np.float64)
            y_w = (xv - m_w) * s_w * g_h[c] + b_h[c]
            want = oracle.f64_to_bf16_rne(y_w)
            got = y[r][:, c].float().cpu().numpy().astype(np.float64)
            tol = _bf16_ulp(want) * 1.0001 + 1e-5 * np.abs(y_w) + 1e-6
            assert np.all(np.abs(got - want) <= tol), (what, c, r)


def test_noalloc_matches_workspace_entry_three_calls():
    g = load_library()
    f = _entry(g)
    stream = torch.cuda.current_stream().cuda_stream

    shapes = [(8, 4, 64, 14, 14, 1), (2, 2, 16000, 16, 32, 2), (4, 2, 2048, 7, 7, 3)]
    for call, (n, B, C, H, W, seed) in enumerate(shapes):
        xs = [workloads.device_normal((B, C, H, W), 0.5, 2.0, 900 + 10 * seed + r, dtype=torch.bfloat16)
              for r in range(n)]
        gamma = workloads.device_normal((C,), 1.0, 0.1, 950 + seed)
        beta = workloads.device_normal((C,), 0.0, 0.1, 960 + seed)

        # existing entry point, caller-allocated workspace
        y_ref = [torch.empty_like(x) for x in xs]
        m_ref, s_ref = torch.empty(C, device="cuda"), torch.empty(C, device="cuda")
        ws = torch.empty(g.syncbn_workspace_bytes(n, B, C, H, W), dtype=torch.uint8, device="cuda")
        g.syncbn_merge_apply(xs, y_ref, m_ref, s_ref, ws, 1e-5, gamma, beta)

        # no-allocation entry point through the C ABI, outputs pre-filled with NaN
        y = [torch.full_like(x, float("nan")) for x in xs]
        m, s = torch.full((C,), float("nan"), device="cuda"), torch.full((C,), float("nan"), device="cuda")
        st = f(_ptrs(xs), n, 1, B, C, H, W, 1e-5, gamma.data_ptr(), beta.data_ptr(), _ptrs(y), 1,
               m.data_ptr(), s.data_ptr(), stream)
        assert st == 0, (call, g.status_string(st))
        sync()

        assert _same_bits(m, m_ref), f"call {call}: mean differs from the workspace entry point"
        assert _same_bits(s, s_ref), f"call {call}: invstd differs from the workspace entry point"
        for r in range(n):
            assert _same_bits(y[r], y_ref[r]), f"call {call}: y[{r}] differs from the workspace entry point"
        chans = sorted({0, 1, C // 2, C - 1})
        _check_oracle_channels(xs, y, m, s, gamma, beta, chans, f"call {call}")


def test_noalloc_rejects_oversize():
    g = load_library()
    f = _entry(g)
    C = 43691                                   # needs 24*C bytes > the 1 MiB array
    assert g.syncbn_workspace_bytes(2, 1, C, 1, 1) > g.syncbn_noalloc_max_workspace_bytes()
    x = [torch.zeros((1, C, 1, 1), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    y = [torch.zeros_like(t) for t in x]
    m, s = torch.empty(C, device="cuda"), torch.empty(C, device="cuda")
    st = f(_ptrs(x), 2, 1, 1, C, 1, 1, 1e-5, None, None, _ptrs(y), 1, m.data_ptr(), s.data_ptr(),
           torch.cuda.current_stream().cuda_stream)
    assert st == g.DDP_ERR_CAPACITY
