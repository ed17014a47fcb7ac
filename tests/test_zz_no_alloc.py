"""syncbn_merge_apply_noalloc, called through the C ABI, against syncbn_merge_apply.

The no-allocation entry point serves callers that cannot allocate device
memory (a host framework that owns the device's memory pool, a memory budget
fixed up front, loops that cannot afford cudaMalloc's implicit
synchronisation): its scratch is a fixed array inside the library.  Two calls
in a row, on different inputs, must each agree with the workspace entry point
on the same inputs, within the SyncBatchNorm tolerances of the parity tests
(mean/invstd 1e-5 relative; y within one bf16 ulp plus 1e-5 relative + 1e-6).

This file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads
from gpu_common import load_library, sync

pytestmark = pytest.mark.gpu


def _ptrs(ts):
    return (ctypes.c_void_p * len(ts))(*[t.data_ptr() for t in ts])


def _bf16_ulp(v):
    v = np.abs(np.asarray(v, np.float64))
    return 2.0 ** (np.floor(np.log2(np.maximum(v, 2.0 ** -126))) - 7)


def _close(a, b, rel, absolute=0.0):
    a = a.float().cpu().numpy().astype(np.float64)
    b = b.float().cpu().numpy().astype(np.float64)
    return bool(np.all(np.abs(a - b) <= rel * np.abs(b) + absolute))


def test_noalloc_matches_workspace_entry_two_calls():
    g = load_library()
    lib = g.lib_handle()
    f = lib.syncbn_merge_apply_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                  ctypes.c_int32, ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    stream = torch.cuda.current_stream().cuda_stream

    for call, (n, B, C, H, W, seed) in enumerate([(8, 4, 64, 14, 14, 1), (4, 2, 2048, 7, 7, 2)]):
        xs = [workloads.device_normal((B, C, H, W), 0.5, 2.0, 900 + 10 * seed + r, dtype=torch.bfloat16)
              for r in range(n)]
        gamma = workloads.device_normal((C,), 1.0, 0.1, 950 + seed)
        beta = workloads.device_normal((C,), 0.0, 0.1, 960 + seed)

        # existing entry point, caller-allocated workspace
        y_ref = [torch.empty_like(x) for x in xs]
        m_ref, s_ref = torch.empty(C, device="cuda"), torch.empty(C, device="cuda")
        ws = torch.empty(g.syncbn_workspace_bytes(n, B, C, H, W), dtype=torch.uint8, device="cuda")
        g.syncbn_merge_apply(xs, y_ref, m_ref, s_ref, ws, 1e-5, gamma, beta)

        # no-allocation entry point through the C ABI
        y = [torch.full_like(x, float("nan")) for x in xs]
        m, s = torch.full((C,), float("nan"), device="cuda"), torch.full((C,), float("nan"), device="cuda")
        st = f(_ptrs(xs), n, 1, B, C, H, W, 1e-5, gamma.data_ptr(), beta.data_ptr(), _ptrs(y), 1,
               m.data_ptr(), s.data_ptr(), stream)
        assert st == 0, (call, g.status_string(st))
        sync()

        assert _close(m, m_ref, 1e-5, 1e-7), f"call {call}: mean"
        assert _close(s, s_ref, 1e-5), f"call {call}: invstd"
        for r in range(n):
            got = y[r].float().cpu().numpy().astype(np.float64)
            ref = y_ref[r].float().cpu().numpy().astype(np.float64)
            tol = _bf16_ulp(ref) * 1.0001 + 1e-5 * np.abs(ref) + 1e-6
            assert np.all(np.abs(got - ref) <= tol), f"call {call}: y[{r}]"


def test_noalloc_rejects_oversize():
    g = load_library()
    lib = g.lib_handle()
    f = lib.syncbn_merge_apply_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                  ctypes.c_int32, ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    C = 43691                                   # needs 24*C bytes > the 1 MiB array
    assert g.syncbn_workspace_bytes(2, 1, C, 1, 1) > g.syncbn_noalloc_max_workspace_bytes()
    x = [torch.zeros((1, C, 1, 1), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    y = [torch.zeros_like(t) for t in x]
    m, s = torch.empty(C, device="cuda"), torch.empty(C, device="cuda")
    st = f(_ptrs(x), 2, 1, 1, C, 1, 1, 1e-5, None, None, _ptrs(y), 1, m.data_ptr(), s.data_ptr(),
           torch.cuda.current_stream().cuda_stream)
    assert st == g.DDP_ERR_CAPACITY
