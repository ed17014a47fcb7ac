"""C-ABI checks that need no GPU: the library loads, exports every function
include/ddp_sync.h declares, the native planner matches the oracle exactly,
and invalid arguments are rejected on the host before any CUDA call."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

import oracle
import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def g():
    import __graft_entry__
    __graft_entry__.build()
    import gradient_sync_ddp_gb300 as pkg
    return pkg


def _declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not fn.endswith(".h"):
            continue
        src = open(os.path.join(ROOT, "include", fn), encoding="utf-8").read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s+\**([A-Za-z_][A-Za-z0-9_]*)\s*\(",
                             src, flags=re.M):
            names.append(m.group(1))
    return names


def test_header_declares_the_boundary():
    names = _declared_functions()
    for required in ("ddp_plan_buckets", "ddp_bucket_allreduce_mean", "ddp_bucket_allreduce_sgd",
                     "syncbn_merge_apply", "syncbn_workspace_bytes", "dist_sampler_indices",
                     "dist_sampler_num_samples", "ddp_status_string", "ddp_last_cuda_error"):
        assert required in names


def test_library_exports_every_declared_symbol(g):
    lib = g.lib_handle()
    for name in _declared_functions():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", g.LIB_PATH], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    for name in _declared_functions():
        assert name in exported, name


def test_status_strings(g):
    for st in (0, -1, -2, -3, -4, -5, -6):
        assert g.status_string(st).startswith("DDP_")
    assert g.version() == "0.1.0"


# --------------------------------------------------------------- planner

def _same_plan(a, b):
    for k in ("buckets", "order", "tensor_offset", "tensor_bucket", "total_elems"):
        assert a[k] == b[k], k


def test_native_planner_resnet50(g):
    num = workloads.numels(workloads.resnet50_layout())
    for cap_mib in (1, 25, 100):
        for eb in (2, 4):
            _same_plan(g.ddp_plan_buckets(num, eb, cap_mib << 20), oracle.plan_buckets(num, eb, cap_mib << 20))


def test_native_planner_gpt2_deep_first(g):
    layout, first = workloads.gpt2_small_layout()
    num = workloads.numels(layout)
    got = g.ddp_plan_buckets(num, 2, 0, g.PLAN_DEEP_FIRST, first)
    _same_plan(got, oracle.plan_buckets(num, 2, 0, oracle.PLAN_DEEP_FIRST, first))
    assert [b[1] for b in got["buckets"]] == [85_017_600, 39_422_208]


def test_native_planner_random(g):
    gen = np.random.Generator(np.random.PCG64(123))
    for _ in range(300):
        T = int(gen.integers(0, 50))
        num = [int(x) for x in gen.integers(0, 100000, T)]
        eb = int(gen.choice([2, 4]))
        cap = int(gen.integers(0, 400000))
        al = int(gen.choice([16, 64, 256, 4096]))
        _same_plan(g.ddp_plan_buckets(num, eb, cap, align_bytes=al), oracle.plan_buckets(num, eb, cap, 0, None, al))
        isf = [bool(x) for x in gen.integers(0, 2, T)]
        _same_plan(g.ddp_plan_buckets(num, eb, cap, g.PLAN_DEEP_FIRST, isf, al),
                   oracle.plan_buckets(num, eb, cap, 1, isf, al))


def test_native_planner_rejects(g):
    lib = g.lib_handle()
    nb = ctypes.c_int32(0)
    tot = ctypes.c_int64(0)
    num = (ctypes.c_int64 * 2)(5, -1)
    o = (ctypes.c_int32 * 2)()
    off = (ctypes.c_int64 * 2)()
    tb = (ctypes.c_int32 * 2)()
    bk = (g.DdpBucket * 2)()
    args = lambda numels, eb, align, mode=0, first=None: lib.ddp_plan_buckets(  # noqa: E731
        2, ctypes.addressof(numels), eb, 100, mode, first, align, ctypes.addressof(bk), 2, ctypes.addressof(nb),
        ctypes.addressof(o), ctypes.addressof(off), ctypes.addressof(tb), ctypes.addressof(tot))
    assert args(num, 4, 256) == g.DDP_ERR_INVALID_ARG                    # negative numel
    ok = (ctypes.c_int64 * 2)(5, 6)
    assert args(ok, 3, 256) == g.DDP_ERR_INVALID_ARG                     # elem_bytes
    assert args(ok, 4, 24) == g.DDP_ERR_INVALID_ARG                      # not a multiple of 16
    assert args(ok, 4, 256, mode=1) == g.DDP_ERR_INVALID_ARG             # DEEP_FIRST needs is_first
    assert args(ok, 4, 256, mode=7) == g.DDP_ERR_INVALID_ARG
    assert args(ok, 4, 256) == g.DDP_OK
    # capacity: three one-tensor buckets into room for one
    num3 = (ctypes.c_int64 * 3)(100, 100, 100)
    o3, off3, tb3, bk1 = (ctypes.c_int32 * 3)(), (ctypes.c_int64 * 3)(), (ctypes.c_int32 * 3)(), (g.DdpBucket * 1)()
    st = lib.ddp_plan_buckets(3, ctypes.addressof(num3), 4, 400, 0, None, 256, ctypes.addressof(bk1), 1,
                              ctypes.addressof(nb), ctypes.addressof(o3), ctypes.addressof(off3),
                              ctypes.addressof(tb3), ctypes.addressof(tot))
    assert st == g.DDP_ERR_CAPACITY and nb.value == 3


# --------------------------------------------------------------- validation (no CUDA call is reached)

FAKE = 1 << 40          # an aligned address that is never dereferenced: every case below fails
                        # validation, or has numel == 0, before any CUDA call


def _ptrs(*addrs):
    return (ctypes.c_void_p * len(addrs))(*addrs)


def test_mean_rejects(g):
    lib = g.lib_handle()
    m = lib.ddp_bucket_allreduce_mean
    two = _ptrs(FAKE, FAKE + 4096)
    assert m(two, 0, 0, 8, FAKE + 8192, 0, None) == g.DDP_ERR_INVALID_ARG          # N = 0
    assert m(_ptrs(*[FAKE] * 17), 17, 0, 8, FAKE + 8192, 0, None) == g.DDP_ERR_INVALID_ARG
    assert m(None, 2, 0, 8, FAKE + 8192, 0, None) == g.DDP_ERR_INVALID_ARG
    assert m(two, 2, 5, 8, FAKE + 8192, 0, None) == g.DDP_ERR_INVALID_ARG          # dtype
    assert m(two, 2, 0, -1, FAKE + 8192, 0, None) == g.DDP_ERR_INVALID_ARG         # numel
    assert m(two, 2, 0, 8, None, 0, None) == g.DDP_ERR_INVALID_ARG
    assert m(_ptrs(FAKE + 4, FAKE + 4096), 2, 0, 8, FAKE + 8192, 0, None) == g.DDP_ERR_ALIGNMENT
    assert m(two, 2, 0, 8, FAKE + 8200, 0, None) == g.DDP_ERR_ALIGNMENT
    assert m(two, 2, 0, 8, FAKE + 8192, 64, None) == g.DDP_ERR_INVALID_ARG         # unknown flag
    assert m(two, 2, 0, 8, FAKE + 8192, 1 | 4, None) == g.DDP_ERR_INVALID_ARG      # tree + ring
    assert m(_ptrs(FAKE, FAKE + 4096, FAKE + 8192), 3, 0, 8, FAKE + 16384, 1, None) == g.DDP_ERR_INVALID_ARG
    assert m(two, 2, 1, 8, FAKE + 8192, 2, None) == g.DDP_ERR_INVALID_ARG          # write-back needs fp32
    assert m(two, 2, 0, 8, FAKE + 16, 0, None) == g.DDP_ERR_INVALID_ARG            # partial overlap
    assert m(two, 2, 1, 8, FAKE, 0, None) == g.DDP_ERR_INVALID_ARG                 # bf16 in place
    # accepted, nothing to do
    assert m(two, 2, 0, 0, FAKE + 8192, 0, None) == g.DDP_OK
    assert m(two, 2, 0, 0, FAKE, 0, None) == g.DDP_OK                              # exact alias, fp32


def test_sgd_rejects(g):
    lib = g.lib_handle()
    s = lib.ddp_bucket_allreduce_sgd
    two = _ptrs(FAKE, FAKE + 4096)
    P, B, G = FAKE + 8192, FAKE + 12288, FAKE + 16384
    assert s(two, 2, 0, 8, None, B, 0.1, 0.9, 0.0, None, 0, None) == g.DDP_ERR_INVALID_ARG
    assert s(two, 2, 0, 8, P, None, 0.1, 0.9, 0.0, None, 0, None) == g.DDP_ERR_INVALID_ARG  # needs buffer
    assert s(two, 2, 0, 8, P, B, 0.1, 0.0, 0.0, None, 0, None) == g.DDP_ERR_INVALID_ARG     # buffer unused
    assert s(two, 2, 0, 8, P, B, float("nan"), 0.9, 0.0, None, 0, None) == g.DDP_ERR_INVALID_ARG
    assert s(two, 2, 0, 8, P, B, 0.1, 0.9, 0.0, None, 1, None) == g.DDP_ERR_INVALID_ARG     # flags reserved
    assert s(two, 2, 0, 8, P + 4, B, 0.1, 0.9, 0.0, None, 0, None) == g.DDP_ERR_ALIGNMENT
    assert s(two, 2, 0, 8, P, P + 16, 0.1, 0.9, 0.0, None, 0, None) == g.DDP_ERR_INVALID_ARG  # overlap
    assert s(two, 2, 0, 8, FAKE, B, 0.1, 0.9, 0.0, None, 0, None) == g.DDP_ERR_INVALID_ARG   # θ on a replica
    assert s(two, 2, 0, 0, P, B, 0.1, 0.9, 0.0, G, 0, None) == g.DDP_OK


def test_syncbn_rejects_and_workspace(g):
    lib = g.lib_handle()
    assert g.syncbn_workspace_bytes(8, 32, 64, 56, 56) > 0
    assert g.syncbn_workspace_bytes(0, 32, 64, 56, 56) == 0
    assert g.syncbn_workspace_bytes(17, 32, 64, 56, 56) == 0
    assert g.syncbn_workspace_bytes(8, 32, 64, 0, 56) == 0
    ws = g.syncbn_workspace_bytes(2, 2, 4, 3, 3)
    x, y = _ptrs(FAKE, FAKE + 4096), _ptrs(FAKE + 8192, FAKE + 12288)
    M, I, W = FAKE + 16384, FAKE + 20480, FAKE + 24576
    f = lib.syncbn_merge_apply
    assert f(x, 2, 1, 2, 4, 3, 3, 1e-5, None, None, y, 1, M, I, W, ws - 1, None) == g.DDP_ERR_CAPACITY
    assert f(x, 2, 1, 2, 4, 3, 3, 0.0, None, None, y, 1, M, I, W, ws, None) == g.DDP_ERR_INVALID_ARG
    assert f(x, 2, 1, 2, 4, 3, 3, 1e-5, None, None, y, 3, M, I, W, ws, None) == g.DDP_ERR_INVALID_ARG
    assert f(x, 2, 1, 2, 4, 3, 3, 1e-5, None, None, y, 1, M, I, W + 8, ws, None) == g.DDP_ERR_ALIGNMENT
    assert f(x, 2, 1, 2, 4, 3, 3, 1e-5, None, None, _ptrs(FAKE + 8192, FAKE + 8200), 1, M, I, W, ws,
             None) == g.DDP_ERR_ALIGNMENT
    assert f(x, 2, 1, 2, 4, 3, 3, 1e-5, None, None, _ptrs(FAKE + 8192, FAKE + 8192), 1, M, I, W, ws,
             None) == g.DDP_ERR_INVALID_ARG                                           # outputs overlap
    assert f(x, 2, 1, 2, 4, 3, 3, 1e-5, None, None, _ptrs(FAKE + 16, FAKE + 12288), 1, M, I, W, ws,
             None) == g.DDP_ERR_INVALID_ARG                                           # y overlaps x


def test_sampler_host_logic(g):
    lib = g.lib_handle()
    for n in range(0, 50):
        for N in range(1, 12):
            for d in (0, 1):
                assert g.dist_sampler_num_samples(n, N, d) == oracle.sampler_num_samples(n, N, bool(d))
    ns = ctypes.c_int64(-7)
    f = lib.dist_sampler_indices
    assert f(10, 3, 3, 0, 0, 1, 0, FAKE, 100, ctypes.addressof(ns), None, None) == g.DDP_ERR_INVALID_ARG
    assert f(10, 3, 0, 0, 0, 1, 0, FAKE, 3, ctypes.addressof(ns), None, None) == g.DDP_ERR_CAPACITY
    assert ns.value == 4
    assert f(10, 3, -1, 0, 0, 1, 0, FAKE, 11, ctypes.addressof(ns), None, None) == g.DDP_ERR_CAPACITY
    assert f(10, 3, 0, 0, 0, 2, 0, FAKE, 100, ctypes.addressof(ns), None, None) == g.DDP_ERR_INVALID_ARG
    assert f(10, 3, 0, 0, 0, 1, 0, FAKE + 4, 100, ctypes.addressof(ns), None, None) == g.DDP_ERR_ALIGNMENT
    assert f(-1, 3, 0, 0, 0, 1, 0, FAKE, 100, ctypes.addressof(ns), None, None) == g.DDP_ERR_INVALID_ARG
    assert f(2, 3, 0, 0, 0, 1, 1, None, 0, ctypes.addressof(ns), None, None) == g.DDP_OK   # n < N, drop_last
    assert ns.value == 0
    r = lib.dist_sampler_indices_from                    # resume offset: 0 <= start <= num_samples
    assert r(10, 3, 0, 0, 0, 1, 0, 5, FAKE, 100, ctypes.addressof(ns), None, None) == g.DDP_ERR_INVALID_ARG
    assert r(10, 3, 0, 0, 0, 1, 0, -1, FAKE, 100, ctypes.addressof(ns), None, None) == g.DDP_ERR_INVALID_ARG
    assert r(10, 3, 0, 0, 0, 1, 0, 1, FAKE, 2, ctypes.addressof(ns), None, None) == g.DDP_ERR_CAPACITY
    assert r(10, 3, -1, 0, 0, 1, 0, 1, FAKE, 8, ctypes.addressof(ns), None, None) == g.DDP_ERR_CAPACITY
    assert r(10, 3, -1, 0, 0, 1, 0, 4, None, 0, ctypes.addressof(ns), None, None) == g.DDP_OK   # nothing left
    assert ns.value == 4


def test_accum_clip_rejects(g):
    lib = g.lib_handle()
    two = _ptrs(FAKE, FAKE + 4096)
    acc = _ptrs(FAKE + 8192, FAKE + 12288)
    a = lib.ddp_bucket_accumulate
    assert a(two, acc, 0, 0, 8, None) == g.DDP_ERR_INVALID_ARG
    assert a(two, acc, 2, 3, 8, None) == g.DDP_ERR_INVALID_ARG
    assert a(two, _ptrs(FAKE + 8192, FAKE + 8200), 2, 0, 8, None) == g.DDP_ERR_ALIGNMENT
    assert a(two, _ptrs(FAKE, FAKE + 12288), 2, 0, 8, None) == g.DDP_ERR_INVALID_ARG      # acc on a micro
    assert a(two, _ptrs(FAKE + 8192, FAKE + 8192), 2, 0, 8, None) == g.DDP_ERR_INVALID_ARG  # acc twice
    assert a(two, acc, 2, 1, 0, None) == g.DDP_OK
    assert g.ddp_norm_workspace_bytes(0) == 0
    assert g.ddp_norm_workspace_bytes(3) == 3 * (2048 * 16 + 16)
    m = lib.ddp_bucket_allreduce_mean_norm
    assert m(two, 2, 0, 8, FAKE + 8192, None, 0, None) == g.DDP_ERR_INVALID_ARG
    assert m(two, 2, 0, 8, FAKE + 8192, FAKE + 65536, -1, None) == g.DDP_ERR_INVALID_ARG
    assert m(two, 2, 0, 8, FAKE + 8192, FAKE + 65544, 0, None) == g.DDP_ERR_ALIGNMENT
    assert m(two, 2, 0, 8, FAKE + 8192, FAKE, 0, None) == g.DDP_ERR_INVALID_ARG           # workspace on a replica
    f = lib.ddp_grad_norm_finalize
    assert f(None, 1, 1.0, None, None, None, None) == g.DDP_ERR_INVALID_ARG
    assert f(FAKE, 0, 1.0, None, None, None, None) == g.DDP_ERR_INVALID_ARG
    assert f(FAKE, 1, float("nan"), None, None, None, None) == g.DDP_ERR_INVALID_ARG
    assert f(FAKE, 1, 1.0, FAKE + 2, None, None, None) == g.DDP_ERR_ALIGNMENT
    assert f(FAKE, 1, 1.0, FAKE + 16, None, None, None) == g.DDP_ERR_INVALID_ARG          # output inside ws
    s = lib.ddp_bucket_sgd
    G, P, B = FAKE, FAKE + 4096, FAKE + 8192
    assert s(G, P, None, 8, 0.1, 0.9, 0.0, None, None, None) == g.DDP_ERR_INVALID_ARG    # needs the buffer
    assert s(G, P, B, 8, 0.1, 0.0, 0.0, None, None, None) == g.DDP_ERR_INVALID_ARG       # buffer unused
    assert s(G, G + 16, B, 8, 0.1, 0.9, 0.0, None, None, None) == g.DDP_ERR_INVALID_ARG  # θ overlaps grad
    assert s(G, P + 4, B, 8, 0.1, 0.9, 0.0, None, None, None) == g.DDP_ERR_ALIGNMENT
    assert s(G, P, B, 8, 0.1, 0.9, 0.0, None, P + 16, None) == g.DDP_ERR_INVALID_ARG     # bf16 copy on θ
    assert s(G, P, B, 0, 0.1, 0.9, 0.0, None, None, None) == g.DDP_OK


def test_absent_buffers_never_overlap(g):
    """NULL optional outputs (no momentum buffer, no scale) are accepted."""
    lib = g.lib_handle()
    two = _ptrs(FAKE, FAKE + 4096)
    assert lib.ddp_bucket_sgd(FAKE, FAKE + 4096, None, 0, 0.1, 0.0, 0.0, None, None, None) == g.DDP_OK
    assert lib.ddp_bucket_allreduce_sgd_cast(two, 2, 0, 8, FAKE + 8192, None, 0.1, 0.0, 0.0, None, None,
                                             None) == g.DDP_ERR_INVALID_ARG                 # cast needs its output
    assert lib.ddp_bucket_allreduce_sgd(two, 2, 0, 0, FAKE + 8192, None, 0.1, 0.0, 0.0, None, 0, None) == g.DDP_OK


def test_bn_stats_rejects(g):
    lib = g.lib_handle()
    u = lib.bn_running_stats_update
    A, B, C, D = FAKE, FAKE + 4096, FAKE + 8192, FAKE + 12288
    assert u(A, B, 0, 0.1, C, D, 8, None) == g.DDP_ERR_INVALID_ARG       # count
    assert u(A, B, 10, 1.5, C, D, 8, None) == g.DDP_ERR_INVALID_ARG      # momentum
    assert u(A, B, 10, 0.1, C, C + 16, 8, None) == g.DDP_ERR_INVALID_ARG # running buffers overlap
    assert u(A, B, 10, 0.1, C + 2, D, 8, None) == g.DDP_ERR_ALIGNMENT
    assert u(A, B, 10, 0.1, C, D, 0, None) == g.DDP_OK
    f = lib.bn_fold_inference_params
    assert f(A, B, None, None, -1.0, 8, C, D, None) == g.DDP_ERR_INVALID_ARG
    assert f(A, B, None, None, 1e-5, 8, A, D, None) == g.DDP_ERR_INVALID_ARG   # output on an input
    assert f(A, B, None, None, 1e-5, 0, C, D, None) == g.DDP_OK


def test_mean_multi_rejects(g):
    lib = g.lib_handle()
    two = _ptrs(FAKE, FAKE + (1 << 20))
    f = lib.ddp_bucket_allreduce_mean_multi
    Bk = g.DdpBucket

    def bk(*pairs):
        arr = (Bk * max(1, len(pairs)))()
        for i, (o, n) in enumerate(pairs):
            arr[i].offset_elems, arr[i].numel = o, n
        return ctypes.addressof(arr), arr

    a, keep = bk((0, 10), (64, 5))
    out = FAKE + (4 << 20)
    assert f(two, 2, 0, a, -1, out, None) == g.DDP_ERR_INVALID_ARG
    assert f(two, 2, 0, a, 1025, out, None) == g.DDP_ERR_INVALID_ARG
    a2, keep2 = bk((64, 5), (0, 10))                                   # not increasing
    assert f(two, 2, 0, a2, 2, out, None) == g.DDP_ERR_INVALID_ARG
    a3, keep3 = bk((0, 10), (6, 5))                                    # overlapping
    assert f(two, 2, 0, a3, 2, out, None) == g.DDP_ERR_INVALID_ARG
    a4, keep4 = bk((0, 10), (66, 5))                                   # 66*4 bytes: not 16-aligned
    assert f(two, 2, 0, a4, 2, out, None) == g.DDP_ERR_ALIGNMENT
    assert f(two, 2, 0, a, 2, FAKE, None) == g.DDP_ERR_INVALID_ARG     # output on replica 0
    assert f(two, 2, 0, a, 0, out, None) == g.DDP_OK
    a5, keep5 = bk((0, 0), (64, 0))
    assert f(two, 2, 0, a5, 2, out, None) == g.DDP_OK                  # empty buckets only


def test_syncbn_channel_parts(g):
    """Which SyncBN calls run as two channel halves on two streams: aligned
    planes with the plane statistics kernel (H*W a multiple of 8 and, for
    bf16, at least 16 vectors; even C, halves of at least 16 channels, 16 MiB
    of input over all replicas), and calls with the per-warp bulk-staged
    statistics (halves of whole channel groups whose run in a sample is a
    whole number of 16-byte vectors, 32 MiB, unaligned planes only).  The planner decides on the
    host, no GPU needed."""
    bf16, f32 = g.BF16, g.F32
    assert g.syncbn_channel_parts(8, bf16, 32, 64, 56, 56) == 2
    assert g.syncbn_channel_parts(8, bf16, 32, 256, 56, 56) == 2
    assert g.syncbn_channel_parts(8, bf16, 32, 512, 28, 28) == 2
    assert g.syncbn_channel_parts(8, bf16, 32, 2048, 7, 7) == 2       # per-warp bulk-staged statistics
    assert g.syncbn_channel_parts(8, f32, 32, 2048, 7, 7) == 1        # fp32 runs: tiled bulk kernel
    assert g.syncbn_channel_parts(8, bf16, 32, 2047, 7, 7) == 1       # odd C
    assert g.syncbn_channel_parts(8, bf16, 32, 512, 7, 7) == 1        # 12.8 MB: under 32 MiB
    assert g.syncbn_channel_parts(8, bf16, 32, 1024, 14, 14) == 2
    assert g.syncbn_channel_parts(8, bf16, 32, 256, 14, 14) == 1      # 26 MB
    assert g.syncbn_channel_parts(8, bf16, 32, 1024, 17, 17) == 2     # groups of 4 channels, runs of 1156
    assert g.syncbn_channel_parts(8, bf16, 32, 1032, 17, 17) == 1     # a half's run of 516*289 elements
    assert g.syncbn_channel_parts(8, bf16, 32, 2048, 8, 8) == 1       # 8 vectors per plane: bulk-staged, aligned
    assert g.syncbn_channel_parts(8, f32, 32, 2048, 8, 8) == 2        # fp32: plane kernel, 16 vectors
    assert g.syncbn_channel_parts(8, bf16, 32, 65, 56, 56) == 1       # odd C
    assert g.syncbn_channel_parts(8, bf16, 32, 30, 56, 56) == 1       # 15 channels per half
    assert g.syncbn_channel_parts(8, bf16, 32, 32, 56, 56) == 2       # 16 per half, 51 MB
    assert g.syncbn_channel_parts(2, bf16, 32, 32, 56, 56) == 1       # 12.8 MB: under 16 MiB
    assert g.syncbn_channel_parts(8, bf16, 32, 64, 28, 29) == 1       # H*W = 812: bulk-staged, 26.6 MB
    for bad in [(0, bf16, 32, 64, 56, 56), (17, bf16, 32, 64, 56, 56), (8, 7, 32, 64, 56, 56),
                (8, bf16, 0, 64, 56, 56), (8, bf16, 32, 64, 0, 56)]:
        with pytest.raises(RuntimeError):
            g.syncbn_channel_parts(*bad)
