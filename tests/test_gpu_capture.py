"""CUDA Graph capture of the entry points other than the bucket average
(which test_gpu_mean covers): a captured call replayed gives the bits of the
same call made eagerly, and the SyncBN path works when its very first call
in a process is made inside a capture (its statistics kernel opts into more
than 48 KiB of shared memory on first use)."""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_common import assert_bit_exact, dev_bf16, dev_f32, host_bits, load_library, sync

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def g():
    return load_library()


def _capture(fn):
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        fn()
    return graph


def test_sampler_in_graph(g):
    n, N = 100_003, 8
    ns = g.dist_sampler_num_samples(n, N, False)
    out = torch.full((N * ns,), -7, dtype=torch.int64, device="cuda")
    graph = _capture(lambda: g.dist_sampler_indices(n, N, -1, 5, 2, True, False, out))
    graph.replay()
    sync()
    want = oracle.dist_sampler_indices(n, N, -1, 5, 2, True, False).reshape(-1)
    np.testing.assert_array_equal(out.cpu().numpy(), want)


def test_sgd_steps_in_graph(g):
    """Three replays of a captured fused SGD step equal three oracle steps."""
    numel, n = 70_001, 8
    gen = np.random.Generator(np.random.PCG64(21))
    theta = (gen.standard_normal(numel) * 0.02).astype(np.float32)
    reps = [workloads.f32_to_bf16_bits((gen.standard_normal(numel) * 0.01).astype(np.float32)) for _ in range(n)]
    d = [dev_bf16(r) for r in reps]
    th_d, b_d = dev_f32(theta), torch.zeros(numel, device="cuda")
    graph = _capture(lambda: g.ddp_bucket_allreduce_sgd(d, th_d, b_d, 0.1, 0.9, 1e-4))
    buf = np.zeros(numel, np.float32)
    th_d.copy_(torch.from_numpy(theta))          # capture does not run the step
    b_d.zero_()
    for _ in range(3):
        graph.replay()
        theta, buf, _ = oracle.sgd_step(reps, theta, buf, 0.1, 0.9, 1e-4, dtype="bf16")
    sync()
    assert_bit_exact(th_d, theta, "theta after 3 replays")
    assert_bit_exact(b_d, buf, "buffer after 3 replays")


@pytest.mark.parametrize("shape", [(4, 4, 64, 7, 7), (2, 3, 16, 28, 28)])
def test_syncbn_in_graph_matches_eager(g, shape):
    n, B, C, H, W = shape
    xs = [dev_bf16(x) for x in workloads.syncbn_input(4, n, B, C, H, W)]
    ws = torch.empty(g.syncbn_workspace_bytes(n, B, C, H, W), dtype=torch.uint8, device="cuda")
    ys_e = [torch.empty_like(x) for x in xs]
    m_e, s_e = torch.empty(C, device="cuda"), torch.empty(C, device="cuda")
    g.syncbn_merge_apply(xs, ys_e, m_e, s_e, ws)
    ys = [torch.empty_like(x) for x in xs]
    m, s = torch.empty(C, device="cuda"), torch.empty(C, device="cuda")
    graph = _capture(lambda: g.syncbn_merge_apply(xs, ys, m, s, ws))
    graph.replay()
    sync()
    np.testing.assert_array_equal(host_bits(m), host_bits(m_e))
    np.testing.assert_array_equal(host_bits(s), host_bits(s_e))
    for r in range(n):
        np.testing.assert_array_equal(host_bits(ys[r]), host_bits(ys_e[r]))


_FIRST_CALL_IN_CAPTURE = r"""
import sys, torch
sys.path.insert(0, sys.argv[1])
import gradient_sync_ddp_gb300 as g
import workloads
n, B, C, H, W = 8, 8, 256, 7, 7
xs = [torch.from_numpy(x.view('int16')).cuda().view(torch.bfloat16) for x in workloads.syncbn_input(4, n, B, C, H, W)]
ws = torch.empty(g.syncbn_workspace_bytes(n, B, C, H, W), dtype=torch.uint8, device='cuda')
ys = [torch.empty_like(x) for x in xs]
m, s = torch.empty(C, device='cuda'), torch.empty(C, device='cuda')
side = torch.cuda.Stream()
side.wait_stream(torch.cuda.current_stream())
graph = torch.cuda.CUDAGraph()
with torch.cuda.graph(graph, stream=side):
    g.syncbn_merge_apply(xs, ys, m, s, ws)          # the first SyncBN call of this process
graph.replay()
torch.cuda.synchronize()
ys2 = [torch.empty_like(x) for x in xs]
m2, s2 = torch.empty(C, device='cuda'), torch.empty(C, device='cuda')
g.syncbn_merge_apply(xs, ys2, m2, s2, ws)
torch.cuda.synchronize()
ok = torch.equal(m.view(torch.int32), m2.view(torch.int32)) and torch.equal(s.view(torch.int32), s2.view(torch.int32))
ok = ok and all(torch.equal(a.view(torch.int16), b.view(torch.int16)) for a, b in zip(ys, ys2))
print('same' if ok else 'differ')
sys.exit(0 if ok else 1)
"""


def test_syncbn_first_call_inside_capture(g):
    """A fresh process whose first SyncBN call (7x7 planes: the bulk-staged
    statistics kernel with 50 KiB of dynamic shared memory) is inside a
    graph capture; the replay equals a later eager call bit for bit."""
    r = subprocess.run([sys.executable, "-c", _FIRST_CALL_IN_CAPTURE, ROOT], capture_output=True, text=True,
                       timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "same" in r.stdout
