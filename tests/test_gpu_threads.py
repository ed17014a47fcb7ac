"""Concurrent calls: the library's per-device caches (device limits,
occupancy, shared-memory opt-ins) are shared between host threads.  Four
threads, each with its own stream and buffers, call the average, the fused
SGD, SyncBN and the sampler at the same time (ctypes releases the GIL during
the foreign call); every result equals the oracle's."""
import threading

import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_common import assert_bit_exact, dev_bf16, dev_f32, load_library

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    return load_library()


def _worker(g, k, results, errors):
    try:
        torch.cuda.set_device(0)
        st = torch.cuda.Stream()
        gen = np.random.Generator(np.random.PCG64(900 + k))
        numel, n = 100_003 + 17 * k, 3 + k
        reps = [gen.standard_normal(numel).astype(np.float32) for _ in range(n)]
        theta = (gen.standard_normal(numel) * 0.02).astype(np.float32)
        xs = workloads.syncbn_input(4, 2, 3, 24 + k, 7, 7)
        with torch.cuda.stream(st):
            d = [dev_f32(r) for r in reps]
            out = torch.empty(numel, device="cuda")
            th = dev_f32(theta)
            buf = torch.zeros(numel, device="cuda")
            xd = [dev_bf16(x) for x in xs]
            ys = [torch.empty_like(x) for x in xd]
            C = 24 + k
            mean, inv = torch.empty(C, device="cuda"), torch.empty(C, device="cuda")
            ws = torch.empty(g.syncbn_workspace_bytes(2, 3, C, 7, 7), dtype=torch.uint8, device="cuda")
            ns = g.dist_sampler_num_samples(50_000, 4, False)
            idx = torch.empty(4 * ns, dtype=torch.int64, device="cuda")
            for _ in range(20):
                g.ddp_bucket_allreduce_mean(d, out, stream=st)
                g.syncbn_merge_apply(xd, ys, mean, inv, ws, stream=st)
                g.dist_sampler_indices(50_000, 4, -1, k, 1, True, False, idx, stream=st)
            g.ddp_bucket_allreduce_sgd(d, th, buf, 0.1, 0.9, 1e-4, stream=st)
        st.synchronize()
        results[k] = (reps, theta, out.cpu(), th.cpu(), idx.cpu().numpy(), xs,
                      mean.cpu().numpy(), inv.cpu().numpy())
    except Exception as e:        # reported by the main thread
        errors.append((k, repr(e)))


def test_four_threads_at_once(g):
    results, errors = {}, []
    ths = [threading.Thread(target=_worker, args=(g, k, results, errors)) for k in range(4)]
    for t in ths:
        t.start()
    for t in ths:
        t.join(timeout=300)
    assert not errors, errors
    for k in range(4):
        reps, theta, out, th, idx, xs, mean, inv = results[k]
        assert_bit_exact(out, oracle.grad_mean(reps), f"thread {k} average")
        th_w, _, _ = oracle.sgd_step(reps, theta, np.zeros_like(theta), 0.1, 0.9, 1e-4)
        assert_bit_exact(th, th_w, f"thread {k} sgd")
        np.testing.assert_array_equal(idx, oracle.dist_sampler_indices(50_000, 4, -1, k, 1, True, False).reshape(-1))
        m_w, s_w, _ = oracle.syncbn(xs, 1e-5)
        assert np.all(np.abs(mean - m_w) <= 1e-5 * np.abs(m_w) + 1e-7 / s_w), f"thread {k} syncbn mean"
        assert np.all(np.abs(inv - s_w) <= 1e-5 * np.abs(s_w)), f"thread {k} syncbn invstd"
