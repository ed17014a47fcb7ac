"""GPU parity: BN running-statistics sync (STATS_COMM + UPDATE_STATS), the
validation-metric mean, the running update and the inference folding."""
import numpy as np
import pytest
import torch

import oracle
from gpu_common import assert_bit_exact, dev_f32, load_library, sync

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    return load_library()


def test_stats_comm_and_update_stats(g):
    """Tech-Renaissance "(24) NCCL通信与分布式数据并行" §十二: every replica's
    B_NEXT [running mean | running var] (ResNet-50's 53 BN layers, 26,560
    values) is mean-all-reduced and copied into B_PREV.  One average with
    write-back: B_PREV gets the average, every B_NEXT the same bits."""
    C = 2 * sum([64] + [64, 64, 256, 256] + [64, 64, 256] * 2 + [128, 128, 512, 512] + [128, 128, 512] * 3
                + [256, 256, 1024, 1024] + [256, 256, 1024] * 5 + [512, 512, 2048, 2048] + [512, 512, 2048] * 2)
    assert C == 2 * 26_560
    gen = np.random.Generator(np.random.PCG64(12))
    nxt = [np.concatenate([gen.standard_normal(C // 2), gen.random(C // 2) + 0.5]).astype(np.float32)
           for _ in range(8)]
    d = [dev_f32(x) for x in nxt]
    prev = torch.full((C,), float("nan"), device="cuda")
    g.ddp_bucket_allreduce_mean(d, prev, flags=g.FLAG_WRITE_BACK_ALL)
    sync()
    want = oracle.grad_mean(nxt)
    assert_bit_exact(prev, want, "B_PREV")
    for r in range(8):
        assert_bit_exact(d[r], want, f"B_NEXT replica {r}")


def test_validation_metric_mean(g):
    """VAL_RESULT_COMM (§十三): sum_loss, sum_top1, sum_top5 of each replica
    averaged: three values."""
    vals = [np.array([2.5 + r, 60.0 + 3 * r, 85.0 + r], np.float32) for r in range(8)]
    out = torch.empty(3, device="cuda")
    g.ddp_bucket_allreduce_mean([dev_f32(v) for v in vals], out)
    sync()
    assert_bit_exact(out, oracle.grad_mean(vals), "metric mean")


def test_running_update(g):
    gen = np.random.Generator(np.random.PCG64(13))
    for C in (1, 7, 2048, 10_001):
        for count, mom in ((802_816, 0.1), (2, 0.5), (1, 0.25)):
            rm = gen.standard_normal(C).astype(np.float32)
            rv = (gen.random(C) + 0.1).astype(np.float32)
            bm = gen.standard_normal(C).astype(np.float32)
            bv = (gen.random(C) * 4).astype(np.float32)
            rm_d, rv_d = dev_f32(rm), dev_f32(rv)
            g.bn_running_stats_update(dev_f32(bm), dev_f32(bv), count, mom, rm_d, rv_d)
            sync()
            wm, wv = oracle.bn_running_update(rm, rv, bm, bv, count, mom)
            assert_bit_exact(rm_d, wm, f"running mean C={C}")
            assert_bit_exact(rv_d, wv, f"running var C={C}")


def test_fold(g):
    gen = np.random.Generator(np.random.PCG64(14))
    for C in (1, 33, 2048):
        rm = gen.standard_normal(C).astype(np.float32)
        rv = (gen.random(C) + 1e-3).astype(np.float32)
        ga = gen.standard_normal(C).astype(np.float32)
        be = gen.standard_normal(C).astype(np.float32)
        for gamma, beta in ((ga, be), (None, None)):
            sc, bi = torch.empty(C, device="cuda"), torch.empty(C, device="cuda")
            g.bn_fold_inference_params(dev_f32(rm), dev_f32(rv), None if gamma is None else dev_f32(gamma),
                                       None if beta is None else dev_f32(beta), 1e-5, sc, bi)
            sync()
            ws, wb = oracle.bn_fold_inference(rm, rv, gamma, beta, 1e-5)
            np.testing.assert_allclose(sc.cpu().numpy(), ws, rtol=1e-6, atol=0)
            np.testing.assert_allclose(bi.cpu().numpy(), wb, rtol=1e-6, atol=1e-6)
