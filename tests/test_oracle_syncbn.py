"""Pins for the oracle's SyncBatchNorm merge + apply (CPU only)."""
import numpy as np
import torch

import oracle
import workloads


def _replicas(N=3, B=4, C=5, H=3, W=7, seed=0, mean=0.5, std=2.0):
    gen = np.random.Generator(np.random.PCG64(seed))
    return [workloads.f32_to_bf16_bits((gen.standard_normal((B, C, H, W)) * std + mean).astype(np.float32))
            for _ in range(N)]


def check_syncbn_two_pass(fn):
    """mean and the biased variance agree with the two-pass definition
    Σ(x − mean)² / M over the concatenated global batch, in fp64."""
    xs = _replicas()
    mean, invstd, _ = fn(xs, 1e-5)
    allx = np.concatenate([oracle.bf16_bits_to_f32(x).astype(np.float64) for x in xs], axis=0)
    m2 = allx.mean(axis=(0, 2, 3))
    v2 = ((allx - m2[None, :, None, None]) ** 2).mean(axis=(0, 2, 3))
    np.testing.assert_allclose(mean, m2, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(invstd, 1 / np.sqrt(v2 + 1e-5), rtol=1e-12)


def test_syncbn_two_pass():
    check_syncbn_two_pass(oracle.syncbn)


def check_syncbn_vs_torch_batch_norm(fn):
    """SyncBatchNorm over N replicas is batch norm over their concatenation
    (AI_Infra notes "1.DataParallel / DDP" §4.3: the synced statistics are
    those of the global batch).  torch.nn.functional.batch_norm in training
    mode, fp64, with affine γ, β, is the independent reference."""
    xs = _replicas(N=4, B=2, C=6, H=5, W=5, seed=1)
    gen = np.random.Generator(np.random.PCG64(2))
    gamma = gen.standard_normal(6)
    beta = gen.standard_normal(6)
    mean, invstd, ys = fn(xs, 1e-5, gamma, beta)
    allx = torch.from_numpy(np.concatenate([oracle.bf16_bits_to_f32(x).astype(np.float64) for x in xs]))
    ref = torch.nn.functional.batch_norm(allx, None, None, torch.from_numpy(gamma), torch.from_numpy(beta),
                                         training=True, eps=1e-5).numpy()
    np.testing.assert_allclose(np.concatenate(ys), ref, rtol=1e-10, atol=1e-12)


def test_syncbn_vs_torch_batch_norm():
    check_syncbn_vs_torch_batch_norm(oracle.syncbn)


def test_syncbn_constant_channel():
    """A constant channel has zero variance: invstd = 1/sqrt(eps), y = β."""
    xs = _replicas(N=2, B=2, C=3, H=2, W=2)
    for x in xs:
        x[:, 1] = 0x4040          # 3.0
    mean, invstd, ys = oracle.syncbn(xs, 1e-5)
    assert mean[1] == 3.0
    assert invstd[1] == 1 / np.sqrt(1e-5)
    assert all(np.all(y[:, 1] == 0.0) for y in ys)


def test_syncbn_stats_at_matches_full():
    xs = _replicas(N=3, B=2, C=4, H=6, W=6, seed=4)
    mean, invstd, _ = oracle.syncbn(xs, 1e-5)
    for c in range(4):
        m, s = oracle.syncbn_stats_at(xs, c, 1e-5)
        assert abs(m - mean[c]) <= 1e-12 * max(1, abs(mean[c]))
        assert abs(s - invstd[c]) <= 1e-12 * invstd[c]


def test_f64_to_bf16_rne_matches_torch():
    """Direct fp64 -> bf16 rounding against torch's fp32 -> bf16 conversion on
    values that are exact in fp32 (so torch's route rounds only once)."""
    gen = np.random.Generator(np.random.PCG64(6))
    x = (gen.standard_normal(200000) * np.exp(gen.uniform(-20, 20, 200000))).astype(np.float32)
    # include exact ties in [1, 2): bf16 spacing there is 2^-7, so 1 + (2k+1)*2^-8
    ties = np.float32(1.0) + (np.arange(128, dtype=np.float32) * 2 + 1) * np.float32(2.0 ** -8)
    x = np.concatenate([x, ties, -ties]).astype(np.float32)
    ours = oracle.f64_to_bf16_rne(x.astype(np.float64))
    t = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(ours, t)
