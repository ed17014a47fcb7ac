"""Pins for the oracle's accumulation, global norm / clipping and non-finite
check (CPU only)."""
import math

import numpy as np
import pytest
import torch

import oracle


def check_no_sync_equivalence(accumulate_fn, mean_fn):
    """AI_Infra notes "1.DataParallel / DDP" §5.2: with the loss divided by
    the accumulation steps K, K local backward passes accumulated under
    no_sync and then averaged over the N replicas give the gradient of one
    pass over all N*K micro-batches.  Linear(128, 10) + cross-entropy, fp64
    autograd (independent of the oracle), N = 4, K = 3, micro-batch 8."""
    g = torch.Generator().manual_seed(11)
    N, K, b = 4, 3, 8
    B = N * K * b
    x = torch.randn(B, 128, generator=g, dtype=torch.float64)
    y = torch.randint(0, 10, (B,), generator=g)
    W = torch.randn(10, 128, generator=g, dtype=torch.float64) * 0.1
    bias = torch.randn(10, generator=g, dtype=torch.float64) * 0.1

    def grad(xs, ys, scale):
        Wp = W.clone().requires_grad_(True)
        bp = bias.clone().requires_grad_(True)
        (torch.nn.functional.cross_entropy(xs @ Wp.T + bp, ys) * scale).backward()
        return torch.cat([Wp.grad.reshape(-1), bp.grad]).numpy()

    full = grad(x, y, 1.0)
    accs = []
    for r in range(N):
        acc = np.zeros(1290)
        for k in range(K):
            s = (r * K + k) * b
            acc = accumulate_fn(acc, grad(x[s:s + b], y[s:s + b], 1.0 / K), "f64")
        accs.append(acc)
    np.testing.assert_allclose(mean_fn(accs, "f64"), full, rtol=1e-12, atol=1e-15)


def test_no_sync_equivalence():
    check_no_sync_equivalence(oracle.accumulate, oracle.grad_mean)


def test_accumulate_is_one_fp32_addition():
    a = np.array([1.0, 2.0 ** 24, -0.0, 1e-40], np.float32)
    m = np.array([2.0 ** -24, 1.0, -0.0, 1e-40], np.float32)
    got = oracle.accumulate(a, m)
    # 1 + 2^-24 rounds to 1 (tie to even); 2^24 + 1 rounds to 2^24; -0 + -0 = -0; subnormals kept
    assert got.tolist()[:2] == [1.0, 2.0 ** 24]
    assert math.copysign(1.0, got[2]) == -1.0
    # a subnormal plus itself: the integer significand doubles exactly (no flush to zero)
    assert got[3:4].view(np.uint32)[0] == 2 * m[3:4].view(np.uint32)[0]
    bf = np.array([0x3F80, 0x4000], np.uint16)                   # 1.0, 2.0
    assert oracle.accumulate(np.zeros(2, np.float32), bf, "bf16").tolist() == [1.0, 2.0]


def check_norm_and_clip(norm_fn, coef_fn):
    """Against torch.nn.utils.clip_grad_norm_ (fp64, CPU): the returned total
    norm and the clipped gradients (g * coefficient)."""
    gen = np.random.Generator(np.random.PCG64(5))
    grads = [gen.standard_normal(n) * s for n, s in ((1000, 0.3), (17, 2.0), (4096, 0.01))]
    for max_norm in (0.5, 1.0, 1e6):
        ps = [torch.nn.Parameter(torch.zeros(len(gr), dtype=torch.float64)) for gr in grads]
        for p, gr in zip(ps, grads):
            p.grad = torch.from_numpy(gr.copy())
        total = float(torch.nn.utils.clip_grad_norm_(ps, max_norm))
        norm = norm_fn(grads)
        assert norm == pytest.approx(total, rel=1e-13)
        c = coef_fn(norm, max_norm)
        for p, gr in zip(ps, grads):
            np.testing.assert_allclose(gr * c, p.grad.numpy(), rtol=1e-13, atol=0)


def test_norm_and_clip_vs_torch():
    check_norm_and_clip(oracle.grad_global_norm, oracle.clip_coefficient)


def test_norm_closed_forms():
    assert oracle.grad_global_norm([[3.0], [4.0]]) == 5.0
    assert oracle.grad_global_norm([[0.0, 0.0]]) == 0.0
    assert oracle.clip_coefficient(5.0, 1.0) == 1.0 / (5.0 + 1e-6)
    assert oracle.clip_coefficient(0.5, 1.0) == 1.0                 # below the threshold: unchanged
    assert oracle.clip_coefficient(5.0, 0.0) == 1.0                 # clipping disabled


def test_nonfinite():
    assert not oracle.any_nonfinite([np.ones(3, np.float32), np.zeros(2, np.float32)])
    assert oracle.any_nonfinite([np.ones(3, np.float32), np.array([0, np.nan], np.float32)])
    assert oracle.any_nonfinite([np.array([-np.inf], np.float32)])
    assert not oracle.any_nonfinite([np.array([3e38], np.float32)])


def test_sgd_from_grad_matches_sgd_step():
    """Without a scale, the step on an averaged gradient is sgd_step's step
    (same operations after the average)."""
    gen = np.random.Generator(np.random.PCG64(9))
    reps = [gen.standard_normal(777).astype(np.float32) for _ in range(4)]
    th = gen.standard_normal(777).astype(np.float32)
    b = gen.standard_normal(777).astype(np.float32)
    th1, b1, g = oracle.sgd_step(reps, th, b, 0.1, 0.9, 1e-4)
    th2, b2 = oracle.sgd_from_grad(g, th, b, 0.1, 0.9, 1e-4)
    assert np.array_equal(th1, th2) and np.array_equal(b1, b2)
    # scale: dyadic example, exact: g=2, scale=0.25 -> d=0.5; θ = 1 - 0.5*0.5 = 0.75
    th3, b3 = oracle.sgd_from_grad(np.array([2.0], np.float32), np.array([1.0], np.float32), None,
                                   0.5, 0.0, 0.0, scale=0.25)
    assert th3[0] == 0.75 and b3 is None


def test_f32_to_bf16_rne_vs_torch():
    """Every class of value against torch's fp32 -> bf16 conversion: random
    magnitudes, exact ties (both parities), the largest values that still
    round to finite, subnormals, signed zeros, infinities; NaN stays NaN."""
    gen = np.random.Generator(np.random.PCG64(21))
    x = (gen.standard_normal(100_000) * np.exp(gen.uniform(-80, 80, 100_000))).astype(np.float32)
    ties = np.array([0x3F808000, 0x3F818000, 0xBF808000, 0x00008000, 0x00018000, 0x7F7F8000, 0x7F7F7FFF],
                    np.uint32).view(np.float32)
    special = np.array([0.0, -0.0, np.inf, -np.inf, 1e-45, -1e-45, 3.4e38], np.float32)
    x = np.concatenate([x, ties, special])
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(oracle.f32_to_bf16_rne(x), want)
    nanbits = oracle.f32_to_bf16_rne(np.array([np.nan], np.float32))
    assert np.isnan(oracle.bf16_bits_to_f32(nanbits))[0]
