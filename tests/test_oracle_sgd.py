"""Pins for the oracle's fused SGD step (CPU only)."""
import numpy as np
import torch

import oracle
from conftest import golden_rows


def check_sgd_golden(sgd_fn):
    """Dyadic worked examples, exact in fp32 (tests/golden/sgd_step.txt)."""
    rows = golden_rows("sgd_step.txt")
    assert len(rows) >= 4
    for reps_s, th_s, buf_s, lr_s, mu_s, wd_s, exp_th, exp_buf, why in rows:
        reps = [np.array([float(v)], dtype=np.float32) for v in reps_s.split()]
        th, b, _ = sgd_fn(reps, np.array([float(th_s)], np.float32), np.array([float(buf_s)], np.float32),
                          float(lr_s), float(mu_s), float(wd_s))
        assert th[0] == np.float32(float(exp_th)), why
        if exp_buf == "none":
            assert b is None, why
        else:
            assert b[0] == np.float32(float(exp_buf)), why


def test_sgd_golden():
    check_sgd_golden(oracle.sgd_step)


def check_sgd_vs_torch(sgd_fn):
    """Three steps against torch.optim.SGD (momentum 0.9, weight decay 1e-4,
    lr 0.1, fp32, CPU) fed the same averaged gradient.  torch rounds its
    operations in a different grouping, so the comparison allows a few fp32
    ulps; a wrong term (sign, factor, order of momentum and decay) is far
    outside that."""
    gen = np.random.Generator(np.random.PCG64(21))
    n, N = 5000, 8
    theta = (gen.standard_normal(n) * 0.02).astype(np.float32)
    p = torch.nn.Parameter(torch.from_numpy(theta.copy()))
    opt = torch.optim.SGD([p], lr=0.1, momentum=0.9, weight_decay=1e-4, foreach=False)
    th, buf = theta.copy(), np.zeros(n, np.float32)
    for step in range(3):
        reps = [(gen.standard_normal(n) * 0.01).astype(np.float32) for _ in range(N)]
        th, buf, g = sgd_fn(reps, th, buf, 0.1, 0.9, 1e-4)
        p.grad = torch.from_numpy(np.mean(np.stack(reps).astype(np.float64), axis=0).astype(np.float32))
        opt.step()
        ref = p.detach().numpy()
        np.testing.assert_allclose(th, ref, rtol=2e-6, atol=1e-8)
        np.testing.assert_allclose(buf, opt.state[p]["momentum_buffer"].numpy(), rtol=1e-5, atol=1e-9)


def test_sgd_vs_torch():
    check_sgd_vs_torch(oracle.sgd_step)


def test_sgd_plain_reduces_to_update_rule():
    """μ = 0, wd = 0: θ − lr·g with g the (exact, small-integer) average;
    no buffer is produced ("1.DataParallel / DDP" §5.3)."""
    reps = [np.full(7, float(r), np.float32) for r in range(4)]       # mean 1.5
    th, b, g = oracle.sgd_step(reps, np.full(7, 10.0, np.float32), None, 0.5, 0.0, 0.0)
    assert b is None
    np.testing.assert_array_equal(g, np.full(7, 1.5, np.float32))
    np.testing.assert_array_equal(th, np.full(7, 9.25, np.float32))


def test_sgd_bf16_replicas():
    """bf16 replicas: the step equals the fp32 step on the exactly widened values."""
    gen = np.random.Generator(np.random.PCG64(8))
    reps = [gen.integers(0x3000, 0x4000, 999).astype(np.uint16) for _ in range(4)]
    th0 = gen.standard_normal(999).astype(np.float32)
    b0 = gen.standard_normal(999).astype(np.float32)
    a = oracle.sgd_step(reps, th0, b0, 0.1, 0.9, 1e-4, dtype="bf16")
    w = oracle.sgd_step([oracle.bf16_bits_to_f32(r) for r in reps], th0, b0, 0.1, 0.9, 1e-4)
    for x, y in zip(a, w):
        assert np.array_equal(x, y)
