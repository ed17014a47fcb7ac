"""GPU parity: ddp_bucket_allreduce_sgd against the oracle, bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_common import assert_bit_exact, dev_bf16, dev_f32, load_library, sync

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    return load_library()


def test_linear_128_10_plain_sgd(g):
    """Linear(128, 10) grads, N = 4, one bucket, mean then SGD lr = 0.1,
    momentum 0 (no buffer)."""
    numel = 1290
    reps = workloads.replica_grads(1, 4, numel, 1.0)
    theta = workloads.params_f32(1, numel, 0.1)
    th_d = dev_f32(theta)
    gout = torch.empty(numel, device="cuda")
    g.ddp_bucket_allreduce_sgd([dev_f32(r) for r in reps], th_d, None, 0.1, 0.0, 0.0, grad_out=gout)
    sync()
    th_w, b_w, g_w = oracle.sgd_step(reps, theta, None, 0.1, 0.0, 0.0)
    assert b_w is None
    assert_bit_exact(th_d, th_w, "theta")
    assert_bit_exact(gout, g_w, "grad")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_momentum_weight_decay_three_steps(g, dtype):
    for n in (1, 3, 8, 16):
        for numel in (1, 5, 4099, 250_007):
            gen = np.random.Generator(np.random.PCG64(n * 31 + numel))
            theta = (gen.standard_normal(numel) * 0.02).astype(np.float32)
            buf = np.zeros(numel, np.float32)
            th_d, b_d = dev_f32(theta), dev_f32(buf)
            gout = torch.empty(numel, device="cuda")
            for step in range(3):
                reps = [(gen.standard_normal(numel) * 0.01).astype(np.float32) for _ in range(n)]
                if dtype == "bf16":
                    reps = [workloads.f32_to_bf16_bits(r) for r in reps]
                d = [dev_f32(r) if dtype == "f32" else dev_bf16(r) for r in reps]
                g.ddp_bucket_allreduce_sgd(d, th_d, b_d, 0.1, 0.9, 1e-4, grad_out=gout if step != 1 else None)
                theta, buf, gm = oracle.sgd_step(reps, theta, buf, 0.1, 0.9, 1e-4, dtype=dtype)
                sync()
                assert_bit_exact(th_d, theta, f"theta {dtype} N={n} numel={numel} step={step}")
                assert_bit_exact(b_d, buf, f"buf {dtype} N={n} numel={numel} step={step}")
                if step != 1:
                    assert_bit_exact(gout, gm, f"grad {dtype} N={n} numel={numel} step={step}")


def test_weight_decay_only_and_adversarial(g):
    gen = np.random.Generator(np.random.PCG64(4))
    numel = 30_001
    reps = [workloads.adversarial_f32(gen, numel) for _ in range(4)]
    theta = workloads.adversarial_f32(gen, numel)
    th_d = dev_f32(theta)
    g.ddp_bucket_allreduce_sgd([dev_f32(r) for r in reps], th_d, None, 0.25, 0.0, 0.5)
    sync()
    with np.errstate(all="ignore"):
        want, _, _ = oracle.sgd_step(reps, theta, None, 0.25, 0.0, 0.5)
    assert_bit_exact(th_d, want, "wd-only adversarial")


def test_gpt2_deep_first_full_size_sampled(g):
    """GPT-2 small layout (124,439,808 params), bf16 grads N(0, 0.01) on 8
    replicas, DEEP/FIRST buckets, fused SGD momentum 0.9, wd 1e-4, lr 0.1,
    three steps from a zero buffer.  Inputs are drawn on the device from
    seeded generators; the oracle recomputes a sample of 2^20 random
    positions plus both ends of each bucket from the same input bits."""
    layout, first = workloads.gpt2_small_layout()
    num = workloads.numels(layout)
    plan = g.ddp_plan_buckets(num, 2, 0, g.PLAN_DEEP_FIRST, first)
    total = plan["total_elems"]
    n = 8
    theta = workloads.device_normal((total,), 0.0, 0.02, workloads.seed_for(3, 99))
    buf = torch.zeros(total, device="cuda")
    gen = np.random.Generator(np.random.PCG64(3))
    idx = [gen.integers(0, total, 1 << 20)]
    for off, numel, _, _ in plan["buckets"]:
        idx += [np.arange(off, off + 4096), np.arange(off + numel - 4096, off + numel)]
    idx = np.unique(np.concatenate(idx))
    idx_d = torch.from_numpy(idx).cuda()
    th_w = theta[idx_d].cpu().numpy()
    b_w = np.zeros(idx.size, np.float32)
    for step in range(3):
        reps = [workloads.device_normal((total,), 0.0, 0.01, workloads.seed_for(3, r) + 1000 * step,
                                        dtype=torch.bfloat16) for r in range(n)]
        for off, numel, _, _ in plan["buckets"]:
            g.ddp_bucket_allreduce_sgd([x[off:off + numel] for x in reps], theta[off:off + numel],
                                       buf[off:off + numel], 0.1, 0.9, 1e-4)
        sample = [x[idx_d].view(torch.int16).cpu().numpy().view(np.uint16) for x in reps]
        th_w, b_w, _ = oracle.sgd_step(sample, th_w, b_w, 0.1, 0.9, 1e-4, dtype="bf16")
        sync()
        assert_bit_exact(theta[idx_d], th_w, f"theta step {step}")
        assert_bit_exact(buf[idx_d], b_w, f"buf step {step}")
        del reps


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_sgd_with_bf16_weight_copy(g, dtype):
    """ddp_bucket_allreduce_sgd_cast: θ as without the copy, and the copy is
    θ rounded to bf16 (nearest, ties to even), bit for bit."""
    for n in (1, 3, 8):
        for numel in (1, 3, 4, 5, 8, 9, 4099, 250_007):
            gen = np.random.Generator(np.random.PCG64(n * 13 + numel))
            theta = (gen.standard_normal(numel) * 0.02).astype(np.float32)
            buf = np.zeros(numel, np.float32)
            reps = [(gen.standard_normal(numel) * 0.01).astype(np.float32) for _ in range(n)]
            if dtype == "bf16":
                reps = [workloads.f32_to_bf16_bits(r) for r in reps]
            d = [dev_f32(r) if dtype == "f32" else dev_bf16(r) for r in reps]
            th_d, b_d = dev_f32(theta), dev_f32(buf)
            low = torch.empty(numel, dtype=torch.bfloat16, device="cuda")
            g.ddp_bucket_allreduce_sgd_cast(d, th_d, b_d, 0.1, 0.9, 1e-4, low)
            sync()
            th_w, b_w, _ = oracle.sgd_step(reps, theta, buf, 0.1, 0.9, 1e-4, dtype=dtype)
            assert_bit_exact(th_d, th_w, f"theta {dtype} N={n} numel={numel}")
            got = low.view(torch.int16).cpu().numpy().view(np.uint16)
            np.testing.assert_array_equal(got, oracle.f32_to_bf16_rne(th_w))


def test_sgd_from_grad_with_bf16_weight_copy(g):
    gen = np.random.Generator(np.random.PCG64(77))
    for numel in (1, 6, 4099, 300_001):
        gr = (gen.standard_normal(numel) * 0.05).astype(np.float32)
        th = (gen.standard_normal(numel) * 0.02).astype(np.float32)
        th_d = dev_f32(th)
        low = torch.empty(numel, dtype=torch.bfloat16, device="cuda")
        sc = torch.tensor([0.5], device="cuda")
        g.ddp_bucket_sgd(dev_f32(gr), th_d, None, 0.1, 0.0, 1e-4, grad_scale=sc, param_bf16=low)
        sync()
        th_w, _ = oracle.sgd_from_grad(gr, th, None, 0.1, 0.0, 1e-4, scale=np.float32(0.5))
        assert_bit_exact(th_d, th_w, f"theta numel={numel}")
        np.testing.assert_array_equal(low.view(torch.int16).cpu().numpy().view(np.uint16), oracle.f32_to_bf16_rne(th_w))
