"""Seeded synthetic inputs shared by the tests, the benchmark and the smoke check.

This module describes *inputs only*: parameter layouts of textbook architectures
(tensor shapes in registration order) and seeded random draws of replica
gradients, parameters and activations.  It holds none of the arithmetic of the
method being tested (no averaging, no optimizer step, no normalisation, no
permutation), so the CPU oracle and the CUDA path can both be fed from it
without sharing any computation.

Seeds follow one rule everywhere: replica ``r`` of workload number ``k`` draws
from ``numpy.random.PCG64(1234 + 100*k + r)``.  Workload numbers:

    1  Linear(128, 10) gradients, 4 replicas            (1290 fp32 elements)
    2  ResNet-50 parameter layout, 8 replicas            (161 tensors, 25,557,032 elements)
    3  GPT-2 small parameter layout, 8 replicas, bf16    (148 tensors, 124,439,808 elements)
    4  SyncBatchNorm activations, 8 replicas x [32,C,H,W] bf16
    5  flat fp32 sweep buffers and DistributedSampler index requests
"""
from __future__ import annotations

import numpy as np

# ---------------------------------------------------------------------------
# parameter layouts (name, shape) in registration order
# ---------------------------------------------------------------------------


def linear_128_10_layout():
    """nn.Linear(128, 10): weight [10, 128] row-major, then bias [10]."""
    return [("weight", (10, 128)), ("bias", (10,))]


def resnet50_layout():
    """torchvision-style ResNet-50 parameters in registration order.

    conv1, bn1, then four stages of bottleneck blocks (3, 4, 6, 3 blocks with
    64, 128, 256, 512 planes, expansion 4; the first block of each stage has a
    1x1 projection "downsample" conv + BN), then fc 2048 -> 1000.  No conv has
    a bias.  161 tensors, 25,557,032 elements.
    """
    out = [("conv1.weight", (64, 3, 7, 7)), ("bn1.weight", (64,)), ("bn1.bias", (64,))]
    inplanes = 64
    for li, (planes, blocks) in enumerate([(64, 3), (128, 4), (256, 6), (512, 3)], start=1):
        for bi in range(blocks):
            p = f"layer{li}.{bi}."
            out += [
                (p + "conv1.weight", (planes, inplanes, 1, 1)),
                (p + "bn1.weight", (planes,)), (p + "bn1.bias", (planes,)),
                (p + "conv2.weight", (planes, planes, 3, 3)),
                (p + "bn2.weight", (planes,)), (p + "bn2.bias", (planes,)),
                (p + "conv3.weight", (planes * 4, planes, 1, 1)),
                (p + "bn3.weight", (planes * 4,)), (p + "bn3.bias", (planes * 4,)),
            ]
            if bi == 0:
                out += [
                    (p + "downsample.0.weight", (planes * 4, inplanes, 1, 1)),
                    (p + "downsample.1.weight", (planes * 4,)),
                    (p + "downsample.1.bias", (planes * 4,)),
                ]
            inplanes = planes * 4
    out += [("fc.weight", (1000, 2048)), ("fc.bias", (1000,))]
    return out


def gpt2_small_layout():
    """GPT-2 small (12 layers, d=768, 12 heads, vocab 50257, context 1024, tied head).

    Returns (layout, is_first).  ``is_first`` marks the tensors that go to the
    FIRST bucket of the two-bucket split: the Tech-Renaissance article
    "(24) NCCL通信与分布式数据并行" §八 puts the BN, FC and first-conv gradient
    regions in FIRST_COMM and the deep-conv region in DEEP_COMM.  For a
    transformer the corresponding reading is: LayerNorm weights/biases (the
    normalisation parameters), the tied token embedding / output head wte (the
    FC), and the position embedding wpe (the input-side layer) are FIRST;
    every attention and MLP weight and bias is DEEP.  148 tensors,
    124,439,808 elements: FIRST 39,422,208, DEEP 85,017,600.
    """
    d, v, ctx, L = 768, 50257, 1024, 12
    layout = [("wte.weight", (v, d)), ("wpe.weight", (ctx, d))]
    first = [True, True]
    for i in range(L):
        p = f"h.{i}."
        blk = [
            (p + "ln_1.weight", (d,), True), (p + "ln_1.bias", (d,), True),
            (p + "attn.c_attn.weight", (d, 3 * d), False), (p + "attn.c_attn.bias", (3 * d,), False),
            (p + "attn.c_proj.weight", (d, d), False), (p + "attn.c_proj.bias", (d,), False),
            (p + "ln_2.weight", (d,), True), (p + "ln_2.bias", (d,), True),
            (p + "mlp.c_fc.weight", (d, 4 * d), False), (p + "mlp.c_fc.bias", (4 * d,), False),
            (p + "mlp.c_proj.weight", (4 * d, d), False), (p + "mlp.c_proj.bias", (d,), False),
        ]
        for name, shape, f in blk:
            layout.append((name, shape))
            first.append(f)
    layout += [("ln_f.weight", (d,)), ("ln_f.bias", (d,))]
    first += [True, True]
    return layout, first


def numels(layout):
    """Element count of each tensor of a layout, as a list of Python ints."""
    out = []
    for _, shape in layout:
        n = 1
        for s in shape:
            n *= int(s)
        out.append(n)
    return out


# SyncBatchNorm activation shapes (C, H, W) with local batch 32.
SYNCBN_SHAPES = [(64, 56, 56), (256, 56, 56), (512, 28, 28), (2048, 7, 7)]
SYNCBN_BATCH = 32

# DistributedSampler request of workload 5: the ImageNet-1k training-set size
# (only the count is used), 8 ranks.
SAMPLER_N_ITEMS = 1_281_167
SAMPLER_REPLICAS = 8

# Flat sweep sizes (bytes) and caps (MiB) of workload 5.
SWEEP_BYTES = [1024 * 4 ** k for k in range(11)]  # 1 KiB .. 1 GiB
SWEEP_REPLICAS = [2, 4, 8, 16]
SWEEP_CAPS_MIB = [1, 25, 100]

# ---------------------------------------------------------------------------
# seeded draws (host, numpy PCG64)
# ---------------------------------------------------------------------------


def seed_for(workload: int, replica: int) -> int:
    return 1234 + 100 * int(workload) + int(replica)


def rng(workload: int, replica: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed_for(workload, replica)))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to the nearest bf16 (ties to even) and return the raw
    16-bit patterns as uint16.  Used only to *make* bf16 inputs; NaN inputs are
    not produced by any generator here."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    u = u + np.uint64(0x7FFF) + lsb
    return (u >> np.uint64(16)).astype(np.uint16)


def normal_f32(gen: np.random.Generator, n: int, mean: float, std: float) -> np.ndarray:
    return (gen.standard_normal(n, dtype=np.float32) * np.float32(std) + np.float32(mean)).astype(np.float32)


def replica_grads(workload: int, n_replicas: int, numel: int, std: float, dtype: str = "f32", mean: float = 0.0):
    """One flat gradient buffer per replica, N(mean, std) drawn per replica.

    dtype "f32" -> float32 arrays; "bf16" -> uint16 arrays holding bf16 bit
    patterns (the fp32 draw rounded to nearest even)."""
    out = []
    for r in range(n_replicas):
        x = normal_f32(rng(workload, r), numel, mean, std)
        out.append(x if dtype == "f32" else f32_to_bf16_bits(x))
    return out


def params_f32(workload: int, numel: int, std: float) -> np.ndarray:
    """Parameter vector theta for an optimizer step; drawn from stream 99 of the workload."""
    return normal_f32(rng(workload, 99), numel, 0.0, std)


def syncbn_input(workload: int, n_replicas: int, batch: int, C: int, H: int, W: int,
                 mean: float = 0.5, std: float = 2.0):
    """Per-replica bf16 activations [batch, C, H, W] (NCHW), as uint16 bit patterns."""
    n = batch * C * H * W
    return [f32_to_bf16_bits(normal_f32(rng(workload, r), n, mean, std)).reshape(batch, C, H, W)
            for r in range(n_replicas)]


def adversarial_f32(gen: np.random.Generator, n: int) -> np.ndarray:
    """fp32 values that stress rounding: mixed magnitudes, subnormals, signed
    zeros, exact ties, infinities and NaNs."""
    kind = gen.integers(0, 8, n)
    x = normal_f32(gen, n, 0.0, 1.0)
    x = np.where(kind == 1, x * np.float32(1e30), x)
    x = np.where(kind == 2, x * np.float32(1e-40), x)            # subnormal range
    x = np.where(kind == 3, np.float32(-0.0), x)
    x = np.where(kind == 4, np.float32(2.0 ** 24) + np.float32(1.0), x)
    x = np.where(kind == 5, np.ldexp(np.float32(1.0), gen.integers(-149, 127, n)).astype(np.float32), x)
    sp = gen.random(n)
    x = np.where(sp < 0.002, np.float32(np.inf), x)
    x = np.where((sp >= 0.002) & (sp < 0.004), np.float32(-np.inf), x)
    x = np.where((sp >= 0.004) & (sp < 0.006), np.float32(np.nan), x)
    return x.astype(np.float32)


# ---------------------------------------------------------------------------
# seeded draws on the device (large perf runs); torch is imported lazily
# ---------------------------------------------------------------------------


def device_normal(shape, mean: float, std: float, seed: int, device="cuda", dtype=None):
    """torch.randn on the device from a seeded generator (fp32), then cast to
    ``dtype`` (torch's own round-to-nearest for bf16)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    x.mul_(std).add_(mean)
    if dtype is not None and dtype != torch.float32:
        x = x.to(dtype)
    return x
