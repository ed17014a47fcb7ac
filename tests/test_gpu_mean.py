"""GPU parity: ddp_bucket_allreduce_mean against the oracle, bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_common import assert_bit_exact, dev_bf16, dev_f32, load_library, sync

pytestmark = pytest.mark.gpu

MiB = 1 << 20


@pytest.fixture(scope="module")
def g():
    return load_library()


def _replicas(n, numel, dtype, seed, std=1.0):
    gen = np.random.Generator(np.random.PCG64(seed))
    out = []
    for _ in range(n):
        x = (gen.standard_normal(numel, dtype=np.float32) * np.float32(std)).astype(np.float32)
        out.append(x if dtype == "f32" else workloads.f32_to_bf16_bits(x))
    return out


def _dev(reps, dtype):
    return [dev_f32(r) if dtype == "f32" else dev_bf16(r) for r in reps]


def _run(g, reps_dev, numel, flags=0, out=None):
    if out is None:
        out = torch.full((max(numel, 1),), float("nan"), device="cuda")
    g.ddp_bucket_allreduce_mean(reps_dev, out, flags=flags, numel=numel)
    sync()
    return out[:numel]


def test_linear_128_10_four_replicas(g):
    """Linear(128, 10) gradient layout (1290 fp32 elements), N = 4 replicas of N(0, 1)."""
    numel = sum(workloads.numels(workloads.linear_128_10_layout()))
    reps = workloads.replica_grads(1, 4, numel, 1.0)
    assert_bit_exact(_run(g, _dev(reps, "f32"), numel), oracle.grad_mean(reps), "linear 128x10")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_sizes_and_replica_counts(g, dtype):
    """Ragged sizes (tails of every length, sub-vector buckets, several grid
    strides) and every replica count class, power of two or not."""
    sizes = [0, 1, 3, 4, 5, 7, 8, 9, 31, 1023, 1290, 4097, 65539, (1 << 20) + 5, 3 * 1216 * 256 * 8 + 13]
    for n in (1, 2, 3, 4, 5, 7, 8, 9, 12, 16):
        for i, numel in enumerate(sizes):
            reps = _replicas(n, numel, dtype, 1000 * n + i)
            got = _run(g, _dev(reps, dtype), numel)
            assert_bit_exact(got, oracle.grad_mean(reps, dtype), f"{dtype} N={n} numel={numel}")


def test_adversarial_values(g):
    """Infinities, NaNs, signed zeros, subnormals, ties at 2^24, huge values."""
    for n in (2, 3, 8, 16):
        gen = np.random.Generator(np.random.PCG64(77 + n))
        reps = [workloads.adversarial_f32(gen, 50_003) for _ in range(n)]
        with np.errstate(all="ignore"):
            want = oracle.grad_mean(reps)
        assert_bit_exact(_run(g, _dev(reps, "f32"), 50_003), want, f"adversarial N={n}")
        bits = [gen.integers(0, 1 << 16, 20_011).astype(np.uint16) for _ in range(n)]
        with np.errstate(all="ignore"):
            want = oracle.grad_mean(bits, "bf16")
        assert_bit_exact(_run(g, _dev(bits, "bf16"), 20_011), want, f"bf16 all patterns N={n}")


def test_golden_cases_on_gpu(g):
    """The hand-derived binary32 cases of tests/golden/mean_rank_order.txt."""
    from conftest import golden_rows
    for n_s, vals_s, exp_s, why in golden_rows("mean_rank_order.txt"):
        vals = [float(t) if t in ("inf", "-inf", "nan") else float.fromhex(t) for t in vals_s.split()]
        exp = float(exp_s) if exp_s in ("inf", "-inf", "nan") else float.fromhex(exp_s)
        reps = [np.full(13, v, dtype=np.float32) for v in vals]
        assert_bit_exact(_run(g, _dev(reps, "f32"), 13), np.full(13, exp, np.float32), why)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_tree_order(g, dtype):
    for n in (1, 2, 4, 8, 16):
        for numel in (1, 7, 4099, 300_001):
            reps = _replicas(n, numel, dtype, 5000 + n + numel)
            got = _run(g, _dev(reps, dtype), numel, flags=g.FLAG_TREE_ORDER)
            assert_bit_exact(got, oracle.grad_mean_tree(reps, dtype), f"tree {dtype} N={n} numel={numel}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_ring_order(g, dtype):
    for n in (1, 2, 3, 4, 5, 8, 13, 16):
        for numel in (1, 2, 3, 7, 17, 1290, 4099, 300_001):
            reps = _replicas(n, numel, dtype, 7000 + n + numel)
            got = _run(g, _dev(reps, dtype), numel, flags=g.FLAG_RING_ORDER)
            want, _ = oracle.ring_allreduce_mean(reps, dtype)
            assert_bit_exact(got, want, f"ring {dtype} N={n} numel={numel}")


def test_write_back_and_in_place(g):
    for flags in (0, g.FLAG_RING_ORDER, g.FLAG_TREE_ORDER):
        n, numel = 4, 100_003
        reps = _replicas(n, numel, "f32", 31 + flags)
        want = (oracle.grad_mean_tree(reps) if flags == g.FLAG_TREE_ORDER else
                oracle.ring_allreduce_mean(reps)[0] if flags == g.FLAG_RING_ORDER else oracle.grad_mean(reps))
        # in place into replica 0 (ncclAllReduce-style)
        d = _dev(reps, "f32")
        g.ddp_bucket_allreduce_mean(d, d[0], flags=flags)
        sync()
        assert_bit_exact(d[0], want, "in place")
        # write back into every replica, out separate
        d = _dev(reps, "f32")
        out = torch.empty(numel, device="cuda")
        g.ddp_bucket_allreduce_mean(d, out, flags=flags | g.FLAG_WRITE_BACK_ALL)
        sync()
        assert_bit_exact(out, want, "write-back out")
        for r in range(n):
            assert_bit_exact(d[r], want, f"write-back replica {r}")
        # write back with out == replica 2
        d = _dev(reps, "f32")
        g.ddp_bucket_allreduce_mean(d, d[2], flags=flags | g.FLAG_WRITE_BACK_ALL)
        sync()
        for r in range(n):
            assert_bit_exact(d[r], want, f"write-back aliased replica {r}")


def _resnet_buffers(g, n=8):
    num = workloads.numels(workloads.resnet50_layout())
    plan = g.ddp_plan_buckets(num, 4, 25 * MiB)
    total = plan["total_elems"]
    reps = workloads.replica_grads(2, n, total, 0.01)
    return plan, reps


def test_resnet50_buckets_full_size(g):
    """ResNet-50 layout (25,557,032 fp32 elements), N = 8, N(0, 0.01), 25 MiB
    buckets: every bucket averaged bit-exactly, padding between buckets left
    untouched."""
    plan, reps = _resnet_buffers(g)
    total = plan["total_elems"]
    d = _dev(reps, "f32")
    out = torch.full((total,), float("nan"), device="cuda")
    for off, numel, _, _ in plan["buckets"]:
        g.ddp_bucket_allreduce_mean([x[off:off + numel] for x in d], out[off:off + numel])
    sync()
    got = out.cpu().numpy()
    for off, numel, _, _ in plan["buckets"]:
        assert_bit_exact(torch.from_numpy(got[off:off + numel]),
                         oracle.grad_mean([r[off:off + numel] for r in reps]), f"bucket at {off}")
    covered = np.zeros(total, bool)
    for off, numel, _, _ in plan["buckets"]:
        covered[off:off + numel] = True
    assert np.isnan(got[~covered]).all()


def test_cuda_graph_capture_of_bucket_launches(g):
    """The per-bucket launches captured once on a side stream into a CUDA
    Graph and replayed give the same bits as the oracle."""
    plan, reps = _resnet_buffers(g, n=4)
    total = plan["total_elems"]
    d = _dev(reps, "f32")
    out = torch.zeros(total, device="cuda")
    side = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for off, numel, _, _ in plan["buckets"]:      # warm-up outside capture
            g.ddp_bucket_allreduce_mean([x[off:off + numel] for x in d], out[off:off + numel])
    torch.cuda.current_stream().wait_stream(side)
    sync()
    out.zero_()
    with torch.cuda.graph(graph, stream=side):
        for off, numel, _, _ in plan["buckets"]:
            g.ddp_bucket_allreduce_mean([x[off:off + numel] for x in d], out[off:off + numel])
    for _ in range(3):
        graph.replay()
    sync()
    got = out.cpu().numpy()
    for off, numel, _, _ in plan["buckets"]:
        assert_bit_exact(torch.from_numpy(got[off:off + numel]),
                         oracle.grad_mean([r[off:off + numel] for r in reps]), f"graph bucket {off}")


def test_sweep_chunked_flat_buffers(g):
    """Flat fp32 buffers split into cap-sized bucket launches (1 and 25 MiB),
    N in {2, 16}, checked whole."""
    for size_bytes in (1024, 64 * 1024, 4 * MiB, 64 * MiB):
        numel = size_bytes // 4
        for n in (2, 16):
            reps = _replicas(n, numel, "f32", size_bytes + n)
            d = _dev(reps, "f32")
            want = oracle.grad_mean(reps)
            for cap in (1 * MiB, 25 * MiB):
                ce = cap // 4
                out = torch.full((numel,), float("nan"), device="cuda")
                for s in range(0, numel, ce):
                    e = min(numel, s + ce)
                    g.ddp_bucket_allreduce_mean([x[s:e] for x in d], out[s:e])
                sync()
                assert_bit_exact(out, want, f"sweep {size_bytes}B N={n} cap={cap}")


def test_sweep_full_size_sampled(g):
    """Flat fp32 buffers of 1 GiB (268,435,456 elements), N in {2, 16}, split
    into cap-sized bucket launches (1, 25, 100 MiB) as the benchmark sweep
    launches them; inputs drawn on the device from seeded generators, 2^20
    sampled outputs plus both ends of every bucket recomputed by the oracle."""
    numel = (1 << 30) // 4
    gen = np.random.Generator(np.random.PCG64(51))
    for n in (2, 16):
        reps = [workloads.device_normal((numel,), 0.0, 1.0, workloads.seed_for(5, r) + 17 * n) for r in range(n)]
        for cap in (1 * MiB, 25 * MiB, 100 * MiB):
            ce = cap // 4
            out = torch.empty(numel, device="cuda")
            starts = list(range(0, numel, ce))
            for s in starts:
                e = min(numel, s + ce)
                g.ddp_bucket_allreduce_mean([x[s:e] for x in reps], out[s:e])
            idx = [gen.integers(0, numel, 1 << 20)]
            for s in starts[:: max(1, len(starts) // 64)]:
                idx += [np.arange(s, min(numel, s + 8)), np.arange(max(0, s - 8), s)]
            idx = np.unique(np.concatenate(idx))
            idx_d = torch.from_numpy(idx).cuda()
            sync()
            want = oracle.grad_mean([x[idx_d].cpu().numpy() for x in reps])
            assert_bit_exact(out[idx_d], want, f"sweep 1 GiB N={n} cap={cap >> 20} MiB")
        del reps


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_multi_bucket_launch_matches_per_bucket(g, dtype):
    """ddp_bucket_allreduce_mean_multi gives, in one launch, the bits of one
    call per bucket: ResNet-50 planned at a 1 MiB cap (66 buckets), ragged and
    tiny buckets, empty buckets, and replica counts of every class."""
    num = workloads.numels(workloads.resnet50_layout())
    elem = 4 if dtype == "f32" else 2
    layouts = [g.ddp_plan_buckets(num, elem, 1 * MiB)]
    custom = [(0, 5), (64, 0), (64, 1), (128, 4093), (4224, 3), (4352, 130_000)]
    layouts.append({"buckets": [(o, m, 0, 0) for o, m in custom], "total_elems": 4352 + 130_000})
    for li, plan in enumerate(layouts):
        total = plan["total_elems"]
        for n in (1, 3, 8, 16):
            reps = _replicas(n, total, dtype, 900 + 10 * n + li)
            d = _dev(reps, dtype)
            out = torch.full((total,), float("nan"), device="cuda")
            g.ddp_bucket_allreduce_mean_multi(d, plan["buckets"], out)
            sync()
            got = out.cpu()
            for off, m, _, _ in plan["buckets"]:
                if m:
                    assert_bit_exact(got[off:off + m], oracle.grad_mean([r[off:off + m] for r in reps], dtype),
                                     f"layout {li} N={n} bucket@{off}")
            covered = np.zeros(total, bool)
            for off, m, _, _ in plan["buckets"]:
                covered[off:off + m] = True
            assert np.isnan(got.numpy()[~covered]).all()


def test_multi_bucket_sweep_full_size_sampled(g):
    """1 GiB flat buffer at a 1 MiB cap: 1024 buckets in one launch, N = 8."""
    numel = (1 << 30) // 4
    ce = MiB // 4
    buckets = [(s, min(ce, numel - s), 0, 0) for s in range(0, numel, ce)]
    assert len(buckets) == 1024
    reps = [workloads.device_normal((numel,), 0.0, 1.0, workloads.seed_for(5, r) + 3) for r in range(8)]
    out = torch.empty(numel, device="cuda")
    g.ddp_bucket_allreduce_mean_multi(reps, buckets, out)
    gen = np.random.Generator(np.random.PCG64(52))
    idx = np.unique(np.concatenate([gen.integers(0, numel, 1 << 20), np.arange(0, numel, ce), np.arange(ce - 1, numel, ce)]))
    idx_d = torch.from_numpy(idx).cuda()
    sync()
    assert_bit_exact(out[idx_d], oracle.grad_mean([x[idx_d].cpu().numpy() for x in reps]), "multi 1 GiB")
