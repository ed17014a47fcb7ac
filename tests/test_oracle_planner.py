"""Pins for the oracle's bucket planner (CPU only)."""
import numpy as np
import pytest

import oracle
import workloads

MiB = 1 << 20


def check_plan_invariants(plan_fn, numels, elem_bytes, cap_bytes, mode=oracle.PLAN_CAP, is_first=None,
                          align_bytes=256):
    """Properties that pin the greedy reverse-order reading without reusing it:
    - every tensor sits in exactly one bucket, buckets are non-empty;
    - concatenating buckets lists tensors last-registered first (CAP), or
      DEEP then FIRST each in reverse order (DEEP_FIRST);
    - inside a bucket tensors are packed back to back; bucket bases are
      aligned and buckets do not overlap;
    - CAP: a bucket exceeds the cap only if it holds one tensor, and every
      closed bucket was closed because the next tensor would overflow it
      (greedy maximality), which determines the partition uniquely."""
    p = plan_fn(numels, elem_bytes, cap_bytes, mode, is_first, align_bytes)
    T = len(numels)
    order, buckets = p["order"], p["buckets"]
    assert sorted(order) == list(range(T))
    align = align_bytes // elem_bytes
    if mode == oracle.PLAN_CAP:
        assert order == list(reversed(range(T)))
    else:
        deep = [t for t in reversed(range(T)) if not is_first[t]]
        first = [t for t in reversed(range(T)) if is_first[t]]
        assert order == deep + first
        assert len(buckets) == (1 if deep else 0) + (1 if first else 0)
    end_prev = 0
    for bi, (off, numel, f, c) in enumerate(buckets):
        assert c >= 1
        assert off % align == 0 and off >= end_prev
        assert off - end_prev < align
        members = order[f:f + c]
        pos = off
        for t in members:
            assert p["tensor_offset"][t] == pos and p["tensor_bucket"][t] == bi
            pos += numels[t]
        assert numel == pos - off
        end_prev = off + numel
        if mode == oracle.PLAN_CAP:
            nbytes = numel * elem_bytes
            if c > 1:
                assert nbytes <= cap_bytes
            if bi + 1 < len(buckets):
                nxt = order[f + c]
                assert nbytes + numels[nxt] * elem_bytes > cap_bytes
    assert p["total_elems"] == (-(-end_prev // align) * align if buckets else 0)
    return p


def test_resnet50_closed_forms():
    """ResNet-50 (161 tensors, 25,557,032 parameters).  At a 100 MiB cap the
    whole model (97.5 MiB of fp32) is one bucket; at 25 MiB the greedy fill
    gives 5 buckets (every bucket must hold < 25 MiB and 97.5 MiB needs at
    least 4); at 1 MiB the conv weights larger than 1 MiB stand alone."""
    num = workloads.numels(workloads.resnet50_layout())
    assert len(num) == 161 and sum(num) == 25_557_032
    p100 = check_plan_invariants(oracle.plan_buckets, num, 4, 100 * MiB)
    assert len(p100["buckets"]) == 1
    p25 = check_plan_invariants(oracle.plan_buckets, num, 4, 25 * MiB)
    assert len(p25["buckets"]) == 5
    assert sum(b[1] for b in p25["buckets"]) == 25_557_032
    p1 = check_plan_invariants(oracle.plan_buckets, num, 4, 1 * MiB)
    big = sum(1 for n in num if n * 4 > MiB)
    assert len(p1["buckets"]) >= big
    # first bucket starts with the last-registered tensor (fc.bias, 1000 elems)
    assert p25["order"][0] == 160 and p25["tensor_offset"][160] == 0


def test_gpt2_deep_first_closed_forms():
    """GPT-2 small, two buckets as in Tech-Renaissance "(24) NCCL通信与分布式
    数据并行" §八: DEEP = 85,017,600 attention/MLP parameters, FIRST =
    39,422,208 (LayerNorms 38,400 + wte 38,597,376 + wpe 786,432), total
    124,439,808."""
    layout, first = workloads.gpt2_small_layout()
    num = workloads.numels(layout)
    assert len(num) == 148 and sum(num) == 124_439_808
    p = check_plan_invariants(oracle.plan_buckets, num, 2, 0, oracle.PLAN_DEEP_FIRST, first)
    (o0, n0, _, c0), (o1, n1, _, c1) = p["buckets"]
    assert (n0, n1) == (85_017_600, 39_422_208)
    assert (c0, c1) == (12 * 8, 12 * 4 + 2 + 2)
    assert o0 == 0 and o1 == 85_017_600           # 85,017,600*2 B is already 256-aligned
    assert 38_597_376 + 786_432 + 12 * 4 * 768 + 2 * 768 == n1


def test_random_layouts_brute_force():
    gen = np.random.Generator(np.random.PCG64(99))
    for trial in range(300):
        T = int(gen.integers(1, 40))
        num = [int(x) for x in gen.integers(0, 5000, T)]
        eb = int(gen.choice([2, 4]))
        cap = int(gen.integers(1, 40000))
        al = int(gen.choice([16, 64, 256]))
        check_plan_invariants(oracle.plan_buckets, num, eb, cap, oracle.PLAN_CAP, None, al)
        isf = [bool(x) for x in gen.integers(0, 2, T)]
        check_plan_invariants(oracle.plan_buckets, num, eb, cap, oracle.PLAN_DEEP_FIRST, isf, al)


def test_tiny_cases():
    p = oracle.plan_buckets([], 4, 100)
    assert p["buckets"] == [] and p["total_elems"] == 0
    p = oracle.plan_buckets([5], 4, 1)                 # larger than the cap: alone
    assert p["buckets"] == [(0, 5, 0, 1)] and p["total_elems"] == 64
    p = oracle.plan_buckets([3, 0, 4], 4, 16)          # 16 B cap: 4 elems fit, then 3
    assert [b[1] for b in p["buckets"]] == [4, 3]
    assert p["tensor_offset"] == [64, 4, 0]
    p = oracle.plan_buckets([4, 4], 4, 32)             # exactly the cap: one bucket
    assert [b[1] for b in p["buckets"]] == [8]
    with pytest.raises(ValueError):
        oracle.plan_buckets([1], 4, 10, align_bytes=6)
