"""Pins for the oracle's alternative summation orders (tree, ring) (CPU only).

Order is checked symbolically: the values are expression trees, so the test
sees exactly which additions the oracle performs and in which grouping.
"""
import numpy as np
import pytest

import oracle
from conftest import golden_rows


class Sym:
    """A symbolic value: a leaf name, a sum of two Syms, or a Sym / int."""

    def __init__(self, node):
        self.node = node

    def __add__(self, other):
        return Sym(("+", self.node, other.node))

    def __radd__(self, other):
        # the +0 start of an accumulator (np.zeros of an object array is int 0)
        assert other == 0
        return Sym(("+", "ZERO", self.node))

    def __truediv__(self, k):
        return Sym(("/", self.node, int(k)))

    def canon(self):
        return _canon(self.node)


def _canon(node):
    if isinstance(node, str):
        return node
    if node[0] == "+":
        a, b = _canon(node[1]), _canon(node[2])
        return ("+",) + tuple(sorted((a, b), key=repr))   # IEEE addition commutes
    return ("/", _canon(node[1]), node[2])


def _parse(expr):
    """Parse '((A00+A10)+A20)+A30' into the canonical tuple form."""
    pos = 0

    def atom():
        nonlocal pos
        if expr[pos] == "(":
            pos += 1
            v = add()
            assert expr[pos] == ")"
            pos += 1
            return v
        start = pos
        while pos < len(expr) and (expr[pos].isalnum() or expr[pos] == "_"):
            pos += 1
        return expr[start:pos]

    def add():
        nonlocal pos
        v = atom()
        while pos < len(expr) and expr[pos] == "+":
            pos += 1
            v = ("+", v, atom())
        return v

    return _canon(add())


def _sym_replicas(N, numel):
    """Replica i, element e -> leaf 'A{i}{chunk(e)}' when numel == N (one
    element per chunk), else 'g{i}_{e}'."""
    out = []
    for i in range(N):
        arr = np.empty(numel, dtype=object)
        for e in range(numel):
            arr[e] = Sym(f"A{i}{e}" if numel == N else f"g{i}_{e}")
        out.append(arr)
    return out


def check_ring_matches_page_tables(ring_fn):
    """The 4-GPU worked example of the AI_Infra notes "1.DataParallel / DDP"
    §2.11: chunk j's fully reduced value σ_j has the grouping the page's
    reduce-scatter tables show (fixture tests/golden/ring_4gpu_sigma.txt),
    and the all-gather divides nothing and adds nothing more."""
    reps = _sym_replicas(4, 4)
    out, bounds = ring_fn(reps, "obj")
    assert bounds == [(0, 1), (1, 2), (2, 3), (3, 4)]
    rows = golden_rows("ring_4gpu_sigma.txt")
    assert len(rows) == 4
    for chunk_s, _holder, expr in rows:
        j = int(chunk_s)
        assert out[j].canon() == ("/", _parse(expr), 4), (j, out[j].canon())


def test_ring_matches_page_tables():
    check_ring_matches_page_tables(oracle.ring_allreduce_mean)


def test_ring_chunking_ragged():
    """numel not divisible by N: chunk lengths differ by at most one, the
    longer chunks first, and together they tile [0, numel)."""
    for numel in (0, 1, 3, 10, 1290, 1291):
        for N in (1, 2, 3, 4, 8):
            reps = [np.zeros(numel, dtype=np.float32) for _ in range(N)]
            _, b = oracle.ring_allreduce_mean(reps, "f32")
            lens = [e - s for s, e in b]
            assert b[0][0] == 0 and b[-1][1] == numel
            assert all(b[i][1] == b[i + 1][0] for i in range(N - 1))
            assert max(lens) - min(lens) <= 1 and lens == sorted(lens, reverse=True)


def test_ring_order_differs_only_by_rounding():
    gen = np.random.Generator(np.random.PCG64(5))
    reps = [gen.standard_normal(4099).astype(np.float32) for _ in range(8)]
    ring, _ = oracle.ring_allreduce_mean(reps, "f32")
    exact = np.mean(np.stack(reps).astype(np.float64), axis=0)
    mag = np.sum(np.abs(np.stack(reps).astype(np.float64)), axis=0) / 8
    assert np.all(np.abs(ring - exact) <= 8 * 2.0 ** -24 * mag)


def check_tree_grouping(tree_fn):
    """Binary-tree order for N = 8: ((g0+g1)+(g2+g3))+((g4+g5)+(g6+g7)), / 8."""
    reps = _sym_replicas(8, 1)
    got = tree_fn(reps, "obj")[0].canon()
    want = ("/", _parse("((g0_0+g1_0)+(g2_0+g3_0))+((g4_0+g5_0)+(g6_0+g7_0))"), 8)
    assert got == want


def test_tree_grouping():
    check_tree_grouping(oracle.grad_mean_tree)


def test_tree_needs_power_of_two():
    with pytest.raises(ValueError):
        oracle.grad_mean_tree([np.zeros(3, np.float32)] * 3)


def test_rank_order_grouping():
    """The rank-ordered average is ((((+0)+g0)+g1)+...)+g_{N-1}, / N
    (Tech-Renaissance "(24) NCCL通信与分布式数据并行" §一: the sum starts from
    zeros_like and adds grad[r] for r = 0..N-1)."""
    got = oracle.grad_mean(_sym_replicas(4, 1), "obj")[0].canon()
    assert got == ("/", _parse("(((ZERO+g0_0)+g1_0)+g2_0)+g3_0"), 4)
