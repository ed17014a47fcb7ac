"""GPU parity: dist_sampler_indices against the oracle, exactly."""
import itertools

import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_common import load_library, sync

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    return load_library()


def _gpu(g, n, N, rank, seed, epoch, shuffle, drop):
    ns = g.dist_sampler_num_samples(n, N, drop)
    cnt = ns if rank >= 0 else ns * N
    out = torch.full((max(cnt, 1),), -7, dtype=torch.int64, device="cuda")
    status = torch.full((1,), 99, dtype=torch.int32, device="cuda")
    got_ns = g.dist_sampler_indices(n, N, rank, seed, epoch, shuffle, drop, out[:cnt] if cnt else None,
                                    walk_status=status)
    sync()
    assert got_ns == ns
    assert status.item() == 0
    res = out[:cnt].cpu().numpy()
    return res if rank >= 0 else res.reshape(N, ns)


def test_small_brute_force(g):
    for n, N, drop, shuf in itertools.product(list(range(0, 34)) + [100, 257], (1, 2, 3, 5, 8, 16),
                                              (False, True), (False, True)):
        for seed, epoch in ((0, 0), (7, 3)):
            want = oracle.dist_sampler_indices(n, N, -1, seed, epoch, shuf, drop)
            np.testing.assert_array_equal(_gpu(g, n, N, -1, seed, epoch, shuf, drop), want.reshape(N, -1))
            r = (n + seed) % N
            np.testing.assert_array_equal(_gpu(g, n, N, r, seed, epoch, shuf, drop),
                                          oracle.dist_sampler_indices(n, N, r, seed, epoch, shuf, drop))


@pytest.mark.parametrize("epoch", [0, 1])
@pytest.mark.parametrize("drop", [False, True])
def test_imagenet_all_ranks(g, epoch, drop):
    """n = 1,281,167 items, N = 8, all ranks, seed 0: every index exact."""
    n, N = workloads.SAMPLER_N_ITEMS, workloads.SAMPLER_REPLICAS
    got = _gpu(g, n, N, -1, 0, epoch, True, drop)
    want = oracle.dist_sampler_indices(n, N, -1, 0, epoch, True, drop)
    np.testing.assert_array_equal(got, want)


def test_large_n_one_rank(g):
    """n above 2^31 (64-bit positions, 32-bit Feistel halves): a rank's list
    is short when N is large; every index checked with the scalar oracle."""
    n, N = (1 << 31) + 11, 1 << 20
    for rank in (0, 5, N - 1):
        got = _gpu(g, n, N, rank, 123, 4, True, False)
        key = 123 + 4
        pos = rank + np.arange(got.size, dtype=np.int64) * N
        want = [oracle.keyed_perm(int(p % n), key, n) for p in pos]
        np.testing.assert_array_equal(got, np.array(want, dtype=np.int64))


def test_seed_epoch_wraparound(g):
    """seed + epoch is taken mod 2^64."""
    a = _gpu(g, 1000, 4, -1, 2 ** 64 - 1, 1, True, False)
    b = _gpu(g, 1000, 4, -1, 0, 0, True, False)
    np.testing.assert_array_equal(a, b)


def test_resume_from_offset(g):
    """dist_sampler_indices_from: entry k is list position start + k of the
    full lists, for one rank and for all ranks (rank-major), every offset
    from 0 to num_samples."""
    for n, N in ((1_281_167, 8), (100_003, 3), (10, 4), (5, 8), (1, 1)):
        for shuffle in (True, False):
            full = oracle.dist_sampler_indices(n, N, -1, 9, 4, shuffle, False)
            ns = full.shape[1]
            for start in sorted({0, 1, ns // 2, max(ns - 1, 0), ns} & set(range(ns + 1))):
                for rank in (-1, 0, N - 1):
                    cnt = (ns - start) * (N if rank < 0 else 1)
                    out = torch.full((max(cnt, 1),), -7, dtype=torch.int64, device="cuda")
                    got_ns = g.dist_sampler_indices_from(n, N, rank, 9, 4, shuffle, False, start,
                                                         out[:cnt] if cnt else None)
                    sync()
                    assert got_ns == ns
                    want = full[:, start:] if rank < 0 else full[rank, start:]
                    np.testing.assert_array_equal(out[:cnt].cpu().numpy(), want.reshape(-1),
                                                  f"n={n} N={N} rank={rank} start={start} shuffle={shuffle}")
