"""Pins for the oracle's DistributedSampler indices (CPU only)."""
import itertools
import math

import numpy as np

import oracle
import workloads


def test_splitmix64_known_answers():
    """Published SplitMix64 outputs for state 0 (the reference generator of
    Steele, Lea & Flood 2014, as used to seed xoshiro/xoroshiro)."""
    assert oracle.splitmix64_stream(0, 3) == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_fmix32_known_answers():
    """MurmurHash3_x86_32 of the empty key is fmix32(seed): the published
    outputs for seeds 1 and 0xFFFFFFFF are 0x514E28B7 and 0x81F16F39; 0 is a
    fixed point."""
    assert oracle.murmur3_fmix32(1) == 0x514E28B7
    assert oracle.murmur3_fmix32(0xFFFFFFFF) == 0x81F16F39
    assert oracle.murmur3_fmix32(0) == 0


def test_round_keys_are_high_halves():
    """Round keys: the high 32 bits of the SplitMix64 outputs from state 0
    (published values above)."""
    assert oracle.feistel_round_keys(0)[:3] == [0xE220A839, 0x6E789E6A, 0x06C45D18]


def test_vectorised_perm_matches_scalar_definition():
    """keyed_perm_all and keyed_perm (scalar Python ints) agree for a domain
    with unequal halves (21 bits) on a sample of indices."""
    n = 1_281_167
    p = oracle.keyed_perm_all(9, n)
    for j in list(range(50)) + list(range(n - 50, n)) + [123_457, 654_321]:
        assert p[j] == oracle.keyed_perm(j, 9, n)


def test_feistel_is_a_bijection_on_its_domain():
    """Every encryption pass permutes [0, 2^bits), bits = ceil(log2 n), for
    odd and even widths up to 12 bits and several keys (brute force), and the
    domain is below 2n."""
    for n in (2, 3, 5, 9, 17, 33, 100, 1000, 3000):
        bits = max(1, (n - 1).bit_length())
        assert (1 << bits) < 2 * n
        for key in (0, 1, 12345, 2 ** 63 + 7):
            img = sorted(oracle.feistel_encrypt(x, key, n) for x in range(1 << bits))
            assert img == list(range(1 << bits))


def check_perm_is_permutation(perm_all, perm_one):
    for n in list(range(0, 70)) + [1000, 4097]:
        for key in (0, 5, 2 ** 64 - 1):
            p = perm_all(key, n)
            assert sorted(p.tolist()) == list(range(n))
            if n <= 70:
                assert [perm_one(j, key, n) for j in range(n)] == p.tolist()


def test_perm_is_permutation():
    check_perm_is_permutation(oracle.keyed_perm_all, oracle.keyed_perm)


def test_perm_depends_on_key():
    a = oracle.keyed_perm_all(0, 1000)
    b = oracle.keyed_perm_all(1, 1000)
    assert not np.array_equal(a, b)


def check_partition_invariants(indices_fn):
    """AI_Infra notes "1.DataParallel / DDP" §4.4: every rank gets
    num_samples indices; without drop_last the ranks together hold every
    index, the total − n extra slots repeat the head of the shuffled list;
    with drop_last they hold total distinct indices; ranks are disjoint apart
    from the repeats; and rank r's list is the shuffled list taken from
    position r with stride N.  Brute force over small n and N."""
    for n, N, drop, shuf in itertools.product(range(0, 41), range(1, 17), (False, True), (False, True)):
        ns = n // N if drop else math.ceil(n / N)
        total = ns * N
        per = [indices_fn(n, N, r, 3, 2, shuf, drop) for r in range(N)]
        allr = indices_fn(n, N, -1, 3, 2, shuf, drop)
        assert allr.shape == (N, ns)
        for r in range(N):
            assert per[r].shape == (ns,)
            assert np.array_equal(per[r], allr[r])
        flat = np.empty(total, dtype=np.int64)       # interleave back into the padded list
        for r in range(N):
            flat[r::N] = per[r]
        if total == 0:
            continue
        assert flat.min() >= 0 and flat.max() < n
        if not drop:
            assert set(flat.tolist()) == set(range(n))
            assert np.array_equal(flat[n:], flat[:total - n] if total - n <= n else flat[np.arange(n, total) % n])
            assert len(set(flat[:n].tolist())) == n
        else:
            assert len(set(flat.tolist())) == total
        if not shuf:
            assert np.array_equal(flat[:min(n, total)], np.arange(min(n, total)))


def test_partition_invariants():
    check_partition_invariants(oracle.dist_sampler_indices)


def test_no_shuffle_matches_page_definition():
    """shuffle=False, drop_last=False: the page's own list operations
    (indices += indices[:total-len]; indices[rank:total:N]) on range(n)."""
    for n, N in [(10, 3), (10, 4), (7, 7), (5, 2), (1281, 8)]:
        ns = math.ceil(n / N)
        total = ns * N
        idx = list(range(n))
        idx += idx[:total - len(idx)]
        for r in range(N):
            assert oracle.dist_sampler_indices(n, N, r, 0, 0, False, False).tolist() == idx[r:total:N]


def test_imagenet_closed_form():
    """n = 1,281,167 over 8 ranks: 160,146 per rank, total 1,281,168, exactly
    one padded slot, at rank 7 / position 160,145, holding π(0)."""
    n, N = workloads.SAMPLER_N_ITEMS, workloads.SAMPLER_REPLICAS
    out = oracle.dist_sampler_indices(n, N, -1, 0, 1, True, False)
    assert out.shape == (8, 160_146)
    assert out[7, 160_145] == out[0, 0]
    flat = out.T.reshape(-1)
    assert np.array_equal(np.sort(flat[:n]), np.arange(n))
    dl = oracle.dist_sampler_indices(n, N, -1, 0, 1, True, True)
    assert dl.shape == (8, 160_145)
