"""CPU oracle for the DDP gradient-synchronisation hot path.

TEST INFRASTRUCTURE ONLY.  This module is the plain, slow, obviously-correct
definition that the CUDA path is checked against.  Only the test suite, the
smoke check and the benchmark's CPU-baseline leg may import it; the product
library never calls it and has no CPU fallback.  It shares no code, table or
constant generator with the CUDA sources.

Sources (web pages; section numbers are the pages' own):
  [TR24]  Tech-Renaissance, "(24) NCCL通信与分布式数据并行"
  [TR16]  Tech-Renaissance, "(16) DTensor"
  [DDP]   AI_Infra notes, "1.DataParallel / DDP" (sgdbs.github.io)
Each function names the section it follows.  Where the pages are silent the
reading taken is stated in the docstring.

Precision: the gradient average, the 1/N scale and the SGD step are fp32 as on
the pages ([TR24] §一 says the local gradients are FP32; [TR24] §九 scales with
a float reciprocal).  Every fp32 operation below is a separate numpy ufunc on
float32 arrays, i.e. one IEEE round-to-nearest-even per operation, no fused
multiply-add.  SyncBatchNorm statistics, which no page fixes, are fp64.

Parity pins: every function here is pinned by tests/test_oracle_*.py against
facts that do not come from this file (worked examples, closed forms,
invariants, brute force, independent library routines).
"""
from __future__ import annotations

import math

import numpy as np

# ---------------------------------------------------------------------------
# bf16 <-> fp32
# ---------------------------------------------------------------------------


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to fp32: the bf16 pattern
    is the top half of the fp32 pattern.  This is the "AMP grad cast" that the
    n_cdg / n_cfg graphs of [TR24] §十一 perform before the all-reduce."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def f64_to_bf16_rne(x: np.ndarray) -> np.ndarray:
    """Round fp64 values to bf16 (nearest, ties to even) directly from the
    fp64 value, returned as fp64 holding the bf16 value.  Used to state the
    expected bf16 outputs of SyncBatchNorm; finite inputs only."""
    x = np.asarray(x, dtype=np.float64)
    out = np.zeros_like(x)
    nz = x != 0
    m, e = np.frexp(x[nz])          # x = m * 2**e, 0.5 <= |m| < 1
    # bf16 has 8 significant bits: scale the mantissa to [128, 256)
    sig = m * 256.0
    r = np.round(sig)               # numpy rounds half to even
    out[nz] = np.ldexp(r, e - 8)
    return out


def _as_f32(g: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return np.ascontiguousarray(g, dtype=np.float32)
    if dtype == "bf16":
        return bf16_bits_to_f32(g)
    if dtype == "f64":
        return np.ascontiguousarray(g, dtype=np.float64)
    if dtype == "obj":              # symbolic values (object arrays), for order checks
        return np.asarray(g, dtype=object)
    raise ValueError(dtype)

# ---------------------------------------------------------------------------
# gradient averaging  ([TR24] §一, §九; [DDP] §4.2)
# ---------------------------------------------------------------------------


def grad_mean(grads, dtype: str = "f32") -> np.ndarray:
    """grad_sync = zeros; for r in 0..N-1: grad_sync += grad[r]; grad_sync /= N.

    [TR24] §一 gives exactly this loop; [DDP] §4.2 sums with an all-reduce and
    then divides by world_size.  The accumulator starts at +0, replicas are
    added in rank order, each addition rounds to the accumulator's precision,
    and the final step is a true division by float(N).  ``dtype`` names how the
    replica arrays are stored: "f32", "bf16" (uint16 bit patterns, widened
    exactly before the sum) or "f64" (used by the data-parallel identity
    check, where the same loop runs in fp64)."""
    n = len(grads)
    if n < 1:
        raise ValueError("need at least one replica")
    first = _as_f32(grads[0], dtype)
    acc = np.zeros(first.shape, dtype=first.dtype)
    for r in range(n):
        acc = acc + _as_f32(grads[r], dtype)
    return acc / first.dtype.type(n)


def grad_mean_tree(grads, dtype: str = "f32") -> np.ndarray:
    """Pairwise (binary-tree) order of the same average, for a power-of-two
    replica count: level by level, neighbours (2i, 2i+1) are added, then the
    total is divided by N.  Tree all-reduce is described in [DDP] §2.13 and
    [TR24] §二; only the summation order differs from grad_mean (the tree has
    no +0 start: the first addition is g0 + g1)."""
    n = len(grads)
    if n < 1 or (n & (n - 1)) != 0:
        raise ValueError("tree order needs a power-of-two replica count")
    level = [_as_f32(g, dtype) for g in grads]
    while len(level) > 1:
        level = [level[2 * i] + level[2 * i + 1] for i in range(len(level) // 2)]
    return level[0] / level[0].dtype.type(n)


def ring_allreduce_mean(grads, dtype: str = "f32"):
    """The average as a ring all-reduce produces it, chunk by chunk.

    [DDP] §2.10-2.11: the flat buffer is cut into N chunks (chunk j = the j-th
    of N near-equal contiguous pieces, the first numel % N pieces one element
    longer).  During reduce-scatter the partial sum of chunk j starts at the
    GPU that owns chunk j (A_jj), travels to GPU j+1, j+2, ... each of which
    adds its own copy, so chunk j is summed in the order j, j+1, ..., j-1
    (mod N) -- the order the page's 4-GPU tables show (σ_0 = ((A_00 + A_10) +
    A_20) + A_30, σ_1 starts from A_11, ...).  The all-gather then copies σ_j
    unchanged to every GPU, and the result is divided by N.

    Returns (mean, chunk_bounds)."""
    n = len(grads)
    gs = [_as_f32(g, dtype) for g in grads]
    numel = gs[0].shape[0]
    base, rem = divmod(numel, n)
    bounds = []
    start = 0
    for j in range(n):
        ln = base + (1 if j < rem else 0)
        bounds.append((start, start + ln))
        start += ln
    out = np.empty(numel, dtype=gs[0].dtype)
    for j, (a, b) in enumerate(bounds):
        acc = gs[j][a:b].copy()
        for step in range(1, n):
            acc = acc + gs[(j + step) % n][a:b]
        out[a:b] = acc / gs[0].dtype.type(n)
    return out, bounds

# ---------------------------------------------------------------------------
# SGD after the sync  ([DDP] §5.3 update rule; momentum / weight decay: reading)
# ---------------------------------------------------------------------------


def sgd_step(grads, theta: np.ndarray, buf, lr: float, momentum: float, weight_decay: float,
             dtype: str = "f32"):
    """One SGD step on the averaged gradient.

    [DDP] §5.3 gives θ_{t+1} = θ_t − η g_t with g_t the averaged gradient, and
    [DDP] §三 (3.1) says every rank runs the same deterministic step on the
    same synced gradient.  The pages give no momentum or weight-decay formula;
    the reading taken is PyTorch's SGD (dampening 0, no Nesterov), each fp32
    operation rounded on its own, in this order:

        g = grad_mean(grads)
        d = g + wd*θ            (only if wd != 0)
        b = μ*buf + d; buf = b; d = b   (only if μ != 0; buf starts at zero)
        θ = θ − lr*d

    Returns (theta_new, buf_new_or_None, g)."""
    f = np.float32
    g = grad_mean(grads, dtype)
    th = np.ascontiguousarray(theta, dtype=np.float32)
    d = g
    if weight_decay != 0.0:
        d = d + f(weight_decay) * th
    b_new = None
    if momentum != 0.0:
        b_new = f(momentum) * np.ascontiguousarray(buf, dtype=np.float32) + d
        d = b_new
    th_new = th - f(lr) * d
    return th_new, b_new, g

# ---------------------------------------------------------------------------
# bucket planning  ([DDP] §3.2 and §4.2; [TR24] §三, §八; [TR16] §四, §六)
# ---------------------------------------------------------------------------

PLAN_CAP = 0
PLAN_DEEP_FIRST = 1


def plan_buckets(numels, elem_bytes: int, cap_bytes: int, mode: int = PLAN_CAP,
                 is_first=None, align_bytes: int = 256):
    """Partition a model's gradient tensors into flat buckets.

    PLAN_CAP ([DDP] §4.2: ``params_in_reverse = list(params)[::-1]`` then
    ``_build_buckets(..., bucket_size_mb=25)``; [DDP] §3.2: buckets follow
    the reverse of registration order because backward produces the last
    layer's gradient first).  ``_build_buckets`` itself is not given; the
    reading is the greedy fill: walk tensors last-registered first, and close
    the open bucket before a tensor whose bytes would push it past the cap.  A
    tensor larger than the cap ends up alone in its bucket.

    PLAN_DEEP_FIRST ([TR24] §八): exactly two buckets, DEEP first (its
    all-reduce overlaps the first layers' backward), then FIRST.  Tensors with
    ``is_first`` true go to FIRST, the rest to DEEP, each in reverse
    registration order.  No cap applies.  An empty group gives no bucket.

    Layout ([TR16] §四 MemoryPlan::finalize, §六 align_up_256): buckets are
    laid out one after another in one flat buffer; tensors are packed without
    gaps inside a bucket; each bucket's base offset is rounded up to
    ``align_bytes``.

    Returns a dict with
      buckets: list of (offset_elems, numel, first, count) where first/count
               index into ``order``;
      order: tensor ids in flat-buffer order;
      tensor_offset: element offset of each tensor id;
      tensor_bucket: bucket index of each tensor id;
      total_elems: flat buffer length (end of the last bucket, aligned)."""
    T = len(numels)
    if align_bytes % elem_bytes != 0:
        raise ValueError("align_bytes must be a multiple of elem_bytes")
    align = align_bytes // elem_bytes
    groups = []
    if mode == PLAN_CAP:
        cur, cur_bytes = [], 0
        for t in reversed(range(T)):
            nb = numels[t] * elem_bytes
            if cur and cur_bytes + nb > cap_bytes:
                groups.append(cur)
                cur, cur_bytes = [], 0
            cur.append(t)
            cur_bytes += nb
        if cur:
            groups.append(cur)
    elif mode == PLAN_DEEP_FIRST:
        deep = [t for t in reversed(range(T)) if not is_first[t]]
        first = [t for t in reversed(range(T)) if is_first[t]]
        groups = [g for g in (deep, first) if g]
    else:
        raise ValueError("unknown mode")

    buckets, order = [], []
    tensor_offset = [0] * T
    tensor_bucket = [0] * T
    cursor = 0
    for bi, grp in enumerate(groups):
        off = cursor
        pos = off
        first_idx = len(order)
        for t in grp:
            tensor_offset[t] = pos
            tensor_bucket[t] = bi
            pos += numels[t]
            order.append(t)
        buckets.append((off, pos - off, first_idx, len(grp)))
        cursor = -(-pos // align) * align
    return {"buckets": buckets, "order": order, "tensor_offset": tensor_offset,
            "tensor_bucket": tensor_bucket, "total_elems": cursor}

# ---------------------------------------------------------------------------
# SyncBatchNorm merge + apply  ([DDP] §4.3; [TR24] §三, §十二)
# ---------------------------------------------------------------------------


def syncbn(xs, eps: float = 1e-5, gamma=None, beta=None, dtype: str = "bf16"):
    """Strict SyncBatchNorm forward over N replicas' activations [B, C, H, W].

    [TR24] §十二: strict SyncBatchNorm all-reduces every rank's per-channel
    sum and sum of squares before the BN finalize/apply; [DDP] §4.3: the
    statistics then cover the whole global batch.  In fp64:
        s_r[c] = Σ x_r[:, c], q_r[c] = Σ x_r[:, c]^2, n_r = B*H*W
        S = Σ_r s_r, Q = Σ_r q_r, M = Σ_r n_r
        mean = S / M,  var = Q / M − mean^2  (biased, as BN normalises with)
        invstd = 1 / sqrt(var + eps)
        y_r = (x_r − mean) * invstd * γ + β
    γ defaults to 1 and β to 0 (the pages give neither).
    Returns (mean[C], invstd[C], [y_r]) all fp64."""
    mean, invstd = syncbn_stats(xs, eps, dtype)
    C = mean.shape[0]
    g = np.ones(C) if gamma is None else np.asarray(gamma, dtype=np.float64)
    b = np.zeros(C) if beta is None else np.asarray(beta, dtype=np.float64)
    ys = [(_to_f64(x, dtype) - mean[None, :, None, None]) * invstd[None, :, None, None] * g[None, :, None, None]
          + b[None, :, None, None] for x in xs]
    return mean, invstd, ys


def _to_f64(x, dtype):
    x = np.asarray(x)
    return bf16_bits_to_f32(x).astype(np.float64) if dtype == "bf16" else np.asarray(x, dtype=np.float64)


def syncbn_stats(xs, eps: float = 1e-5, dtype: str = "bf16"):
    """The merged statistics of ``syncbn`` for every channel: per replica r
    the fp64 sums s_r[c] = Σ x_r[:, c] and q_r[c] = Σ x_r[:, c]^2 over its
    B*H*W elements ([TR24] §十二: each rank's sum and sum of squares), then
    S = Σ_r s_r, Q = Σ_r q_r, M = Σ_r n_r, mean = S/M,
    var = Q/M − mean^2, invstd = 1/sqrt(var + eps).  One replica is widened
    to fp64 at a time, so full-size inputs fit in host memory.
    Returns (mean[C], invstd[C]) fp64."""
    S = Q = None
    M = 0
    for x in xs:
        x = _to_f64(x, dtype)
        s, q = x.sum(axis=(0, 2, 3)), (x * x).sum(axis=(0, 2, 3))
        S = s if S is None else S + s
        Q = q if Q is None else Q + q
        M += x.shape[0] * x.shape[2] * x.shape[3]
    mean = S / M
    var = Q / M - mean * mean
    return mean, 1.0 / np.sqrt(var + eps)


def syncbn_stats_at(xs, c: int, eps: float = 1e-5, dtype: str = "bf16"):
    """mean and invstd of one channel only (same definition as ``syncbn``),
    for spot checks on full-size inputs."""
    S = Q = 0.0
    M = 0
    for x in xs:
        v = np.asarray(x)[:, c]
        v = bf16_bits_to_f32(v).astype(np.float64) if dtype == "bf16" else v.astype(np.float64)
        S += v.sum()
        Q += (v * v).sum()
        M += v.size
    mean = S / M
    var = Q / M - mean * mean
    return mean, 1.0 / math.sqrt(var + eps)

# ---------------------------------------------------------------------------
# DistributedSampler  ([DDP] §4.4)
# ---------------------------------------------------------------------------

_M64 = (1 << 64) - 1
_M32 = (1 << 32) - 1
SPLITMIX_GAMMA = 0x9E3779B97F4A7C15
FEISTEL_ROUNDS = 4
WALK_CAP = 4096


def splitmix64_mix(z: int) -> int:
    """The SplitMix64 output function (Steele, Lea & Flood, "Fast splittable
    pseudorandom number generators", OOPSLA 2014), on Python ints mod 2^64."""
    z &= _M64
    z ^= z >> 30
    z = (z * 0xBF58476D1CE4E5B9) & _M64
    z ^= z >> 27
    z = (z * 0x94D049BB133111EB) & _M64
    return z ^ (z >> 31)


def splitmix64_stream(state: int, count: int):
    """First ``count`` outputs of SplitMix64 seeded with ``state``: the state
    advances by the golden-ratio increment before each output."""
    out = []
    for _ in range(count):
        state = (state + SPLITMIX_GAMMA) & _M64
        out.append(splitmix64_mix(state))
    return out


def murmur3_fmix32(h: int) -> int:
    """The 32-bit finalizer of MurmurHash3 (A. Appleby, public domain): two
    xor-shift / multiply steps and a last xor-shift, on Python ints mod 2^32."""
    h &= _M32
    h ^= h >> 16
    h = (h * 0x85EBCA6B) & _M32
    h ^= h >> 13
    h = (h * 0xC2B2AE35) & _M32
    return h ^ (h >> 16)


def feistel_round_keys(key: int):
    """k_0..k_3: the high 32 bits of the first four SplitMix64 outputs from
    state ``key``."""
    return [z >> 32 for z in splitmix64_stream(key, FEISTEL_ROUNDS)]


def _feistel_params(n: int):
    """Half widths of the network for a domain of n values: bits =
    ceil(log2 n) (at least 1) split into a high half of ceil(bits/2) bits and
    a low half of floor(bits/2) bits, so the domain 2^bits is below 2n.  For
    n < 2^62 both halves fit in 31 bits."""
    bits = max(1, (n - 1).bit_length())      # smallest bits with 2^bits >= n
    h_lo = bits // 2
    h_hi = bits - h_lo
    return h_hi, h_lo, (1 << h_hi) - 1, (1 << h_lo) - 1


def feistel_encrypt(x: int, key: int, n: int) -> int:
    """One pass of the keyed Feistel network on bits = ceil(log2 n) bits.
    x is split into a high half H (ceil(bits/2) bits) and a low half L
    (floor(bits/2) bits); with the round keys k_i of feistel_round_keys, even
    rounds set H ^= fmix32(L ^ k_i) mod 2^|H|, odd rounds L ^= fmix32(H ^ k_i)
    mod 2^|L|.  Each round undoes itself, so the pass is a bijection of
    [0, 2^bits) whatever the round function."""
    h_hi, h_lo, m_hi, m_lo = _feistel_params(n)
    rk = feistel_round_keys(key)
    H, L = x >> h_lo, x & m_lo
    for i in range(FEISTEL_ROUNDS):
        if i % 2 == 0:
            H ^= murmur3_fmix32(L ^ rk[i]) & m_hi
        else:
            L ^= murmur3_fmix32(H ^ rk[i]) & m_lo
    return (H << h_lo) | L


def keyed_perm(j: int, key: int, n: int) -> int:
    """π_key(j) for j in [0, n): Feistel encryption with cycle walking (encrypt
    again while the value is >= n).  Returns -1 if the walk exceeds WALK_CAP
    encryptions (never observed; both sides report it as an error).

    [DDP] §4.4 shuffles with torch.randperm(n, generator seeded with
    seed+epoch).  torch's generator stream is not reproducible outside torch,
    so the reading is: any permutation keyed by seed+epoch that every rank
    computes identically; this keyed Feistel permutation is the one used."""
    if n <= 1:
        return j
    y = feistel_encrypt(j, key, n)
    steps = 1
    while y >= n:
        if steps >= WALK_CAP:
            return -1
        y = feistel_encrypt(y, key, n)
        steps += 1
    return y


def keyed_perm_all(key: int, n: int) -> np.ndarray:
    """π_key(0..n-1) for every index, numpy-vectorised version of keyed_perm
    (same arithmetic on uint32 halves; wrapping multiplication mod 2^32)."""
    if n <= 1:
        return np.arange(n, dtype=np.int64)
    h_hi, h_lo, m_hi, m_lo = _feistel_params(n)
    rk = [np.uint32(k) for k in feistel_round_keys(key)]
    mh, ml, hl = np.uint32(m_hi), np.uint32(m_lo), np.uint64(h_lo)

    def fmix(h):
        h = h ^ (h >> np.uint32(16))
        h = h * np.uint32(0x85EBCA6B)
        h = h ^ (h >> np.uint32(13))
        h = h * np.uint32(0xC2B2AE35)
        return h ^ (h >> np.uint32(16))

    def enc(x):
        H, L = (x >> hl).astype(np.uint32), (x & np.uint64(m_lo)).astype(np.uint32)
        for i in range(FEISTEL_ROUNDS):
            if i % 2 == 0:
                H = H ^ (fmix(L ^ rk[i]) & mh)
            else:
                L = L ^ (fmix(H ^ rk[i]) & ml)
        return (H.astype(np.uint64) << hl) | L.astype(np.uint64)

    with np.errstate(over="ignore"):
        y = enc(np.arange(n, dtype=np.uint64))
        steps = 1
        todo = y >= np.uint64(n)
        while todo.any():
            if steps >= WALK_CAP:
                raise RuntimeError("cycle walk exceeded its cap")
            y[todo] = enc(y[todo])
            steps += 1
            todo = y >= np.uint64(n)
    return y.astype(np.int64)


def sampler_num_samples(n: int, n_replicas: int, drop_last: bool) -> int:
    """[DDP] §4.4: floor(n/N) with drop_last, else ceil(n/N)."""
    return n // n_replicas if drop_last else -(-n // n_replicas)


def dist_sampler_indices(n: int, n_replicas: int, rank: int, seed: int, epoch: int,
                         shuffle: bool = True, drop_last: bool = False) -> np.ndarray:
    """The indices rank ``rank`` draws in epoch ``epoch`` ([DDP] §4.4).

        num_samples = drop_last ? n // N : ceil(n / N);  total = num_samples * N
        base = shuffle ? π_{seed+epoch}(0..n-1) : 0..n-1
        padded: base extended by repeating from its head up to total
                (drop_last: base cut to total)
        out = padded[rank : total : N]

    ``rank`` = -1 returns every rank's list stacked rank-major [N, num_samples].
    Padding repeats the head cyclically (padded[j] = base[j mod n]); that is
    the page's ``indices += indices[:total-len]`` whenever total - n <= n,
    which holds whenever n >= N - 1."""
    ns = sampler_num_samples(n, n_replicas, drop_last)
    total = ns * n_replicas
    key = (seed + epoch) & _M64
    base = keyed_perm_all(key, n) if shuffle else np.arange(n, dtype=np.int64)
    if total == 0:
        padded = np.zeros(0, dtype=np.int64)
    else:
        padded = base[np.arange(total, dtype=np.int64) % n]
    if rank >= 0:
        return padded[rank:total:n_replicas].copy()
    return np.stack([padded[r:total:n_replicas] for r in range(n_replicas)]) if n_replicas else padded

# ---------------------------------------------------------------------------
# gradient accumulation, global norm / clipping, non-finite check
# ([DDP] §5.2; [TR24] §十一 NaN-check graph)
# ---------------------------------------------------------------------------


def accumulate(acc: np.ndarray, micro: np.ndarray, dtype: str = "f32") -> np.ndarray:
    """acc + micro in fp32: one micro-step of gradient accumulation under
    no_sync ([DDP] §5.2: backward adds the new gradient into .grad; the
    all-reduce runs only after the last micro-step).  dtype "f64" runs the
    same addition in fp64 (used by the no_sync identity check)."""
    acc_t = np.float64 if dtype == "f64" else np.float32
    return np.ascontiguousarray(acc, dtype=acc_t) + _as_f32(micro, dtype)


def grad_global_norm(grads) -> float:
    """L2 norm of all averaged gradients together, in fp64: the quantity
    clip_grad_norm_ computes after accumulation and the all-reduce
    ([DDP] §5.2, point ③)."""
    total = 0.0
    for g in grads:
        g64 = np.asarray(g, dtype=np.float64)
        total += float(np.dot(g64, g64))
    return math.sqrt(total)


def clip_coefficient(norm: float, max_norm: float) -> float:
    """The factor clip_grad_norm_ multiplies gradients by: max_norm divided by
    (norm + 1e-6), never above 1.  max_norm <= 0 disables clipping (factor 1).
    The pages only name clip_grad_norm_(..., 1.0); the formula is PyTorch's."""
    if max_norm <= 0.0:
        return 1.0
    return min(1.0, max_norm / (norm + 1e-6))


def any_nonfinite(grads) -> bool:
    """True if any averaged gradient element is NaN or infinite (the role of
    the NaN-check graph n_ncg in [TR24] §十一)."""
    return any(not np.all(np.isfinite(np.asarray(g, dtype=np.float64))) for g in grads)


def sgd_from_grad(g: np.ndarray, theta: np.ndarray, buf, lr: float, momentum: float, weight_decay: float,
                  scale=None):
    """The SGD step of sgd_step on an already averaged gradient, optionally
    multiplied first by a clipping factor (one fp32 rounding):
        d = g*scale (if scale is given); d = d + wd*θ; b = μ*buf + d; θ = θ − lr*b
    Returns (theta_new, buf_new_or_None)."""
    f = np.float32
    d = np.ascontiguousarray(g, dtype=np.float32)
    if scale is not None:
        d = d * f(scale)
    th = np.ascontiguousarray(theta, dtype=np.float32)
    if weight_decay != 0.0:
        d = d + f(weight_decay) * th
    b_new = None
    if momentum != 0.0:
        b_new = f(momentum) * np.ascontiguousarray(buf, dtype=np.float32) + d
        d = b_new
    return th - f(lr) * d, b_new

# ---------------------------------------------------------------------------
# BN running statistics and inference folding ([TR24] §十二)
# ---------------------------------------------------------------------------


def bn_running_update(running_mean, running_var, batch_mean, batch_var, count: int, momentum: float):
    """One running-statistics update from a batch's mean and biased variance
    over `count` values per channel.  [TR24] §十二 keeps per-rank running
    statistics (B_NEXT_MEAN / B_NEXT_VAR) that are then mean-all-reduced; the
    update rule itself is not on the pages — the reading is PyTorch's BN:
        r_mean = (1 − m)·r_mean + m·batch_mean
        r_var  = (1 − m)·r_var  + m·batch_var·count/(count − 1)
    in fp32, each operation rounded on its own; (1 − m) and count/(count−1)
    are computed in fp64 and rounded to fp32 once."""
    f = np.float32
    keep = f(1.0 - momentum)
    mom = f(momentum)
    corr = f(count / (count - 1)) if count > 1 else f(1.0)
    rm = keep * np.asarray(running_mean, np.float32) + mom * np.asarray(batch_mean, np.float32)
    unb = np.asarray(batch_var, np.float32) * corr
    rv = keep * np.asarray(running_var, np.float32) + mom * unb
    return rm, rv


def bn_fold_inference(running_mean, running_var, gamma, beta, eps: float):
    """UPDATE_BN_INF_PARAMS of [TR24] §十二: the per-channel scale and bias
    that make BN at inference one multiply-add, y = x·eq_scale + eq_bias.
    Reading (standard BN folding), in fp64:
        eq_scale = γ / sqrt(running_var + eps),  eq_bias = β − running_mean·eq_scale"""
    rm = np.asarray(running_mean, np.float64)
    rv = np.asarray(running_var, np.float64)
    g = np.ones_like(rm) if gamma is None else np.asarray(gamma, np.float64)
    b = np.zeros_like(rm) if beta is None else np.asarray(beta, np.float64)
    scale = g / np.sqrt(rv + eps)
    return scale, b - rm * scale


def f32_to_bf16_rne(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest, ties to even; a
    NaN stays a NaN.  The low-precision copy of the updated master weights
    ([TR16] §六: FP32 master weights and a half-width compute copy, refreshed
    by one whole-region cast after the update)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    nan = (u & 0x7FFFFFFF) > 0x7F800000
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    r = np.where(nan, (u >> 16) | 0x40, r)
    return r.astype(np.uint16)
