// N-replica bucket average (the single-GPU form of the gradient all-reduce)
// and the same average fused with the SGD step.
//
// Definition: Tech-Renaissance "(24) NCCL通信与分布式数据并行" §一 — grad_sync
// starts at zero, grad[r] is added for r = 0..N-1, then divided by float(N);
// §九 — the all-reduce sums and a scale kernel multiplies by 1/world_size
// (here one pass: the replicas are read once, the average written once).
// AI_Infra notes "1.DataParallel / DDP" §2.11 (ring order) and §2.13 (tree
// order) give the alternative summation orders; §5.3 the SGD update.
//
// GB300 design: the kernel is HBM-bound ((N+1)*4 bytes per fp32 element), so
// each thread streams one 16-byte vector from every replica (all N loads are
// issued before the first add, N*16 bytes in flight per thread), keeps the
// adds in the exact rank order with __fadd_rn (no contraction), and writes
// the fp32 result with a streaming store.  The grid strides over the bucket:
// one wave of resident CTAs (occupancy calculator x SMs) for ordinary
// buckets, several waves for launches long enough to give each thread many
// vectors (see launch_wave); launches use programmatic dependent launch so
// back-to-back bucket kernels overlap launch and tail.  The
// replica pointers travel in a __grid_constant__ parameter block, so a
// launch is self-contained and capturable into a CUDA Graph.
#include <cstdint>

#include "common.cuh"
#include "host_common.h"

namespace ddp {
namespace {

struct RepPtrs {
    const void* p[DDP_MAX_REPLICAS];
};

enum Order { kRank = 0, kTree = 1, kRing = 2 };

struct MeanParams {
    RepPtrs rep;
    float* out;
    float4* norm_slots;   // NORM: per-CTA (Σout² hi, lo, non-finite flag, 0), one per CTA
    int32_t* norm_count;  // NORM: number of CTAs that wrote a slot
    int64_t numel;
    int64_t ring_base;  // ring chunk j has ring_base + (j < ring_rem) elements
    int64_t ring_rem;
    int32_t n;
    int32_t pow2;       // n is a power of two: scale by the exact reciprocal
    float inv_n;
};

// acc / n.  For n = 2^k, acc * 2^-k is the same real number as acc / 2^k, so
// both round to the same fp32 value (subnormal results included); otherwise
// a true IEEE division.
__device__ __forceinline__ float scale_by_n(float acc, int32_t pow2, float inv_n, int32_t n) {
    return pow2 ? __fmul_rn(acc, inv_n) : __fdiv_rn(acc, static_cast<float>(n));
}

// Ring chunk holding element e: N near-equal contiguous chunks, the first
// `rem` of them one element longer.
__device__ __forceinline__ int ring_chunk(int64_t e, int64_t base, int64_t rem) {
    const int64_t big = rem * (base + 1);
    return e < big ? static_cast<int>(e / (base + 1)) : static_cast<int>(rem + (e - big) / base);
}

template <bool BF16, int ORDER>
__device__ float mean_one(const MeanParams& a, int64_t e) {
    const int n = a.n;
    float acc;
    if constexpr (ORDER == kRank) {
        acc = 0.0f;
        for (int r = 0; r < n; ++r) acc = __fadd_rn(acc, load_elem<BF16>(a.rep.p[r], e));
    } else if constexpr (ORDER == kTree) {
        float t[DDP_MAX_REPLICAS];
        for (int r = 0; r < n; ++r) t[r] = load_elem<BF16>(a.rep.p[r], e);
        for (int w = n; w > 1; w >>= 1)
            for (int i = 0; i < w / 2; ++i) t[i] = __fadd_rn(t[2 * i], t[2 * i + 1]);
        acc = t[0];
    } else {
        const int j = ring_chunk(e, a.ring_base, a.ring_rem);
        acc = load_elem<BF16>(a.rep.p[j], e);
        for (int s = 1; s < n; ++s) {
            int r = j + s;
            r -= (r >= n) ? n : 0;
            acc = __fadd_rn(acc, load_elem<BF16>(a.rep.p[r], e));
        }
    }
    return scale_by_n(acc, a.pow2, a.inv_n, n);
}

// NORM: also reduce Σ out² and "any out non-finite" over the CTA and store
// them in the CTA's slot (side output for gradient clipping and the NaN check).
template <int NMAX, bool BF16, int ORDER, bool WB, bool NC, bool NORM = false>
__global__ void __launch_bounds__(kThreads) mean_kernel(const __grid_constant__ MeanParams a) {
    constexpr int VEC = BF16 ? 8 : 4;   // elements per 16-byte input vector
    constexpr int ESZ = BF16 ? 2 : 4;
    const int n = a.n;
    const int64_t nvec = a.numel / VEC;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    const int64_t gtid = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
    float nsq = 0.0f;       // NORM: this thread's Σ out²
    bool nonfinite = false; // NORM: this thread saw a NaN or infinity
    pdl_enter();

    for (int64_t v = gtid; v < nvec; v += stride) {
        const int64_t e0 = v * VEC;
        float res[VEC];
        bool done = false;
        uint4 raw[NMAX];
        if constexpr (ORDER == kRing) {
            const int j0 = ring_chunk(e0, a.ring_base, a.ring_rem);
            const int j1 = ring_chunk(e0 + VEC - 1, a.ring_base, a.ring_rem);
            if (j0 == j1) {
                // load replicas rotated so that raw[s] is replica (j0 + s) mod n
#pragma unroll
                for (int s = 0; s < NMAX; ++s) {
                    if (s < n) {
                        int r = j0 + s;
                        r -= (r >= n) ? n : 0;
                        raw[s] = ld16<NC>(static_cast<const char*>(a.rep.p[r]) + e0 * ESZ);
                    }
                }
#pragma unroll
                for (int k = 0; k < VEC; ++k) {
                    float acc = vec_elem<BF16>(raw[0], k);
#pragma unroll
                    for (int s = 1; s < NMAX; ++s)
                        if (s < n) acc = __fadd_rn(acc, vec_elem<BF16>(raw[s], k));
                    res[k] = scale_by_n(acc, a.pow2, a.inv_n, n);
                }
            } else {
#pragma unroll
                for (int k = 0; k < VEC; ++k) res[k] = mean_one<BF16, kRing>(a, e0 + k);
            }
            done = true;
        }
        if (!done) {
#pragma unroll
            for (int r = 0; r < NMAX; ++r)
                if (r < n) raw[r] = ld16<NC>(static_cast<const char*>(a.rep.p[r]) + e0 * ESZ);
#pragma unroll
            for (int k = 0; k < VEC; ++k) {
                float acc;
                if constexpr (ORDER == kRank) {
                    acc = 0.0f;
#pragma unroll
                    for (int r = 0; r < NMAX; ++r)
                        if (r < n) acc = __fadd_rn(acc, vec_elem<BF16>(raw[r], k));
                } else {
                    float t[NMAX];
#pragma unroll
                    for (int r = 0; r < NMAX; ++r) t[r] = (r < n) ? vec_elem<BF16>(raw[r], k) : 0.0f;
#pragma unroll
                    for (int w = NMAX; w > 1; w >>= 1)
                        if (w <= n) {
#pragma unroll
                            for (int i = 0; i < w / 2; ++i) t[i] = __fadd_rn(t[2 * i], t[2 * i + 1]);
                        }
                    acc = t[0];
                }
                res[k] = scale_by_n(acc, a.pow2, a.inv_n, n);
            }
        }
        if constexpr (NORM) {
#pragma unroll
            for (int k = 0; k < VEC; ++k) {
                nsq = fmaf(res[k], res[k], nsq);
                nonfinite |= (__float_as_uint(res[k]) & 0x7f800000u) == 0x7f800000u;
            }
        }
#pragma unroll
        for (int q = 0; q < VEC / 4; ++q) {
            const uint4 o = f4_bits(res[4 * q], res[4 * q + 1], res[4 * q + 2], res[4 * q + 3]);
            st16(a.out + e0 + 4 * q, o);
            if constexpr (WB) {
#pragma unroll
                for (int r = 0; r < NMAX; ++r)
                    if (r < n && a.rep.p[r] != a.out)
                        st16(const_cast<float*>(static_cast<const float*>(a.rep.p[r])) + e0 + 4 * q, o);
            }
        }
    }

    // ragged tail: the last numel % VEC elements, one per thread of block 0
    const int64_t tail0 = nvec * VEC;
    if (gtid < a.numel - tail0) {
        const int64_t e = tail0 + gtid;
        const float m = mean_one<BF16, ORDER>(a, e);
        a.out[e] = m;
        if constexpr (NORM) {
            nsq = fmaf(m, m, nsq);
            nonfinite |= (__float_as_uint(m) & 0x7f800000u) == 0x7f800000u;
        }
        if constexpr (WB) {
            for (int r = 0; r < n; ++r)
                if (a.rep.p[r] != a.out) const_cast<float*>(static_cast<const float*>(a.rep.p[r]))[e] = m;
        }
    }
    if constexpr (NORM) {
        const bool any_nf = __syncthreads_or(nonfinite);
        FF s{nsq, 0.0f}, unused{0.0f, 0.0f};
        block_sum2_ff(s, unused);
        if (threadIdx.x == 0) {
            a.norm_slots[blockIdx.x] = make_float4(s.hi, s.lo, any_nf ? 1.0f : 0.0f, 0.0f);
            if (blockIdx.x == 0) *a.norm_count = static_cast<int32_t>(gridDim.x);
        }
    }
}

struct SgdParams {
    RepPtrs rep;
    float* param;
    float* buf;
    float* gout;
    __nv_bfloat16* lowp;   // optional bf16 copy of the updated θ
    int64_t numel;
    int32_t n;
    int32_t pow2;
    float inv_n;
    float lr, mom, wd;
};

// d = g + wd*θ; b = μ*buf + d; θ = θ − lr*b — each operation rounded on its own.
__device__ __forceinline__ void sgd_elem(const SgdParams& a, float g, float& th, float& b) {
    float d = g;
    if (a.wd != 0.0f) d = __fadd_rn(d, __fmul_rn(a.wd, th));
    if (a.mom != 0.0f) {
        b = __fadd_rn(__fmul_rn(a.mom, b), d);
        d = b;
    }
    th = __fsub_rn(th, __fmul_rn(a.lr, d));
}

template <int NMAX, bool BF16>
__global__ void __launch_bounds__(kThreads) sgd_kernel(const __grid_constant__ SgdParams a) {
    constexpr int VEC = BF16 ? 8 : 4;
    constexpr int ESZ = BF16 ? 2 : 4;
    const int n = a.n;
    const bool has_mom = a.mom != 0.0f;
    const int64_t nvec = a.numel / VEC;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    const int64_t gtid = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
    pdl_enter();

    for (int64_t v = gtid; v < nvec; v += stride) {
        const int64_t e0 = v * VEC;
        uint4 raw[NMAX];
#pragma unroll
        for (int r = 0; r < NMAX; ++r)
            if (r < n) raw[r] = ld16<true>(static_cast<const char*>(a.rep.p[r]) + e0 * ESZ);
        uint4 thv[VEC / 4], bv[VEC / 4];
#pragma unroll
        for (int q = 0; q < VEC / 4; ++q) {
            thv[q] = ld16<false>(a.param + e0 + 4 * q);
            bv[q] = has_mom ? ld16<false>(a.buf + e0 + 4 * q) : make_uint4(0, 0, 0, 0);
        }
        float th[VEC], b[VEC], g[VEC];
#pragma unroll
        for (int k = 0; k < VEC; ++k) {
            float acc = 0.0f;
#pragma unroll
            for (int r = 0; r < NMAX; ++r)
                if (r < n) acc = __fadd_rn(acc, vec_elem<BF16>(raw[r], k));
            g[k] = scale_by_n(acc, a.pow2, a.inv_n, n);
            th[k] = vec_elem<false>(thv[k / 4], k % 4);
            b[k] = vec_elem<false>(bv[k / 4], k % 4);
            sgd_elem(a, g[k], th[k], b[k]);
        }
        if (a.lowp != nullptr) {
            if constexpr (VEC == 8)
                st16(a.lowp + e0, make_uint4(pack_bf16x2(th[0], th[1]), pack_bf16x2(th[2], th[3]),
                                             pack_bf16x2(th[4], th[5]), pack_bf16x2(th[6], th[7])));
            else
                st8(a.lowp + e0, make_uint2(pack_bf16x2(th[0], th[1]), pack_bf16x2(th[2], th[3])));
        }
#pragma unroll
        for (int q = 0; q < VEC / 4; ++q) {
            st16(a.param + e0 + 4 * q, f4_bits(th[4 * q], th[4 * q + 1], th[4 * q + 2], th[4 * q + 3]));
            if (has_mom) st16(a.buf + e0 + 4 * q, f4_bits(b[4 * q], b[4 * q + 1], b[4 * q + 2], b[4 * q + 3]));
            if (a.gout != nullptr)
                st16(a.gout + e0 + 4 * q, f4_bits(g[4 * q], g[4 * q + 1], g[4 * q + 2], g[4 * q + 3]));
        }
    }

    const int64_t tail0 = nvec * VEC;
    if (gtid < a.numel - tail0) {
        const int64_t e = tail0 + gtid;
        float acc = 0.0f;
        for (int r = 0; r < n; ++r) acc = __fadd_rn(acc, load_elem<BF16>(a.rep.p[r], e));
        const float g = scale_by_n(acc, a.pow2, a.inv_n, n);
        float th = a.param[e];
        float b = has_mom ? a.buf[e] : 0.0f;
        sgd_elem(a, g, th, b);
        a.param[e] = th;
        if (has_mom) a.buf[e] = b;
        if (a.gout != nullptr) a.gout[e] = g;
        if (a.lowp != nullptr) a.lowp[e] = __float2bfloat16_rn(th);
    }
}

// ---------------------------------------------------------------- host side

// Grid of the streaming kernels.  One grid-stride wave of resident CTAs is
// the default; a launch long enough that one wave would give every thread
// at least kMultiWaveVecs vectors gets up to kWaves waves instead (each
// thread still at least kMinVecsPerThread vectors).  Measured on GB300:
// fused SGD over GPT-2-small buckets 6.58 -> 7.24 TB/s and the bf16 average
// 6.89 -> 7.19 TB/s with 16 waves (8 vectors per thread at least).  With the
// thresholds lowered to 8 and 2, the 25 MiB fp32 buckets (14 vectors per
// thread at one wave) also run several waves of short CTAs: the ResNet-50
// step 7.08 -> 7.13 TB/s (one launch alone 27.62 -> 27.35 us), SGD 7.35 ->
// 7.39, the bf16 average 7.23 -> 7.33, ring / tree order 6.87 / 6.87 -> 6.94
// / 7.06 TB/s; thresholds 8 and 1 were within noise of these.
constexpr int kWaves = 16;
constexpr int64_t kMultiWaveVecs = 8;
constexpr int64_t kMinVecsPerThread = 2;

template <typename Params>
int launch_wave(void (*kernel)(Params), int64_t nvec, cudaStream_t s, const Params& p, int max_grid = 1 << 30) {
    int wave = 0;
    const int st = one_wave_grid(reinterpret_cast<const void*>(kernel), kThreads, INT64_MAX, &wave);
    if (st != DDP_OK) return st;
    const int64_t threads = static_cast<int64_t>(wave) * kThreads;
    int64_t g = (nvec + kThreads - 1) / kThreads;                 // one vector per thread at most
    if (nvec >= kMultiWaveVecs * threads) {
        g = (nvec + kThreads * kMinVecsPerThread - 1) / (kThreads * kMinVecsPerThread);
        if (g > static_cast<int64_t>(kWaves) * wave) g = static_cast<int64_t>(kWaves) * wave;
    } else if (g > wave) {
        g = wave;
    }
    if (g < 1) g = 1;
    int grid = static_cast<int>(g);
    if (grid > max_grid) grid = max_grid;
    return launch_pdl(kernel, dim3(static_cast<unsigned>(grid)), kThreads, s, p);
}

template <int NMAX, bool BF16, int ORDER, bool WB, bool NC>
int launch_mean(const MeanParams& p, int64_t nvec, cudaStream_t s) {
    return launch_wave(mean_kernel<NMAX, BF16, ORDER, WB, NC>, nvec, s, p);
}

template <int NMAX, bool BF16, int ORDER>
int dispatch_mean_mode(const MeanParams& p, int64_t nvec, cudaStream_t s, bool wb, bool aliased) {
    if constexpr (BF16) {
        return launch_mean<NMAX, true, ORDER, false, true>(p, nvec, s);
    } else {
        if (wb) return launch_mean<NMAX, false, ORDER, true, false>(p, nvec, s);
        if (aliased) return launch_mean<NMAX, false, ORDER, false, false>(p, nvec, s);
        return launch_mean<NMAX, false, ORDER, false, true>(p, nvec, s);
    }
}

template <int NMAX, bool BF16>
int dispatch_mean_order(const MeanParams& p, int64_t nvec, cudaStream_t s, int order, bool wb, bool aliased) {
    switch (order) {
        case kTree: return dispatch_mean_mode<NMAX, BF16, kTree>(p, nvec, s, wb, aliased);
        case kRing: return dispatch_mean_mode<NMAX, BF16, kRing>(p, nvec, s, wb, aliased);
        default: return dispatch_mean_mode<NMAX, BF16, kRank>(p, nvec, s, wb, aliased);
    }
}

template <bool BF16>
int dispatch_mean(const MeanParams& p, int64_t nvec, cudaStream_t s, int order, bool wb, bool aliased) {
    if (p.n <= 4) return dispatch_mean_order<4, BF16>(p, nvec, s, order, wb, aliased);
    if (p.n <= 8) return dispatch_mean_order<8, BF16>(p, nvec, s, order, wb, aliased);
    return dispatch_mean_order<16, BF16>(p, nvec, s, order, wb, aliased);
}

template <bool BF16>
int dispatch_sgd(const SgdParams& p, int64_t nvec, cudaStream_t s) {
    if (p.n <= 4) return launch_wave(sgd_kernel<4, BF16>, nvec, s, p);
    if (p.n <= 8) return launch_wave(sgd_kernel<8, BF16>, nvec, s, p);
    return launch_wave(sgd_kernel<16, BF16>, nvec, s, p);
}

bool is_pow2(int n) { return n > 0 && (n & (n - 1)) == 0; }

// Shared validation of the replica list.
int check_replicas(const void* const* replicas, int32_t n, int32_t dtype, int64_t numel) {
    if (replicas == nullptr || n < 1 || n > DDP_MAX_REPLICAS) return DDP_ERR_INVALID_ARG;
    if (dtype != DDP_F32 && dtype != DDP_BF16) return DDP_ERR_INVALID_ARG;
    if (numel < 0 || numel > INT64_MAX / 16) return DDP_ERR_INVALID_ARG;
    for (int r = 0; r < n; ++r) {
        if (replicas[r] == nullptr && numel > 0) return DDP_ERR_INVALID_ARG;
        if (!aligned16(replicas[r])) return DDP_ERR_ALIGNMENT;
    }
    return DDP_OK;
}

}  // namespace
}  // namespace ddp

using namespace ddp;

extern "C" int ddp_bucket_allreduce_mean(const void* const* replicas, int32_t n_replicas, int32_t in_dtype,
                                         int64_t numel, float* out, uint32_t flags, void* stream) {
    int st = check_replicas(replicas, n_replicas, in_dtype, numel);
    if (st != DDP_OK) return st;
    if (out == nullptr && numel > 0) return DDP_ERR_INVALID_ARG;
    if (!aligned16(out)) return DDP_ERR_ALIGNMENT;
    const uint32_t known = DDP_FLAG_TREE_ORDER | DDP_FLAG_WRITE_BACK_ALL | DDP_FLAG_RING_ORDER;
    if (flags & ~known) return DDP_ERR_INVALID_ARG;
    const bool tree = flags & DDP_FLAG_TREE_ORDER, ring = flags & DDP_FLAG_RING_ORDER;
    const bool wb = flags & DDP_FLAG_WRITE_BACK_ALL;
    if (tree && ring) return DDP_ERR_INVALID_ARG;
    if (tree && !is_pow2(n_replicas)) return DDP_ERR_INVALID_ARG;
    if (wb && in_dtype != DDP_F32) return DDP_ERR_INVALID_ARG;

    const size_t esz = in_dtype == DDP_BF16 ? 2 : 4;
    const size_t in_bytes = static_cast<size_t>(numel) * esz, out_bytes = static_cast<size_t>(numel) * 4;
    bool aliased = false;
    for (int r = 0; r < n_replicas; ++r) {
        if (static_cast<const void*>(out) == replicas[r] && in_dtype == DDP_F32) {
            aliased = true;
        } else if (overlaps(out, out_bytes, replicas[r], in_bytes)) {
            return DDP_ERR_INVALID_ARG;
        }
        if (wb)   // replicas are written: they must be disjoint or identical
            for (int q = 0; q < r; ++q)
                if (replicas[q] != replicas[r] && overlaps(replicas[q], in_bytes, replicas[r], in_bytes))
                    return DDP_ERR_INVALID_ARG;
    }
    if (numel == 0) return DDP_OK;

    MeanParams p{};
    for (int r = 0; r < n_replicas; ++r) p.rep.p[r] = replicas[r];
    p.out = out;
    p.numel = numel;
    p.n = n_replicas;
    p.pow2 = is_pow2(n_replicas);
    p.inv_n = 1.0f / static_cast<float>(n_replicas);   // exact when n is a power of two
    p.ring_base = numel / n_replicas;
    p.ring_rem = numel % n_replicas;
    const int order = tree ? kTree : ring ? kRing : kRank;
    const int64_t nvec = numel / (in_dtype == DDP_BF16 ? 8 : 4);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return in_dtype == DDP_BF16 ? dispatch_mean<true>(p, nvec, s, order, wb, aliased)
                                : dispatch_mean<false>(p, nvec, s, order, wb, aliased);
}

static int allreduce_sgd_impl(const void* const* replicas, int32_t n_replicas, int32_t in_dtype, int64_t numel,
                              float* param, float* momentum_buf, float lr, float momentum, float weight_decay,
                              float* grad_out, void* param_bf16, uint32_t flags, void* stream) {
    int st = check_replicas(replicas, n_replicas, in_dtype, numel);
    if (st != DDP_OK) return st;
    if (flags != 0 || (param == nullptr && numel > 0)) return DDP_ERR_INVALID_ARG;
    if (!(lr == lr) || !(momentum == momentum) || !(weight_decay == weight_decay)) return DDP_ERR_INVALID_ARG;
    const bool has_mom = momentum != 0.0f;
    if (has_mom && momentum_buf == nullptr && numel > 0) return DDP_ERR_INVALID_ARG;
    if (!has_mom && momentum_buf != nullptr) return DDP_ERR_INVALID_ARG;
    if (!aligned16(param) || (momentum_buf && !aligned16(momentum_buf)) || (grad_out && !aligned16(grad_out)) ||
        !aligned16(param_bf16))
        return DDP_ERR_ALIGNMENT;
    const size_t esz = in_dtype == DDP_BF16 ? 2 : 4;
    const size_t in_bytes = static_cast<size_t>(numel) * esz, fb = static_cast<size_t>(numel) * 4;
    const void* outs[4] = {param, momentum_buf, grad_out, param_bf16};
    const size_t ob[4] = {fb, fb, fb, static_cast<size_t>(numel) * 2};
    for (int i = 0; i < 4; ++i) {
        if (outs[i] == nullptr) continue;
        for (int j = 0; j < i; ++j)
            if (overlaps(outs[i], ob[i], outs[j], ob[j])) return DDP_ERR_INVALID_ARG;
        for (int r = 0; r < n_replicas; ++r)
            if (overlaps(outs[i], ob[i], replicas[r], in_bytes)) return DDP_ERR_INVALID_ARG;
    }
    if (numel == 0) return DDP_OK;

    SgdParams p{};
    for (int r = 0; r < n_replicas; ++r) p.rep.p[r] = replicas[r];
    p.param = param;
    p.buf = momentum_buf;
    p.gout = grad_out;
    p.lowp = static_cast<__nv_bfloat16*>(param_bf16);
    p.numel = numel;
    p.n = n_replicas;
    p.pow2 = is_pow2(n_replicas);
    p.inv_n = 1.0f / static_cast<float>(n_replicas);
    p.lr = lr;
    p.mom = momentum;
    p.wd = weight_decay;
    const int64_t nvec = numel / (in_dtype == DDP_BF16 ? 8 : 4);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return in_dtype == DDP_BF16 ? dispatch_sgd<true>(p, nvec, s) : dispatch_sgd<false>(p, nvec, s);
}


extern "C" int ddp_bucket_allreduce_sgd(const void* const* replicas, int32_t n_replicas, int32_t in_dtype,
                                        int64_t numel, float* param, float* momentum_buf,
                                        float lr, float momentum, float weight_decay,
                                        float* grad_out, uint32_t flags, void* stream) {
    return allreduce_sgd_impl(replicas, n_replicas, in_dtype, numel, param, momentum_buf, lr, momentum, weight_decay,
                              grad_out, nullptr, flags, stream);
}

extern "C" int ddp_bucket_allreduce_sgd_cast(const void* const* replicas, int32_t n_replicas, int32_t in_dtype,
                                             int64_t numel, float* param, float* momentum_buf, float lr,
                                             float momentum, float weight_decay, float* grad_out, void* param_bf16,
                                             void* stream) {
    if (param_bf16 == nullptr && numel > 0) return DDP_ERR_INVALID_ARG;
    return allreduce_sgd_impl(replicas, n_replicas, in_dtype, numel, param, momentum_buf, lr, momentum, weight_decay,
                              grad_out, param_bf16, 0u, stream);
}

// ---------------------------------------------------------------- average with a norm side output

namespace ddp {
namespace {

template <bool BF16>
int dispatch_mean_norm(const MeanParams& p, int64_t nvec, cudaStream_t s, bool aliased) {
    if (p.n <= 4)
        return aliased ? launch_wave(mean_kernel<4, BF16, kRank, false, false, true>, nvec, s, p, DDP_NORM_SLOTS)
                       : launch_wave(mean_kernel<4, BF16, kRank, false, true, true>, nvec, s, p, DDP_NORM_SLOTS);
    if (p.n <= 8)
        return aliased ? launch_wave(mean_kernel<8, BF16, kRank, false, false, true>, nvec, s, p, DDP_NORM_SLOTS)
                       : launch_wave(mean_kernel<8, BF16, kRank, false, true, true>, nvec, s, p, DDP_NORM_SLOTS);
    return aliased ? launch_wave(mean_kernel<16, BF16, kRank, false, false, true>, nvec, s, p, DDP_NORM_SLOTS)
                   : launch_wave(mean_kernel<16, BF16, kRank, false, true, true>, nvec, s, p, DDP_NORM_SLOTS);
}

}  // namespace
}  // namespace ddp

extern "C" int ddp_bucket_allreduce_mean_norm(const void* const* replicas, int32_t n_replicas, int32_t in_dtype,
                                              int64_t numel, float* out, void* norm_ws, int32_t bucket_index,
                                              void* stream) {
    int st = check_replicas(replicas, n_replicas, in_dtype, numel);
    if (st != DDP_OK) return st;
    if (norm_ws == nullptr || bucket_index < 0 || (out == nullptr && numel > 0)) return DDP_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(norm_ws)) return DDP_ERR_ALIGNMENT;
    const size_t esz = in_dtype == DDP_BF16 ? 2 : 4;
    const size_t in_bytes = static_cast<size_t>(numel) * esz, out_bytes = static_cast<size_t>(numel) * 4;
    char* slot = static_cast<char*>(norm_ws) + static_cast<size_t>(bucket_index) * kNormBucketBytes;
    bool aliased = false;
    for (int r = 0; r < n_replicas; ++r) {
        if (static_cast<const void*>(out) == replicas[r] && in_dtype == DDP_F32) aliased = true;
        else if (overlaps(out, out_bytes, replicas[r], in_bytes)) return DDP_ERR_INVALID_ARG;
        if (overlaps(slot, kNormBucketBytes, replicas[r], in_bytes)) return DDP_ERR_INVALID_ARG;
    }
    if (overlaps(slot, kNormBucketBytes, out, out_bytes)) return DDP_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (numel == 0) {      // an empty bucket contributes nothing: record zero CTAs
        const cudaError_t e = cudaMemsetAsync(slot + kNormSlotBytes, 0, sizeof(int32_t), s);
        return e == cudaSuccess ? DDP_OK : cuda_fail(e);
    }
    MeanParams p{};
    for (int r = 0; r < n_replicas; ++r) p.rep.p[r] = replicas[r];
    p.out = out;
    p.numel = numel;
    p.n = n_replicas;
    p.pow2 = is_pow2(n_replicas);
    p.inv_n = 1.0f / static_cast<float>(n_replicas);
    p.norm_slots = reinterpret_cast<float4*>(slot);
    p.norm_count = reinterpret_cast<int32_t*>(slot + kNormSlotBytes);
    const int64_t nvec = numel / (in_dtype == DDP_BF16 ? 8 : 4);
    return in_dtype == DDP_BF16 ? dispatch_mean_norm<true>(p, nvec, s, aliased)
                                : dispatch_mean_norm<false>(p, nvec, s, aliased);
}

// ---------------------------------------------------------------- several buckets in one launch

namespace ddp {
namespace {

constexpr int kMultiMaxBuckets = DDP_MULTI_MAX_BUCKETS;
constexpr int kChunk = 128;                 // vectors per warp chunk (4 per lane)

struct MultiParams {
    RepPtrs rep;                            // replica flat-buffer bases
    float* out;                             // output flat-buffer base
    int32_t n;
    int32_t pow2;
    float inv_n;
    int32_t n_buckets;
    int64_t off[kMultiMaxBuckets];          // bucket offsets (elements)
    int64_t numel[kMultiMaxBuckets];
    int32_t chunk_start[kMultiMaxBuckets + 1];   // prefix sums of chunks per bucket
};

template <int NMAX, bool BF16>
__global__ void __launch_bounds__(kThreads) mean_multi_kernel(const __grid_constant__ MultiParams a) {
    constexpr int VEC = BF16 ? 8 : 4;
    constexpr int ESZ = BF16 ? 2 : 4;
    const int n = a.n;
    const int lane = threadIdx.x % 32;
    const int warps = gridDim.x * (kThreads / 32);
    const int total = a.chunk_start[a.n_buckets];
    pdl_enter();
    for (int c = blockIdx.x * (kThreads / 32) + threadIdx.x / 32; c < total; c += warps) {
        int lo = 0, hi = a.n_buckets - 1;    // bucket b with chunk_start[b] <= c < chunk_start[b+1] (warp-uniform)
        while (lo < hi) {
            const int mid = (lo + hi + 1) / 2;
            if (a.chunk_start[mid] <= c) lo = mid;
            else hi = mid - 1;
        }
        const int b = lo;
        const int64_t off = a.off[b], numel = a.numel[b];
        const int64_t nvec = numel / VEC;
        const int64_t v0 = static_cast<int64_t>(c - a.chunk_start[b]) * kChunk;
#pragma unroll 1
        for (int j = 0; j < kChunk / 32; ++j) {
            const int64_t v = v0 + j * 32 + lane;
            if (v >= nvec) break;
            const int64_t e0 = off + v * VEC;
            uint4 raw[NMAX];
#pragma unroll
            for (int r = 0; r < NMAX; ++r)
                if (r < n) raw[r] = ld16<true>(static_cast<const char*>(a.rep.p[r]) + e0 * ESZ);
            float res[VEC];
#pragma unroll
            for (int k = 0; k < VEC; ++k) {
                float acc = 0.0f;
#pragma unroll
                for (int r = 0; r < NMAX; ++r)
                    if (r < n) acc = __fadd_rn(acc, vec_elem<BF16>(raw[r], k));
                res[k] = scale_by_n(acc, a.pow2, a.inv_n, n);
            }
#pragma unroll
            for (int q = 0; q < VEC / 4; ++q)
                st16(a.out + e0 + 4 * q, f4_bits(res[4 * q], res[4 * q + 1], res[4 * q + 2], res[4 * q + 3]));
        }
        // the bucket's last chunk also averages its ragged tail
        if (c == a.chunk_start[b + 1] - 1 && lane < numel - nvec * VEC) {
            const int64_t e = off + nvec * VEC + lane;
            float acc = 0.0f;
            for (int r = 0; r < n; ++r) acc = __fadd_rn(acc, load_elem<BF16>(a.rep.p[r], e));
            a.out[e] = scale_by_n(acc, a.pow2, a.inv_n, n);
        }
    }
}

template <bool BF16>
int dispatch_multi(const MultiParams& p, int64_t total_chunks, cudaStream_t s) {
    void (*kernel)(MultiParams) = p.n <= 4 ? mean_multi_kernel<4, BF16>
                                : p.n <= 8 ? mean_multi_kernel<8, BF16> : mean_multi_kernel<16, BF16>;
    int grid = 0;
    const int64_t need = (total_chunks + kThreads / 32 - 1) / (kThreads / 32);
    const int st = one_wave_grid(reinterpret_cast<const void*>(kernel), kThreads, need, &grid);
    if (st != DDP_OK) return st;
    return launch_pdl(kernel, dim3(static_cast<unsigned>(grid)), kThreads, s, p);
}

}  // namespace
}  // namespace ddp

extern "C" int ddp_bucket_allreduce_mean_multi(const void* const* replica_bases, int32_t n_replicas,
                                               int32_t in_dtype, const ddp_bucket* buckets, int32_t n_buckets,
                                               float* out_base, void* stream) {
    if (n_buckets < 0 || n_buckets > DDP_MULTI_MAX_BUCKETS || (n_buckets > 0 && buckets == nullptr))
        return DDP_ERR_INVALID_ARG;
    int64_t span = 0;               // elements from the base to the end of the last bucket
    int64_t prev_end = 0;
    for (int b = 0; b < n_buckets; ++b) {
        const int64_t o = buckets[b].offset_elems, m = buckets[b].numel;
        if (o < 0 || m < 0 || o < prev_end || m > INT64_MAX / 16 - o) return DDP_ERR_INVALID_ARG;
        prev_end = o + m;
        span = prev_end;
    }
    int st = check_replicas(replica_bases, n_replicas, in_dtype, span);
    if (st != DDP_OK) return st;
    if (out_base == nullptr && span > 0) return DDP_ERR_INVALID_ARG;
    if (!aligned16(out_base)) return DDP_ERR_ALIGNMENT;
    const int64_t esz = in_dtype == DDP_BF16 ? 2 : 4;
    for (int b = 0; b < n_buckets; ++b)
        if ((buckets[b].offset_elems * esz) % 16 != 0 || (buckets[b].offset_elems * 4) % 16 != 0)
            return DDP_ERR_ALIGNMENT;
    for (int b = 0; b < n_buckets; ++b) {
        const int64_t o = buckets[b].offset_elems, m = buckets[b].numel;
        for (int r = 0; r < n_replicas; ++r)
            if (overlaps(out_base + o, static_cast<size_t>(m) * 4, replica_bases[r],
                         static_cast<size_t>(span) * esz))
                return DDP_ERR_INVALID_ARG;
    }
    if (span == 0) return DDP_OK;
    static thread_local MultiParams p;      // ~20 KB: kept off the stack
    p = MultiParams{};
    for (int r = 0; r < n_replicas; ++r) p.rep.p[r] = replica_bases[r];
    p.out = out_base;
    p.n = n_replicas;
    p.pow2 = is_pow2(n_replicas);
    p.inv_n = 1.0f / static_cast<float>(n_replicas);
    p.n_buckets = n_buckets;
    const int64_t vec = in_dtype == DDP_BF16 ? 8 : 4;
    int64_t chunks = 0;
    for (int b = 0; b < n_buckets; ++b) {
        p.off[b] = buckets[b].offset_elems;
        p.numel[b] = buckets[b].numel;
        p.chunk_start[b] = static_cast<int32_t>(chunks);
        const int64_t nv = buckets[b].numel / vec;
        chunks += buckets[b].numel == 0 ? 0 : (nv == 0 ? 1 : (nv + kChunk - 1) / kChunk +
                                                            ((buckets[b].numel % vec) != 0 && nv % kChunk == 0 ? 1 : 0));
        if (chunks > INT32_MAX / 2) return DDP_ERR_UNSUPPORTED;
    }
    p.chunk_start[n_buckets] = static_cast<int32_t>(chunks);
    if (chunks == 0) return DDP_OK;        // only empty buckets
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return in_dtype == DDP_BF16 ? dispatch_multi<true>(p, chunks, s) : dispatch_multi<false>(p, chunks, s);
}
