// Gradient accumulation under no_sync, the global gradient norm with
// clipping and the non-finite check, and the SGD step on an averaged
// gradient.
//
// AI_Infra notes "1.DataParallel / DDP" §5.2: micro-steps only add their
// gradient into .grad (the loss divided by the accumulation steps); the
// all-reduce runs once after the last micro-step; clip_grad_norm_ is applied
// to the synced gradient before the optimizer step.  Tech-Renaissance
// "(24) NCCL通信与分布式数据并行" §十一: a NaN-check graph runs after the
// gradient syncs.
//
// The bucket average with the Σg² side output lives with the other average
// kernels (allreduce.cu); this file holds the rest of the flow:
//   accumulate_kernel   acc[r] += micro[r] for all replicas in one launch:
//                       (esz + 8) bytes per element and replica, HBM-bound.
//   norm_finalize_kernel  one CTA: adds every bucket's per-CTA partials in a
//                       fixed order (float-float), then one thread computes
//                       the norm and clip factor in fp64.
//   sgd_grad_kernel     d = g·scale, weight decay, momentum, θ update:
//                       4 + 16 bytes per element, HBM-bound.
#include <cstdint>

#include "common.cuh"
#include "host_common.h"

namespace ddp {
namespace {

constexpr int kAccWaves = 16;

struct AccParams {
    const void* micro[DDP_MAX_REPLICAS];
    float* acc[DDP_MAX_REPLICAS];
    int64_t numel;
};

// grid (x: CTAs over the vectors, grid-stride, y: replica)
template <bool BF16>
__global__ void __launch_bounds__(kThreads) accumulate_kernel(const __grid_constant__ AccParams a) {
    constexpr int VEC = BF16 ? 8 : 4;
    constexpr int ESZ = BF16 ? 2 : 4;
    const int r = blockIdx.y;
    const char* m = static_cast<const char*>(a.micro[r]);
    float* acc = a.acc[r];
    const int64_t nvec = a.numel / VEC;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    const int64_t gtid = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
    pdl_enter();
    for (int64_t v0 = gtid; v0 < nvec; v0 += 2 * stride) {
        uint4 mv[2], av[2][VEC / 4];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int64_t v = v0 + u * stride;
            if (v < nvec) {
                mv[u] = ld16<true>(m + v * VEC * ESZ);
#pragma unroll
                for (int q = 0; q < VEC / 4; ++q) av[u][q] = ld16<false>(acc + v * VEC + 4 * q);
            }
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int64_t v = v0 + u * stride;
            if (v >= nvec) continue;
#pragma unroll
            for (int q = 0; q < VEC / 4; ++q) {
                float o[4];
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    o[k] = __fadd_rn(vec_elem<false>(av[u][q], k), vec_elem<BF16>(mv[u], 4 * q + k));
                st16(acc + v * VEC + 4 * q, f4_bits(o[0], o[1], o[2], o[3]));
            }
        }
    }
    const int64_t tail0 = nvec * VEC;
    if (gtid < a.numel - tail0) {
        const int64_t e = tail0 + gtid;
        acc[e] = __fadd_rn(acc[e], load_elem<BF16>(m, e));
    }
}

constexpr int kFinalizeThreads = 1024;

struct FinalizeParams {
    const char* ws;
    float* norm_out;
    float* coef_out;
    int32_t* nonfinite_out;
    int32_t n_buckets;
    float max_norm;
};

__global__ void __launch_bounds__(kFinalizeThreads) norm_finalize_kernel(const __grid_constant__ FinalizeParams a) {
    __shared__ FF sh[kFinalizeThreads / 32];
    pdl_enter();
    FF s{0.0f, 0.0f};
    bool nf = false;
    for (int b = 0; b < a.n_buckets; ++b) {
        const char* base = a.ws + static_cast<size_t>(b) * kNormBucketBytes;
        const int32_t cnt = *reinterpret_cast<const int32_t*>(base + kNormSlotBytes);
        const float4* slots = reinterpret_cast<const float4*>(base);
        for (int i = threadIdx.x; i < cnt; i += kFinalizeThreads) {
            const float4 v = slots[i];
            s = ff_add(s, FF{v.x, v.y});
            nf |= v.z != 0.0f;
        }
    }
    const bool any_nf = __syncthreads_or(nf);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s = ff_add(s, ff_shfl_down(s, o));
    if (threadIdx.x % 32 == 0) sh[threadIdx.x / 32] = s;
    __syncthreads();
    if (threadIdx.x != 0) return;
    FF t = sh[0];
    for (int w = 1; w < kFinalizeThreads / 32; ++w) t = ff_add(t, sh[w]);
    const double norm = sqrt(static_cast<double>(t.hi) + static_cast<double>(t.lo));
    double coef = 1.0;
    if (a.max_norm > 0.0f) {
        coef = static_cast<double>(a.max_norm) / (norm + 1e-6);
        if (coef > 1.0) coef = 1.0;
    }
    if (a.norm_out) *a.norm_out = static_cast<float>(norm);
    if (a.coef_out) *a.coef_out = static_cast<float>(coef);
    if (a.nonfinite_out) *a.nonfinite_out = any_nf ? 1 : 0;
}

struct SgdGradParams {
    const float* grad;
    float* param;
    float* buf;
    const float* scale;
    __nv_bfloat16* lowp;   // optional bf16 copy of the updated θ
    int64_t numel;
    float lr, mom, wd;
};

__device__ __forceinline__ void sgd_from_grad(const SgdGradParams& a, float g, float sc, bool has_scale,
                                              float& th, float& b) {
    float d = has_scale ? __fmul_rn(g, sc) : g;
    if (a.wd != 0.0f) d = __fadd_rn(d, __fmul_rn(a.wd, th));
    if (a.mom != 0.0f) {
        b = __fadd_rn(__fmul_rn(a.mom, b), d);
        d = b;
    }
    th = __fsub_rn(th, __fmul_rn(a.lr, d));
}

__global__ void __launch_bounds__(kThreads) sgd_grad_kernel(const __grid_constant__ SgdGradParams a) {
    const int64_t nvec = a.numel / 4;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    const int64_t gtid = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
    const bool has_mom = a.mom != 0.0f;
    const bool has_scale = a.scale != nullptr;
    pdl_enter();
    const float sc = has_scale ? *a.scale : 1.0f;
    for (int64_t v0 = gtid; v0 < nvec; v0 += 2 * stride) {
        uint4 gv[2], tv[2], bv[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int64_t v = v0 + u * stride;
            if (v < nvec) {
                gv[u] = ld16<true>(a.grad + 4 * v);
                tv[u] = ld16<false>(a.param + 4 * v);
                bv[u] = has_mom ? ld16<false>(a.buf + 4 * v) : make_uint4(0, 0, 0, 0);
            }
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int64_t v = v0 + u * stride;
            if (v >= nvec) continue;
            float th[4], b[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                th[k] = vec_elem<false>(tv[u], k);
                b[k] = vec_elem<false>(bv[u], k);
                sgd_from_grad(a, vec_elem<false>(gv[u], k), sc, has_scale, th[k], b[k]);
            }
            st16(a.param + 4 * v, f4_bits(th[0], th[1], th[2], th[3]));
            if (has_mom) st16(a.buf + 4 * v, f4_bits(b[0], b[1], b[2], b[3]));
            if (a.lowp != nullptr) st8(a.lowp + 4 * v, make_uint2(pack_bf16x2(th[0], th[1]), pack_bf16x2(th[2], th[3])));
        }
    }
    const int64_t tail0 = nvec * 4;
    if (gtid < a.numel - tail0) {
        const int64_t e = tail0 + gtid;
        float th = a.param[e];
        float b = has_mom ? a.buf[e] : 0.0f;
        sgd_from_grad(a, a.grad[e], sc, has_scale, th, b);
        a.param[e] = th;
        if (has_mom) a.buf[e] = b;
        if (a.lowp != nullptr) a.lowp[e] = __float2bfloat16_rn(th);
    }
}

}  // namespace
}  // namespace ddp

using namespace ddp;

extern "C" size_t ddp_norm_workspace_bytes(int32_t n_buckets) {
    return n_buckets < 1 ? 0 : static_cast<size_t>(n_buckets) * kNormBucketBytes;
}

extern "C" int ddp_bucket_accumulate(const void* const* micro, float* const* acc, int32_t n_replicas,
                                     int32_t in_dtype, int64_t numel, void* stream) {
    if (micro == nullptr || acc == nullptr || n_replicas < 1 || n_replicas > DDP_MAX_REPLICAS)
        return DDP_ERR_INVALID_ARG;
    if ((in_dtype != DDP_F32 && in_dtype != DDP_BF16) || numel < 0 || numel > INT64_MAX / 16)
        return DDP_ERR_INVALID_ARG;
    const size_t mb = static_cast<size_t>(numel) * (in_dtype == DDP_BF16 ? 2 : 4), ab = static_cast<size_t>(numel) * 4;
    for (int r = 0; r < n_replicas; ++r) {
        if (numel > 0 && (micro[r] == nullptr || acc[r] == nullptr)) return DDP_ERR_INVALID_ARG;
        if (!aligned16(micro[r]) || !aligned16(acc[r])) return DDP_ERR_ALIGNMENT;
    }
    for (int r = 0; r < n_replicas; ++r) {
        for (int q = 0; q < n_replicas; ++q) {
            if (overlaps(acc[r], ab, micro[q], mb)) return DDP_ERR_INVALID_ARG;
            if (q < r && overlaps(acc[r], ab, acc[q], ab)) return DDP_ERR_INVALID_ARG;
        }
    }
    if (numel == 0) return DDP_OK;
    AccParams p{};
    for (int r = 0; r < n_replicas; ++r) {
        p.micro[r] = micro[r];
        p.acc[r] = acc[r];
    }
    p.numel = numel;
    const bool bf16 = in_dtype == DDP_BF16;
    const int64_t nvec = numel / (bf16 ? 8 : 4);
    void (*kernel)(AccParams) = bf16 ? accumulate_kernel<true> : accumulate_kernel<false>;
    int wave = 0;
    int st = one_wave_grid(reinterpret_cast<const void*>(kernel), kThreads, INT64_MAX, &wave);
    if (st != DDP_OK) return st;
    // kAccWaves waves of resident CTAs over all replicas, not one grid-stride wave: measured on
    // GB300 (8 x 124M bf16 + fp32), 1 wave moved 6.05 TB/s, 2 waves 6.48, 8 waves 6.87
    int64_t gx = (nvec + kThreads - 1) / kThreads;
    const int64_t cap = (kAccWaves * static_cast<int64_t>(wave) + n_replicas - 1) / n_replicas;
    if (gx > cap) gx = cap;
    if (gx < 1) gx = 1;
    return launch_pdl(kernel, dim3(static_cast<unsigned>(gx), static_cast<unsigned>(n_replicas)), kThreads,
                      static_cast<cudaStream_t>(stream), p);
}

extern "C" int ddp_grad_norm_finalize(const void* norm_ws, int32_t n_buckets, float max_norm, float* norm_out,
                                      float* clip_coef_out, int32_t* nonfinite_out, void* stream) {
    if (norm_ws == nullptr || n_buckets < 1 || !(max_norm == max_norm)) return DDP_ERR_INVALID_ARG;
    if (!aligned16(norm_ws) || (reinterpret_cast<uintptr_t>(norm_out) & 3u) ||
        (reinterpret_cast<uintptr_t>(clip_coef_out) & 3u) || (reinterpret_cast<uintptr_t>(nonfinite_out) & 3u))
        return DDP_ERR_ALIGNMENT;
    const size_t wsb = ddp_norm_workspace_bytes(n_buckets);
    if (overlaps(norm_out, 4, norm_ws, wsb) || overlaps(clip_coef_out, 4, norm_ws, wsb) ||
        overlaps(nonfinite_out, 4, norm_ws, wsb))
        return DDP_ERR_INVALID_ARG;
    FinalizeParams p{};
    p.ws = static_cast<const char*>(norm_ws);
    p.norm_out = norm_out;
    p.coef_out = clip_coef_out;
    p.nonfinite_out = nonfinite_out;
    p.n_buckets = n_buckets;
    p.max_norm = max_norm;
    return launch_pdl(norm_finalize_kernel, dim3(1), kFinalizeThreads, static_cast<cudaStream_t>(stream), p);
}

extern "C" int ddp_bucket_sgd(const float* grad, float* param, float* momentum_buf, int64_t numel, float lr,
                              float momentum, float weight_decay, const float* grad_scale, void* param_bf16,
                              void* stream) {
    if (numel < 0 || numel > INT64_MAX / 16) return DDP_ERR_INVALID_ARG;
    if (!(lr == lr) || !(momentum == momentum) || !(weight_decay == weight_decay)) return DDP_ERR_INVALID_ARG;
    const bool has_mom = momentum != 0.0f;
    if (!has_mom && momentum_buf != nullptr) return DDP_ERR_INVALID_ARG;
    if (numel > 0 && (grad == nullptr || param == nullptr || (has_mom && momentum_buf == nullptr)))
        return DDP_ERR_INVALID_ARG;
    if (!aligned16(grad) || !aligned16(param) || !aligned16(momentum_buf) || !aligned16(param_bf16) ||
        (reinterpret_cast<uintptr_t>(grad_scale) & 3u))
        return DDP_ERR_ALIGNMENT;
    const size_t b = static_cast<size_t>(numel) * 4, hb = static_cast<size_t>(numel) * 2;
    if (overlaps(grad, b, param, b) || overlaps(grad, b, momentum_buf, b) || overlaps(param, b, momentum_buf, b) ||
        overlaps(grad_scale, 4, param, b) || overlaps(grad_scale, 4, momentum_buf, b) ||
        overlaps(param_bf16, hb, grad, b) || overlaps(param_bf16, hb, param, b) ||
        overlaps(param_bf16, hb, momentum_buf, b) || overlaps(param_bf16, hb, grad_scale, 4))
        return DDP_ERR_INVALID_ARG;
    if (numel == 0) return DDP_OK;
    SgdGradParams p{};
    p.grad = grad;
    p.param = param;
    p.buf = momentum_buf;
    p.scale = grad_scale;
    p.lowp = static_cast<__nv_bfloat16*>(param_bf16);
    p.numel = numel;
    p.lr = lr;
    p.mom = momentum;
    p.wd = weight_decay;
    int grid = 0;
    const int st = one_wave_grid(reinterpret_cast<const void*>(sgd_grad_kernel), kThreads,
                                 (numel / 4 + kThreads - 1) / kThreads, &grid);
    if (st != DDP_OK) return st;
    return launch_pdl(sgd_grad_kernel, dim3(static_cast<unsigned>(grid)), kThreads,
                      static_cast<cudaStream_t>(stream), p);
}
