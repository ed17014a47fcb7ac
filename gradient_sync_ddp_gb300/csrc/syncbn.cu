// Strict SyncBatchNorm forward across N replicas on one GPU: per-channel
// statistics of the global batch, merged in fp64, then the normalisation.
//
// Tech-Renaissance "(24) NCCL通信与分布式数据并行" §十二: strict SyncBatchNorm
// all-reduces every rank's sum and sum of squares before BN finalize/apply.
// AI_Infra notes "1.DataParallel / DDP" §4.3: the synced statistics are those
// of the whole global batch (one extra all-reduce per BN layer).
//
// Three launches on the caller's stream:
//   1. stats  — grid (C, S): CTA (c, s) reduces slice s of the N*batch planes
//      of channel c (each plane is H*W contiguous elements of one replica and
//      one sample).  Threads stream 16-byte vectors when a plane's length is
//      a multiple of the vector width, single elements otherwise.  The sums
//      are shifted by K_c, the channel's first element (replica 0, sample 0):
//      d = x − K_c, and Σd, Σd² are accumulated, so Q/M − mean² never
//      subtracts two large nearly equal numbers when |mean| >> std.  Each
//      vector is summed pairwise in fp32, a thread accumulates at most a few
//      hundred elements in fp32, and the CTA combines its threads in fp64
//      into workspace partials.
//   2. merge  — one thread per channel sums the S partials in fixed order in
//      fp64: with m' = Σd/M, mean = K_c + m', var = Σd²/M − m'² (the same
//      S/M and Q/M − mean² up to rounding), invstd = 1/sqrt(var + eps); it
//      stores per channel (m_hi, m_lo, scale, β) where m_hi + m_lo is the
//      mean as an fp32 pair and scale = invstd·γ.
//   3. apply  — y = ((x − m_hi) − m_lo)·scale + β over every replica, 16-byte
//      vectors in and out.  x − m_hi is exact when x is near the mean
//      (Sterbenz), so no cancellation error is amplified by a large invstd
//      (the form x·scale + (β − mean·scale) would lose it).
// Traffic: x is read twice and y written once (2+2+2 bytes per bf16 element).
#include <cstdint>
#include <mutex>

#include "common.cuh"
#include "host_common.h"

namespace ddp {
namespace {

constexpr int kTargetCtas = 2048;   // stats CTAs aimed for (~1.7 waves of 8 CTAs on 152 SMs)

struct BnParams {
    const void* x[DDP_MAX_REPLICAS];
    void* y[DDP_MAX_REPLICAS];
    const float* gamma;
    const float* beta;
    float* mean_out;
    float* invstd_out;
    double2* partial;   // [C][S] (sum, sum of squares)
    float4* coef;       // [C] (m_hi, m_lo, scale, beta)
    FastDiv div_unit;   // per-plane unit count (vectors or elements per plane)
    FastDiv div_batch;  // batch
    FastDiv div_hw;     // H*W
    FastDiv div_c;      // C
    int32_t n, batch, C, HW, S;
    float eps;
};

__device__ __forceinline__ void block_sum2(double& a, double& b) {
    __shared__ double sh[2][kThreads / 32];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        a += __shfl_down_sync(0xffffffffu, a, o);
        b += __shfl_down_sync(0xffffffffu, b, o);
    }
    const int w = threadIdx.x / 32, l = threadIdx.x % 32;
    if (l == 0) {
        sh[0][w] = a;
        sh[1][w] = b;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        a = 0.0;
        b = 0.0;
        for (int i = 0; i < kThreads / 32; ++i) {
            a += sh[0][i];
            b += sh[1][i];
        }
    }
}

template <bool BF16, bool VEC>
__global__ void __launch_bounds__(kThreads) bn_stats_kernel(const __grid_constant__ BnParams a) {
    constexpr int W = VEC ? (BF16 ? 8 : 4) : 1;    // elements per access
    constexpr int ESZ = BF16 ? 2 : 4;
    const int c = blockIdx.x, s = blockIdx.y;
    const int P = a.n * a.batch;
    const int p0 = static_cast<int>(static_cast<int64_t>(P) * s / a.S);
    const int p1 = static_cast<int>(static_cast<int64_t>(P) * (s + 1) / a.S);
    const uint32_t units = static_cast<uint32_t>(a.HW / W);     // accesses per plane
    const uint32_t total = static_cast<uint32_t>(p1 - p0) * units;
    pdl_enter();

    const float K = load_elem<BF16>(a.x[0], static_cast<int64_t>(c) * a.HW);   // shift: x[0][0, c, 0, 0]
    float acc_s = 0.0f, acc_q = 0.0f;
    for (uint32_t t = threadIdx.x; t < total; t += kThreads) {
        const uint32_t pl_off = fdiv(t, a.div_unit);
        const uint32_t u = t - pl_off * units;
        const uint32_t pl = static_cast<uint32_t>(p0) + pl_off;
        const uint32_t r = fdiv(pl, a.div_batch);
        const uint32_t b = pl - r * static_cast<uint32_t>(a.batch);
        const int64_t elem = (static_cast<int64_t>(b) * a.C + c) * a.HW + static_cast<int64_t>(u) * W;
        const char* p = static_cast<const char*>(a.x[r]) + elem * ESZ;
        if constexpr (VEC) {
            const uint4 raw = ld16<true>(p);
            float e[W], q[W];
#pragma unroll
            for (int k = 0; k < W; ++k) {
                e[k] = __fsub_rn(vec_elem<BF16>(raw, k), K);
                q[k] = e[k] * e[k];
            }
#pragma unroll
            for (int w = W; w > 1; w >>= 1)
#pragma unroll
                for (int k = 0; k < w / 2; ++k) {
                    e[k] = e[2 * k] + e[2 * k + 1];
                    q[k] = q[2 * k] + q[2 * k + 1];
                }
            acc_s += e[0];
            acc_q += q[0];
        } else {
            const float v = __fsub_rn(load_elem<BF16>(p, 0), K);
            acc_s += v;
            acc_q += v * v;
        }
    }
    double ds = acc_s, dq = acc_q;
    block_sum2(ds, dq);
    if (threadIdx.x == 0) a.partial[static_cast<int64_t>(c) * a.S + s] = make_double2(ds, dq);
}

template <bool BF16>
__global__ void __launch_bounds__(kThreads) bn_merge_kernel(const __grid_constant__ BnParams a) {
    const int c = blockIdx.x * kThreads + threadIdx.x;
    pdl_enter();
    if (c >= a.C) return;
    double S = 0.0, Q = 0.0;
    for (int s = 0; s < a.S; ++s) {
        const double2 v = a.partial[static_cast<int64_t>(c) * a.S + s];
        S += v.x;
        Q += v.y;
    }
    const double M = static_cast<double>(a.n) * a.batch * a.HW;
    const double K = static_cast<double>(load_elem<BF16>(a.x[0], static_cast<int64_t>(c) * a.HW));
    const double ms = S / M;
    const double mean = K + ms;
    const double var = Q / M - ms * ms;
    const double invstd = 1.0 / sqrt(var + static_cast<double>(a.eps));
    const double g = a.gamma ? static_cast<double>(a.gamma[c]) : 1.0;
    const double b = a.beta ? static_cast<double>(a.beta[c]) : 0.0;
    const float m_hi = static_cast<float>(mean);
    a.mean_out[c] = m_hi;
    a.invstd_out[c] = static_cast<float>(invstd);
    a.coef[c] = make_float4(m_hi, static_cast<float>(mean - static_cast<double>(m_hi)),
                            static_cast<float>(invstd * g), static_cast<float>(b));
}

// ((x − m_hi) − m_lo)·scale + β with k = (m_hi, m_lo, scale, β)
__device__ __forceinline__ float normalize(float x, float4 k) {
    return fmaf(__fsub_rn(__fsub_rn(x, k.x), k.y), k.z, k.w);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const uint32_t l = __bfloat16_as_ushort(__float2bfloat16_rn(lo));
    const uint32_t h = __bfloat16_as_ushort(__float2bfloat16_rn(hi));
    return l | (h << 16);
}

// CVEC: H*W is a multiple of 8, so the 8 elements of one access share a channel.
template <bool BF16_IN, bool BF16_OUT, bool CVEC, bool NC>
__global__ void __launch_bounds__(kThreads) bn_apply_kernel(const __grid_constant__ BnParams a) {
    const int r = blockIdx.y;
    const char* x = static_cast<const char*>(a.x[r]);
    char* y = static_cast<char*>(a.y[r]);
    constexpr int ISZ = BF16_IN ? 2 : 4, OSZ = BF16_OUT ? 2 : 4;
    const uint32_t E = static_cast<uint32_t>(a.batch) * a.C * a.HW;
    const uint32_t nvec = E / 8;
    const uint32_t stride = gridDim.x * kThreads;
    const uint32_t gtid = blockIdx.x * kThreads + threadIdx.x;
    pdl_enter();
    for (uint32_t v = gtid; v < nvec; v += stride) {
        const uint32_t e0 = v * 8;
        float xv[8];
        if constexpr (BF16_IN) {
            const uint4 raw = ld16<NC>(x + static_cast<int64_t>(e0) * ISZ);
#pragma unroll
            for (int k = 0; k < 8; ++k) xv[k] = vec_elem<true>(raw, k);
        } else {
            const uint4 r0 = ld16<NC>(x + static_cast<int64_t>(e0) * ISZ);
            const uint4 r1 = ld16<NC>(x + static_cast<int64_t>(e0) * ISZ + 16);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                xv[k] = vec_elem<false>(r0, k);
                xv[4 + k] = vec_elem<false>(r1, k);
            }
        }
        float yv[8];
        if constexpr (CVEC) {
            const uint32_t pl = fdiv(e0, a.div_hw);
            const uint32_t c = pl - fdiv(pl, a.div_c) * static_cast<uint32_t>(a.C);
            const float4 k4 = __ldg(a.coef + c);
#pragma unroll
            for (int k = 0; k < 8; ++k) yv[k] = normalize(xv[k], k4);
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint32_t pl = fdiv(e0 + k, a.div_hw);
                const uint32_t c = pl - fdiv(pl, a.div_c) * static_cast<uint32_t>(a.C);
                yv[k] = normalize(xv[k], __ldg(a.coef + c));
            }
        }
        if constexpr (BF16_OUT) {
            st16(y + static_cast<int64_t>(e0) * OSZ,
                 make_uint4(pack_bf16x2(yv[0], yv[1]), pack_bf16x2(yv[2], yv[3]), pack_bf16x2(yv[4], yv[5]),
                            pack_bf16x2(yv[6], yv[7])));
        } else {
            st16(y + static_cast<int64_t>(e0) * OSZ, f4_bits(yv[0], yv[1], yv[2], yv[3]));
            st16(y + static_cast<int64_t>(e0) * OSZ + 16, f4_bits(yv[4], yv[5], yv[6], yv[7]));
        }
    }
    // tail: E % 8 elements
    const uint32_t t0 = nvec * 8;
    if (gtid < E - t0) {
        const uint32_t e = t0 + gtid;
        const float xe = load_elem<BF16_IN>(x, e);
        const uint32_t pl = fdiv(e, a.div_hw);
        const uint32_t c = pl - fdiv(pl, a.div_c) * static_cast<uint32_t>(a.C);
        const float ye = normalize(xe, a.coef[c]);
        if constexpr (BF16_OUT) reinterpret_cast<__nv_bfloat16*>(y)[e] = __float2bfloat16_rn(ye);
        else reinterpret_cast<float*>(y)[e] = ye;
    }
}

// slices per channel for the stats grid
int stats_slices(int32_t n, int32_t batch, int32_t C) {
    const int P = n * batch;
    int S = (kTargetCtas + C - 1) / C;
    if (S > P) S = P;
    if (S < 1) S = 1;
    return S;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool valid_sizes(int32_t n, int32_t batch, int32_t C, int32_t H, int32_t W) {
    if (n < 1 || n > DDP_MAX_REPLICAS || batch < 1 || C < 1 || H < 1 || W < 1) return false;
    const int64_t hw = static_cast<int64_t>(H) * W;
    const int64_t per = static_cast<int64_t>(batch) * C * hw;
    // 32-bit index arithmetic inside the kernels
    return hw < (int64_t(1) << 31) && per < (int64_t(1) << 31) &&
           static_cast<int64_t>(n) * batch * hw < (int64_t(1) << 31);
}

template <bool BF16_IN, bool BF16_OUT>
int launch_apply(const BnParams& p, bool cvec, bool nc, dim3 grid, cudaStream_t s) {
    if (cvec) {
        if (nc) return launch_pdl(bn_apply_kernel<BF16_IN, BF16_OUT, true, true>, grid, kThreads, s, p);
        return launch_pdl(bn_apply_kernel<BF16_IN, BF16_OUT, true, false>, grid, kThreads, s, p);
    }
    if (nc) return launch_pdl(bn_apply_kernel<BF16_IN, BF16_OUT, false, true>, grid, kThreads, s, p);
    return launch_pdl(bn_apply_kernel<BF16_IN, BF16_OUT, false, false>, grid, kThreads, s, p);
}

}  // namespace
}  // namespace ddp

using namespace ddp;

extern "C" size_t syncbn_workspace_bytes(int32_t n_replicas, int32_t batch, int32_t C, int32_t H, int32_t W) {
    if (!valid_sizes(n_replicas, batch, C, H, W)) return 0;
    const int S = stats_slices(n_replicas, batch, C);
    return align_up(static_cast<size_t>(C) * S * sizeof(double2), 16) + static_cast<size_t>(C) * sizeof(float4);
}

extern "C" int syncbn_merge_apply(const void* const* x, int32_t n_replicas, int32_t in_dtype,
                                  int32_t batch, int32_t C, int32_t H, int32_t W, float eps,
                                  const float* gamma, const float* beta,
                                  void* const* y, int32_t out_dtype, float* mean_out, float* invstd_out,
                                  void* workspace, size_t workspace_bytes, void* stream) {
    if (x == nullptr || y == nullptr || mean_out == nullptr || invstd_out == nullptr || workspace == nullptr)
        return DDP_ERR_INVALID_ARG;
    if (!valid_sizes(n_replicas, batch, C, H, W)) return DDP_ERR_INVALID_ARG;
    if ((in_dtype != DDP_F32 && in_dtype != DDP_BF16) || (out_dtype != DDP_F32 && out_dtype != DDP_BF16))
        return DDP_ERR_INVALID_ARG;
    if (!(eps > 0.0f) || !(eps < 3.0e38f)) return DDP_ERR_INVALID_ARG;
    if (workspace_bytes < syncbn_workspace_bytes(n_replicas, batch, C, H, W)) return DDP_ERR_CAPACITY;
    if (!aligned16(workspace) || ((uintptr_t)mean_out & 3u) || ((uintptr_t)invstd_out & 3u) ||
        ((uintptr_t)gamma & 3u) || ((uintptr_t)beta & 3u))
        return DDP_ERR_ALIGNMENT;
    const size_t E = static_cast<size_t>(batch) * C * H * W;
    const size_t ib = E * (in_dtype == DDP_BF16 ? 2 : 4), ob = E * (out_dtype == DDP_BF16 ? 2 : 4);
    bool in_place_any = false;
    for (int r = 0; r < n_replicas; ++r) {
        if (x[r] == nullptr || y[r] == nullptr) return DDP_ERR_INVALID_ARG;
        if (!aligned16(x[r]) || !aligned16(y[r])) return DDP_ERR_ALIGNMENT;
    }
    for (int r = 0; r < n_replicas; ++r) {
        for (int q = 0; q < n_replicas; ++q) {
            const bool same = (x[q] == y[r]) && q == r && in_dtype == out_dtype;
            if (same) in_place_any = true;
            else if (overlaps(y[r], ob, x[q], ib)) return DDP_ERR_INVALID_ARG;
        }
        for (int q = 0; q < r; ++q)
            if (overlaps(y[r], ob, y[q], ob)) return DDP_ERR_INVALID_ARG;
        if (overlaps(y[r], ob, workspace, workspace_bytes) || overlaps(y[r], ob, mean_out, C * 4u) ||
            overlaps(y[r], ob, invstd_out, C * 4u))
            return DDP_ERR_INVALID_ARG;
    }

    BnParams p{};
    for (int r = 0; r < n_replicas; ++r) {
        p.x[r] = x[r];
        p.y[r] = y[r];
    }
    p.gamma = gamma;
    p.beta = beta;
    p.mean_out = mean_out;
    p.invstd_out = invstd_out;
    p.n = n_replicas;
    p.batch = batch;
    p.C = C;
    p.HW = H * W;
    p.S = stats_slices(n_replicas, batch, C);
    p.eps = eps;
    char* ws = static_cast<char*>(workspace);
    p.partial = reinterpret_cast<double2*>(ws);
    ws += align_up(static_cast<size_t>(C) * p.S * sizeof(double2), 16);
    p.coef = reinterpret_cast<float4*>(ws);

    const bool bf16_in = in_dtype == DDP_BF16;
    const int wvec = bf16_in ? 8 : 4;
    const bool vec = (p.HW % wvec) == 0;
    p.div_unit = make_fastdiv(static_cast<uint32_t>(vec ? p.HW / wvec : p.HW));
    p.div_batch = make_fastdiv(static_cast<uint32_t>(batch));
    p.div_hw = make_fastdiv(static_cast<uint32_t>(p.HW));
    p.div_c = make_fastdiv(static_cast<uint32_t>(C));

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const dim3 sgrid(static_cast<unsigned>(C), static_cast<unsigned>(p.S));
    int st;
    if (bf16_in) st = vec ? launch_pdl(bn_stats_kernel<true, true>, sgrid, kThreads, s, p)
                          : launch_pdl(bn_stats_kernel<true, false>, sgrid, kThreads, s, p);
    else st = vec ? launch_pdl(bn_stats_kernel<false, true>, sgrid, kThreads, s, p)
                  : launch_pdl(bn_stats_kernel<false, false>, sgrid, kThreads, s, p);
    if (st != DDP_OK) return st;
    const dim3 mgrid(static_cast<unsigned>((C + kThreads - 1) / kThreads));
    st = bf16_in ? launch_pdl(bn_merge_kernel<true>, mgrid, kThreads, s, p)
                 : launch_pdl(bn_merge_kernel<false>, mgrid, kThreads, s, p);
    if (st != DDP_OK) return st;

    DeviceInfo d;
    if ((st = current_device_info(&d)) != DDP_OK) return st;
    const int64_t nvec = static_cast<int64_t>(E / 8);
    int64_t gx = (nvec + kThreads - 1) / kThreads;
    const int64_t resident = static_cast<int64_t>(d.sm_count) * (d.max_threads_per_sm / kThreads);
    int64_t cap = (resident + n_replicas - 1) / n_replicas;
    if (gx > cap) gx = cap;
    if (gx < 1) gx = 1;
    const dim3 agrid(static_cast<unsigned>(gx), static_cast<unsigned>(n_replicas));
    const bool cvec = (p.HW % 8) == 0;
    const bool nc = !in_place_any;
    const bool bf16_out = out_dtype == DDP_BF16;
    if (bf16_in) return bf16_out ? launch_apply<true, true>(p, cvec, nc, agrid, s) : launch_apply<true, false>(p, cvec, nc, agrid, s);
    return bf16_out ? launch_apply<false, true>(p, cvec, nc, agrid, s) : launch_apply<false, false>(p, cvec, nc, agrid, s);
}

// ---------------------------------------------------------------- variant without a caller workspace
//
// Some callers cannot hand this library a workspace because they cannot
// allocate device memory themselves: code embedded in a host framework whose
// memory pool owns the whole device and forbids side allocations, code run
// under a fixed device-memory budget reserved up front, or step loops where
// cudaMalloc's implicit device synchronisation is not acceptable.  For them
// the statistics scratch lives in a fixed array compiled into this library.
namespace ddp {
namespace {

constexpr size_t kStaticScratchBytes = size_t(1) << 20;   // 1 MiB per device that loads the library

__device__ __align__(256) unsigned char g_syncbn_scratch[kStaticScratchBytes];

constexpr int kMaxScratchDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxScratchDevices] = {};

// Device address of g_syncbn_scratch on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up once
// per device (with that device current) and cached.
int static_scratch(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= kMaxScratchDevices) return DDP_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_syncbn_scratch);
        if (e != cudaSuccess) return cuda_fail(e);
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return DDP_OK;
}

}  // namespace
}  // namespace ddp

extern "C" size_t syncbn_noalloc_max_workspace_bytes(void) { return ddp::kStaticScratchBytes; }

extern "C" int syncbn_merge_apply_noalloc(const void* const* x, int32_t n_replicas, int32_t in_dtype,
                                          int32_t batch, int32_t C, int32_t H, int32_t W, float eps,
                                          const float* gamma, const float* beta,
                                          void* const* y, int32_t out_dtype, float* mean_out, float* invstd_out,
                                          void* stream) {
    const size_t need = syncbn_workspace_bytes(n_replicas, batch, C, H, W);
    if (need == 0) return DDP_ERR_INVALID_ARG;
    if (need > ddp::kStaticScratchBytes) return DDP_ERR_CAPACITY;
    void* ws = nullptr;
    const int st = ddp::static_scratch(&ws);
    if (st != DDP_OK) return st;
    return syncbn_merge_apply(x, n_replicas, in_dtype, batch, C, H, W, eps, gamma, beta, y, out_dtype, mean_out,
                              invstd_out, ws, ddp::kStaticScratchBytes, stream);
}
