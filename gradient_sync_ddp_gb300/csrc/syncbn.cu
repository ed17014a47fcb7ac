// Strict SyncBatchNorm forward across N replicas on one GPU: per-channel
// statistics of the global batch, merged in float-float, then the normalisation.
//
// Tech-Renaissance "(24) NCCL通信与分布式数据并行" §十二: strict SyncBatchNorm
// all-reduces every rank's sum and sum of squares before BN finalize/apply.
// AI_Infra notes "1.DataParallel / DDP" §4.3: the synced statistics are those
// of the whole global batch (one extra all-reduce per BN layer).
//
// Three launches on the caller's stream (large calls: three for each channel
// half, the second half on a side stream joined back before the call
// returns):
//   1. stats  — per-channel partial sums over slices of the N*batch samples.
//      The sums are shifted by K_c, the channel's first element (replica 0,
//      sample 0): d = x − K_c, and Σd, Σd² are accumulated, so Q/M − mean²
//      never subtracts two large nearly equal numbers when |mean| >> std.
//      The kernel depends on the plane (H*W contiguous elements of one
//      sample and channel):
//        plane kernel — H*W a multiple of the 16-byte vector and at least
//          64 vectors long (56x56, 28x28):
//          CTA (c, s) streams its planes with 16-byte loads, a warp at a
//          time over 64-vector chunks of one plane, two element positions
//          per packed f32x2 instruction.
//        bulk-staged kernel — unaligned planes at least one vector long
//          (7x7, 14x14, 3x3) and aligned bf16 ones under 16 vectors (8x8, 4x4):
//          a CTA owns G consecutive channels (G*H*W about
//          2K elements) and a slice of the samples; for one sample those G
//          channels are one contiguous run, copied into shared memory by one
//          bulk asynchronous copy (each warp streaming its own runs through
//          two buffers, or, for runs too long for that, tiles of runs per
//          CTA), and each lane sums a contiguous range of one channel's plane
//          there.
//        staged group kernel — planes shorter than a vector (1x1, 2x2):
//          runs are copied to shared memory and reduced per channel there.
//        element kernel — unaligned planes too long to stage (111x111).
//      Every kernel reads a run's ragged end element by element, so no
//      access leaves the replica buffer.
//      Threads accumulate at most a few hundred elements in fp32 (vectors
//      summed pairwise); the CTA combines threads in float-float (pairs of
//      fp32, ~48 significant bits: GB300's fp64 pipe is too narrow for
//      reductions) and stores one fp32 (sum, sum of squares) partial per
//      channel and slice.
//   2. merge  — one warp per channel sums the S partials in a fixed order in
//      float-float (fp32 pairs), then its lane 0 finalises in float-float:
//      m' = Σd/M, mean = K_c + m' and var = Σd²/M − m'² (the same S/M and
//      Q/M − mean² up to rounding); in fp32, invstd = 1/sqrt(var + eps) with
//      IEEE-rounded sqrt and divide.  With the mean as an fp32 pair
//      m_hi + m_lo and scale = invstd·γ, it stores per channel (m_hi, scale,
//      shift), shift = β − m_lo·scale rounded once.
//   3. apply  — y = (x − m_hi)·scale + shift over every replica, 16-byte
//      vectors in and out, the channel computed once per 8-element vector
//      (or, where the grid stride is a whole number of samples, once per
//      thread), element pairs in packed f32x2 arithmetic.  x − m_hi is
//      exact when x is near the mean (Sterbenz), so no cancellation error
//      is amplified by a large invstd; only the mean's tiny low part goes
//      into the shift (the form x·scale + (β − mean·scale) would lose that
//      protection).
// Traffic: x is read twice and y written once (2+2+2 bytes per bf16 element).
// The statistics kernels read x through the coherent path with the default
// L2 policy and the apply walks replicas and vectors in the reverse order,
// so the apply's second read of x finds the part of x still in L2 (all of
// it when x is smaller than L2) before the part that has left it.
#include <cstdint>
#include <map>
#include <mutex>
#include <utility>

#include "common.cuh"
#include "host_common.h"

namespace ddp {
namespace {

constexpr int kTargetCtas = 2048;        // stats CTAs aimed for (about two waves on 152 SMs)
constexpr int64_t kMaxPartials = 65536;  // C*S bound: fp32 partials stay <= 512 KiB
constexpr int kRunElems = 2048;          // channels per group: G*H*W <= this (G >= 1)
constexpr int kStageBytes = 32768;       // shared staging buffer per CTA (staged group kernel)
constexpr int kPlaneVecsPerThread = 24;  // plane statistics: slices sized for this many vectors per thread
constexpr int kPlaneMinVecs = 16;        // aligned bf16 planes of fewer vectors: bulk-staged statistics
constexpr int kApplyWaves = 16;          // apply grid: at most this many waves of 8 CTAs per SM
constexpr int kApplyVecs = 8;            // apply grid: at least this many 16-byte vectors per thread

struct BnParams {
    const void* x[DDP_MAX_REPLICAS];
    void* y[DDP_MAX_REPLICAS];
    const float* gamma;
    const float* beta;
    float* mean_out;
    float* invstd_out;
    float2* partial;    // [C][S] (Σd, Σd²) per channel and slice
    float4* coef;       // [C] (m_hi, scale, shift, unused)
    FastDiv div_unit;   // plane kernel: accesses per plane; group kernel: 16-byte vectors per staging slot
    FastDiv div_batch;  // batch
    FastDiv div_hw;     // H*W
    FastDiv div_c;      // C
    FastDiv div_s;      // S, valid when ps_small
    int32_t ps_small;   // n*batch*S < 2^31: slice bounds in 32-bit arithmetic
    int32_t n, batch, C, HW, S;
    int32_t G;          // group kernel: channels per CTA (power of two)
    int32_t R;          // group kernel: runs staged per tile
    int32_t slot_bytes; // group kernel: shared bytes per staged run
    int32_t tc_log2;    // bulk kernel: log2 of the lanes per channel (see plan_stats)
    int32_t vec_reads;  // bulk kernel: every lane's range starts 16-byte aligned (16-byte shared reads)
    uint64_t buf_fl;    // bulk kernel: replica bytes rounded down to 16 (copies stop there)
    float eps;
    float inv_hi, inv_lo;  // 1 / (n * batch * H * W) as a float pair
    int32_t tree_top;      // merge: first shuffle offset (lanes >= min(S, 32) hold no sums)
    FastDiv div_vs8;       // apply mode 3: 8-element vectors per sample (C*H*W/8)
    // channel range of this launch sequence: [0, C) for a whole call, half of it for each of
    // the two channel halves a call may run concurrently (plane statistics, apply mode 0)
    int32_t c_base, c_end;
    int32_t parted;        // 1: [c_base, c_end) is a strict part of [0, C)
    FastDiv div_vp;        // parted apply: 8-element vectors of one sample within the part
    uint32_t vs_full;      // parted apply: 8-element vectors per sample (C*H*W/8)
    uint32_t v_base;       // parted apply: the part's first vector within a sample (c_base*H*W/8)
};

template <bool BF16>
__device__ __forceinline__ float shared_elem(const unsigned char* p, int e) {
    if constexpr (BF16) return __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const unsigned short*>(p)[e]) << 16);
    else return reinterpret_cast<const float*>(p)[e];
}

// Two fp32 values in one 64-bit register pair, for the packed f32x2
// arithmetic of the sm_100 family: one instruction does both lanes, each
// rounded to nearest even exactly as the scalar add, subtract or fused
// multiply-add would.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}

// Elements (2j, 2j + 1) of a 16-byte vector of 8 bf16 or 4 fp32 values, as an fp32 pair.
template <bool BF16>
__device__ __forceinline__ uint64_t vec_pair(const uint4& v, int j) {
    if constexpr (BF16) {
        const uint32_t w = j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w;
        return f2_pack(bf16_lo(w), bf16_hi(w));
    } else {
        return j == 0 ? f2_pack(__uint_as_float(v.x), __uint_as_float(v.y))
                      : f2_pack(__uint_as_float(v.z), __uint_as_float(v.w));
    }
}

// Samples [p0, p1) of slice s: p_k = floor(P*k/S) with P = n*batch.
__device__ __forceinline__ void slice_bounds(const BnParams& a, int s, int& p0, int& p1) {
    const int P = a.n * a.batch;
    if (a.ps_small) {
        p0 = static_cast<int>(fdiv(static_cast<uint32_t>(P * s), a.div_s));
        p1 = static_cast<int>(fdiv(static_cast<uint32_t>(P * (s + 1)), a.div_s));
    } else {
        p0 = static_cast<int>(static_cast<int64_t>(P) * s / a.S);
        p1 = static_cast<int>(static_cast<int64_t>(P) * (s + 1) / a.S);
    }
}

// Start of the statistics kernels: wait for the previous grid in the stream
// (full completion and memory flush) before letting this call's merge and
// apply launch.  The apply reads its first vectors of x before its own wait,
// which is safe only once every kernel issued before this call (one of them
// may have written x, e.g. the previous layer's apply) has completed.
__device__ __forceinline__ void pdl_wait_then_release() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Group kernel, grid (ceil(C/G), S).
template <bool BF16>
__global__ void __launch_bounds__(kThreads) bn_stats_group_kernel(const __grid_constant__ BnParams a) {
    constexpr int ESZ = BF16 ? 2 : 4;
    __shared__ __align__(16) unsigned char stage[kStageBytes];
    __shared__ float red[2][kThreads];
    const int c0 = blockIdx.x * a.G, s = blockIdx.y;
    const int Gc = min(a.G, a.C - c0);            // channels of this group
    const int Tc = kThreads / a.G;                // threads per channel
    const int cl = threadIdx.x / Tc, k = threadIdx.x - cl * Tc;
    const bool active = cl < Gc;
    int p0, p1;
    slice_bounds(a, s, p0, p1);
    const uint64_t run_bytes = static_cast<uint64_t>(Gc) * a.HW * ESZ;
    const uint32_t vslot = static_cast<uint32_t>(a.slot_bytes / 16);
    pdl_wait_then_release();   // must stay the wait-then-release form: the apply reads x before its own wait
    const float K = active ? load_elem<BF16>(a.x[0], static_cast<int64_t>(c0 + cl) * a.HW) : 0.0f;

    float acc_s = 0.0f, acc_q = 0.0f;
    for (int t0 = p0; t0 < p1; t0 += a.R) {
        const int nr = min(a.R, p1 - t0);
        // stage runs t0 .. t0+nr-1
        const uint32_t total = static_cast<uint32_t>(nr) * vslot;
        for (uint32_t t = threadIdx.x; t < total; t += kThreads) {
            const uint32_t j = fdiv(t, a.div_unit);
            const uint32_t v = t - j * vslot;
            const uint32_t pl = static_cast<uint32_t>(t0) + j;
            const uint32_t r = fdiv(pl, a.div_batch);
            const uint32_t b = pl - r * static_cast<uint32_t>(a.batch);
            const char* base = static_cast<const char*>(a.x[r]);
            const uint64_t a0 = (static_cast<uint64_t>(b) * a.C + c0) * a.HW * ESZ;   // run bytes [a0, a1)
            const uint64_t a1 = a0 + run_bytes;
            const uint64_t a0al = a0 & ~uint64_t(15), a1fl = a1 & ~uint64_t(15);
            const uint64_t src = a0al + 16ull * v;
            unsigned char* dst = stage + j * a.slot_bytes + 16 * v;
            if (src < a1fl) {
                *reinterpret_cast<uint4*>(dst) = ld16_keep(base + src);
            } else if (src < a1) {                      // ragged end, element by element
                const uint64_t lo = src > a0 ? src : a0;
                const uint64_t hi = (src + 16 < a1) ? src + 16 : a1;
                for (uint64_t q = lo; q < hi; q += ESZ) {
                    if constexpr (BF16)
                        *reinterpret_cast<unsigned short*>(stage + j * a.slot_bytes + (q - a0al)) =
                            *reinterpret_cast<const unsigned short*>(base + q);
                    else
                        *reinterpret_cast<float*>(stage + j * a.slot_bytes + (q - a0al)) =
                            *reinterpret_cast<const float*>(base + q);
                }
            }
        }
        __syncthreads();
        if (active) {
            for (int j = 0; j < nr; ++j) {
                const uint32_t pl = static_cast<uint32_t>(t0 + j);
                const uint32_t r = fdiv(pl, a.div_batch);
                const uint32_t b = pl - r * static_cast<uint32_t>(a.batch);
                const uint32_t pre = static_cast<uint32_t>(((static_cast<uint64_t>(b) * a.C + c0) * a.HW * ESZ) & 15u);
                const unsigned char* run = stage + j * a.slot_bytes + pre;
                const int e0 = cl * a.HW;
                for (int e = k; e < a.HW; e += Tc) {
                    const float d = __fsub_rn(shared_elem<BF16>(run, e0 + e), K);
                    acc_s += d;
                    acc_q += d * d;
                }
            }
        }
        __syncthreads();
    }
    red[0][threadIdx.x] = acc_s;
    red[1][threadIdx.x] = acc_q;
    __syncthreads();
    if (threadIdx.x < Gc) {
        FF S{0.0f, 0.0f}, Q{0.0f, 0.0f};
        for (int i = 0; i < Tc; ++i) {
            S = ff_add(S, FF{red[0][threadIdx.x * Tc + i], 0.0f});
            Q = ff_add(Q, FF{red[1][threadIdx.x * Tc + i], 0.0f});
        }
        a.partial[static_cast<int64_t>(c0 + threadIdx.x) * a.S + s] =
            make_float2(__fadd_rn(S.hi, S.lo), __fadd_rn(Q.hi, Q.lo));
    }
}

// Bulk-staged kernel, grid (ceil(C/G), S), for H*W >= the vector width W
// and not a multiple of it (7x7, 14x14, 3x3, ...), or (bf16) a multiple of
// it shorter than 16 vectors (8x8, 4x4).  A run (one sample's G
// consecutive channels) is contiguous in memory; the 16-byte aligned blocks
// that cover it are copied into shared memory by one bulk asynchronous copy
// (the copy engine moves them without registers; completion is counted on
// an mbarrier).  Only where the replica buffer ends inside a block is the
// run's end read with plain loads.  A tile is up to kBulkRuns runs; two
// tile buffers alternate, so the copy of tile t+2 runs while tile t+1 is
// summed.  Tiles stay small (at most 4 runs of <= 8 KiB) so that 6 CTAs fit
// per SM: on 8 x [32, 2048, 7, 7] bf16, 4-5 runs per tile (6 CTAs per SM)
// beat 8 runs (4 CTAs per SM) by 3 %, and 2-3 runs or two waves of CTAs
// were slower.  Warp w sums run w of the tile; within a run, lane l owns a
// contiguous range of one channel's plane (Tc = 2^tc_log2 lanes share a
// plane: 32/G for G < 32, up to one 16-byte vector per lane on short aligned
// planes, else one lane per plane, for channels l, l+32, ...), so every
// element it reads belongs to its channel and needs no mask.  Each wait for a copy is
// bounded (about a second of globaltimer): on expiry the CTA writes NaN
// partials for its channels, which makes the statistics NaN, instead of
// waiting on.
constexpr int kBulkRuns = 4;             // runs per tile
constexpr int kBulkBufMax = 32768;        // bytes per tile buffer at most
constexpr uint64_t kCopyWaitNs = 1000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// One poll of the barrier's phase; the thread may be suspended for up to
// kPollSuspendNs while the phase is incomplete.
constexpr uint32_t kPollSuspendNs = 100000;

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(kPollSuspendNs)
        : "memory");
    return ok != 0;
}

// Sum (x - K) and (x - K)^2 over `count` elements starting at byte `byte0`
// of the shared buffer `buf` (element aligned; 32-bit words read).
template <bool BF16>
__device__ __forceinline__ void sum_range(const unsigned char* buf, uint32_t byte0, uint32_t count, float K,
                                          bool vec_reads, float& acc_s, float& acc_q) {
    // element pairs in packed f32x2 accumulators, a ragged first or last element in scalar ones
    float s0 = 0.0f, q0 = 0.0f;
    const uint64_t K2 = f2_pack(K, K);
    uint64_t s2 = f2_pack(0.0f, 0.0f), q2 = s2;
    auto add_pair = [&](float lo, float hi) {
        const uint64_t d = f2_sub(f2_pack(lo, hi), K2);
        s2 = f2_add(s2, d);
        q2 = f2_fma(d, d, q2);
    };
    if constexpr (BF16) {
        const uint32_t* w = reinterpret_cast<const uint32_t*>(buf);
        uint32_t h = byte0 >> 1;
        const uint32_t hend = h + count;
        if ((h & 1u) && h < hend) {                          // odd start: high half of a word
            const float d = __fsub_rn(bf16_hi(w[h >> 1]), K);
            s0 += d;
            q0 = fmaf(d, d, q0);
            ++h;
        }
        if (vec_reads) {                                     // every lane's range 16-byte aligned
            for (; h + 8 <= hend; h += 8) {
                const uint4 q = *reinterpret_cast<const uint4*>(w + (h >> 1));
                add_pair(bf16_lo(q.x), bf16_hi(q.x));
                add_pair(bf16_lo(q.y), bf16_hi(q.y));
                add_pair(bf16_lo(q.z), bf16_hi(q.z));
                add_pair(bf16_lo(q.w), bf16_hi(q.w));
            }
        }
        for (; h + 8 <= hend; h += 8) {
            uint32_t v[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) v[i] = w[(h >> 1) + i];
#pragma unroll
            for (int i = 0; i < 4; ++i) add_pair(bf16_lo(v[i]), bf16_hi(v[i]));
        }
        for (; h + 2 <= hend; h += 2) {
            const uint32_t v = w[h >> 1];
            add_pair(bf16_lo(v), bf16_hi(v));
        }
        if (h < hend) {                                      // last element: low half of a word
            const float d = __fsub_rn(bf16_lo(w[h >> 1]), K);
            s0 += d;
            q0 = fmaf(d, d, q0);
        }
    } else {
        const float* f = reinterpret_cast<const float*>(buf) + (byte0 >> 2);
        uint32_t i = 0;
        for (; i + 4 <= count; i += 4) {
            add_pair(f[i], f[i + 1]);
            add_pair(f[i + 2], f[i + 3]);
        }
        for (; i < count; ++i) {
            const float d = __fsub_rn(f[i], K);
            s0 += d;
            q0 = fmaf(d, d, q0);
        }
    }
    float sl, sh, ql, qh;
    f2_unpack(s2, sl, sh);
    f2_unpack(q2, ql, qh);
    acc_s += (s0 + sl) + sh;
    acc_q += (q0 + ql) + qh;
}

template <bool BF16, int CPL>
__global__ void __launch_bounds__(kThreads) bn_stats_bulk_kernel(const __grid_constant__ BnParams a) {
    constexpr int ESZ = BF16 ? 2 : 4;
    constexpr int kWarps = kThreads / 32;
    extern __shared__ __align__(128) unsigned char smem[];   // two tile buffers of R * slot_bytes
    __shared__ uint64_t bar[2];
    const int c0 = a.c_base + blockIdx.x * a.G, s = blockIdx.y;
    const int Gc = min(a.G, a.c_end - c0);
    const int HW = a.HW;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int p0, p1;
    slice_bounds(a, s, p0, p1);
    const int R = a.R;                                       // runs per tile
    const int ntiles = (p1 - p0 + R - 1) / R;
    const uint32_t buf_bytes = static_cast<uint32_t>(R) * a.slot_bytes;
    const uint32_t run_bytes = static_cast<uint32_t>(Gc) * HW * ESZ;
    // this lane's CPL channels (lane/Tc, then every 32/Tc-th) and its element range, part
    // lane%Tc of Tc = 2^tc_log2 equal parts of a plane (the splits are shifts)
    const int Tc = 1 << a.tc_log2;
    const int part = lane & (Tc - 1);
    const uint32_t e_lo = (static_cast<uint32_t>(HW) * part) >> a.tc_log2;
    const uint32_t e_hi = (static_cast<uint32_t>(HW) * (part + 1)) >> a.tc_log2;
    int cl[CPL];
    float K[CPL], acc_s[CPL], acc_q[CPL];
    pdl_wait_then_release();   // must stay the wait-then-release form: the apply reads x before its own wait
#pragma unroll
    for (int m = 0; m < CPL; ++m) {
        cl[m] = (lane >> a.tc_log2) + (32 >> a.tc_log2) * m;
        K[m] = cl[m] < Gc ? load_elem<BF16>(a.x[0], static_cast<int64_t>(c0 + cl[m]) * HW) : 0.0f;
        acc_s[m] = 0.0f;
        acc_q[m] = 0.0f;
    }
    if (threadIdx.x == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&bar[0])) : "memory");
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&bar[1])) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();

    // Copy tile t into buffer t & 1 (warp 0): each lane handles runs lane, lane+32, ...
    auto issue = [&](int t) {
        const int tb = p0 + t * R, nr = min(R, p1 - tb);
        unsigned char* buf = smem + (t & 1) * buf_bytes;
        uint64_t* b = &bar[t & 1];
        uint32_t tx = 0;
        for (int j = lane; j < nr; j += 32) {
            const uint32_t pl = static_cast<uint32_t>(tb + j);
            const uint32_t r = fdiv(pl, a.div_batch);
            const uint32_t bb = pl - r * static_cast<uint32_t>(a.batch);
            const uint64_t a0 = (static_cast<uint64_t>(bb) * a.C + c0) * HW * ESZ, a1 = a0 + run_bytes;
            const uint64_t hi = min((a1 + 15) & ~uint64_t(15), a.buf_fl);
            tx += static_cast<uint32_t>(hi - (a0 & ~uint64_t(15)));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) tx += __shfl_xor_sync(0xffffffffu, tx, o);
        if (lane == 0)
            asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(b)), "r"(tx)
                         : "memory");
        __syncwarp();
        for (int j = lane; j < nr; j += 32) {
            const uint32_t pl = static_cast<uint32_t>(tb + j);
            const uint32_t r = fdiv(pl, a.div_batch);
            const uint32_t bb = pl - r * static_cast<uint32_t>(a.batch);
            const uint64_t a0 = (static_cast<uint64_t>(bb) * a.C + c0) * HW * ESZ, a1 = a0 + run_bytes;
            const uint64_t a0al = a0 & ~uint64_t(15);
            const uint64_t hi = min((a1 + 15) & ~uint64_t(15), a.buf_fl);
            unsigned char* dst = buf + j * a.slot_bytes;
            const char* src = static_cast<const char*>(a.x[r]);
            asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                             smem_u32(dst)),
                         "l"(src + a0al), "r"(static_cast<uint32_t>(hi - a0al)), "r"(smem_u32(b))
                         : "memory");
            for (uint64_t q = hi; q < a1; q += ESZ) {             // the buffer ends inside the last block
                if constexpr (BF16) *reinterpret_cast<unsigned short*>(dst + (q - a0al)) = *reinterpret_cast<const unsigned short*>(src + q);
                else *reinterpret_cast<float*>(dst + (q - a0al)) = *reinterpret_cast<const float*>(src + q);
            }
        }
    };
    if (warp == 0) {
        issue(0);
        if (ntiles > 1) issue(1);
    }

    bool failed = false;
    int fail_t = 0;
    for (int t = 0; t < ntiles; ++t) {
        // thread 0 waits for the tile's copies; the others wait at the CTA barrier (no issue slots)
        bool timed_out = false;
        const uint32_t parity = static_cast<uint32_t>(t >> 1) & 1u;
        if (threadIdx.x == 0 && !mbar_try_wait(&bar[t & 1], parity)) {
            const uint64_t start = global_ns();
            while (!mbar_try_wait(&bar[t & 1], parity)) {
                if (global_ns() - start > kCopyWaitNs) {
                    timed_out = true;
                    break;
                }
            }
        }
        if (__syncthreads_or(timed_out)) {                    // also orders warp 0's plain tail stores
            failed = true;
            fail_t = t;
            break;
        }
        const int tb = p0 + t * R, nr = min(R, p1 - tb);
        const unsigned char* buf = smem + (t & 1) * buf_bytes;
        for (int j = warp; j < nr; j += kWarps) {
            const uint32_t pl = static_cast<uint32_t>(tb + j);
            const uint32_t r = fdiv(pl, a.div_batch);
            const uint32_t bb = pl - r * static_cast<uint32_t>(a.batch);
            const uint32_t pre = static_cast<uint32_t>(((static_cast<uint64_t>(bb) * a.C + c0) * HW * ESZ) & 15u);
            const unsigned char* run = buf + j * a.slot_bytes;
#pragma unroll
            for (int m = 0; m < CPL; ++m) {
                if (cl[m] < Gc)
                    sum_range<BF16>(run, pre + (static_cast<uint32_t>(cl[m]) * HW + e_lo) * ESZ, e_hi - e_lo, K[m],
                                    a.vec_reads != 0, acc_s[m], acc_q[m]);
            }
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // reads done before the next bulk writes
        __syncthreads();
        if (warp == 0 && t + 2 < ntiles) issue(t + 2);
    }
    if (failed) {
        // let the copies in flight (the failed tile's and the next one's) land, bounded, before the
        // shared memory is reused
        if (threadIdx.x == 0)
            for (int u = fail_t; u < ntiles && u < fail_t + 2; ++u) {
                const uint32_t pu = static_cast<uint32_t>(u >> 1) & 1u;
                const uint64_t start = global_ns();
                while (!mbar_try_wait(&bar[u & 1], pu) && global_ns() - start <= kCopyWaitNs) {
                }
            }
        __syncthreads();
    }

    // combine: smem holds [warp][m][lane] sums, then one thread per channel adds the warps' and
    // lanes' shares in a fixed order in float-float
    float* red_s = reinterpret_cast<float*>(smem);
    float* red_q = red_s + kWarps * CPL * 32;
#pragma unroll
    for (int m = 0; m < CPL; ++m) {
        red_s[(warp * CPL + m) * 32 + lane] = acc_s[m];
        red_q[(warp * CPL + m) * 32 + lane] = acc_q[m];
    }
    __syncthreads();
    if (threadIdx.x < Gc) {
        const int c = threadIdx.x;
        const int cps = 32 >> a.tc_log2;          // channels per 32 lanes
        const int m = c / cps;
        const int l0 = (c % cps) << a.tc_log2;
        const int nl = Tc;
        FF S{0.0f, 0.0f}, Q{0.0f, 0.0f};
        for (int w = 0; w < kWarps; ++w)
            for (int l = l0; l < l0 + nl; ++l) {
                S = ff_add(S, FF{red_s[(w * CPL + m) * 32 + l], 0.0f});
                Q = ff_add(Q, FF{red_q[(w * CPL + m) * 32 + l], 0.0f});
            }
        a.partial[static_cast<int64_t>(c0 + c) * a.S + s] =
            failed ? make_float2(__int_as_float(0x7fc00000), __int_as_float(0x7fc00000))
                   : make_float2(__fadd_rn(S.hi, S.lo), __fadd_rn(Q.hi, Q.lo));
    }
}

// Bulk-staged kernel with a pipeline per warp, same grid, planes and lane
// mapping as the tiled kernel above, in CTAs of bulkw_threads(CPL) threads:
// warp w of a CTA of k warps owns runs w, w + k, ... of the CTA's slice and
// streams them through kBulkWarpRuns buffers of its own, each completed on
// its own mbarrier, which every lane of the warp waits on itself; a buffer
// is refilled as soon as its warp has summed it.
// No CTA barrier sits inside the loop, so a warp never waits for another
// warp's copies or sums.  Used where the warps' buffers fit in
// kBulkWarpMaxSmem (short runs: 7x7, 14x14, 8x8 bf16); measured on
// 8 x [32, C, H, W] bf16 (us per call, tiled -> per warp): 2048x7x7 29.0 ->
// 28.2, 256x14x14 20.6 -> 18.4, 2048x8x8 46.7 -> 41.5, 512x7x7 15.1 -> 13.2,
// 1024x14x14 52.3 either way; three buffers per warp were no better.  A
// wait that runs out marks the CTA failed; the warp then lets its copies in
// flight land (bounded) before the shared memory is reused.
constexpr int kBulkWarpRuns = 2;
constexpr int kBulkWarpMaxSmem = 72 * 1024;

// Threads per CTA of the per-warp kernel: 4 warps where a lane holds one or
// two channels (twice the CTAs, each with a quarter of the SM's run
// buffers: split 7x7 calls 25.7 -> 24.8 us, 1024x14x14 49.3 -> 48.5), 8
// where it holds four or eight (short aligned planes: 8x8 41.2 against
// 42.1 us with 4 warps).
__host__ __device__ constexpr int bulkw_threads(int cpl) { return cpl >= 4 ? 256 : 128; }

template <bool BF16, int CPL>
__global__ void __launch_bounds__(bulkw_threads(CPL)) bn_stats_bulkw_kernel(const __grid_constant__ BnParams a) {
    constexpr int ESZ = BF16 ? 2 : 4;
    constexpr int kT = bulkw_threads(CPL);
    constexpr int kWarps = kT / 32;
    constexpr int NB = kBulkWarpRuns;                         // runs in flight per warp
    extern __shared__ __align__(128) unsigned char smem[];   // NB run buffers per warp
    __shared__ uint64_t bar[kWarps][NB];
    const int c0 = a.c_base + blockIdx.x * a.G, s = blockIdx.y;
    const int Gc = min(a.G, a.c_end - c0);
    const int HW = a.HW;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int p0, p1;
    slice_bounds(a, s, p0, p1);
    const uint32_t run_bytes = static_cast<uint32_t>(Gc) * HW * ESZ;
    const int Tc = 1 << a.tc_log2;
    const int part = lane & (Tc - 1);
    const uint32_t e_lo = (static_cast<uint32_t>(HW) * part) >> a.tc_log2;
    const uint32_t e_hi = (static_cast<uint32_t>(HW) * (part + 1)) >> a.tc_log2;
    int cl[CPL];
    float K[CPL], acc_s[CPL], acc_q[CPL];
    pdl_wait_then_release();   // must stay the wait-then-release form: the apply reads x before its own wait
#pragma unroll
    for (int m = 0; m < CPL; ++m) {
        cl[m] = (lane >> a.tc_log2) + (32 >> a.tc_log2) * m;
        K[m] = cl[m] < Gc ? load_elem<BF16>(a.x[0], static_cast<int64_t>(c0 + cl[m]) * HW) : 0.0f;
        acc_s[m] = 0.0f;
        acc_q[m] = 0.0f;
    }
    if (lane == 0) {
        for (int i = 0; i < NB; ++i)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&bar[warp][i])) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncwarp();
    unsigned char* wbuf = smem + static_cast<uint32_t>(warp) * NB * a.slot_bytes;
    const int span = p1 - p0;
    const int nrun = span > warp ? (span - warp + kWarps - 1) / kWarps : 0;
    auto issue = [&](int k) {                                 // lane 0: run k of this warp into buffer k % NB
        const uint32_t pl = static_cast<uint32_t>(p0 + warp + k * kWarps);
        const uint32_t r = fdiv(pl, a.div_batch);
        const uint32_t bb = pl - r * static_cast<uint32_t>(a.batch);
        const uint64_t a0 = (static_cast<uint64_t>(bb) * a.C + c0) * HW * ESZ, a1 = a0 + run_bytes;
        const uint64_t a0al = a0 & ~uint64_t(15);
        const uint64_t hi = min((a1 + 15) & ~uint64_t(15), a.buf_fl);
        unsigned char* dst = wbuf + (k % NB) * a.slot_bytes;
        const char* src = static_cast<const char*>(a.x[r]);
        uint64_t* bp = &bar[warp][k % NB];
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bp)),
                     "r"(static_cast<uint32_t>(hi - a0al))
                     : "memory");
        asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                         smem_u32(dst)),
                     "l"(src + a0al), "r"(static_cast<uint32_t>(hi - a0al)), "r"(smem_u32(bp))
                     : "memory");
        for (uint64_t q = hi; q < a1; q += ESZ) {
            if constexpr (BF16) *reinterpret_cast<unsigned short*>(dst + (q - a0al)) = *reinterpret_cast<const unsigned short*>(src + q);
            else *reinterpret_cast<float*>(dst + (q - a0al)) = *reinterpret_cast<const float*>(src + q);
        }
    };
    if (lane == 0)
        for (int k = 0; k < NB && k < nrun; ++k) issue(k);
    __syncwarp();
    bool failed = false;
    int k = 0;
    for (; k < nrun; ++k) {
        const uint32_t parity = static_cast<uint32_t>(k / NB) & 1u;
        bool to = false;
        if (!mbar_try_wait(&bar[warp][k % NB], parity)) {
            const uint64_t start = global_ns();
            while (!mbar_try_wait(&bar[warp][k % NB], parity)) {
                if (global_ns() - start > kCopyWaitNs) {
                    to = true;
                    break;
                }
            }
        }
        if (__any_sync(0xffffffffu, to)) {
            failed = true;
            break;
        }
        __syncwarp();                                         // lane 0's plain tail stores
        const uint32_t pl = static_cast<uint32_t>(p0 + warp + k * kWarps);
        const uint32_t r = fdiv(pl, a.div_batch);
        const uint32_t bb = pl - r * static_cast<uint32_t>(a.batch);
        const uint32_t pre = static_cast<uint32_t>(((static_cast<uint64_t>(bb) * a.C + c0) * HW * ESZ) & 15u);
        const unsigned char* run = wbuf + (k % NB) * a.slot_bytes;
#pragma unroll
        for (int m = 0; m < CPL; ++m) {
            if (cl[m] < Gc)
                sum_range<BF16>(run, pre + (static_cast<uint32_t>(cl[m]) * HW + e_lo) * ESZ, e_hi - e_lo, K[m],
                                a.vec_reads != 0, acc_s[m], acc_q[m]);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0 && k + NB < nrun) issue(k + NB);
        __syncwarp();
    }
    if (failed) {                                             // let this warp's copies in flight land (bounded)
        for (int j = k; j < nrun && j < k + NB; ++j) {
            const uint32_t parity = static_cast<uint32_t>(j / NB) & 1u;
            const uint64_t start = global_ns();
            while (!mbar_try_wait(&bar[warp][j % NB], parity) && global_ns() - start <= kCopyWaitNs) {
            }
        }
    }
    failed = __syncthreads_or(failed);
    float* red_s = reinterpret_cast<float*>(smem);
    float* red_q = red_s + kWarps * CPL * 32;
#pragma unroll
    for (int m = 0; m < CPL; ++m) {
        red_s[(warp * CPL + m) * 32 + lane] = acc_s[m];
        red_q[(warp * CPL + m) * 32 + lane] = acc_q[m];
    }
    __syncthreads();
    auto combine = [&](int c) {
        const int cps = 32 >> a.tc_log2;
        const int m = c / cps;
        const int l0 = (c % cps) << a.tc_log2;
        const int nl = Tc;
        FF S{0.0f, 0.0f}, Q{0.0f, 0.0f};
        for (int w = 0; w < kWarps; ++w)
            for (int l = l0; l < l0 + nl; ++l) {
                S = ff_add(S, FF{red_s[(w * CPL + m) * 32 + l], 0.0f});
                Q = ff_add(Q, FF{red_q[(w * CPL + m) * 32 + l], 0.0f});
            }
        a.partial[static_cast<int64_t>(c0 + c) * a.S + s] =
            failed ? make_float2(__int_as_float(0x7fc00000), __int_as_float(0x7fc00000))
                   : make_float2(__fadd_rn(S.hi, S.lo), __fadd_rn(Q.hi, Q.lo));
    };
    if constexpr (kT >= kThreads) {                           // G <= kThreads: a thread per channel
        if (threadIdx.x < Gc) combine(threadIdx.x);
    } else {
        for (int c = threadIdx.x; c < Gc; c += kT) combine(c);
    }
}

// Plane kernel, grid (C, S), for H*W a multiple of the 16-byte vector width
// W: CTA (c, s) reduces channel c over its slice of planes.  A warp owns a
// chunk of 64 consecutive vectors of one plane (lane l reads vectors l and
// l + 32 of the chunk: coalesced), so the plane and address arithmetic is
// done once per chunk; each warp handles two chunks per iteration, four
// 16-byte loads in flight per lane.
constexpr int kChunkVecs = 64;

template <bool BF16>
__global__ void __launch_bounds__(kThreads, 5) bn_stats_plane_kernel(const __grid_constant__ BnParams a) {
    constexpr int W = BF16 ? 8 : 4;    // elements per 16-byte access
    constexpr int ESZ = BF16 ? 2 : 4;
    constexpr int kWarps = kThreads / 32;
    const int c = a.c_base + blockIdx.x, s = blockIdx.y;
    const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
    int p0, p1;
    slice_bounds(a, s, p0, p1);
    const uint32_t units = static_cast<uint32_t>(a.HW / W);                     // vectors per plane
    const uint32_t cpp = (units + kChunkVecs - 1) / kChunkVecs;                  // chunks per plane
    const uint32_t total = static_cast<uint32_t>(p1 - p0) * cpp;
    pdl_wait_then_release();   // must stay the wait-then-release form: the apply reads x before its own wait
    const float K = load_elem<BF16>(a.x[0], static_cast<int64_t>(c) * a.HW);   // shift: x[0][0, c, 0, 0]
    // one (Σd, Σd²) pair per element position of the vector: each sums one element per vector (as
    // many terms as a per-vector total would), at one add and one fused multiply-add per element,
    // done two positions per packed f32x2 instruction
    constexpr int NP = W / 2;
    const uint64_t K2 = f2_pack(K, K);
    uint64_t s2[NP], q2[NP];
#pragma unroll
    for (int j = 0; j < NP; ++j) s2[j] = q2[j] = f2_pack(0.0f, 0.0f);
    for (uint32_t ch0 = warp; ch0 < total; ch0 += 2 * kWarps) {
        uint4 raw[2][2];
        bool ok[2][2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const uint32_t ch = ch0 + i * kWarps;                               // warp-uniform
            const uint32_t pl_off = fdiv(ch, a.div_unit);
            const uint32_t cc = ch - pl_off * cpp;
            const uint32_t pl = static_cast<uint32_t>(p0) + pl_off;
            const uint32_t r = fdiv(pl, a.div_batch);
            const uint32_t b = pl - r * static_cast<uint32_t>(a.batch);
            const char* base = static_cast<const char*>(a.x[ch < total ? r : 0]) +
                               (static_cast<int64_t>(b) * a.C + c) * a.HW * ESZ;
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const uint32_t v = cc * kChunkVecs + u * 32 + lane;
                ok[i][u] = ch < total && v < units;
                raw[i][u] = ok[i][u] ? ld16_keep(base + static_cast<int64_t>(v) * 16) : make_uint4(0, 0, 0, 0);
            }
        }
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                if (!ok[i][u]) continue;
#pragma unroll
                for (int j = 0; j < NP; ++j) {
                    const uint64_t d = f2_sub(vec_pair<BF16>(raw[i][u], j), K2);
                    s2[j] = f2_add(s2[j], d);
                    q2[j] = f2_fma(d, d, q2[j]);
                }
            }
    }
    float ps[W], pq[W];
#pragma unroll
    for (int j = 0; j < NP; ++j) {
        f2_unpack(s2[j], ps[2 * j], ps[2 * j + 1]);
        f2_unpack(q2[j], pq[2 * j], pq[2 * j + 1]);
    }
#pragma unroll
    for (int w = W; w > 1; w >>= 1)
#pragma unroll
        for (int k = 0; k < w / 2; ++k) {
            ps[k] = ps[2 * k] + ps[2 * k + 1];
            pq[k] = pq[2 * k] + pq[2 * k + 1];
        }
    FF fs{ps[0], 0.0f}, fq{pq[0], 0.0f};
    block_sum2_ff(fs, fq);
    if (threadIdx.x == 0)
        a.partial[static_cast<int64_t>(c) * a.S + s] = make_float2(__fadd_rn(fs.hi, fs.lo), __fadd_rn(fq.hi, fq.lo));
}

// Element kernel, grid (C, S): planes that are neither vector aligned nor
// small enough to stage (e.g. 111x111); single-element loads.
template <bool BF16>
__global__ void __launch_bounds__(kThreads) bn_stats_element_kernel(const __grid_constant__ BnParams a) {
    const int c = blockIdx.x, s = blockIdx.y;
    int p0, p1;
    slice_bounds(a, s, p0, p1);
    pdl_wait_then_release();   // must stay the wait-then-release form: the apply reads x before its own wait
    const float K = load_elem<BF16>(a.x[0], static_cast<int64_t>(c) * a.HW);
    float acc_s = 0.0f, acc_q = 0.0f;
    for (int pl = p0; pl < p1; ++pl) {
        const int r = pl / a.batch, b = pl - r * a.batch;
        const void* base = static_cast<const char*>(a.x[r]) +
                           (static_cast<int64_t>(b) * a.C + c) * a.HW * (BF16 ? 2 : 4);
        for (int e = threadIdx.x; e < a.HW; e += kThreads) {
            const float d = __fsub_rn(load_elem<BF16>(base, e), K);
            acc_s += d;
            acc_q += d * d;
        }
    }
    FF fs{acc_s, 0.0f}, fq{acc_q, 0.0f};
    block_sum2_ff(fs, fq);
    if (threadIdx.x == 0)
        a.partial[static_cast<int64_t>(c) * a.S + s] = make_float2(__fadd_rn(fs.hi, fs.lo), __fadd_rn(fq.hi, fq.lo));
}

// Float-float product: Dekker's product with the exact low part of
// a.hi·b.hi from a fused multiply-add, plus the cross terms.
__device__ __forceinline__ FF ff_mul(FF a, FF b) {
    const float p = __fmul_rn(a.hi, b.hi);
    const float e = fmaf(a.hi, b.hi, -p);
    const float t = fmaf(a.hi, b.lo, fmaf(a.lo, b.hi, e));
    const float hi = __fadd_rn(p, t);
    return FF{hi, __fsub_rn(t, __fsub_rn(hi, p))};
}

// CTA of 32 warps = 32 channels.  Warp w adds channel (32·blockIdx + w)'s S
// partials in float-float (lane l takes slices l, l + 32, ..., then a fixed
// shuffle tree only as deep as the lanes that hold sums); warp 0 then
// finalises the 32 channels, one per lane, in float-float on the fp32 pipe
// (GB300's fp64 pipe is narrow: a dozen dependent fp64 operations cost more
// than the rest of the merge): m' = Σd/M, mean = K_c + m',
// var = Σd²/M − m'², invstd = 1/sqrt(var + eps) in fp32 with IEEE sqrt and
// divide, and the coefficients (m_hi, scale, shift) with
// shift = β − m_lo·scale rounded once.
constexpr int kMergeThreads = 1024;

template <bool BF16>
__global__ void __launch_bounds__(kMergeThreads) bn_merge_kernel(const __grid_constant__ BnParams a) {
    __shared__ FF sums[2][32];
    const int w = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int c = a.c_base + blockIdx.x * 32 + w;
    const int cc = a.c_base + blockIdx.x * 32 + lane;   // warp 0: the channel this lane finalises
    pdl_enter();
    // warp 0 fetches its channels' shift K, gamma and beta while the partials are summed
    float Kc = 0.0f, gc = 1.0f, bc = 0.0f;
    if (w == 0 && cc < a.c_end) {
        Kc = load_elem<BF16>(a.x[0], static_cast<int64_t>(cc) * a.HW);
        if (a.gamma) gc = a.gamma[cc];
        if (a.beta) bc = a.beta[cc];
    }
    FF S{0.0f, 0.0f}, Q{0.0f, 0.0f};
    if (c < a.c_end) {
        const float2* p = a.partial + static_cast<int64_t>(c) * a.S;
        int s0 = lane;
        for (; s0 + 96 < a.S; s0 += 128) {           // four independent loads in flight
            const float2 v0 = p[s0], v1 = p[s0 + 32], v2 = p[s0 + 64], v3 = p[s0 + 96];
            S = ff_add(ff_add(S, FF{v0.x, 0.0f}), ff_add(FF{v1.x, 0.0f}, ff_add(FF{v2.x, 0.0f}, FF{v3.x, 0.0f})));
            Q = ff_add(ff_add(Q, FF{v0.y, 0.0f}), ff_add(FF{v1.y, 0.0f}, ff_add(FF{v2.y, 0.0f}, FF{v3.y, 0.0f})));
        }
        for (; s0 < a.S; s0 += 32) {
            const float2 v = p[s0];
            S = ff_add(S, FF{v.x, 0.0f});
            Q = ff_add(Q, FF{v.y, 0.0f});
        }
    }
    for (int o = a.tree_top; o > 0; o >>= 1) {    // lanes >= min(S, 32) hold zeros
        S = ff_add(S, ff_shfl_down(S, o));
        Q = ff_add(Q, ff_shfl_down(Q, o));
    }
    if (lane == 0) {
        sums[0][w] = S;
        sums[1][w] = Q;
    }
    __syncthreads();
    if (w != 0 || cc >= a.c_end) return;
    const FF inv{a.inv_hi, a.inv_lo};            // 1/M as a float pair
    const FF ms = ff_mul(sums[0][lane], inv);    // mean of the shifted values
    const FF mean = ff_add(FF{Kc, 0.0f}, ms);
    const FF ms2 = ff_mul(ms, ms);
    const FF var = ff_add(ff_mul(sums[1][lane], inv), FF{-ms2.hi, -ms2.lo});
    const FF ve = ff_add(var, FF{a.eps, 0.0f});
    const float invstd = 1.0f / sqrtf(ve.hi);
    a.mean_out[cc] = mean.hi;
    a.invstd_out[cc] = invstd;
    // y = (x − mean)·scale + β = (x − m_hi)·scale + (β − m_lo·scale): the low part of the mean
    // goes into the shift (one rounding), so x − m_hi is the apply's only subtraction
    const float scale = invstd * gc;
    a.coef[cc] = make_float4(mean.hi, scale, fmaf(-mean.lo, scale, bc), 0.0f);
}

// (x − m_hi)·scale + shift with k = (m_hi, scale, shift, unused)
__device__ __forceinline__ float normalize(float x, float4 k) {
    return fmaf(__fsub_rn(x, k.x), k.y, k.z);
}

// The same for elements (2j, 2j + 1) of a pair, with each element's coefficients
__device__ __forceinline__ uint64_t normalize2(uint64_t x2, const float4& ka, const float4& kb) {
    return f2_fma(f2_sub(x2, f2_pack(ka.x, kb.x)), f2_pack(ka.y, kb.y), f2_pack(ka.z, kb.z));
}

__device__ __forceinline__ uint32_t channel_of(uint32_t e, const BnParams& a) {
    const uint32_t pl = fdiv(e, a.div_hw);
    return pl - fdiv(pl, a.div_c) * static_cast<uint32_t>(a.C);
}

// CMODE: 0 = H*W a multiple of 8 (one channel per 8-element vector);
//        1 = H*W >= 8 (at most one channel boundary inside a vector);
//        2 = H*W < 8 (channel per element);
//        3 = as 1, with the grid stride a whole number of samples: every
//            vector a thread visits sits at the same position of its
//            sample, so the thread finds its channels and packs their
//            coefficients once, before its loop;
//        4 = as 0, over the channels [c_base, c_end) only: the launch's
//            vectors are those channels' runs in each sample;
//        5 = as 3 over the channels [c_base, c_end) only (the part's run in
//            a sample a whole number of vectors, the grid stride a whole
//            number of such runs).
template <bool BF16_IN, bool BF16_OUT, int CMODE, bool NC>
__global__ void __launch_bounds__(kThreads) bn_apply_kernel(const __grid_constant__ BnParams a) {
    // replicas and vectors are visited in the reverse of the statistics pass's order (its last CTAs
    // read the last samples), so the x still in L2 from that pass is read first
    const int r = gridDim.y - 1 - blockIdx.y;
    const char* x = static_cast<const char*>(a.x[r]);
    char* y = static_cast<char*>(a.y[r]);
    constexpr int ISZ = BF16_IN ? 2 : 4, OSZ = BF16_OUT ? 2 : 4;
    const uint32_t E = static_cast<uint32_t>(a.batch) * (a.c_end - a.c_base) * a.HW;   // this launch's elements
    const uint32_t nvec = E / 8;
    const uint32_t stride = gridDim.x * kThreads;
    const uint32_t gtid = blockIdx.x * kThreads + threadIdx.x;
    // vector index within the replica of this launch's vector vr (modes 4 and 5: a part of the
    // channels)
    auto full_vec = [&](uint32_t vr) -> uint32_t {
        if constexpr (CMODE == 4 || CMODE == 5) {
            const uint32_t b = fdiv(vr, a.div_vp);
            return b * a.vs_full + a.v_base + (vr - b * static_cast<uint32_t>(a.div_vp.d));
        }
        return vr;
    };
    // the loads of 4 vectors, issued before any arithmetic
    uint4 raw[4][2];
    auto load4 = [&](uint32_t v0) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const uint32_t v = v0 + u * stride;
            if (v < nvec) {
                const uint32_t vr = full_vec(nvec - 1 - v);   // reverse order
                raw[u][0] = ld16<NC>(x + static_cast<int64_t>(vr) * 8 * ISZ);
                if constexpr (!BF16_IN) raw[u][1] = ld16<NC>(x + static_cast<int64_t>(vr) * 8 * ISZ + 16);
            }
        }
    };
    // the first iteration's x before the wait, overlapping the merge: x depends on no kernel of
    // this call, and the statistics kernel let this one launch only after every earlier kernel
    // in the stream had completed; the coefficients are read after the wait
    if (gtid < nvec) load4(gtid);
    pdl_enter();
    // modes 3 and 5: the coefficient pairs of this thread's element positions (fixed for all its
    // vectors)
    uint64_t M2[4], S2[4], T2[4];
    if constexpr (CMODE == 3 || CMODE == 5) {
        float4 kA = make_float4(0.0f, 0.0f, 0.0f, 0.0f), kB = kA;
        uint32_t eb = 8;
        if (gtid < nvec) {
            const uint32_t vr = nvec - 1 - gtid;
            uint32_t e0;                                    // element offset in the sample
            if constexpr (CMODE == 3) e0 = (vr - fdiv(vr, a.div_vs8) * static_cast<uint32_t>(a.div_vs8.d)) * 8;
            else e0 = (a.v_base + vr - fdiv(vr, a.div_vp) * static_cast<uint32_t>(a.div_vp.d)) * 8;
            const uint32_t cA = fdiv(e0, a.div_hw);
            eb = (cA + 1) * static_cast<uint32_t>(a.HW) - e0;
            kA = __ldg(a.coef + cA);
            kB = eb < 8 ? __ldg(a.coef + cA + 1) : kA;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float4& lo = static_cast<uint32_t>(2 * j) < eb ? kA : kB;
            const float4& hi = static_cast<uint32_t>(2 * j + 1) < eb ? kA : kB;
            M2[j] = f2_pack(lo.x, hi.x);
            S2[j] = f2_pack(lo.y, hi.y);
            T2[j] = f2_pack(lo.z, hi.z);
        }
    }
    for (uint32_t v0 = gtid; v0 < nvec; v0 += 4 * stride) {
        if (v0 != gtid) load4(v0);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const uint32_t v = v0 + u * stride;
            if (v >= nvec) continue;
            const uint32_t e0 = full_vec(nvec - 1 - v) * 8;
            uint64_t xv[4];                                 // element pairs (2j, 2j + 1)
#pragma unroll
            for (int j = 0; j < 4; ++j)
                xv[j] = BF16_IN ? vec_pair<true>(raw[u][0], j) : vec_pair<false>(raw[u][j >> 1], j & 1);
            uint64_t yv2[4];
            if constexpr (CMODE == 0 || CMODE == 4) {
                const float4 k4 = __ldg(a.coef + channel_of(e0, a));
#pragma unroll
                for (int j = 0; j < 4; ++j) yv2[j] = normalize2(xv[j], k4, k4);
            } else if constexpr (CMODE == 1) {
                const uint32_t pl = fdiv(e0, a.div_hw);
                const uint32_t cross = static_cast<uint32_t>(a.HW) - (e0 - pl * static_cast<uint32_t>(a.HW));
                const uint32_t c0 = pl - fdiv(pl, a.div_c) * static_cast<uint32_t>(a.C);
                const float4 k0 = __ldg(a.coef + c0);
                const float4 k1 = cross < 8 ? __ldg(a.coef + (c0 + 1 == static_cast<uint32_t>(a.C) ? 0 : c0 + 1)) : k0;
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    yv2[j] = normalize2(xv[j], static_cast<uint32_t>(2 * j) < cross ? k0 : k1,
                                        static_cast<uint32_t>(2 * j + 1) < cross ? k0 : k1);
            } else if constexpr (CMODE == 3 || CMODE == 5) {
#pragma unroll
                for (int j = 0; j < 4; ++j) yv2[j] = f2_fma(f2_sub(xv[j], M2[j]), S2[j], T2[j]);
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    yv2[j] = normalize2(xv[j], __ldg(a.coef + channel_of(e0 + 2 * j, a)),
                                        __ldg(a.coef + channel_of(e0 + 2 * j + 1, a)));
            }
            float yv[8];
#pragma unroll
            for (int j = 0; j < 4; ++j) f2_unpack(yv2[j], yv[2 * j], yv[2 * j + 1]);
            if constexpr (BF16_OUT) {
                st16(y + static_cast<int64_t>(e0) * OSZ,
                     make_uint4(pack_bf16x2(yv[0], yv[1]), pack_bf16x2(yv[2], yv[3]), pack_bf16x2(yv[4], yv[5]),
                                pack_bf16x2(yv[6], yv[7])));
            } else {
                st16(y + static_cast<int64_t>(e0) * OSZ, f4_bits(yv[0], yv[1], yv[2], yv[3]));
                st16(y + static_cast<int64_t>(e0) * OSZ + 16, f4_bits(yv[4], yv[5], yv[6], yv[7]));
            }
        }
    }
    // tail: E % 8 elements
    const uint32_t t0 = nvec * 8;
    if (gtid < E - t0) {
        const uint32_t e = t0 + gtid;
        const float ye = normalize(load_elem<BF16_IN>(x, e), a.coef[channel_of(e, a)]);
        if constexpr (BF16_OUT) reinterpret_cast<__nv_bfloat16*>(y)[e] = __float2bfloat16_rn(ye);
        else reinterpret_cast<float*>(y)[e] = ye;
    }
}

// ---------------------------------------------------------------- launch planning (host)

// Launch with `smem` bytes of dynamic shared memory and programmatic stream
// serialisation; the opt-in above 48 KiB is set once per kernel and device.
int launch_pdl_smem(void (*kernel)(BnParams), dim3 grid, int smem, cudaStream_t s, const BnParams& p,
                    int block = kThreads) {
    static std::mutex mu;
    static std::map<std::pair<const void*, int>, int> granted;   // (kernel, device) -> bytes allowed
    if (smem > 48 * 1024) {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return cuda_fail(e);
        std::lock_guard<std::mutex> lock(mu);
        auto key = std::make_pair(reinterpret_cast<const void*>(kernel), dev);
        auto it = granted.find(key);
        if (it == granted.end() || it->second < smem) {
            e = cudaFuncSetAttribute(reinterpret_cast<const void*>(kernel), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     smem);
            if (e != cudaSuccess) return cuda_fail(e);
            granted[key] = smem;
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(static_cast<unsigned>(block));
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, p);
    if (e != cudaSuccess) return cuda_fail(e);
    return check_launch();
}

// Channels per lane of the bulk-staged kernel: G * (lanes per channel) / 32.
template <bool BF16>
int launch_bulk(int cpl, dim3 grid, int smem, cudaStream_t s, const BnParams& p) {
    switch (cpl) {
        case 1: return launch_pdl_smem(bn_stats_bulk_kernel<BF16, 1>, grid, smem, s, p);
        case 2: return launch_pdl_smem(bn_stats_bulk_kernel<BF16, 2>, grid, smem, s, p);
        case 4: return launch_pdl_smem(bn_stats_bulk_kernel<BF16, 4>, grid, smem, s, p);
        default: return launch_pdl_smem(bn_stats_bulk_kernel<BF16, 8>, grid, smem, s, p);
    }
}

template <bool BF16>
int launch_bulkw(int cpl, dim3 grid, int smem, cudaStream_t s, const BnParams& p) {
    switch (cpl) {
        case 1: return launch_pdl_smem(bn_stats_bulkw_kernel<BF16, 1>, grid, smem, s, p, bulkw_threads(1));
        case 2: return launch_pdl_smem(bn_stats_bulkw_kernel<BF16, 2>, grid, smem, s, p, bulkw_threads(2));
        case 4: return launch_pdl_smem(bn_stats_bulkw_kernel<BF16, 4>, grid, smem, s, p, bulkw_threads(4));
        default: return launch_pdl_smem(bn_stats_bulkw_kernel<BF16, 8>, grid, smem, s, p, bulkw_threads(8));
    }
}

enum StatsKind { kPlaneVec, kPlaneScalar, kBulk, kBulkWarp, kStaged };

struct StatsPlan {
    StatsKind kind;
    int G, S, R, slot_bytes;
    int smem;           // bulk kernel: dynamic shared bytes (two tile buffers)
    int tc_log2, cpl;   // bulk kernel: log2 of the lanes per channel, channels per lane
    bool split;         // the call runs as two channel halves on two streams
    bool vec_reads;     // bulk kernel: every lane's range starts on a 16-byte boundary of its run
};

// Slices of the bulk kernel: about one resident wave of CTAs, so that each
// CTA streams several tiles through its two buffers.  kWaveSms is GB300's
// SM count; on another part only the slice count (not the result's
// correctness) depends on it.
constexpr int kWaveSms = 152;

int bulk_slices(int n_groups, int P, int C, int smem, int cpl, int ctas_per_256) {
    int per_sm = (227 * 1024) / (smem + 1024);              // shared memory per SM, 1 KiB reserved per CTA
    // registers: 6 CTAs of 256 threads with one channel per lane (40 registers), 5 with two (48),
    // 4 with four or eight (59-64); twice as many CTAs of 128 threads
    const int reg_cap = (cpl >= 4 ? 4 : (cpl == 2 ? 5 : 6)) * ctas_per_256;
    if (per_sm > reg_cap) per_sm = reg_cap;
    if (per_sm < 1) per_sm = 1;
    int64_t S = static_cast<int64_t>(kWaveSms) * per_sm / n_groups;
    if (S > P) S = P;
    const int64_t cap = kMaxPartials / C;
    if (S > cap) S = cap;
    if (S < 1) S = 1;
    return static_cast<int>(S);
}

int pow2_floor(int v) {
    int p = 1;
    while (p * 2 <= v) p *= 2;
    return p;
}

// Channels per group of the group kernel: the largest power of two <= 256
// with G*H*W <= kRunElems (at least 1), and no larger than C allows.
int group_channels(int C, int HW) {
    int G = 1;
    while (G < kThreads && static_cast<int64_t>(2 * G) * HW <= kRunElems) G *= 2;
    const int cap = pow2_floor(C);
    return G < cap ? G : cap;
}

int slices_for(int n_groups, int P, int C) {
    int64_t S = (kTargetCtas + n_groups - 1) / n_groups;
    if (S > P) S = P;
    const int64_t cap = kMaxPartials / C;
    if (S > cap) S = cap;
    if (S < 1) S = 1;
    return static_cast<int>(S);
}

int slot_bytes_for(int G, int HW, int esz) {
    return static_cast<int>((static_cast<int64_t>(G) * HW * esz + 14 + 15) / 16 * 16);
}

// Whether a call runs as two channel halves on two streams (the first half's
// statistics, merge and apply on the caller's stream, the second half's on a
// side stream), so that each half's launches fill the other's gaps: the
// three launches of a call depend on each other, and between them the
// memory idles through a grid's drain, the merge and the next ramp.  Taken
// where the input over all replicas is large enough and the channels split
// evenly into whole statistics units: aligned planes with the plane kernel
// (even C, halves of at least 16 channels, 16 MiB), and unaligned planes
// with the per-warp bulk-staged kernel (halves of whole channel groups whose
// run in a sample is a whole number of 16-byte vectors, 32 MiB).  Measured
// on 8 x [32, C, H, W] bf16 with inputs rotated past L2 (us per call, one
// sequence -> two halves): 64x56x56 46.1 -> 45.5, 256x56x56 188.5 -> 181.9,
// 512x28x28 95.9 -> 92.0, 64x28x28 22.9 -> 19.7, 2048x7x7 27.9 -> 25.4,
// 1024x14x14 52.3 -> 49.3; 256x14x14 (26 MB) gained nothing, and short
// aligned planes on the bulk kernel lost (2048x8x8 41.1 -> 43.6, 8192x4x4
// 41.0 -> 43.0).  Both halves
// use one slice count, fitted to a half, so the sums, and every output bit,
// are those of the call run as one sequence with that count.
constexpr int64_t kSplitMinBytes = int64_t(16) << 20;       // x over all replicas, plane statistics
constexpr int64_t kSplitBulkMinBytes = int64_t(32) << 20;   // x over all replicas, bulk-staged statistics
constexpr int kSplitMinChannels = 16;                         // per half

// Aligned planes of at least kPlaneMinVecs vectors: plane kernel with
// 16-byte loads.  A warp reads 64-vector chunks of one plane, so shorter
// planes leave lanes idle; measured on 8 x [32, C, H, W] bf16 with about
// 67 MB of input, plane kernel against bulk-staged kernel (us per call):
// 4x4 203 / 46, 4x8 113 / 46, 8x8 70 / 47, 8x16 47 / 48, 16x16 36 / 52,
// 16x24 30 / 36.  Shorter aligned bf16 planes and unaligned planes at
// least one vector long: bulk-staged kernel (runs of G channels).
// Short aligned fp32 planes stay with the plane kernel: there a lane adds
// fewer fp32 values per accumulator (the bulk kernel adds a lane's whole
// plane into one pair, and on fp32 2x4 planes its means were off by up to
// 1.5e-7 standard deviations; bf16 differences add exactly).  Planes
// shorter than a vector: staged group kernel.  Unaligned planes too long to
// fit a group's run in the shared buffer: plane kernel with element loads.
StatsPlan plan_stats(int n, int batch, int C, int HW, int esz) {
    StatsPlan sp{};
    const int P = n * batch;
    const int W = 16 / esz;
    const int G = group_channels(C, HW);
    const int slot = slot_bytes_for(G, HW, esz);
    const bool fits = slot <= kStageBytes;
    if (HW % W == 0 && (HW / W >= kPlaneMinVecs || esz == 4 || !fits)) sp.kind = kPlaneVec;
    else if (!fits) sp.kind = kPlaneScalar;
    else sp.kind = HW >= W ? kBulk : kStaged;
    if (sp.kind == kBulk) {
        sp.G = G;
        sp.slot_bytes = slot;
        sp.R = kBulkBufMax / slot < kBulkRuns ? kBulkBufMax / slot : kBulkRuns;
        // lanes per channel: 32/G for G < 32 (each a contiguous part of the plane), else one; on
        // short aligned planes, up to one 16-byte vector per lane where the plane's vector count
        // allows (at most 8 channels per lane), so that eight lanes read 128 contiguous bytes of
        // shared memory: with a lane per channel, every lane of a warp read the same bank on
        // 128-byte planes (8x8 bf16: 85 us per call against 47)
        int tl = 0;
        while ((G << tl) < 32) ++tl;
        if (HW % W == 0) {
            const int vp = HW / W;
            int t = 0;
            while (t < 5 && vp % (2 << t) == 0 && (G << (t + 1)) <= 32 * 8) ++t;
            if (t > tl) tl = t;
        }
        sp.tc_log2 = tl;
        sp.cpl = (G << tl) / 32;
        // aligned runs and parts of whole 16-byte vectors: warp-uniform, so no lane takes the
        // other loop (on 7x7 planes, per-lane alignment tests cost 28.3 -> 32.7 us)
        sp.vec_reads = esz == 2 && HW % W == 0 && (HW / W) % (1 << tl) == 0;
        const int red = kThreads * sp.cpl * 2 * static_cast<int>(sizeof(float));
        if ((kThreads / 32) * kBulkWarpRuns * slot <= kBulkWarpMaxSmem) {
            sp.kind = kBulkWarp;
            const int bt = bulkw_threads(sp.cpl);
            const int warp_bufs = (bt / 32) * kBulkWarpRuns * slot;
            const int redw = bt * sp.cpl * 2 * static_cast<int>(sizeof(float));
            sp.smem = warp_bufs > redw ? warp_bufs : redw;
        } else {
            sp.smem = 2 * sp.R * slot > red ? 2 * sp.R * slot : red;
        }
        const int64_t bytes = static_cast<int64_t>(n) * batch * C * HW * esz;
        sp.split = sp.kind == kBulkWarp && HW % W != 0 && C % 2 == 0 && C / 2 >= kSplitMinChannels &&
                   (C / 2) % G == 0 && (static_cast<int64_t>(C / 2) * HW) % 8 == 0 && bytes >= kSplitBulkMinBytes;
        sp.S = bulk_slices(((sp.split ? C / 2 : C) + G - 1) / G, P, C, sp.smem, sp.cpl,
                           sp.kind == kBulkWarp ? kThreads / bulkw_threads(sp.cpl) : 1);
    } else if (sp.kind == kStaged) {
        sp.G = G;
        sp.slot_bytes = slot;
        sp.R = kStageBytes / slot;
        sp.S = slices_for((C + G - 1) / G, P, C);
    } else {
        sp.G = 1;
        sp.slot_bytes = 0;
        sp.R = 0;
        sp.S = slices_for(C, P, C);
        if (sp.kind == kPlaneVec) {
            // slices by work per thread, about kPlaneVecsPerThread 16-byte vectors each (measured on
            // 8 x [32,C,56|28,..] bf16: 24 beat the fixed CTA target, 8-12 and 32 were slower)
            const int64_t vecs = static_cast<int64_t>(P) * (HW / W);
            int64_t S = vecs / (static_cast<int64_t>(kThreads) * kPlaneVecsPerThread);
            if (S > P) S = P;
            if (S > kMaxPartials / C) S = kMaxPartials / C;
            if (S < 1) S = 1;
            sp.S = static_cast<int>(S);
            sp.split = HW % 8 == 0 && C % 2 == 0 && C / 2 >= kSplitMinChannels &&
                       static_cast<int64_t>(n) * batch * C * HW * esz >= kSplitMinBytes;
        }
    }
    return sp;
}

// Slice count of the plane kernel within [ceil(cap/2), cap] that fills its
// last wave of resident CTAs best: the smallest ceil(C*S / wave) / (C*S),
// the larger S on ties.  (Measured on 8 x [32,C,H,W] bf16 with 760 resident
// CTAs: 64x56x56 ran at 0.93 of copy bandwidth with 11 slices, one wave,
// against 0.86 with 16, two waves of which the second was a third full.)
int plane_slices_for_wave(int C, int cap, int64_t wave) {
    int best = cap;
    int64_t best_w = 0, best_g = 1;   // ceil(grid / wave) and grid of the best so far
    for (int S = cap; S >= (cap + 1) / 2; --S) {
        const int64_t g = static_cast<int64_t>(C) * S;
        const int64_t w = (g + wave - 1) / wave;
        if (best_w == 0 || w * best_g < best_w * g) {
            best = S;
            best_w = w;
            best_g = g;
        }
    }
    return best;
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

// Partials needed by any plan of these sizes (fp32 or bf16 input).
int64_t max_partials(int32_t n, int32_t batch, int32_t C, int32_t HW) {
    int64_t m = 0;
    for (int esz : {2, 4}) {
        const StatsPlan sp = plan_stats(n, batch, C, HW, esz);
        const int64_t v = static_cast<int64_t>(C) * sp.S;
        if (v > m) m = v;
    }
    return m;
}

template <bool BF16_IN, bool BF16_OUT, int CMODE>
int launch_apply_mode(const BnParams& p, bool nc, dim3 grid, cudaStream_t s) {
    if (nc) return launch_pdl(bn_apply_kernel<BF16_IN, BF16_OUT, CMODE, true>, grid, kThreads, s, p);
    return launch_pdl(bn_apply_kernel<BF16_IN, BF16_OUT, CMODE, false>, grid, kThreads, s, p);
}

template <bool BF16_IN, bool BF16_OUT>
int launch_apply(const BnParams& p, int cmode, bool nc, dim3 grid, cudaStream_t s) {
    if (cmode == 0) return launch_apply_mode<BF16_IN, BF16_OUT, 0>(p, nc, grid, s);
    if (cmode == 1) return launch_apply_mode<BF16_IN, BF16_OUT, 1>(p, nc, grid, s);
    if (cmode == 3) return launch_apply_mode<BF16_IN, BF16_OUT, 3>(p, nc, grid, s);
    if (cmode == 4) return launch_apply_mode<BF16_IN, BF16_OUT, 4>(p, nc, grid, s);
    if (cmode == 5) return launch_apply_mode<BF16_IN, BF16_OUT, 5>(p, nc, grid, s);
    return launch_apply_mode<BF16_IN, BF16_OUT, 2>(p, nc, grid, s);
}


bool split_channels(const StatsPlan& sp) { return sp.split; }

// A side stream and its fork and join events, one per host thread and
// device, created on the thread's first split call outside stream capture
// (a call that finds none while its stream is capturing runs unsplit, with
// the same results).  Destroyed when the thread exits; stale after
// cudaDeviceReset.
struct SideStream {
    cudaStream_t s = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
    ~SideStream() {
        if (s) cudaStreamDestroy(s);
        if (fork) cudaEventDestroy(fork);
        if (join) cudaEventDestroy(join);
    }
};
constexpr int kMaxSideDevices = 64;

SideStream* side_stream(cudaStream_t caller) {
    thread_local SideStream table[kMaxSideDevices];
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    if (dev < 0 || dev >= kMaxSideDevices) return nullptr;
    SideStream& h = table[dev];
    if (h.s != nullptr) return &h;
    // a failed query or creation leaves no error behind for the launches' own checks to report
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(caller, &cs) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    if (cs != cudaStreamCaptureStatusNone) return nullptr;
    cudaStream_t st = nullptr;
    cudaEvent_t f = nullptr, j = nullptr;
    if (cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&f, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&j, cudaEventDisableTiming) != cudaSuccess) {
        (void)cudaGetLastError();
        if (st) cudaStreamDestroy(st);
        if (f) cudaEventDestroy(f);
        return nullptr;
    }
    h.s = st;
    h.fork = f;
    h.join = j;
    return &h;
}

// The three launches of a call (statistics, merge, apply) for the channels
// [p.c_base, p.c_end), on stream s.
int launch_sequence(BnParams p, const StatsPlan& sp, bool bf16_in, bool bf16_out, bool nc, cudaStream_t s) {
    int st;
    if (sp.kind == kBulk || sp.kind == kBulkWarp || sp.kind == kStaged) {
        p.div_unit = make_fastdiv(static_cast<uint32_t>(sp.slot_bytes / 16));
        const dim3 grid(static_cast<unsigned>((p.c_end - p.c_base + sp.G - 1) / sp.G), static_cast<unsigned>(sp.S));
        if (sp.kind == kBulk)
            st = bf16_in ? launch_bulk<true>(sp.cpl, grid, sp.smem, s, p) : launch_bulk<false>(sp.cpl, grid, sp.smem, s, p);
        else if (sp.kind == kBulkWarp)
            st = bf16_in ? launch_bulkw<true>(sp.cpl, grid, sp.smem, s, p) : launch_bulkw<false>(sp.cpl, grid, sp.smem, s, p);
        else
            st = bf16_in ? launch_pdl(bn_stats_group_kernel<true>, grid, kThreads, s, p)
                         : launch_pdl(bn_stats_group_kernel<false>, grid, kThreads, s, p);
    } else {
        const int wv = bf16_in ? 8 : 4;             // elements per 16-byte vector
        const dim3 grid(static_cast<unsigned>(p.c_end - p.c_base), static_cast<unsigned>(sp.S));
        if (sp.kind == kPlaneVec) {
            const uint32_t units = static_cast<uint32_t>(p.HW / wv);
            p.div_unit = make_fastdiv((units + kChunkVecs - 1) / kChunkVecs);
            st = bf16_in ? launch_pdl(bn_stats_plane_kernel<true>, grid, kThreads, s, p)
                         : launch_pdl(bn_stats_plane_kernel<false>, grid, kThreads, s, p);
        } else {
            st = bf16_in ? launch_pdl(bn_stats_element_kernel<true>, grid, kThreads, s, p)
                         : launch_pdl(bn_stats_element_kernel<false>, grid, kThreads, s, p);
        }
    }
    if (st != DDP_OK) return st;
    const dim3 mgrid(static_cast<unsigned>((p.c_end - p.c_base + 31) / 32));
    st = bf16_in ? launch_pdl(bn_merge_kernel<true>, mgrid, kMergeThreads, s, p)
                 : launch_pdl(bn_merge_kernel<false>, mgrid, kMergeThreads, s, p);
    if (st != DDP_OK) return st;

    DeviceInfo d;
    if ((st = current_device_info(&d)) != DDP_OK) return st;
    const int64_t nvec = static_cast<int64_t>(p.batch) * (p.c_end - p.c_base) * p.HW / 8;
    // at least kApplyVecs vectors per thread (two passes of its 4-vector unroll), and at most
    // kApplyWaves waves counted at the SM's thread limit (8 CTAs of 256 threads; registers
    // allow 5-6, so the grid runs more real waves): several waves stream faster than one
    // grid-stride wave, and grids rounded to whole real waves measured slower
    int64_t gx = (nvec + static_cast<int64_t>(kThreads) * kApplyVecs - 1) / (static_cast<int64_t>(kThreads) * kApplyVecs);
    const int64_t resident = static_cast<int64_t>(d.sm_count) * (d.max_threads_per_sm / kThreads);
    int64_t cap = (kApplyWaves * resident + p.n - 1) / p.n;
    if (gx > cap) gx = cap;
    if (gx < 1) gx = 1;
    int cmode = (p.HW % 8) == 0 ? (p.parted ? 4 : 0) : (p.HW >= 8 ? 1 : 2);
    const int64_t run_elems = static_cast<int64_t>(p.c_end - p.c_base) * p.HW;   // a sample's run of this launch
    if (cmode == 1 && run_elems % 8 == 0) {
        // mode 3 (5 for a part): a grid stride (gx*kThreads vectors) that is a whole number of the
        // launch's runs, with gx the multiple of the smallest such count nearest to the size
        // chosen above (a part is split off only where its run is a whole number of vectors)
        const int64_t vs8 = run_elems / 8;
        int64_t gcd = kThreads, tmp = vs8;
        while (tmp != 0) {                                  // gcd(kThreads, vs8)
            const int64_t q = gcd % tmp;
            gcd = tmp;
            tmp = q;
        }
        const int64_t m0 = vs8 / gcd;                       // CTAs per whole number of samples
        int64_t g3 = (gx + m0 / 2) / m0 * m0;
        if (g3 < m0) g3 = m0;
        if (g3 <= 2 * gx + m0 && g3 * kThreads <= (int64_t(1) << 31) / 4) {
            gx = g3;
            cmode = p.parted ? 5 : 3;
            p.div_vs8 = make_fastdiv(static_cast<uint32_t>(vs8));
        }
    }
    if (p.parted && cmode != 4 && cmode != 5) return DDP_ERR_UNSUPPORTED;   // excluded by the split rule
    const dim3 agrid(static_cast<unsigned>(gx), static_cast<unsigned>(p.n));
    if (bf16_in) return bf16_out ? launch_apply<true, true>(p, cmode, nc, agrid, s) : launch_apply<true, false>(p, cmode, nc, agrid, s);
    return bf16_out ? launch_apply<false, true>(p, cmode, nc, agrid, s) : launch_apply<false, false>(p, cmode, nc, agrid, s);
}

}  // namespace
}  // namespace ddp

using namespace ddp;

extern "C" size_t syncbn_workspace_bytes(int32_t n_replicas, int32_t batch, int32_t C, int32_t H, int32_t W) {
    if (!valid_sizes(n_replicas, batch, C, H, W)) return 0;
    const int64_t parts = max_partials(n_replicas, batch, C, H * W);
    return align_up(static_cast<size_t>(parts) * sizeof(float2), 16) + static_cast<size_t>(C) * sizeof(float4);
}

extern "C" int syncbn_channel_parts(int32_t n_replicas, int32_t in_dtype, int32_t batch, int32_t C, int32_t H,
                                    int32_t W) {
    if (!valid_sizes(n_replicas, batch, C, H, W) || (in_dtype != DDP_F32 && in_dtype != DDP_BF16))
        return DDP_ERR_INVALID_ARG;
    const int esz = in_dtype == DDP_BF16 ? 2 : 4;
    const StatsPlan sp = plan_stats(n_replicas, batch, C, H * W, esz);
    return split_channels(sp) ? 2 : 1;
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

    const bool bf16_in = in_dtype == DDP_BF16;
    const int esz = bf16_in ? 2 : 4;
    StatsPlan sp = plan_stats(n_replicas, batch, C, H * W, esz);
    const bool split = split_channels(sp);
    int st;
    if (sp.kind == kPlaneVec) {
        // the plan's slice count sizes the workspace; the launch may take fewer to end on a full wave
        DeviceInfo d;
        if ((st = current_device_info(&d)) != DDP_OK) return st;
        int per_sm = 1;
        st = resident_blocks_per_sm(bf16_in ? reinterpret_cast<const void*>(bn_stats_plane_kernel<true>)
                                            : reinterpret_cast<const void*>(bn_stats_plane_kernel<false>),
                                    kThreads, &per_sm);
        if (st != DDP_OK) return st;
        // a split call fits the wave of each half, and runs with that slice count also where it
        // finds no side stream (then as one sequence, with the same sums)
        sp.S = plane_slices_for_wave(split ? C / 2 : C, sp.S, static_cast<int64_t>(d.sm_count) * per_sm);
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
    p.S = sp.S;
    p.G = sp.G;
    p.R = sp.R;
    p.slot_bytes = sp.slot_bytes;
    p.buf_fl = (static_cast<uint64_t>(batch) * C * p.HW * esz) & ~uint64_t(15);
    p.tc_log2 = sp.tc_log2;
    p.vec_reads = sp.vec_reads ? 1 : 0;
    p.eps = eps;
    const double inv_count = 1.0 / (static_cast<double>(n_replicas) * batch * p.HW);
    p.inv_hi = static_cast<float>(inv_count);
    p.inv_lo = static_cast<float>(inv_count - static_cast<double>(p.inv_hi));
    const int lanes = sp.S < 32 ? sp.S : 32;      // lanes of a merge warp that hold sums
    int top = 1;
    while (top < lanes) top *= 2;
    p.tree_top = top / 2;                           // 0 for a single slice
    char* ws = static_cast<char*>(workspace);
    p.partial = reinterpret_cast<float2*>(ws);
    ws += align_up(static_cast<size_t>(C) * p.S * sizeof(float2), 16);
    p.coef = reinterpret_cast<float4*>(ws);
    p.div_batch = make_fastdiv(static_cast<uint32_t>(batch));
    p.ps_small = static_cast<int64_t>(n_replicas) * batch * sp.S < (int64_t(1) << 31) ? 1 : 0;
    if (p.ps_small) p.div_s = make_fastdiv(static_cast<uint32_t>(sp.S));
    p.div_hw = make_fastdiv(static_cast<uint32_t>(p.HW));
    p.div_c = make_fastdiv(static_cast<uint32_t>(C));

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool nc = !in_place_any;
    const bool bf16_out = out_dtype == DDP_BF16;
    p.c_base = 0;
    p.c_end = C;
    SideStream* side = nullptr;
    if (split) side = side_stream(s);
    if (side == nullptr) return launch_sequence(p, sp, bf16_in, bf16_out, nc, s);

    // two channel halves, the second on the side stream: each half's merge and apply overlap the
    // other's statistics and apply instead of leaving the memory idle between the launches
    BnParams q = p;
    const int half = C / 2;
    p.c_end = half;
    q.c_base = half;
    for (BnParams* h : {&p, &q}) {
        h->parted = 1;
        h->div_vp = make_fastdiv(static_cast<uint32_t>(static_cast<int64_t>(half) * p.HW / 8));
        h->vs_full = static_cast<uint32_t>(static_cast<int64_t>(C) * p.HW / 8);
        h->v_base = static_cast<uint32_t>(static_cast<int64_t>(h->c_base) * p.HW / 8);
    }
    cudaError_t e = cudaEventRecord(side->fork, s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(side->s, side->fork, 0);
    if (e != cudaSuccess) return cuda_fail(e);
    st = launch_sequence(p, sp, bf16_in, bf16_out, nc, s);
    if (st == DDP_OK) st = launch_sequence(q, sp, bf16_in, bf16_out, nc, side->s);
    // the join is recorded whatever happened, so that the caller's stream (or its capture) never
    // leaves the side stream's work unjoined
    e = cudaEventRecord(side->join, side->s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, side->join, 0);
    if (st != DDP_OK) return st;
    return e == cudaSuccess ? DDP_OK : cuda_fail(e);
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
// per device (with that device current) and cached for the life of the
// process.  A cudaDeviceReset of that device leaves the cached address stale
// (the module is loaded again into a new context), so this entry point is not
// for processes that reset a device and keep using it.
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
    // only the bytes this call needs are handed on, so the capacity and overlap checks cover exactly those
    return syncbn_merge_apply(x, n_replicas, in_dtype, batch, C, H, W, eps, gamma, beta, y, out_dtype, mean_out,
                              invstd_out, ws, need, stream);
}
