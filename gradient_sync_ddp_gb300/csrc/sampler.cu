// DistributedSampler index lists, one thread per output index.
//
// AI_Infra notes "1.DataParallel / DDP" §4.4: num_samples = ceil(n/N) (or
// floor with drop_last), total = num_samples*N; the list 0..n-1 is shuffled
// with a generator seeded by seed+epoch (the same on every rank, so no
// communication is needed), padded by repeating its head up to total (or cut
// to total), and rank r takes positions r, r+N, r+2N, ...
//
// The shuffle is a keyed permutation that any thread evaluates for any
// position on its own: a 4-round Feistel network on bits = ceil(log2 n) bits
// (halves of ceil(bits/2) and floor(bits/2) bits, so the domain is below 2n;
// for n < 2^62 each half fits in 31 bits), round keys = the high 32 bits of
// the first four SplitMix64 outputs from state seed+epoch (Steele, Lea &
// Flood, OOPSLA 2014), round function = the MurmurHash3 32-bit finalizer
// (Appleby) truncated to the half's width, and cycle walking (encrypt again
// while the value is >= n; under two encryptions per index on average).
// Each walk is bounded: after 4096 encryptions the output is -1 and the
// index is counted in a status word instead of looping on.  The kernel is
// integer-ALU bound (4 rounds x 2 32-bit multiplies per encryption); the
// 8-byte output per index is its only memory traffic.
#include <cstdint>

#include "common.cuh"
#include "host_common.h"

namespace ddp {
namespace {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;
constexpr int kRounds = 4;
constexpr int kWalkCap = 4096;
constexpr int kBlocksPerSm = 2;                    // target CTAs per SM (fewer if occupancy caps it)
constexpr int kWalks = 1;                          // independent walks per lane
constexpr int64_t kMinItemsPerWarp = 64;
constexpr int kWarpsPerBlock = kThreads / 32;

struct SamplerParams {
    int64_t* out;
    int32_t* status;
    uint32_t rk[kRounds];
    uint64_t n;          // items
    uint32_t mask_hi;    // 2^h_hi - 1
    uint32_t mask_lo;    // 2^h_lo - 1
    int64_t ns;          // num_samples
    int64_t count;       // outputs to write
    int64_t per_warp;    // slots per pool
    int64_t pools;       // ceil(count / per_warp)
    FastDiv ns_div;      // division by ns, valid when small != 0
    int32_t small;       // count < 2^31
    int32_t N;           // replicas
    int32_t rank;        // -1: all ranks, rank-major
    int32_t h_lo;        // width of the low half
    int32_t shuffle;
};

uint64_t splitmix64_mix(uint64_t z) {
    z ^= z >> 30;
    z *= 0xBF58476D1CE4E5B9ull;
    z ^= z >> 27;
    z *= 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

__device__ __forceinline__ uint32_t fmix32(uint32_t h) {
    h ^= h >> 16;
    h *= 0x85EBCA6Bu;
    h ^= h >> 13;
    h *= 0xC2B2AE35u;
    return h ^ (h >> 16);
}

// x = (H, L) with H the high ceil(bits/2) bits and L the low floor(bits/2)
// bits; even rounds H ^= fmix32(L ^ k_i) mod 2^|H|, odd rounds L ^= fmix32(H
// ^ k_i) mod 2^|L|.  Every round undoes itself, so the pass is a bijection.
template <typename U>
__device__ __forceinline__ U encrypt(U x, const SamplerParams& a) {
    uint32_t H = static_cast<uint32_t>(x >> a.h_lo), L = static_cast<uint32_t>(x) & a.mask_lo;
#pragma unroll
    for (int i = 0; i < kRounds; ++i) {
        if (i % 2 == 0) H ^= fmix32(L ^ a.rk[i]) & a.mask_hi;
        else L ^= fmix32(H ^ a.rk[i]) & a.mask_lo;
    }
    return (static_cast<U>(H) << a.h_lo) | L;
}

// Output slot i -> unshuffled index: slot (r, s) of the rank-major output
// holds padded-list position r + s*N; padding repeats the head.  U = uint32_t
// is used only when n <= 2^31 and count < 2^31; then every position is below
// total < n + N < 2^32 and the whole computation fits 32 bits.
template <typename U>
__device__ __forceinline__ U base_index(int64_t i, const SamplerParams& a) {
    U r, s;
    if (a.rank >= 0) {
        r = static_cast<U>(a.rank);
        s = static_cast<U>(i);
    } else {
        if constexpr (sizeof(U) == 4) r = fdiv(static_cast<uint32_t>(i), a.ns_div);
        else r = static_cast<U>(i / a.ns);
        s = static_cast<U>(i) - r * static_cast<U>(a.ns);
    }
    const U pos = r + s * static_cast<U>(a.N);
    const U n = static_cast<U>(a.n);
    if (pos < n) return pos;
    return pos - n < n ? pos - n : pos % n;    // pos >= 2n only when N > n
}

// Warps take pools of per_warp consecutive output slots (grid-stride over
// pools; the host sizes pools so that the grid is kBlocksPerSm CTAs on every
// SM).  Each lane carries kWalks independent cycle walks, so a warp acts as
// 32*kWalks virtual lanes and two dependency chains interleave.  Walk
// lengths are geometric: instead of idling until the slowest walk of the
// warp has finished, a virtual lane whose walk ends writes its index and
// takes the pool's next unclaimed slot (ballot + prefix count), so every
// iteration is one encryption per virtual lane until the pool runs dry.  The
// body is written with selects rather than branches; lanes without a slot
// compute on a clamped copy and store nothing.
template <typename U>
__global__ void __launch_bounds__(kThreads) sampler_kernel(const __grid_constant__ SamplerParams a) {
    const int lane = threadIdx.x & 31;
    const unsigned lanes_below = (1u << lane) - 1u;
    const U n = static_cast<U>(a.n);
    const int64_t warps = static_cast<int64_t>(gridDim.x) * kWarpsPerBlock;
    for (int64_t pool = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) / 32; pool < a.pools;
         pool += warps) {
        const int64_t begin = pool * a.per_warp;
        const int32_t len = static_cast<int32_t>(min(a.per_warp, a.count - begin));
        int64_t* out = a.out + begin;
        if (!(a.shuffle && a.n > 1)) {
            for (int32_t o = lane; o < len; o += 32) out[o] = static_cast<int64_t>(base_index<U>(begin + o, a));
            continue;
        }
        int32_t off[kWalks];                       // slot of each walk, relative to begin
        U y[kWalks];
        int32_t steps[kWalks];                     // encryptions applied to y
        bool live[kWalks];
#pragma unroll
        for (int v = 0; v < kWalks; ++v) {
            off[v] = v * 32 + lane;
            live[v] = off[v] < len;
            y[v] = base_index<U>(begin + min(off[v], len - 1), a);
            steps[v] = 0;
        }
        int32_t next = 32 * kWalks;                // first unclaimed slot of the pool
        while (true) {
            bool any_live = false;
#pragma unroll
            for (int v = 0; v < kWalks; ++v) any_live |= live[v];
            if (!__any_sync(0xffffffffu, any_live)) break;
            bool done[kWalks];
            int capped = 0;
#pragma unroll
            for (int v = 0; v < kWalks; ++v) {
                y[v] = encrypt<U>(y[v], a);
                ++steps[v];
                const bool hit = y[v] < n;
                done[v] = live[v] && (hit || steps[v] >= kWalkCap);
                if (done[v]) out[off[v]] = hit ? static_cast<int64_t>(y[v]) : int64_t(-1);
                capped += (done[v] && !hit) ? 1 : 0;
            }
            if (capped && a.status) atomicAdd(a.status, capped);   // walk bound reached: never observed
#pragma unroll
            for (int v = 0; v < kWalks; ++v) {
                const unsigned fin = __ballot_sync(0xffffffffu, done[v]);
                const int32_t o = next + __popc(fin & lanes_below);
                next += __popc(fin);
                const U yb = base_index<U>(begin + min(o, len - 1), a);
                off[v] = done[v] ? o : off[v];
                live[v] = done[v] ? o < len : live[v];
                y[v] = done[v] ? yb : y[v];
                steps[v] = done[v] ? 0 : steps[v];
            }
        }
    }
}

}  // namespace
}  // namespace ddp

using namespace ddp;

extern "C" int64_t dist_sampler_num_samples(int64_t n_items, int32_t n_replicas, int32_t drop_last) {
    if (n_items < 0 || n_items >= (int64_t(1) << 62) || n_replicas < 1 || (drop_last != 0 && drop_last != 1))
        return -1;
    return drop_last ? n_items / n_replicas : (n_items + n_replicas - 1) / n_replicas;
}

extern "C" int dist_sampler_indices(int64_t n_items, int32_t n_replicas, int32_t rank,
                                    uint64_t seed, uint64_t epoch, int32_t shuffle, int32_t drop_last,
                                    int64_t* out, int64_t out_capacity, int64_t* num_samples_out,
                                    int32_t* walk_status, void* stream) {
    if (num_samples_out == nullptr) return DDP_ERR_INVALID_ARG;
    if (shuffle != 0 && shuffle != 1) return DDP_ERR_INVALID_ARG;
    const int64_t ns = dist_sampler_num_samples(n_items, n_replicas, drop_last);
    if (ns < 0 || rank < -1 || rank >= n_replicas || out_capacity < 0) return DDP_ERR_INVALID_ARG;
    *num_samples_out = ns;
    const int64_t count = rank >= 0 ? ns : ns * n_replicas;
    if (out_capacity < count) return DDP_ERR_CAPACITY;
    if (count > 0 && out == nullptr) return DDP_ERR_INVALID_ARG;
    if (out != nullptr && (reinterpret_cast<uintptr_t>(out) & 7u)) return DDP_ERR_ALIGNMENT;
    if (walk_status != nullptr && (reinterpret_cast<uintptr_t>(walk_status) & 3u)) return DDP_ERR_ALIGNMENT;
    if (walk_status != nullptr && overlaps(walk_status, 4, out, static_cast<size_t>(count) * 8))
        return DDP_ERR_INVALID_ARG;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (walk_status != nullptr) {
        cudaError_t e = cudaMemsetAsync(walk_status, 0, sizeof(int32_t), s);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    if (count == 0) return DDP_OK;

    SamplerParams p{};
    p.out = out;
    p.status = walk_status;
    const uint64_t key = seed + epoch;            // mod 2^64
    uint64_t state = key;
    for (int i = 0; i < kRounds; ++i) {           // SplitMix64 stream from `key`
        state += kGamma;
        p.rk[i] = static_cast<uint32_t>(splitmix64_mix(state) >> 32);
    }
    const uint64_t n = static_cast<uint64_t>(n_items);
    int bits = 1;
    while (bits < 62 && (uint64_t(1) << bits) < n) ++bits;   // smallest bits >= 1 with 2^bits >= n
    p.h_lo = bits / 2;                                        // both halves <= 31 bits
    p.mask_lo = static_cast<uint32_t>((uint64_t(1) << p.h_lo) - 1);
    p.mask_hi = static_cast<uint32_t>((uint64_t(1) << (bits - p.h_lo)) - 1);
    p.n = n;
    p.ns = ns;
    p.count = count;
    p.small = count < (int64_t(1) << 31) ? 1 : 0;
    if (p.small) p.ns_div = make_fastdiv(static_cast<uint32_t>(ns));
    p.N = n_replicas;
    p.rank = rank;
    p.shuffle = shuffle;

    const bool narrow = n <= (uint64_t(1) << 31) && p.small;
    const void* kernel = narrow ? reinterpret_cast<const void*>(sampler_kernel<uint32_t>)
                                : reinterpret_cast<const void*>(sampler_kernel<uint64_t>);
    DeviceInfo dev;
    int st = current_device_info(&dev);
    if (st != DDP_OK) return st;
    int per_sm = 1;
    if ((st = resident_blocks_per_sm(kernel, kThreads, &per_sm)) != DDP_OK) return st;
    const int64_t target_warps = static_cast<int64_t>(dev.sm_count) * (per_sm < kBlocksPerSm ? per_sm : kBlocksPerSm) *
                                 kWarpsPerBlock;
    p.per_warp = (count + target_warps - 1) / target_warps;
    if (p.per_warp < kMinItemsPerWarp) p.per_warp = kMinItemsPerWarp;
    if (p.per_warp > (int64_t(1) << 30)) p.per_warp = int64_t(1) << 30;   // pool offsets stay int32
    p.pools = (count + p.per_warp - 1) / p.per_warp;
    const int grid = static_cast<int>((p.pools + kWarpsPerBlock - 1) / kWarpsPerBlock);   // <= target blocks
    // plain launch: the status word's memset just before must complete first
    if (narrow) sampler_kernel<uint32_t><<<grid, kThreads, 0, s>>>(p);
    else sampler_kernel<uint64_t><<<grid, kThreads, 0, s>>>(p);
    return check_launch();
}
