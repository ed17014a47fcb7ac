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
// (halves of ceil(bits/2) and floor(bits/2) bits, so the domain is below
// 2n), round keys = the first four SplitMix64 outputs from state seed+epoch,
// round function = the SplitMix64 output mix (Steele, Lea & Flood, OOPSLA
// 2014) truncated to the half's width, and cycle walking (encrypt again
// while the value is >= n; under two encryptions per index on average).  Each walk is bounded: after 4096
// encryptions the thread writes -1 and counts the index in a status word
// instead of looping on.  The kernel is integer-ALU bound (~4 rounds x
// ~1.6 walks x 2 64-bit multiplies per index); the 8-byte output per index
// is its only memory traffic.  Threads stream through several output slots
// so that lanes of a warp stay busy although walk lengths differ.
#include <cstdint>

#include "common.cuh"
#include "host_common.h"

namespace ddp {
namespace {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;
constexpr int kRounds = 4;
constexpr int kWalkCap = 4096;

struct SamplerParams {
    int64_t* out;
    int32_t* status;
    uint64_t rk[kRounds];
    uint64_t n;          // items
    uint64_t mask_hi;    // 2^h_hi - 1
    uint64_t mask_lo;    // 2^h_lo - 1
    int64_t ns;          // num_samples
    int64_t count;       // outputs to write
    int32_t N;           // replicas
    int32_t rank;        // -1: all ranks, rank-major
    int32_t h_lo;        // width of the low half
    int32_t shuffle;
};

__host__ __device__ __forceinline__ uint64_t mix64(uint64_t z) {
    z ^= z >> 30;
    z *= 0xBF58476D1CE4E5B9ull;
    z ^= z >> 27;
    z *= 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

// x = (H, L) with H the high ceil(bits/2) bits and L the low floor(bits/2)
// bits; even rounds H ^= mix64(L ^ k_i) mod 2^|H|, odd rounds L ^= mix64(H ^
// k_i) mod 2^|L|.  Every round undoes itself, so the pass is a bijection.
__device__ __forceinline__ uint64_t encrypt(uint64_t x, const SamplerParams& a) {
    uint64_t H = x >> a.h_lo, L = x & a.mask_lo;
#pragma unroll
    for (int i = 0; i < kRounds; ++i) {
        if (i % 2 == 0) H ^= mix64(L ^ a.rk[i]) & a.mask_hi;
        else L ^= mix64(H ^ a.rk[i]) & a.mask_lo;
    }
    return (H << a.h_lo) | L;
}

// Position -> unshuffled index for output slot i.
__device__ __forceinline__ uint64_t base_index(int64_t i, const SamplerParams& a) {
    int64_t r, s;
    if (a.rank >= 0) {
        r = a.rank;
        s = i;
    } else {
        r = i / a.ns;
        s = i - r * a.ns;
    }
    const uint64_t pos = static_cast<uint64_t>(r) + static_cast<uint64_t>(s) * static_cast<uint64_t>(a.N);
    return pos < a.n ? pos : pos % a.n;       // padding repeats the head
}

// Each thread owns output slots gtid, gtid + T, gtid + 2T, ... (T = grid
// threads, about 8 slots per thread).  Cycle-walk lengths are geometric, so
// instead of idling until the slowest lane of the warp has finished one
// index, a thread starts its next slot as soon as one is done: every loop
// iteration is exactly one encryption for every lane.
__global__ void __launch_bounds__(kThreads) sampler_kernel(const __grid_constant__ SamplerParams a) {
    const int64_t T = static_cast<int64_t>(gridDim.x) * kThreads;
    int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
    if (!(a.shuffle && a.n > 1)) {
        for (; i < a.count; i += T) a.out[i] = static_cast<int64_t>(base_index(i, a));
        return;
    }
    if (i >= a.count) return;
    uint64_t y = base_index(i, a);
    int steps = 0;                             // encryptions applied to y
    while (true) {
        if (steps > 0 && (y < a.n || steps >= kWalkCap)) {
            if (y < a.n) {
                a.out[i] = static_cast<int64_t>(y);
            } else {                           // walk bound reached: never observed
                a.out[i] = -1;
                if (a.status) atomicAdd(a.status, 1);
            }
            i += T;
            if (i >= a.count) break;
            y = base_index(i, a);
            steps = 0;
        }
        y = encrypt(y, a);
        ++steps;
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
        p.rk[i] = mix64(state);
    }
    const uint64_t n = static_cast<uint64_t>(n_items);
    int bits = 1;
    while (bits < 63 && (uint64_t(1) << bits) < n) ++bits;   // smallest bits >= 1 with 2^bits >= n
    p.h_lo = bits / 2;
    p.mask_lo = (uint64_t(1) << p.h_lo) - 1;
    p.mask_hi = (uint64_t(1) << (bits - p.h_lo)) - 1;
    p.n = n;
    p.ns = ns;
    p.count = count;
    p.N = n_replicas;
    p.rank = rank;
    p.shuffle = shuffle;

    int grid = 0;
    constexpr int64_t kSlotsPerThread = 4;
    const int st = one_wave_grid(reinterpret_cast<const void*>(sampler_kernel), kThreads,
                                 (count + kSlotsPerThread * kThreads - 1) / (kSlotsPerThread * kThreads), &grid);
    if (st != DDP_OK) return st;
    // plain launch: the status word's memset just before must complete first
    sampler_kernel<<<grid, kThreads, 0, s>>>(p);
    return check_launch();
}
