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
constexpr int kBlocksPerSm = 3;                    // target CTAs per SM (fewer if occupancy caps it)
constexpr int64_t kMinItemsPerWarp = 64;
constexpr int kSamplerThreads = 256;               // threads per CTA
constexpr int kWarpsPerBlock = kSamplerThreads / 32;

struct SamplerParams {
    int64_t* out;
    int32_t* status;
    uint32_t rk[kRounds];   // round keys
    uint32_t rkx[kRounds];  // k ^ (k >> 16): the key after fmix32's first xor-shift
    uint32_t sh16;          // 2^16 and 2^19: __umulhi(h, 2^(32-s)) == h >> s, which
    uint32_t sh19;          //   issues on the multiply pipe instead of the integer ALU
    uint32_t p2lo;          // 2^h_lo
    uint32_t mask_hi;       // 2^h_hi - 1
    uint32_t mask_lo;       // 2^h_lo - 1
    int32_t h_lo;           // width of the low half
    uint64_t n;             // items
    int64_t ns;             // num_samples (length of a rank's list)
    int64_t start;          // first list position written (resume offset)
    int64_t row_len;        // ns - start: output slots per rank
    int64_t per_warp;       // slots per pool; pools never cross a row
    int64_t pools_per_row;  // ceil(ns / per_warp)
    int64_t pools;          // rows * pools_per_row
    int32_t N;              // replicas
    int32_t rank;           // -1: all ranks, rank-major rows
    int32_t shuffle;
};

uint64_t splitmix64_mix(uint64_t z) {
    z ^= z >> 30;
    z *= 0xBF58476D1CE4E5B9ull;
    z ^= z >> 27;
    z *= 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

// fmix32(x ^ k), the MurmurHash3 32-bit finalizer, with its shifts written
// as multiply-highs.  NARROW: x < 2^16, so x >> 16 == 0 and the first
// xor-shift of x ^ k is x ^ (k ^ (k >> 16)) (shifts distribute over xor).
template <bool NARROW>
__device__ __forceinline__ uint32_t round_fn(uint32_t x, int i, const SamplerParams& a) {
    uint32_t h;
    if constexpr (NARROW) {
        h = x ^ a.rkx[i];
    } else {
        h = x ^ a.rk[i];
        h ^= __umulhi(h, a.sh16);
    }
    h *= 0x85EBCA6Bu;
    h ^= __umulhi(h, a.sh19);
    h *= 0xC2B2AE35u;
    return h ^ __umulhi(h, a.sh16);
}

// One pass of the network on x = H * 2^h_lo + L, H the high ceil(bits/2)
// bits and L the low floor(bits/2) bits: even rounds H ^= fmix32(L ^ k_i)
// mod 2^|H|, odd rounds L ^= fmix32(H ^ k_i) mod 2^|L|.  Every round undoes
// itself, so the pass is a bijection.  The halves are carried as 32-bit words
// whose bits above the half's width are don't-cares: a round's output is
// xored in unmasked, and the mask is applied where the half is read (fused
// with the key xor), which is the same arithmetic mod 2^|half|.
template <bool NARROW, typename U>
__device__ __forceinline__ U encrypt(U x, const SamplerParams& a) {
    uint32_t L = static_cast<uint32_t>(x);                  // bits above h_lo: don't-care
    uint32_t H = static_cast<uint32_t>(x >> a.h_lo);        // exact: x < 2^bits
    H ^= round_fn<NARROW>(L & a.mask_lo, 0, a);
    L ^= round_fn<NARROW>(H & a.mask_hi, 1, a);
    H ^= round_fn<NARROW>(L & a.mask_lo, 2, a);
    L ^= round_fn<NARROW>(H & a.mask_hi, 3, a);
    return static_cast<U>(H & a.mask_hi) * a.p2lo + (L & a.mask_lo);
}

// Padded-list position -> unshuffled index: padding repeats the head.
template <typename U>
__device__ __forceinline__ U wrap(U pos, U n) {
    if (pos < n) return pos;
    return pos - n < n ? pos - n : pos % n;    // pos >= 2n only when N > n
}

// Unshuffled index of slot s of a pool whose first slot is position pos0.
// PAD: the pool holds padded positions (>= n); otherwise no wrap is needed.
template <typename U, bool PAD>
__device__ __forceinline__ U slot_index(U pos0, int32_t s, U N, U n) {
    const U pos = pos0 + static_cast<U>(s) * N;
    return PAD ? wrap<U>(pos, n) : pos;
}

// The walks of one pool: per_warp consecutive slots 0 .. len-1 of one rank's
// row, slot s holding padded-list position pos0 + s*N.  Cycle-walk lengths
// are geometric: instead of idling until the slowest lane of the warp has
// finished, a lane whose walk ends writes its index and takes the pool's
// next unclaimed slot (ballot + prefix count), so every iteration is one
// encryption per lane until the pool runs dry.  The body uses selects, not
// branches; a lane without a slot walks a copy of the last slot and stores
// nothing.  The walk bound can only be reached once the loop has run
// kWalkCap times, so its check sits behind that warp-uniform test.
template <typename U, bool PAD>
__device__ __forceinline__ void walk_pool(const SamplerParams& a, int64_t* out, U pos0, int32_t len, int lane) {
    constexpr bool kNarrow = sizeof(U) == 4;
    const unsigned lanes_below = (1u << lane) - 1u;
    const U n = static_cast<U>(a.n), N = static_cast<U>(a.N);
    const int32_t last = len - 1;
    int32_t off = lane;                           // this lane's slot in the pool
    U x = slot_index<U, PAD>(pos0, min(off, last), N, n);
    int32_t deadline = kWalkCap;                  // loop count at which this lane's walk gives up
    int32_t next = 32;                            // first unclaimed slot of the pool
    for (int32_t it = 1;; ++it) {
        const bool live = off < len;
        if (!__any_sync(0xffffffffu, live)) break;
        x = encrypt<kNarrow>(x, a);
        const bool hit = x < n;
        if (live && hit) out[off] = static_cast<int64_t>(x);
        bool done = hit;
        if (it >= kWalkCap) {                     // warp-uniform; never reached in practice
            const bool give_up = !hit && it >= deadline;
            if (live && give_up) {
                out[off] = -1;
                if (a.status) atomicAdd(a.status, 1);
            }
            done = done || give_up;
        }
        const unsigned fin = __ballot_sync(0xffffffffu, done);
        const int32_t o = next + __popc(fin & lanes_below);
        next += __popc(fin);
        const U xn = slot_index<U, PAD>(pos0, min(o, last), N, n);
        off = done ? o : off;
        x = done ? xn : x;
        deadline = done ? it + kWalkCap : deadline;
    }
}

// Warps take pools grid-stride; the host sizes pools so that the grid is
// kBlocksPerSm CTAs on every SM.  U is uint32_t when n <= 2^31: then every
// position is below total < n + N < 2^32 and both halves below 2^16.
template <typename U>
__global__ void __launch_bounds__(kSamplerThreads) sampler_kernel(const __grid_constant__ SamplerParams a) {
    const int lane = threadIdx.x & 31;
    const U n = static_cast<U>(a.n);
    const U N = static_cast<U>(a.N);
    const int64_t warps = static_cast<int64_t>(gridDim.x) * kWarpsPerBlock;
    for (int64_t pool = (static_cast<int64_t>(blockIdx.x) * kSamplerThreads + threadIdx.x) / 32; pool < a.pools;
         pool += warps) {
        const int64_t row = pool / a.pools_per_row;
        const int64_t s0 = (pool - row * a.pools_per_row) * a.per_warp;
        const int32_t len = static_cast<int32_t>(min(a.per_warp, a.row_len - s0));
        const int64_t r = a.rank >= 0 ? a.rank : row;
        int64_t* out = a.out + (a.rank >= 0 ? 0 : row * a.row_len) + s0;
        const U pos0 = static_cast<U>(r) + static_cast<U>(a.start + s0) * N;
        if (!(a.shuffle && a.n > 1)) {
            for (int32_t o = lane; o < len; o += 32) out[o] = static_cast<int64_t>(wrap<U>(pos0 + o * N, n));
            continue;
        }
        if (pos0 + static_cast<U>(len - 1) * N >= n) walk_pool<U, true>(a, out, pos0, len, lane);
        else walk_pool<U, false>(a, out, pos0, len, lane);
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

extern "C" int dist_sampler_indices_from(int64_t n_items, int32_t n_replicas, int32_t rank,
                                         uint64_t seed, uint64_t epoch, int32_t shuffle, int32_t drop_last,
                                         int64_t start, int64_t* out, int64_t out_capacity,
                                         int64_t* num_samples_out, int32_t* walk_status, void* stream) {
    if (num_samples_out == nullptr) return DDP_ERR_INVALID_ARG;
    if (shuffle != 0 && shuffle != 1) return DDP_ERR_INVALID_ARG;
    const int64_t ns = dist_sampler_num_samples(n_items, n_replicas, drop_last);
    if (ns < 0 || rank < -1 || rank >= n_replicas || out_capacity < 0) return DDP_ERR_INVALID_ARG;
    *num_samples_out = ns;
    if (start < 0 || start > ns) return DDP_ERR_INVALID_ARG;
    const int64_t row_len = ns - start;
    const int64_t count = rank >= 0 ? row_len : row_len * n_replicas;
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
        p.rkx[i] = p.rk[i] ^ (p.rk[i] >> 16);
    }
    p.sh16 = 1u << 16;
    p.sh19 = 1u << 19;
    const uint64_t n = static_cast<uint64_t>(n_items);
    int bits = 1;
    while (bits < 62 && (uint64_t(1) << bits) < n) ++bits;   // smallest bits >= 1 with 2^bits >= n
    p.h_lo = bits / 2;                                        // both halves <= 31 bits
    p.p2lo = 1u << p.h_lo;
    p.mask_lo = p.p2lo - 1u;
    p.mask_hi = static_cast<uint32_t>((uint64_t(1) << (bits - p.h_lo)) - 1);
    p.n = n;
    p.ns = ns;
    p.start = start;
    p.row_len = row_len;
    p.N = n_replicas;
    p.rank = rank;
    p.shuffle = shuffle;

    const bool narrow = n <= (uint64_t(1) << 31);
    const void* kernel = narrow ? reinterpret_cast<const void*>(sampler_kernel<uint32_t>)
                                : reinterpret_cast<const void*>(sampler_kernel<uint64_t>);
    DeviceInfo dev;
    int st = current_device_info(&dev);
    if (st != DDP_OK) return st;
    int per_sm = 1;
    if ((st = resident_blocks_per_sm(kernel, kSamplerThreads, &per_sm)) != DDP_OK) return st;
    const int64_t target_warps = static_cast<int64_t>(dev.sm_count) * (per_sm < kBlocksPerSm ? per_sm : kBlocksPerSm) *
                                 kWarpsPerBlock;
    p.per_warp = (count + target_warps - 1) / target_warps;
    if (p.per_warp < kMinItemsPerWarp) p.per_warp = kMinItemsPerWarp;
    if (p.per_warp > (int64_t(1) << 30)) p.per_warp = int64_t(1) << 30;   // pool offsets stay int32
    p.pools_per_row = (row_len + p.per_warp - 1) / p.per_warp;
    p.pools = (rank >= 0 ? 1 : n_replicas) * p.pools_per_row;
    const int64_t need = (p.pools + kWarpsPerBlock - 1) / kWarpsPerBlock;
    const int64_t wave = static_cast<int64_t>(dev.sm_count) * per_sm;
    const int grid = static_cast<int>(need < wave ? need : wave);
    // plain launch: the status word's memset just before must complete first
    if (narrow) sampler_kernel<uint32_t><<<grid, kSamplerThreads, 0, s>>>(p);
    else sampler_kernel<uint64_t><<<grid, kSamplerThreads, 0, s>>>(p);
    return check_launch();
}

extern "C" int dist_sampler_indices(int64_t n_items, int32_t n_replicas, int32_t rank,
                                    uint64_t seed, uint64_t epoch, int32_t shuffle, int32_t drop_last,
                                    int64_t* out, int64_t out_capacity, int64_t* num_samples_out,
                                    int32_t* walk_status, void* stream) {
    return dist_sampler_indices_from(n_items, n_replicas, rank, seed, epoch, shuffle, drop_last, 0, out,
                                     out_capacity, num_samples_out, walk_status, stream);
}
