// Device helpers shared by the library's kernels: 16-byte global accesses
// with explicit cache policy, and the exact bf16 -> fp32 widening.
#pragma once

#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace ddp {

constexpr int kThreads = 256;

// 16-byte global load.  NC = true: read-only (non-coherent) path without L1
// allocation, for buffers the kernel never writes; every element is read
// exactly once, so nothing is worth caching.  NC = false: coherent streaming
// load, for buffers the same kernel also writes (in-place updates).
template <bool NC>
__device__ __forceinline__ uint4 ld16(const void* p) {
    uint4 v;
    if constexpr (NC) {
        asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
            : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
            : "l"(p));
    } else {
        asm volatile("ld.global.cs.v4.u32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                     : "l"(p)
                     : "memory");
    }
    return v;
}

// 16-byte global load through the coherent path with the default L2 policy,
// for data that a later kernel reads again (SyncBN's x: read by the
// statistics pass, then by the apply).  The read-only path of ld16<true>
// does not keep lines in L2 for another kernel: on GB300 a second pass over
// 51 MB read that way ran at 14.3 us against 9.8 us after plain loads.
__device__ __forceinline__ uint4 ld16_keep(const void* p) {
    uint4 v;
    asm volatile("ld.global.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

// 16-byte streaming store (evict-first: the result is not re-read by this kernel).
__device__ __forceinline__ void st16(void* p, uint4 v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// 8-byte streaming store.
__device__ __forceinline__ void st8(void* p, uint2 v) {
    asm volatile("st.global.cs.v2.u32 [%0], {%1,%2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
}

// Two fp32 values rounded to bf16 (nearest, ties to even), element 0 in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const uint32_t l = __bfloat16_as_ushort(__float2bfloat16_rn(lo));
    const uint32_t h = __bfloat16_as_ushort(__float2bfloat16_rn(hi));
    return l | (h << 16);
}

__device__ __forceinline__ uint4 f4_bits(float a, float b, float c, float d) {
    return make_uint4(__float_as_uint(a), __float_as_uint(b), __float_as_uint(c), __float_as_uint(d));
}

// bf16 -> fp32 is exact: the bf16 pattern is the high half of the fp32 pattern.
// A 32-bit word holds two bf16 values, element 0 in the low half.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Element k of a 16-byte vector holding 4 fp32 or 8 bf16 values, as fp32.
template <bool BF16>
__device__ __forceinline__ float vec_elem(const uint4& v, int k) {
    const uint32_t w = (k >> (BF16 ? 1 : 0)) == 0 ? v.x : (k >> (BF16 ? 1 : 0)) == 1 ? v.y
                     : (k >> (BF16 ? 1 : 0)) == 2 ? v.z : v.w;
    if constexpr (BF16) return (k & 1) ? bf16_hi(w) : bf16_lo(w);
    else return __uint_as_float(w);
}

// One element of a flat fp32 or bf16 buffer, as fp32 (scalar path).
template <bool BF16>
__device__ __forceinline__ float load_elem(const void* base, int64_t e) {
    if constexpr (BF16) {
        const unsigned short h = reinterpret_cast<const unsigned short*>(base)[e];
        return __uint_as_float(static_cast<uint32_t>(h) << 16);
    } else {
        return reinterpret_cast<const float*>(base)[e];
    }
}

// Programmatic dependent launch.  Every kernel of this library is launched
// with programmatic stream serialisation allowed, so its launch (and the
// scheduling of its CTAs on SMs freed by the previous kernel) overlaps the
// tail of the kernel before it on the stream.  Correctness does not depend on
// what that previous kernel was: each kernel first lets its own dependents
// launch, then waits for the full completion (and memory flush) of the grid
// it depends on before it touches global memory.
__device__ __forceinline__ void pdl_enter() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

}  // namespace ddp

namespace ddp {

// Division of unsigned 32-bit values n < 2^31 by a fixed divisor 1 <= d < 2^31
// with one multiply-high, add and shift (Granlund & Montgomery, "Division by
// invariant integers using multiplication", PLDI 1994, round-up variant):
// s = ceil(log2 d), m = floor(2^32 (2^s - d) / d) + 1, q = (mulhi(n, m) + n) >> s.
struct FastDiv {
    uint32_t d, m, s;
};

inline FastDiv make_fastdiv(uint32_t d) {
    FastDiv f{d, 0, 0};
    while ((uint64_t(1) << f.s) < d) ++f.s;
    f.m = static_cast<uint32_t>(((uint64_t(1) << 32) * ((uint64_t(1) << f.s) - d)) / d + 1);
    return f;
}

__device__ __forceinline__ uint32_t fdiv(uint32_t n, const FastDiv& f) {
    return (__umulhi(n, f.m) + n) >> f.s;
}

}  // namespace ddp

namespace ddp {

// Float-float arithmetic: a value is hi + lo, kept with fp32 operations only
// (Knuth's TwoSum, then a renormalising Fast2Sum), about 48 significant bits.
// GB300's FP64 pipe is narrow (one 32-lane fp64 instruction occupies it for
// many cycles), so the reductions here avoid fp64 and use this instead; the
// order of every reduction is fixed, so results are deterministic.
struct FF {
    float hi, lo;
};

__device__ __forceinline__ FF ff_add(FF a, FF b) {
    const float s = __fadd_rn(a.hi, b.hi);
    const float bb = __fsub_rn(s, a.hi);
    const float e = __fadd_rn(__fsub_rn(a.hi, __fsub_rn(s, bb)), __fsub_rn(b.hi, bb));
    const float t = __fadd_rn(e, __fadd_rn(a.lo, b.lo));
    const float hi = __fadd_rn(s, t);
    return FF{hi, __fsub_rn(t, __fsub_rn(hi, s))};
}

__device__ __forceinline__ FF ff_shfl_down(FF v, int o) {
    return FF{__shfl_down_sync(0xffffffffu, v.hi, o), __shfl_down_sync(0xffffffffu, v.lo, o)};
}

// Sum of two per-thread values over the CTA in float-float, result in thread 0.
__device__ __forceinline__ void block_sum2_ff(FF& a, FF& b) {
    __shared__ FF sh[2][kThreads / 32];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        a = ff_add(a, ff_shfl_down(a, o));
        b = ff_add(b, ff_shfl_down(b, o));
    }
    const int w = threadIdx.x / 32, l = threadIdx.x % 32;
    if (l == 0) {
        sh[0][w] = a;
        sh[1][w] = b;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        a = sh[0][0];
        b = sh[1][0];
        for (int i = 1; i < kThreads / 32; ++i) {
            a = ff_add(a, sh[0][i]);
            b = ff_add(b, sh[1][i]);
        }
    }
}

}  // namespace ddp
