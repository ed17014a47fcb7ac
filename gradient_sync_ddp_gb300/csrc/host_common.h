// Host-side helpers shared by the library's translation units: status
// bookkeeping, pointer checks and a per-device cache of launch limits.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "ddp_sync.h"

namespace ddp {

// Norm workspace: per bucket DDP_NORM_SLOTS float4 slots (one per CTA of the
// bucket's launch: Σout² as a float-float pair, a non-finite flag) followed by
// the number of CTAs that wrote a slot, padded to 16 bytes.
constexpr size_t kNormSlotBytes = static_cast<size_t>(DDP_NORM_SLOTS) * 16;
constexpr size_t kNormBucketBytes = kNormSlotBytes + 16;

// Record a CUDA error for ddp_last_cuda_error() and return DDP_ERR_CUDA.
int cuda_fail(cudaError_t e);

// After a kernel launch: DDP_OK, or DDP_ERR_CUDA if the launch failed.
int check_launch();

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// [a, a+na) and [b, b+nb) share at least one byte (a NULL pointer is an
// absent buffer and overlaps nothing).
inline bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return a != nullptr && b != nullptr && na > 0 && nb > 0 && x < y + nb && y < x + na;
}

struct DeviceInfo {
    int device;
    int sm_count;
    int max_threads_per_sm;
};

// Launch limits of the current device, queried once per device and cached.
int current_device_info(DeviceInfo* out);

// Resident CTAs per SM of `func` at `block` threads (occupancy calculator),
// cached per kernel and device.
int resident_blocks_per_sm(const void* func, int block, int* out);

// Launch kernel<<<grid, block, 0, s>>>(params) with programmatic stream
// serialisation allowed (the kernel must begin with pdl_enter()).
template <typename Params>
int launch_pdl(void (*kernel)(Params), dim3 grid, int block, cudaStream_t s, const Params& params) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(static_cast<unsigned>(block));
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, params);
    if (e != cudaSuccess) return cuda_fail(e);
    return check_launch();
}

// One wave of `kernel`: SMs x resident CTAs per SM, capped at need_blocks (>= 1).
inline int one_wave_grid(const void* kernel, int block, int64_t need_blocks, int* grid) {
    DeviceInfo d;
    int st = current_device_info(&d);
    if (st != DDP_OK) return st;
    int per_sm = 1;
    if ((st = resident_blocks_per_sm(kernel, block, &per_sm)) != DDP_OK) return st;
    const int64_t wave = static_cast<int64_t>(d.sm_count) * per_sm;
    if (need_blocks < 1) need_blocks = 1;
    *grid = static_cast<int>(need_blocks < wave ? need_blocks : wave);
    return DDP_OK;
}

}  // namespace ddp
