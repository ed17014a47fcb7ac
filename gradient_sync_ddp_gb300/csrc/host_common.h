// Host-side helpers shared by the library's translation units: status
// bookkeeping, pointer checks and a per-device cache of launch limits.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime_api.h>

#include "ddp_sync.h"

namespace ddp {

// Record a CUDA error for ddp_last_cuda_error() and return DDP_ERR_CUDA.
int cuda_fail(cudaError_t e);

// After a kernel launch: DDP_OK, or DDP_ERR_CUDA if the launch failed.
int check_launch();

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// [a, a+na) and [b, b+nb) share at least one byte.
inline bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return na > 0 && nb > 0 && x < y + nb && y < x + na;
}

struct DeviceInfo {
    int device;
    int sm_count;
    int max_threads_per_sm;
};

// Launch limits of the current device, queried once per device and cached.
int current_device_info(DeviceInfo* out);

}  // namespace ddp
