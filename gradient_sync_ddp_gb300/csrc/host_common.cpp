// Status strings, thread-local CUDA error and the per-device launch-limit cache.
#include "host_common.h"

#include <map>
#include <mutex>
#include <utility>

namespace ddp {

namespace {
thread_local int g_last_cuda_error = 0;

constexpr int kMaxDevices = 64;
std::mutex g_info_mu;
DeviceInfo g_info[kMaxDevices];
bool g_info_valid[kMaxDevices] = {};
}  // namespace

int cuda_fail(cudaError_t e) {
    g_last_cuda_error = static_cast<int>(e);
    return DDP_ERR_CUDA;
}

int check_launch() {
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? DDP_OK : cuda_fail(e);
}

int current_device_info(DeviceInfo* out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices) return DDP_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_info_mu);
    if (!g_info_valid[dev]) {
        DeviceInfo d{};
        d.device = dev;
        if ((e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return cuda_fail(e);
        if ((e = cudaDeviceGetAttribute(&d.max_threads_per_sm, cudaDevAttrMaxThreadsPerMultiProcessor, dev)) !=
            cudaSuccess)
            return cuda_fail(e);
        g_info[dev] = d;
        g_info_valid[dev] = true;
    }
    *out = g_info[dev];
    return DDP_OK;
}

int resident_blocks_per_sm(const void* func, int block, int* out) {
    static std::mutex mu;
    static std::map<std::pair<const void*, int>, int> cache;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    std::lock_guard<std::mutex> lock(mu);
    auto key = std::make_pair(func, dev * 4096 + block);
    auto it = cache.find(key);
    if (it == cache.end()) {
        int n = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, func, block, 0);
        if (e != cudaSuccess) return cuda_fail(e);
        if (n < 1) n = 1;
        it = cache.emplace(key, n).first;
    }
    *out = it->second;
    return DDP_OK;
}

}  // namespace ddp

extern "C" const char* ddp_status_string(int status) {
    switch (status) {
        case DDP_OK: return "DDP_OK";
        case DDP_ERR_INVALID_ARG: return "DDP_ERR_INVALID_ARG: invalid argument";
        case DDP_ERR_ALIGNMENT: return "DDP_ERR_ALIGNMENT: device pointer not 16-byte aligned";
        case DDP_ERR_CAPACITY: return "DDP_ERR_CAPACITY: output or workspace too small";
        case DDP_ERR_CUDA: return "DDP_ERR_CUDA: a CUDA call failed";
        case DDP_ERR_UNSUPPORTED: return "DDP_ERR_UNSUPPORTED: not supported";
        case DDP_ERR_TIMEOUT: return "DDP_ERR_TIMEOUT: bounded loop ran out";
        default: return "unknown ddp_status";
    }
}

extern "C" int ddp_last_cuda_error(void) { return ddp::g_last_cuda_error; }

extern "C" const char* ddp_sync_version(void) { return "0.1.0"; }
