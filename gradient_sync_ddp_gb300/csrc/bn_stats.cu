// BatchNorm running statistics and inference folding.
//
// Tech-Renaissance "(24) NCCL通信与分布式数据并行" §十二: each rank's forward
// writes its batch statistics into running statistics (B_NEXT_MEAN /
// B_NEXT_VAR); STATS_COMM mean-all-reduces them every batch and UPDATE_STATS
// copies the synced values into B_PREV_* for the next batch — on one GPU that
// is ddp_bucket_allreduce_mean over the replicas' [mean | var] buffers with
// out = the B_PREV buffer and DDP_FLAG_WRITE_BACK_ALL; UPDATE_BN_INF_PARAMS
// finally folds the running statistics into eq_scale / eq_bias.  This file
// holds the two per-channel kernels around that: the running update
// (PyTorch's momentum blend with the unbiased variance) and the folding.
// Both touch C floats per array; they are launch-latency bound.
#include <cstdint>

#include "common.cuh"
#include "host_common.h"

namespace ddp {
namespace {

struct RunParams {
    const float* bmean;
    const float* bvar;
    float* rmean;
    float* rvar;
    int32_t C;
    float keep, mom, corr;   // fl(1 - momentum), momentum, fl(count / (count - 1))
};

__global__ void __launch_bounds__(kThreads) running_update_kernel(const __grid_constant__ RunParams a) {
    const int c = blockIdx.x * kThreads + threadIdx.x;
    pdl_enter();
    if (c >= a.C) return;
    a.rmean[c] = __fadd_rn(__fmul_rn(a.keep, a.rmean[c]), __fmul_rn(a.mom, a.bmean[c]));
    a.rvar[c] = __fadd_rn(__fmul_rn(a.keep, a.rvar[c]), __fmul_rn(a.mom, __fmul_rn(a.bvar[c], a.corr)));
}

struct FoldParams {
    const float* rmean;
    const float* rvar;
    const float* gamma;
    const float* beta;
    float* scale;
    float* bias;
    int32_t C;
    float eps;
};

__global__ void __launch_bounds__(kThreads) fold_kernel(const __grid_constant__ FoldParams a) {
    const int c = blockIdx.x * kThreads + threadIdx.x;
    pdl_enter();
    if (c >= a.C) return;
    const double g = a.gamma ? static_cast<double>(a.gamma[c]) : 1.0;
    const double b = a.beta ? static_cast<double>(a.beta[c]) : 0.0;
    const double sc = g / sqrt(static_cast<double>(a.rvar[c]) + static_cast<double>(a.eps));
    a.scale[c] = static_cast<float>(sc);
    a.bias[c] = static_cast<float>(b - static_cast<double>(a.rmean[c]) * sc);
}

bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace
}  // namespace ddp

using namespace ddp;

extern "C" int bn_running_stats_update(const float* batch_mean, const float* batch_var, int64_t count,
                                       float momentum, float* running_mean, float* running_var, int32_t C,
                                       void* stream) {
    if (C < 0 || count < 1 || !(momentum >= 0.0f && momentum <= 1.0f)) return DDP_ERR_INVALID_ARG;
    if (C > 0 && (batch_mean == nullptr || batch_var == nullptr || running_mean == nullptr || running_var == nullptr))
        return DDP_ERR_INVALID_ARG;
    if (!aligned4(batch_mean) || !aligned4(batch_var) || !aligned4(running_mean) || !aligned4(running_var))
        return DDP_ERR_ALIGNMENT;
    const size_t b = static_cast<size_t>(C) * 4;
    if (overlaps(running_mean, b, running_var, b) || overlaps(running_mean, b, batch_mean, b) ||
        overlaps(running_mean, b, batch_var, b) || overlaps(running_var, b, batch_mean, b) ||
        overlaps(running_var, b, batch_var, b))
        return DDP_ERR_INVALID_ARG;
    if (C == 0) return DDP_OK;
    RunParams p{batch_mean, batch_var, running_mean, running_var, C,
                static_cast<float>(1.0 - static_cast<double>(momentum)), momentum,
                count > 1 ? static_cast<float>(static_cast<double>(count) / static_cast<double>(count - 1)) : 1.0f};
    return launch_pdl(running_update_kernel, dim3(static_cast<unsigned>((C + kThreads - 1) / kThreads)), kThreads,
                      static_cast<cudaStream_t>(stream), p);
}

extern "C" int bn_fold_inference_params(const float* running_mean, const float* running_var, const float* gamma,
                                        const float* beta, float eps, int32_t C, float* scale_out, float* bias_out,
                                        void* stream) {
    if (C < 0 || !(eps >= 0.0f) || !(eps < 3.0e38f)) return DDP_ERR_INVALID_ARG;
    if (C > 0 && (running_mean == nullptr || running_var == nullptr || scale_out == nullptr || bias_out == nullptr))
        return DDP_ERR_INVALID_ARG;
    if (!aligned4(running_mean) || !aligned4(running_var) || !aligned4(gamma) || !aligned4(beta) ||
        !aligned4(scale_out) || !aligned4(bias_out))
        return DDP_ERR_ALIGNMENT;
    const size_t b = static_cast<size_t>(C) * 4;
    const void* ins[4] = {running_mean, running_var, gamma, beta};
    for (const void* q : ins)
        if (overlaps(scale_out, b, q, b) || overlaps(bias_out, b, q, b)) return DDP_ERR_INVALID_ARG;
    if (overlaps(scale_out, b, bias_out, b)) return DDP_ERR_INVALID_ARG;
    if (C == 0) return DDP_OK;
    FoldParams p{running_mean, running_var, gamma, beta, scale_out, bias_out, C, eps};
    return launch_pdl(fold_kernel, dim3(static_cast<unsigned>((C + kThreads - 1) / kThreads)), kThreads,
                      static_cast<cudaStream_t>(stream), p);
}
