/*
 * The rank-ordered gradient average in plain C.
 *
 * TEST INFRASTRUCTURE: timing context for the CPU baseline, pinned
 * bit-exact to oracle.grad_mean (tests/test_oracle_cref.py); nothing in the
 * product links or calls it.
 *
 * Tech-Renaissance "(24) NCCL通信与分布式数据并行" §一: grad_sync starts at
 * zero, each replica's gradient is added in rank order, and the sum is
 * divided by float(N).  Compiled with -ffp-contract=off and without
 * fast-math, so every addition and the division round once to fp32, exactly
 * as the definition states.  The threaded variant splits the elements into
 * contiguous ranges; each element's additions keep the same order, so both
 * give the same bits.
 */
#include <stdint.h>

#ifdef _OPENMP
#include <omp.h>
#endif

static void mean_range(const float* const* g, int32_t n, int64_t lo, int64_t hi, float* out) {
    const float fn = (float)n;
    for (int64_t i = lo; i < hi; ++i) {
        float acc = 0.0f;
        for (int32_t r = 0; r < n; ++r) acc = acc + g[r][i];
        out[i] = acc / fn;
    }
}

void oracle_grad_mean_f32(const float* const* g, int32_t n, int64_t numel, float* out) {
    mean_range(g, n, 0, numel, out);
}

void oracle_grad_mean_f32_threads(const float* const* g, int32_t n, int64_t numel, float* out) {
#ifdef _OPENMP
#pragma omp parallel
    {
        const int64_t t = omp_get_thread_num(), T = omp_get_num_threads();
        mean_range(g, n, numel * t / T, numel * (t + 1) / T, out);
    }
#else
    mean_range(g, n, 0, numel, out);
#endif
}

int32_t oracle_threads(void) {
#ifdef _OPENMP
    return (int32_t)omp_get_max_threads();
#else
    return 1;
#endif
}
