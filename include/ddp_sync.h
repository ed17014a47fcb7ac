/*
 * ddp_sync.h — C ABI of the GB300 (sm_103a) DDP gradient-synchronisation library
 * (libddp_sync.so).
 *
 * The library implements, on one GPU, the data-parallel hot path of DDP
 * training: N model replicas' gradients are N resident device buffers, and the
 * library averages them bucket by bucket (optionally fused with the bf16 ->
 * fp32 widen and an SGD step), merges SyncBatchNorm statistics across the
 * replicas and applies the normalisation, and produces DistributedSampler
 * index lists; a host-side tracker tells when a bucket's gradients are all
 * ready.
 *
 * Sources (web pages, cited by title and section):
 *   [TR24] Tech-Renaissance, "(24) NCCL通信与分布式数据并行"
 *   [TR16] Tech-Renaissance, "(16) DTensor"
 *   [DDP]  AI_Infra notes, "1.DataParallel / DDP"
 *
 * Conventions shared by every entry point
 *   - Plain C types only.  Device pointers are CUDA device addresses on the
 *     current device; host pointers are ordinary host memory.  `stream` is a
 *     cudaStream_t passed as void* (NULL = the legacy default stream).
 *   - Ownership: the caller owns every buffer.  No entry point allocates or
 *     frees memory, synchronises the device, or keeps a pointer after it
 *     returns.  Host arrays (e.g. the list of replica pointers) are read
 *     during the call only; their contents are copied into the kernel's
 *     launch parameters, so the calls may be captured into a CUDA Graph.
 *   - Asynchrony: work is enqueued on `stream` and the call returns at once.
 *     Results are valid once the stream has reached that point.  Calls on
 *     disjoint buffers (e.g. different buckets) may be issued on different
 *     streams: the GPU then starts one launch on the SMs the previous one
 *     frees instead of after its whole grid.
 *   - Errors: every entry point returns an int status (ddp_status below) and
 *     never throws or aborts.  Arguments are validated on the host before any
 *     CUDA call; an invalid call enqueues nothing and leaves every buffer
 *     untouched.  A failed kernel launch returns DDP_ERR_CUDA and the CUDA
 *     error code is available from ddp_last_cuda_error() on the same thread.
 *   - Alignment: every device pointer must be 16-byte aligned
 *     (DDP_ERR_ALIGNMENT otherwise); bucket offsets from ddp_plan_buckets are
 *     256-byte aligned, so pointers into planned buffers always qualify.
 *   - Replica count: 1 <= n_replicas <= DDP_MAX_REPLICAS.
 *   - Empty requests: with numel == 0 (or an empty sampler list) nothing is
 *     enqueued and the data pointers may be NULL.
 *   - Arithmetic: no fused multiply-add in the bit-exact paths, IEEE
 *     round-to-nearest-even on every fp32 operation, subnormals preserved.
 */
#ifndef DDP_SYNC_H
#define DDP_SYNC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DDP_MAX_REPLICAS 16

typedef enum {
    DDP_OK = 0,
    DDP_ERR_INVALID_ARG = -1,   /* null pointer, negative size, bad enum, bad overlap */
    DDP_ERR_ALIGNMENT = -2,     /* a device pointer is not 16-byte aligned */
    DDP_ERR_CAPACITY = -3,      /* an output array or workspace is too small */
    DDP_ERR_CUDA = -4,          /* a CUDA call failed; see ddp_last_cuda_error() */
    DDP_ERR_UNSUPPORTED = -5,   /* valid request the library does not implement */
    DDP_ERR_TIMEOUT = -6        /* a bounded wait or loop ran out (see each entry) */
} ddp_status;

typedef enum { DDP_F32 = 0, DDP_BF16 = 1 } ddp_dtype;

/* bucket planning modes */
enum { DDP_PLAN_CAP = 0, DDP_PLAN_DEEP_FIRST = 1 };

/* summation-order / output flags of the all-reduce entry points */
enum {
    DDP_FLAG_TREE_ORDER = 1u,      /* pairwise tree order (power-of-two N) */
    DDP_FLAG_WRITE_BACK_ALL = 2u,  /* also store the result into every replica (fp32 only) */
    DDP_FLAG_RING_ORDER = 4u       /* chunk-rotated order of a ring all-reduce */
};

/* One bucket of a plan: a contiguous range of the flat gradient buffer. */
typedef struct {
    int64_t offset_elems;   /* first element of the bucket in the flat buffer */
    int64_t numel;          /* elements in the bucket (tensors packed back to back) */
    int32_t first;          /* index into `order` of the bucket's first tensor */
    int32_t count;          /* number of tensors in the bucket */
} ddp_bucket;

/*
 * ddp_plan_buckets — partition a model's gradient tensors into flat buckets.
 *
 * [DDP] §3.2 and §4.2: buckets are built over the parameters in reverse
 * registration order (the last layer's gradient is ready first) with a size
 * cap (25 MB by default).  [TR24] §八: the two-bucket split, DEEP first,
 * then FIRST.  [TR16] §四/§六: one flat buffer, bucket bases aligned.
 *
 *   n_tensors       number of tensors T (>= 0)
 *   numels          host int64[T], element count of each tensor in
 *                   registration order (each >= 0)
 *   elem_bytes      bytes per gradient element (2 or 4)
 *   cap_bytes       DDP_PLAN_CAP: close a bucket before a tensor whose bytes
 *                   would push it past cap_bytes (a tensor larger than the
 *                   cap is alone); ignored for DDP_PLAN_DEEP_FIRST.  >= 0.
 *   mode            DDP_PLAN_CAP or DDP_PLAN_DEEP_FIRST
 *   is_first        host uint8[T] (DDP_PLAN_DEEP_FIRST only, else may be
 *                   NULL): nonzero puts the tensor in the FIRST bucket.
 *   align_bytes     bucket base alignment in bytes: a positive multiple of
 *                   elem_bytes and of 16 (256 = [TR16] align_up_256)
 *   buckets         host ddp_bucket[max_buckets], written [0, *n_buckets)
 *   n_buckets       host int32*, receives the number of buckets
 *   order           host int32[T]: tensor ids in flat-buffer order
 *   tensor_offset   host int64[T]: element offset of each tensor id
 *   tensor_bucket   host int32[T]: bucket of each tensor id
 *   total_elems     host int64*: flat buffer length, end of the last bucket
 *                   rounded up to the alignment
 * Host-only; no CUDA call.  Returns DDP_ERR_CAPACITY (with *n_buckets set to
 * the number needed) if max_buckets is too small.
 */
int ddp_plan_buckets(int32_t n_tensors, const int64_t* numels, int32_t elem_bytes, int64_t cap_bytes,
                     int32_t mode, const uint8_t* is_first, int32_t align_bytes,
                     ddp_bucket* buckets, int32_t max_buckets, int32_t* n_buckets,
                     int32_t* order, int64_t* tensor_offset, int32_t* tensor_bucket,
                     int64_t* total_elems);

/*
 * Bucket readiness (the reducer's bookkeeping; host side, no CUDA call).
 *
 * [DDP] §3.2 and §4.2: every parameter's gradient hook marks the parameter
 * ready in its bucket, and a bucket's all-reduce is issued as soon as all of
 * its parameters are ready, while backward still runs for earlier layers.
 * [DDP] §3.3: a parameter skipped by the forward pass never gets a gradient,
 * so its bucket never completes and the job waits forever;
 * find_unused_parameters marks such parameters as needing no communication.
 * Here marking a parameter unused counts it as ready: its gradient slice is
 * averaged as it stands, so the caller zeroes it for the step, as PyTorch's
 * reducer does.  The wait for the remaining buckets is bounded and reports
 * the first parameter that was never marked instead of hanging.
 *
 * All functions are thread-safe (hooks may fire on several threads).  The
 * tracker copies what it needs from the arguments; the caller frees nothing
 * but the tracker itself (ddp_reducer_destroy).
 */
typedef struct ddp_reducer ddp_reducer;   /* opaque */

/*
 * ddp_reducer_create — tracker for n_tensors parameters in n_buckets buckets.
 *   tensor_bucket  host int32[n_tensors]: bucket of each parameter (as from
 *                  ddp_plan_buckets), each in [0, n_buckets); every bucket
 *                  must hold at least one parameter
 *   out            receives the tracker
 * DDP_ERR_INVALID_ARG on a bad count, bucket index or empty bucket.
 */
int ddp_reducer_create(int32_t n_tensors, const int32_t* tensor_bucket, int32_t n_buckets, ddp_reducer** out);

/* Free the tracker (NULL is allowed). */
void ddp_reducer_destroy(ddp_reducer* r);

/*
 * ddp_reducer_mark_ready — parameter `tensor`'s gradient is ready.
 *   bucket_done  receives the bucket this mark completed (all of its
 *                parameters now marked; the caller launches its average),
 *                or -1.  Each bucket is reported exactly once per iteration.
 * DDP_ERR_INVALID_ARG if tensor is out of range or already marked in this
 * iteration (a gradient hook fired twice).
 */
int ddp_reducer_mark_ready(ddp_reducer* r, int32_t tensor, int32_t* bucket_done);

/* ddp_reducer_mark_unused — like mark_ready, for a parameter the forward
 * pass did not use in this iteration ([DDP] §3.3, find_unused_parameters). */
int ddp_reducer_mark_unused(ddp_reducer* r, int32_t tensor, int32_t* bucket_done);

/*
 * ddp_reducer_wait_all — wait until every bucket of this iteration is
 * complete, for at most timeout_us microseconds (>= 0; 0 only checks).
 *   first_missing  receives the lowest parameter index not yet marked, or -1
 *                  when all are (may be NULL)
 * DDP_OK when all buckets are complete; DDP_ERR_TIMEOUT when the time ran
 * out first (the [DDP] §3.3 hang, reported instead of waited out).
 */
int ddp_reducer_wait_all(ddp_reducer* r, int64_t timeout_us, int32_t* first_missing);

/* Start the next iteration: every parameter unmarked, no bucket complete. */
int ddp_reducer_reset(ddp_reducer* r);

/* Buckets completed so far in this iteration, in completion order: writes up
 * to max_out bucket indices into order_out and the count into *n_done. */
int ddp_reducer_completed(const ddp_reducer* r, int32_t* order_out, int32_t max_out, int32_t* n_done);

/*
 * ddp_reducer_take_ready — every bucket that completed since the previous
 * take (or since create / reset), for one grouped launch.
 *
 * [DDP] §3.2: buckets fire as they fill.  When hooks complete buckets faster
 * than the caller launches them (the end of backward; small caps, where one
 * launch per bucket is latency-bound), the caller takes all the completed
 * buckets at once and averages them with one
 * ddp_bucket_allreduce_mean_multi call instead of one call per bucket.
 *   timeout_us   >= 0: if no completed bucket is waiting, wait up to this
 *                long for one (0: do not wait); no wait once every bucket of
 *                the iteration has been taken
 *   buckets_out  host int32[max_out] (max_out >= 1): the buckets taken, in
 *                increasing bucket index order (a plan's offset order, as
 *                ddp_bucket_allreduce_mean_multi wants); when more than
 *                max_out are waiting, the lowest max_out are taken and the
 *                rest stay for the next take
 *   n_out        receives the number taken (0 when the wait ran out, or
 *                when every bucket has been taken)
 * Each bucket is taken exactly once per iteration.  The bucket_done result
 * of the mark calls is independent of taking: a caller uses one or the
 * other to decide what to launch.
 * DDP_ERR_INVALID_ARG on a NULL pointer, max_out < 1 or timeout_us < 0.
 */
int ddp_reducer_take_ready(ddp_reducer* r, int64_t timeout_us, int32_t* buckets_out, int32_t max_out,
                           int32_t* n_out);

/*
 * ddp_bucket_allreduce_mean — average one bucket over N replicas.
 *
 * [TR24] §一: grad_sync = 0; for r in 0..N-1: grad_sync += grad[r];
 * grad_sync /= float(N).  [TR24] §九 / [DDP] §4.2: sum all-reduce then
 * scale by 1/world_size, fused here into one pass.  [TR24] §十一: an AMP
 * gradient cast precedes the all-reduce; bf16 replicas are widened to fp32
 * exactly inside the same pass.
 *
 *   replicas    host array of n_replicas device pointers, replica r's bucket
 *               (numel elements of in_dtype, 16-byte aligned)
 *   n_replicas  N, 1..DDP_MAX_REPLICAS
 *   in_dtype    DDP_F32 or DDP_BF16
 *   numel       elements in the bucket (>= 0; 0 enqueues nothing)
 *   out         device float[numel], 16-byte aligned: the fp32 average.  It
 *               may be exactly equal to a replica pointer when in_dtype is
 *               DDP_F32 (in place, like ncclAllReduce); any other overlap
 *               with a replica is rejected.
 *   flags       0 = rank order (bit-exact with the definition above; the
 *               1/N scale is a multiply by the exact reciprocal when N is a
 *               power of two and a true division otherwise — identical
 *               results); DDP_FLAG_TREE_ORDER = ((g0+g1)+(g2+g3))+... then
 *               /N (N a power of two); DDP_FLAG_RING_ORDER = element e of
 *               chunk j (N near-equal contiguous chunks, longer ones first)
 *               is summed g_j, g_j+1, ..., g_j-1 (mod N) then /N, the order
 *               of the ring all-reduce of [DDP] §2.11; DDP_FLAG_WRITE_BACK_ALL
 *               (DDP_F32 only) also stores the average into every replica.
 *               TREE and RING are exclusive.
 *   stream      cudaStream_t as void*
 */
int ddp_bucket_allreduce_mean(const void* const* replicas, int32_t n_replicas, int32_t in_dtype,
                              int64_t numel, float* out, uint32_t flags, void* stream);

#define DDP_MULTI_MAX_BUCKETS 1024

/*
 * ddp_bucket_allreduce_mean_multi — ddp_bucket_allreduce_mean (rank order)
 * for several buckets of one flat layout in a single launch.
 *
 * [DDP] §3.2 and [TR24] §三: small buckets mean many launches; when several
 * buckets are ready at the same time (the end of backward, the FIRST bucket
 * of [TR24] §八 together with late DEEP tensors, a sweep of small caps) one
 * launch serves them all and pays the launch latency once.  The result is
 * bit for bit that of one ddp_bucket_allreduce_mean call per bucket.
 *   replica_bases  host array of n_replicas device pointers: each replica's
 *                  flat gradient buffer (16-byte aligned)
 *   buckets        host ddp_bucket[n_buckets] in increasing, non-overlapping
 *                  offset order (e.g. a plan's buckets; first/count unused);
 *                  offset_elems·4 and offset_elems·elem_bytes must be
 *                  multiples of 16 (planned 256-byte offsets are)
 *   n_buckets      0 .. DDP_MULTI_MAX_BUCKETS
 *   out_base       device float*: the flat output buffer; bucket b's average
 *                  goes to out_base + offset_elems; must not overlap the
 *                  replicas (no in-place form)
 */
int ddp_bucket_allreduce_mean_multi(const void* const* replica_bases, int32_t n_replicas, int32_t in_dtype,
                                    const ddp_bucket* buckets, int32_t n_buckets, float* out_base, void* stream);

/*
 * ddp_bucket_allreduce_sgd — average one bucket and apply the SGD step.
 *
 * [DDP] §5.3: θ ← θ − η·g with g the synced average; [DDP] §3.1: every rank
 * applies the same deterministic step.  [TR24] §九 (note) suggests folding
 * the 1/world_size into the optimizer kernel; this entry does that.
 * Momentum and weight decay follow PyTorch's SGD (dampening 0, no
 * Nesterov), each fp32 operation rounded separately:
 *     g = mean (as ddp_bucket_allreduce_mean, rank order)
 *     d = g + weight_decay*θ                 (if weight_decay != 0)
 *     b = momentum*buf + d; buf = b; d = b   (if momentum != 0)
 *     θ = θ − lr*d
 *
 *   replicas, n_replicas, in_dtype, numel   as for the mean
 *   param         device float[numel], θ, updated in place
 *   momentum_buf  device float[numel], updated in place; required iff
 *                 momentum != 0 (else must be NULL).  Start it at zero.
 *   lr, momentum, weight_decay   finite fp32 scalars
 *   grad_out      device float[numel] or NULL: also store g
 *   flags         0 (reserved)
 * param, momentum_buf and grad_out must not overlap each other or any
 * replica.
 */
int ddp_bucket_allreduce_sgd(const void* const* replicas, int32_t n_replicas, int32_t in_dtype,
                             int64_t numel, float* param, float* momentum_buf,
                             float lr, float momentum, float weight_decay,
                             float* grad_out, uint32_t flags, void* stream);

/*
 * ---- gradient accumulation, global norm with clipping, non-finite check ----
 *
 * [DDP] §5.2: with gradient accumulation, micro-steps run under no_sync (the
 * gradient is only added into .grad locally, loss divided by the number of
 * steps), the all-reduce runs once after the last micro-step, and
 * clip_grad_norm_ is applied to the synced gradient before the optimizer
 * step.  [TR24] §十一: a NaN-check graph (n_ncg) runs after the gradient
 * syncs.  Flow on one GPU:
 *   micro-steps:  ddp_bucket_accumulate (acc[r] += micro[r], every replica)
 *   last step:    ddp_bucket_allreduce_mean_norm for each bucket (average +
 *                 per-CTA Σg², non-finite flag), ddp_grad_norm_finalize
 *                 (norm, clip factor, flag; all in device memory, no host
 *                 sync), ddp_bucket_sgd for each bucket with the clip factor.
 */

/*
 * ddp_bucket_accumulate — acc[r][i] = acc[r][i] + (float)micro[r][i] for every
 * replica r (one fp32 rounding per element; bf16 micro gradients are widened
 * exactly).
 *   micro       host array of n_replicas device pointers, numel in_dtype each
 *   acc         host array of n_replicas device pointers, numel float each,
 *               updated in place; no acc buffer may overlap another buffer of
 *               the call
 */
int ddp_bucket_accumulate(const void* const* micro, float* const* acc, int32_t n_replicas, int32_t in_dtype,
                          int64_t numel, void* stream);

#define DDP_NORM_SLOTS 2048

/* Bytes of the norm workspace for n_buckets buckets (0 if n_buckets < 1). */
size_t ddp_norm_workspace_bytes(int32_t n_buckets);

/*
 * ddp_bucket_allreduce_mean_norm — ddp_bucket_allreduce_mean in rank order
 * (same bits in out), plus a side output for clipping: the bucket's Σ out[i]²
 * (per-CTA partials, fp32 per thread, float-float per CTA) and whether any
 * out[i] is NaN or infinite, stored in slot `bucket_index` of norm_ws.
 *   norm_ws       device buffer of ddp_norm_workspace_bytes(n_buckets) bytes,
 *                 16-byte aligned; each bucket of a step writes its own slot
 *   bucket_index  0 .. n_buckets-1
 * flags are not taken (rank order, no write-back).
 */
int ddp_bucket_allreduce_mean_norm(const void* const* replicas, int32_t n_replicas, int32_t in_dtype,
                                   int64_t numel, float* out, void* norm_ws, int32_t bucket_index, void* stream);

/*
 * ddp_grad_norm_finalize — combine the slots of buckets 0..n_buckets-1 (all
 * written in this step) into, in device memory:
 *   norm_out       sqrt(Σ over every bucket of Σ out²)   (float)
 *   clip_coef_out  min(1, max_norm / (norm + 1e-6)); 1 if max_norm <= 0
 *                  (clip_grad_norm_'s factor)            (float)
 *   nonfinite_out  1 if any averaged gradient element is NaN or infinite,
 *                  else 0                                (int32)
 * Any of the three outputs may be NULL.  One small kernel; no host sync.
 */
int ddp_grad_norm_finalize(const void* norm_ws, int32_t n_buckets, float max_norm, float* norm_out,
                           float* clip_coef_out, int32_t* nonfinite_out, void* stream);

/*
 * ddp_bucket_sgd — the SGD step of ddp_bucket_allreduce_sgd applied to an
 * already averaged gradient, optionally scaled first by a device scalar:
 *     d = grad * (*grad_scale)        (if grad_scale != NULL; one rounding)
 *     d = d + weight_decay*θ; b = momentum*buf + d; buf = b; θ = θ − lr*b
 *   grad          device float[numel] (the averaged gradient), read only
 *   param, momentum_buf, lr, momentum, weight_decay   as ddp_bucket_allreduce_sgd
 *   grad_scale    device float or NULL, e.g. clip_coef_out of
 *                 ddp_grad_norm_finalize
 *   param_bf16    device bf16[numel] or NULL: also store the updated θ
 *                 rounded to bf16 (as ddp_bucket_allreduce_sgd_cast)
 */
int ddp_bucket_sgd(const float* grad, float* param, float* momentum_buf, int64_t numel, float lr,
                   float momentum, float weight_decay, const float* grad_scale, void* param_bf16, void* stream);

/*
 * ddp_bucket_allreduce_sgd_cast — ddp_bucket_allreduce_sgd that also stores
 * the updated θ rounded to bf16 (nearest, ties to even) into param_bf16.
 *
 * [TR16] §六: master weights are FP32, the compute copy half width, and one
 * whole-region cast refreshes the compute copy after the update.  Writing
 * the copy from the update kernel costs its 2-byte store per element and
 * saves the cast pass (a 4-byte read and the same store).
 *   param_bf16    device bf16[numel], 16-byte aligned, overlapping nothing
 *                 else of the call
 * flags are not taken.
 */
int ddp_bucket_allreduce_sgd_cast(const void* const* replicas, int32_t n_replicas, int32_t in_dtype,
                                  int64_t numel, float* param, float* momentum_buf, float lr, float momentum,
                                  float weight_decay, float* grad_out, void* param_bf16, void* stream);

/*
 * syncbn_workspace_bytes — device workspace that syncbn_merge_apply needs
 * for these sizes (0 for invalid sizes).
 */
size_t syncbn_workspace_bytes(int32_t n_replicas, int32_t batch, int32_t C, int32_t H, int32_t W);

/*
 * syncbn_channel_parts — how syncbn_merge_apply runs these sizes: 2 when it
 * splits the channels into two halves on two streams (see "Streams" under
 * syncbn_merge_apply; each half is three launches), 1 when it runs one
 * sequence of three launches on the caller's stream, DDP_ERR_INVALID_ARG
 * for invalid sizes or dtype.  A call that finds no side stream of its
 * thread while its stream captures runs one sequence even where this
 * returns 2.
 */
int syncbn_channel_parts(int32_t n_replicas, int32_t in_dtype, int32_t batch, int32_t C, int32_t H, int32_t W);

/*
 * syncbn_merge_apply — strict SyncBatchNorm forward across N replicas.
 *
 * [TR24] §十二: strict SyncBatchNorm all-reduces each rank's per-channel sum
 * and sum of squares before BN finalize/apply.  [DDP] §4.3: the statistics
 * are those of the global batch.  Per channel c:
 *     S = Σ_r Σ x_r[:,c],  Q = Σ_r Σ x_r[:,c]²,  M = N·batch·H·W
 *     mean = S/M,  var = Q/M − mean²  (biased),  invstd = 1/sqrt(var + eps)
 *     y_r = (x_r − mean)·invstd·γ + β
 * Sums are shifted by each channel's first element (so Q/M − mean² does
 * not cancel when |mean| >> std); threads accumulate a few hundred
 * elements in fp32, each CTA combines its threads in float-float (pairs of
 * fp32) and stores one fp32 partial per channel and slice of the samples,
 * and a merge kernel sums the partials and finalises in float-float; the
 * apply runs in fp32.
 *
 *   x            host array of n_replicas device pointers, each
 *                [batch, C, H, W] NCHW contiguous, in_dtype elements
 *   in_dtype     DDP_BF16 or DDP_F32
 *   batch,C,H,W  local batch and shape, each >= 1
 *   eps          > 0
 *   gamma, beta  device float[C] or NULL (γ = 1, β = 0)
 *   y            host array of n_replicas device pointers, same shape,
 *                out_dtype elements; y[r] may equal x[r] when the dtypes
 *                match (in place), no other overlap
 *   mean_out, invstd_out   device float[C] each
 *   workspace    device buffer of >= syncbn_workspace_bytes(...) bytes,
 *                16-byte aligned, contents ignored on entry; calls whose
 *                kernels may overlap on the GPU (different streams without
 *                ordering) need different workspaces, or they race on the
 *                partial sums
 * Streams: large inputs whose channels split evenly into the statistics
 * kernels' units (an even C; see syncbn_channel_parts) run as two
 * channel halves, the second on a side stream that the library keeps per
 * host thread and device (created on the thread's first such call made
 * outside stream capture; a call that finds none while its stream captures
 * runs as one sequence).  The side stream waits on an event recorded on
 * `stream` and `stream` waits on its join event before the call returns,
 * so the call stays ordered on `stream` and capturable; both forms give the
 * same bits.  After cudaDeviceReset the thread's side stream is stale.
 */
int syncbn_merge_apply(const void* const* x, int32_t n_replicas, int32_t in_dtype,
                       int32_t batch, int32_t C, int32_t H, int32_t W, float eps,
                       const float* gamma, const float* beta,
                       void* const* y, int32_t out_dtype, float* mean_out, float* invstd_out,
                       void* workspace, size_t workspace_bytes, void* stream);

/*
 * syncbn_merge_apply_noalloc — syncbn_merge_apply without a caller workspace.
 *
 * The pages have no counterpart: this entry point exists for callers that
 * cannot allocate device memory themselves (code inside a host framework
 * whose memory pool owns the device and forbids side allocations, code under
 * a device-memory budget fixed up front, step loops that cannot afford
 * cudaMalloc's implicit device synchronisation).  It allocates nothing and
 * frees nothing; its scratch is a fixed array of
 * syncbn_noalloc_max_workspace_bytes() bytes (1 MiB) compiled into the
 * library, held by every GPU that loads the library until the process exits.
 *
 *   Arguments, results and errors are those of syncbn_merge_apply, without
 *   workspace/workspace_bytes.  Sizes whose syncbn_workspace_bytes(...)
 *   exceeds the fixed array are rejected with DDP_ERR_CAPACITY (every shape
 *   with C <= 43690 fits: the planner keeps every workspace within 1 MiB
 *   for those).
 *   Set-up: the first call on each device looks up the array's device
 *   address (cudaGetSymbolAddress, with that device current) and caches it;
 *   make that first call before any stream capture.  The address stays
 *   cached for the life of the process: after a cudaDeviceReset of that
 *   device it is stale (the module is loaded again into the new context),
 *   so a process that resets a device must not call this entry point on it
 *   again; it can use syncbn_merge_apply with a workspace instead.
 *   The capacity and overlap checks of syncbn_merge_apply apply to the
 *   syncbn_workspace_bytes(...) bytes at the start of the array that the
 *   call uses.
 *   Sharing: every call on a device uses the same array, which keeps the last
 *   call's contents (nothing in it needs to start at zero).  Calls whose
 *   kernels overlap on the GPU (different streams without ordering between
 *   them) race on the array and give wrong results; order them on one stream
 *   or with events.
 */
int syncbn_merge_apply_noalloc(const void* const* x, int32_t n_replicas, int32_t in_dtype,
                               int32_t batch, int32_t C, int32_t H, int32_t W, float eps,
                               const float* gamma, const float* beta,
                               void* const* y, int32_t out_dtype, float* mean_out, float* invstd_out,
                               void* stream);

/* Size in bytes of the fixed scratch array used by syncbn_merge_apply_noalloc. */
size_t syncbn_noalloc_max_workspace_bytes(void);

/*
 * ---- BatchNorm running statistics ([TR24] §十二) ----
 * STATS_COMM + UPDATE_STATS (mean all-reduce of every rank's running mean /
 * var, then copy into the "previous" buffers) is ddp_bucket_allreduce_mean
 * over the replicas' [mean | var] buffers with out = the previous-statistics
 * buffer and DDP_FLAG_WRITE_BACK_ALL; the validation-metric mean
 * (VAL_RESULT_COMM, [TR24] §十三) is the same call on the metric sums.  The
 * two entries below are the per-channel steps around it.
 */

/*
 * bn_running_stats_update — running statistics from one batch (PyTorch's
 * rule; the pages do not give one):
 *   running_mean = (1 − momentum)·running_mean + momentum·batch_mean
 *   running_var  = (1 − momentum)·running_var  + momentum·batch_var·count/(count − 1)
 * fp32, each operation rounded on its own; (1 − momentum) and
 * count/(count − 1) are rounded to fp32 once on the host.
 *   batch_mean, batch_var      device float[C] (biased batch variance)
 *   count                      values per channel in the batch (>= 1)
 *   momentum                   in [0, 1]
 *   running_mean, running_var  device float[C], updated in place
 */
int bn_running_stats_update(const float* batch_mean, const float* batch_var, int64_t count, float momentum,
                            float* running_mean, float* running_var, int32_t C, void* stream);

/*
 * bn_fold_inference_params — UPDATE_BN_INF_PARAMS: eq_scale = γ/sqrt(var + eps),
 * eq_bias = β − mean·eq_scale (fp64 inside, fp32 out), so inference BN is
 * y = x·eq_scale + eq_bias.  gamma / beta may be NULL (1 / 0).
 */
int bn_fold_inference_params(const float* running_mean, const float* running_var, const float* gamma,
                             const float* beta, float eps, int32_t C, float* scale_out, float* bias_out,
                             void* stream);

/*
 * dist_sampler_num_samples — indices per rank ([DDP] §4.4):
 * floor(n/N) with drop_last, else ceil(n/N).  -1 on invalid input.
 */
int64_t dist_sampler_num_samples(int64_t n_items, int32_t n_replicas, int32_t drop_last);

/*
 * dist_sampler_indices — DistributedSampler index lists.
 *
 * [DDP] §4.4: num_samples = drop_last ? n/N : ceil(n/N); total =
 * num_samples·N; the (shuffled) list 0..n-1 is padded by repeating its head
 * up to total (or cut to total with drop_last); rank r takes positions
 * r, r+N, r+2N, ...  The shuffle is a permutation keyed by seed+epoch so
 * every rank agrees without communication: a 4-round Feistel network on
 * ceil(log2 n) bits (a high half of ceil(bits/2) bits and a low half of
 * floor(bits/2) bits, updated alternately) whose round keys are the high 32
 * bits of the first four SplitMix64 outputs from state seed+epoch and whose
 * round function is the MurmurHash3 32-bit finalizer of (half ^ key),
 * truncated to the other half's width, with cycle walking into [0, n).
 *
 *   n_items        n >= 0 (< 2^62)
 *   n_replicas     N >= 1
 *   rank           0..N-1 for one rank's list, or -1 for all ranks,
 *                  rank-major [N][num_samples]
 *   seed, epoch    the permutation key is seed + epoch (mod 2^64)
 *   shuffle, drop_last   0 or 1
 *   out            device int64[out_capacity]
 *   out_capacity   elements available at out; must be >= num_samples
 *                  (rank >= 0) or N·num_samples (rank == -1), else
 *                  DDP_ERR_CAPACITY with *num_samples_out still set
 *   num_samples_out  host int64*, receives num_samples (computed on the host)
 *   walk_status    device int32 or NULL: set to 0, then to the number of
 *                  indices whose cycle walk exceeded 4096 encryptions (those
 *                  outputs are -1).  Never observed; the bound keeps every
 *                  thread's loop finite.
 */
int dist_sampler_indices(int64_t n_items, int32_t n_replicas, int32_t rank,
                         uint64_t seed, uint64_t epoch, int32_t shuffle, int32_t drop_last,
                         int64_t* out, int64_t out_capacity, int64_t* num_samples_out,
                         int32_t* walk_status, void* stream);

/*
 * dist_sampler_indices_from — the same lists from position `start` on
 * (resuming an epoch part-way: each rank has already consumed the first
 * `start` indices of its list, e.g. start = steps done × per-rank batch).
 *   start   0 <= start <= num_samples, else DDP_ERR_INVALID_ARG
 *   out     num_samples − start indices (rank >= 0), or all ranks rank-major
 *           [N][num_samples − start] (rank == -1); out_capacity counts
 *           those.  Entry k is list position start + k of dist_sampler_indices.
 * Everything else as dist_sampler_indices (which is this call with start 0).
 */
int dist_sampler_indices_from(int64_t n_items, int32_t n_replicas, int32_t rank,
                              uint64_t seed, uint64_t epoch, int32_t shuffle, int32_t drop_last,
                              int64_t start, int64_t* out, int64_t out_capacity, int64_t* num_samples_out,
                              int32_t* walk_status, void* stream);

/* Human-readable name of a ddp_status value (static string). */
const char* ddp_status_string(int status);

/* CUDA error code (cudaError_t as int) of the last DDP_ERR_CUDA on this thread. */
int ddp_last_cuda_error(void);

/* Library version, e.g. "0.1.0". */
const char* ddp_sync_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DDP_SYNC_H */
