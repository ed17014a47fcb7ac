// Bucket readiness: the reducer's bookkeeping of which gradients are ready.
//
// AI_Infra notes "1.DataParallel / DDP" §3.2 and §4.2: a gradient hook marks
// its parameter ready in its bucket; once every parameter of a bucket is
// ready, the bucket's all-reduce is issued (asynchronously, while backward
// continues).  §3.3: a parameter the forward pass skipped never gets a
// gradient, so its bucket never fills and every rank waits forever unless
// the parameter is marked as needing no communication
// (find_unused_parameters).  Here the wait is bounded and the parameter that
// was never marked is reported.
//
// §3.2 also has buckets fire as they fill; when hooks complete several
// buckets faster than the caller launches them (the end of backward, small
// caps), ddp_reducer_take_ready hands over every bucket completed since the
// previous take at once, so they can go out as one grouped launch.
//
// Host code only.  One mutex guards the state; a condition variable wakes
// ddp_reducer_wait_all and ddp_reducer_take_ready when a bucket completes.
// Marking is O(1): each bucket keeps the number of parameters still missing.
#include <chrono>
#include <condition_variable>
#include <cstdint>
#include <mutex>
#include <new>
#include <vector>

#include "ddp_sync.h"

struct ddp_reducer {
    std::mutex mu;
    std::condition_variable cv;
    std::vector<int32_t> tensor_bucket;   // bucket of each parameter
    std::vector<int32_t> bucket_size;     // parameters per bucket
    std::vector<int32_t> missing;         // parameters not yet marked, per bucket
    std::vector<uint8_t> marked;          // per parameter: 0 no, 1 ready, 2 unused
    std::vector<int32_t> done_order;      // buckets completed this iteration, in order
    std::vector<uint8_t> taken;           // per bucket: handed out by ddp_reducer_take_ready
    int32_t n_taken = 0;                  // buckets handed out this iteration
    int32_t buckets_left = 0;
};

namespace {

int mark(ddp_reducer* r, int32_t tensor, int32_t* bucket_done, uint8_t how) {
    if (r == nullptr || bucket_done == nullptr) return DDP_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(r->mu);
    if (tensor < 0 || tensor >= static_cast<int32_t>(r->tensor_bucket.size())) return DDP_ERR_INVALID_ARG;
    if (r->marked[tensor] != 0) return DDP_ERR_INVALID_ARG;          // the hook fired twice
    r->marked[tensor] = how;
    const int32_t b = r->tensor_bucket[tensor];
    *bucket_done = -1;
    if (--r->missing[b] == 0) {
        *bucket_done = b;
        r->done_order.push_back(b);
        --r->buckets_left;
        r->cv.notify_all();
    }
    return DDP_OK;
}

}  // namespace

extern "C" int ddp_reducer_create(int32_t n_tensors, const int32_t* tensor_bucket, int32_t n_buckets,
                                  ddp_reducer** out) {
    if (out == nullptr) return DDP_ERR_INVALID_ARG;
    *out = nullptr;
    if (n_tensors < 1 || n_buckets < 1 || n_buckets > n_tensors || tensor_bucket == nullptr)
        return DDP_ERR_INVALID_ARG;
    std::vector<int32_t> size(static_cast<size_t>(n_buckets), 0);
    for (int32_t t = 0; t < n_tensors; ++t) {
        const int32_t b = tensor_bucket[t];
        if (b < 0 || b >= n_buckets) return DDP_ERR_INVALID_ARG;
        ++size[b];
    }
    for (int32_t b = 0; b < n_buckets; ++b)
        if (size[b] == 0) return DDP_ERR_INVALID_ARG;              // a bucket that could never complete
    ddp_reducer* r = new (std::nothrow) ddp_reducer;
    if (r == nullptr) return DDP_ERR_CAPACITY;
    r->tensor_bucket.assign(tensor_bucket, tensor_bucket + n_tensors);
    r->bucket_size = size;
    r->missing = size;
    r->marked.assign(static_cast<size_t>(n_tensors), 0);
    r->done_order.reserve(static_cast<size_t>(n_buckets));
    r->taken.assign(static_cast<size_t>(n_buckets), 0);
    r->buckets_left = n_buckets;
    *out = r;
    return DDP_OK;
}

extern "C" void ddp_reducer_destroy(ddp_reducer* r) { delete r; }

extern "C" int ddp_reducer_mark_ready(ddp_reducer* r, int32_t tensor, int32_t* bucket_done) {
    return mark(r, tensor, bucket_done, 1);
}

extern "C" int ddp_reducer_mark_unused(ddp_reducer* r, int32_t tensor, int32_t* bucket_done) {
    return mark(r, tensor, bucket_done, 2);
}

extern "C" int ddp_reducer_wait_all(ddp_reducer* r, int64_t timeout_us, int32_t* first_missing) {
    if (r == nullptr || timeout_us < 0) return DDP_ERR_INVALID_ARG;
    std::unique_lock<std::mutex> lock(r->mu);
    const bool all = r->cv.wait_for(lock, std::chrono::microseconds(timeout_us), [r] { return r->buckets_left == 0; });
    if (first_missing != nullptr) {
        *first_missing = -1;
        for (size_t t = 0; t < r->marked.size(); ++t)
            if (r->marked[t] == 0) {
                *first_missing = static_cast<int32_t>(t);
                break;
            }
    }
    return all ? DDP_OK : DDP_ERR_TIMEOUT;
}

extern "C" int ddp_reducer_reset(ddp_reducer* r) {
    if (r == nullptr) return DDP_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(r->mu);
    r->missing = r->bucket_size;
    r->marked.assign(r->marked.size(), 0);
    r->done_order.clear();
    r->taken.assign(r->taken.size(), 0);
    r->n_taken = 0;
    r->buckets_left = static_cast<int32_t>(r->bucket_size.size());
    return DDP_OK;
}

extern "C" int ddp_reducer_take_ready(ddp_reducer* r, int64_t timeout_us, int32_t* buckets_out, int32_t max_out,
                                      int32_t* n_out) {
    if (r == nullptr || n_out == nullptr || buckets_out == nullptr || max_out < 1 || timeout_us < 0)
        return DDP_ERR_INVALID_ARG;
    std::unique_lock<std::mutex> lock(r->mu);
    const int32_t nb = static_cast<int32_t>(r->bucket_size.size());
    auto pending = [r] { return static_cast<int32_t>(r->done_order.size()) > r->n_taken; };
    // wait for a completed bucket not yet handed out, unless every bucket has been handed out already
    if (!pending() && r->n_taken < nb && timeout_us > 0)
        r->cv.wait_for(lock, std::chrono::microseconds(timeout_us), [&] { return pending(); });
    // completed, not yet handed out: in bucket index order (a plan's offset order), lowest first
    int32_t n = 0;
    for (int32_t b = 0; b < nb && n < max_out; ++b) {
        if (r->missing[b] == 0 && !r->taken[b]) {
            r->taken[b] = 1;
            buckets_out[n++] = b;
        }
    }
    r->n_taken += n;
    *n_out = n;
    return DDP_OK;
}

extern "C" int ddp_reducer_completed(const ddp_reducer* r, int32_t* order_out, int32_t max_out, int32_t* n_done) {
    if (r == nullptr || n_done == nullptr || max_out < 0 || (max_out > 0 && order_out == nullptr))
        return DDP_ERR_INVALID_ARG;
    ddp_reducer* m = const_cast<ddp_reducer*>(r);
    std::lock_guard<std::mutex> lock(m->mu);
    const int32_t n = static_cast<int32_t>(m->done_order.size());
    for (int32_t i = 0; i < n && i < max_out; ++i) order_out[i] = m->done_order[i];
    *n_done = n;
    return DDP_OK;
}
