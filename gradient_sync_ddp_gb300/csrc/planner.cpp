// Bucket planner: partitions a model's gradient tensors into flat, aligned
// buckets (host only, no CUDA call).
//
// Reverse-registration greedy fill with a byte cap: AI_Infra notes
// "1.DataParallel / DDP" §3.2 (buckets follow the backward order, 25 MB
// default) and §4.2 (params[::-1] handed to the bucket builder).
// Two-bucket DEEP/FIRST split: Tech-Renaissance "(24) NCCL通信与分布式数据并行"
// §八.  Cursor layout with aligned bases: Tech-Renaissance "(16) DTensor" §四
// (MemoryPlan::finalize walks a cursor) and §六 (slots rounded up to 256 B).
#include <cstdint>
#include <vector>

#include "ddp_sync.h"

namespace {

int64_t round_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

}  // namespace

extern "C" int ddp_plan_buckets(int32_t n_tensors, const int64_t* numels, int32_t elem_bytes, int64_t cap_bytes,
                                int32_t mode, const uint8_t* is_first, int32_t align_bytes,
                                ddp_bucket* buckets, int32_t max_buckets, int32_t* n_buckets,
                                int32_t* order, int64_t* tensor_offset, int32_t* tensor_bucket,
                                int64_t* total_elems) {
    if (n_tensors < 0 || n_buckets == nullptr || total_elems == nullptr) return DDP_ERR_INVALID_ARG;
    if (n_tensors > 0 && (numels == nullptr || order == nullptr || tensor_offset == nullptr ||
                          tensor_bucket == nullptr))
        return DDP_ERR_INVALID_ARG;
    if (elem_bytes != 2 && elem_bytes != 4) return DDP_ERR_INVALID_ARG;
    if (align_bytes <= 0 || align_bytes % elem_bytes != 0 || align_bytes % 16 != 0) return DDP_ERR_INVALID_ARG;
    if (cap_bytes < 0 || max_buckets < 0 || (max_buckets > 0 && buckets == nullptr)) return DDP_ERR_INVALID_ARG;
    if (mode != DDP_PLAN_CAP && mode != DDP_PLAN_DEEP_FIRST) return DDP_ERR_INVALID_ARG;
    if (mode == DDP_PLAN_DEEP_FIRST && n_tensors > 0 && is_first == nullptr) return DDP_ERR_INVALID_ARG;
    const int64_t kMaxElems = INT64_MAX / 8;
    for (int32_t t = 0; t < n_tensors; ++t)
        if (numels[t] < 0 || numels[t] > kMaxElems) return DDP_ERR_INVALID_ARG;

    // 1. groups of tensor ids, in flat order
    std::vector<std::vector<int32_t>> groups;
    if (mode == DDP_PLAN_CAP) {
        std::vector<int32_t> cur;
        int64_t cur_bytes = 0;
        for (int32_t t = n_tensors - 1; t >= 0; --t) {
            const int64_t nb = numels[t] * elem_bytes;
            if (!cur.empty() && cur_bytes + nb > cap_bytes) {
                groups.push_back(cur);
                cur.clear();
                cur_bytes = 0;
            }
            cur.push_back(t);
            cur_bytes += nb;
        }
        if (!cur.empty()) groups.push_back(cur);
    } else {
        std::vector<int32_t> deep, first;
        for (int32_t t = n_tensors - 1; t >= 0; --t) (is_first[t] ? first : deep).push_back(t);
        if (!deep.empty()) groups.push_back(deep);
        if (!first.empty()) groups.push_back(first);
    }

    const int32_t nb = static_cast<int32_t>(groups.size());
    *n_buckets = nb;
    if (nb > max_buckets) return DDP_ERR_CAPACITY;

    // 2. layout: a cursor over the flat buffer, bucket bases aligned
    const int64_t align = align_bytes / elem_bytes;
    int64_t cursor = 0;
    int32_t pos_in_order = 0;
    for (int32_t b = 0; b < nb; ++b) {
        const int64_t base = cursor;
        int64_t pos = base;
        buckets[b].offset_elems = base;
        buckets[b].first = pos_in_order;
        buckets[b].count = static_cast<int32_t>(groups[b].size());
        for (int32_t t : groups[b]) {
            tensor_offset[t] = pos;
            tensor_bucket[t] = b;
            order[pos_in_order++] = t;
            pos += numels[t];
        }
        buckets[b].numel = pos - base;
        cursor = round_up(pos, align);
    }
    *total_elems = cursor;
    return DDP_OK;
}
