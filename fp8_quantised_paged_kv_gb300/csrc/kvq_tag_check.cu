// kvq_tag_check.cu -- the separate batched KV-cache integrity pass.
//
// Every physical page carries a tag that changes whenever the page is
// reassigned; each request records the tag it expects for each of its
// pages; before decode reads the cache the check compares the two and aborts
// the request on any mismatch.  It runs as its own batched pass rather than
// inside the attention kernel, so no attention thread group races with it
// (blog post "Smaller, faster, safer", page-2 mirror section "KV Cache
// 完整性检查"; page-3 mirror section "一个不能出错的共享缓存").
//
// One warp per request scans the ceil(L / page_size) entries it uses with
// coalesced loads of the block-table and expected-tag rows, gathers the live
// tags, and OR-reduces with __any_sync.  Lane 0 writes the flag (0 or 1).
#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr int kTagThreads = 256;

__global__ void __launch_bounds__(kTagThreads) tag_check_kernel(TagCheckArgs a)
{
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int64_t r = static_cast<int64_t>(blockIdx.x) * (kTagThreads / 32) + warp;
    if (r >= a.batch)
        return;
    const int64_t len = a.seq_lens[r] > 0 ? a.seq_lens[r] : 0;
    int64_t used = (len + a.page_size - 1) / a.page_size;
    bool bad = false;
    if (used > a.max_pages_per_seq) {
        bad = true;
        used = a.max_pages_per_seq;
    }
    const int32_t *bt = a.block_table + r * a.max_pages_per_seq;
    const uint32_t *exp = a.expected_tags + r * a.max_pages_per_seq;
    for (int64_t i = lane; i < used; i += 32) {
        const int32_t p = __ldg(bt + i);
        if (p < 0 || p >= a.num_pages || __ldg(a.page_tags + p) != __ldg(exp + i))
            bad = true;
    }
    bad = __any_sync(0xFFFFFFFFu, bad);
    if (lane == 0)
        a.abort_flags[r] = bad ? 1 : 0;
}

} // namespace

cudaError_t launch_tag_check(const TagCheckArgs &a, cudaStream_t stream)
{
    if (a.batch == 0)
        return cudaSuccess;
    const int per_block = kTagThreads / 32;
    const unsigned blocks = static_cast<unsigned>((a.batch + per_block - 1) / per_block);
    tag_check_kernel<<<blocks, kTagThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

} // namespace kvq
