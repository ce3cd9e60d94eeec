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
// One CTA per request: its threads take the ceil(L / page_size) entries the
// request uses in one strided pass (coalesced block-table and expected-tag
// loads, one gather of the live tag each), OR-reduce with __syncthreads_or,
// and thread 0 writes the flag (0 or 1).  A 513-page request costs one round
// of dependent loads instead of 17 rounds on a single warp.
#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr int kTagThreads = 128;

__global__ void __launch_bounds__(kTagThreads) tag_check_kernel(TagCheckArgs a)
{
    const int64_t r = blockIdx.x;
    const int64_t len = a.seq_lens[r] > 0 ? a.seq_lens[r] : 0;
    int64_t used = (len + a.page_size - 1) / a.page_size;
    bool bad = false;
    if (used > a.max_pages_per_seq) {
        bad = true;
        used = a.max_pages_per_seq;
    }
    const int32_t *bt = a.block_table + r * a.max_pages_per_seq;
    const uint32_t *exp = a.expected_tags + r * a.max_pages_per_seq;
    for (int64_t i = threadIdx.x; i < used; i += kTagThreads) {
        const int32_t p = __ldg(bt + i);
        const uint32_t want = __ldg(exp + i);
        if (p < 0 || p >= a.num_pages || __ldg(a.page_tags + p) != want)
            bad = true;
    }
    bad = __syncthreads_or(bad);
    if (threadIdx.x == 0)
        a.abort_flags[r] = bad ? 1 : 0;
}

} // namespace

cudaError_t launch_tag_check(const TagCheckArgs &a, cudaStream_t stream)
{
    if (a.batch == 0)
        return cudaSuccess;
    tag_check_kernel<<<static_cast<unsigned>(a.batch), kTagThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

} // namespace kvq
