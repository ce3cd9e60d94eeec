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
// One CTA per request: its 256 threads take the ceil(L / page_size) entries
// the request uses, 1,024 per pass, issuing every block-table and
// expected-tag load of the pass before the live-tag gathers, so a pass costs
// two rounds of dependent loads; OR-reduce with __syncthreads_or; thread 0
// writes the flag (0 or 1).
#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr int kTagThreads = 256;
constexpr int kTagUnroll = 4;          // entries per thread per pass: all loads issued before any use

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
    for (int64_t base = 0; base < used; base += kTagThreads * kTagUnroll) {
        int32_t p[kTagUnroll];
        uint32_t want[kTagUnroll], live[kTagUnroll];
#pragma unroll
        for (int k = 0; k < kTagUnroll; ++k) {
            const int64_t i = base + k * kTagThreads + threadIdx.x;
            p[k] = i < used ? __ldg(bt + i) : 0;
            want[k] = i < used ? __ldg(exp + i) : 0u;
        }
#pragma unroll
        for (int k = 0; k < kTagUnroll; ++k) {
            const bool in_range = p[k] >= 0 && p[k] < a.num_pages;
            live[k] = in_range ? __ldg(a.page_tags + p[k]) : 0u;
        }
#pragma unroll
        for (int k = 0; k < kTagUnroll; ++k) {
            const int64_t i = base + k * kTagThreads + threadIdx.x;
            if (i < used && (p[k] < 0 || p[k] >= a.num_pages || live[k] != want[k]))
                bad = true;
        }
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
