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
// One CTA per request: its 512 threads take the ceil(L / page_size) entries
// the request uses, 4,096 per pass, issuing every block-table and
// expected-tag load of the pass before the live-tag gathers, so a pass costs
// two rounds of dependent loads; OR-reduce with __syncthreads_or; thread 0
// writes the flag (0 or 1).
#include "kvq_rowops.cuh"

namespace kvq {
namespace {

constexpr int kTagThreads = 512;

#ifdef KVQ_PHASE_STAMPS
// Instrumented build only: %globaltimer at entry (point 0) and when the flag
// is written (1) by thread 0 of every CTA of the last launch.
constexpr int kTagStampCtas = 4096;
__device__ unsigned long long g_tag_stamps[kTagStampCtas * 2];
__device__ __forceinline__ void tag_stamp(int point)
{
    if (threadIdx.x == 0 && blockIdx.x < kTagStampCtas)
        g_tag_stamps[blockIdx.x * 2 + point] = global_timer_ns();
}
#define KVQ_TAG_STAMP(p) tag_stamp(p)
#else
#define KVQ_TAG_STAMP(p) ((void)0)
#endif

__global__ void __launch_bounds__(kTagThreads) tag_check_kernel(TagCheckArgs a)
{
    KVQ_TAG_STAMP(0);
    grid_launch_dependents();              // a dependent decode launch may begin now
    const int64_t r = blockIdx.x;
    const bool bad = tag_check_request<8>(a.block_table, a.expected_tags, a.seq_lens, a.page_tags,
                                          a.max_pages_per_seq, a.page_size, a.num_pages, r);
    if (threadIdx.x == 0)
        a.abort_flags[r] = bad ? 1 : 0;
    KVQ_TAG_STAMP(1);
}

} // namespace

cudaError_t launch_tag_check(const TagCheckArgs &a, cudaStream_t stream)
{
    if (a.batch == 0)
        return cudaSuccess;
    tag_check_kernel<<<static_cast<unsigned>(a.batch), kTagThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

#ifdef KVQ_PHASE_STAMPS
cudaError_t read_tag_stamps(unsigned long long *host, size_t count)
{
    const size_t n = count < static_cast<size_t>(kTagStampCtas * 2) ? count : kTagStampCtas * 2;
    return cudaMemcpyFromSymbol(host, g_tag_stamps, n * sizeof(unsigned long long));
}
#endif

} // namespace kvq
