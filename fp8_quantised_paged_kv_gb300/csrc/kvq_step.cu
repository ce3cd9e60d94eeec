// kvq_step.cu -- the two passes that precede attention in a decode step,
// fused into one launch: the batched per-page tag check (blog post
// "Smaller, faster, safer", page-2 mirror section "KV Cache 完整性检查";
// page-3 mirror section "一个不能出错的共享缓存") and the quantise-on-append
// of each request's new token (page-1 mirror section "量化KV缓存").
//
// One CTA per request r, whose new token is token r.  The CTA first issues
// the loads of the token's K/V rows, slot and scales, then tag-checks the
// request's pages (the same computation as tag_check_kernel), writes the
// abort flag, and stores the token's codes only if the request passed.  The
// check still runs, and finishes, before anything of the request is written;
// the fusion only removes a launch and overlaps the two sets of loads.
#include "kvq_rowops.cuh"

namespace kvq {
namespace {

constexpr int kStepThreads = 512;

#ifdef KVQ_PHASE_STAMPS
// Instrumented build only: %globaltimer at entry (point 0) and exit (1) of
// thread 0 of every CTA of the last launch.
constexpr int kCheckStampCtas = 4096;
__device__ unsigned long long g_check_stamps[kCheckStampCtas * 2];
__device__ __forceinline__ void check_stamp(int point)
{
    if (threadIdx.x == 0 && blockIdx.x < kCheckStampCtas)
        g_check_stamps[blockIdx.x * 2 + point] = global_timer_ns();
}
#define KVQ_CHECK_STAMP(p) check_stamp(p)
#else
#define KVQ_CHECK_STAMP(p) ((void)0)
#endif
constexpr int kMaxRowsPerPass = kStepThreads / kThreadsPerRow;   // 32 rows (K and V of 16 heads)

template <bool kBf16Cache>
__global__ void __launch_bounds__(kStepThreads) tag_check_append_kernel(TagCheckArgs t, AppendArgs a)
{
    KVQ_CHECK_STAMP(0);
    grid_launch_dependents();              // a dependent decode launch may begin now
    const int64_t r = blockIdx.x;
    const int rows = 2 * a.num_kv_heads;
    const int part = threadIdx.x % kThreadsPerRow;
    // loads of this request's new token (first pass of rows), before the check
    const int row0 = threadIdx.x / kThreadsPerRow;
    uint4 x = make_uint4(0, 0, 0, 0);
    float scale = 1.f;
    if (row0 < rows) {
        const bool is_v = row0 >= a.num_kv_heads;
        const int h = is_v ? row0 - a.num_kv_heads : row0;
        x = __ldg(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(is_v ? a.v_new : a.k_new) +
                                                  (r * a.num_kv_heads + h) * kHeadDim + part * 8));
        scale = kBf16Cache ? 1.f : __ldg((is_v ? a.v_scale : a.k_scale) + h);
    }
    const int64_t slot = __ldg(a.slot_mapping + r);

    const bool bad = tag_check_request<8>(t.block_table, t.expected_tags, t.seq_lens, t.page_tags,
                                          t.max_pages_per_seq, t.page_size, t.num_pages, r);
    if (threadIdx.x == 0)
        t.abort_flags[r] = bad ? 1 : 0;
    KVQ_CHECK_STAMP(1);
    if (bad || slot < 0 || slot >= a.num_slots)
        return;
    const int64_t page = slot / a.page_size;
    const int64_t off = slot % a.page_size;
    for (int row = row0; row < rows; row += kMaxRowsPerPass) {
        const bool is_v = row >= a.num_kv_heads;
        const int h = is_v ? row - a.num_kv_heads : row;
        if (row != row0) {
            x = __ldg(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(is_v ? a.v_new : a.k_new) +
                                                      (r * a.num_kv_heads + h) * kHeadDim + part * 8));
            scale = kBf16Cache ? 1.f : __ldg((is_v ? a.v_scale : a.k_scale) + h);
        }
        const int64_t dst_row = (page * a.num_kv_heads + h) * a.page_size + off;
        void *cache = is_v ? a.v_cache : a.k_cache;
        void *dst = kBf16Cache ? static_cast<void *>(static_cast<uint16_t *>(cache) + dst_row * kHeadDim)
                               : static_cast<void *>(static_cast<uint8_t *>(cache) + dst_row * kHeadDim);
        store_row_part<kBf16Cache>(dst, part, x, scale);
    }
}

} // namespace

cudaError_t launch_tag_check_append(const TagCheckArgs &t, const AppendArgs &a, cudaStream_t stream)
{
    if (t.batch == 0)
        return cudaSuccess;

    if (a.bf16_cache)
        tag_check_append_kernel<true><<<static_cast<unsigned>(t.batch), kStepThreads, 0, stream>>>(t, a);
    else
        tag_check_append_kernel<false><<<static_cast<unsigned>(t.batch), kStepThreads, 0, stream>>>(t, a);
    return cudaGetLastError();
}

#ifdef KVQ_PHASE_STAMPS
cudaError_t read_check_stamps(unsigned long long *host, size_t count)
{
    const size_t n = count < static_cast<size_t>(kCheckStampCtas * 2) ? count : kCheckStampCtas * 2;
    return cudaMemcpyFromSymbol(host, g_check_stamps, n * sizeof(unsigned long long));
}
#endif

} // namespace kvq
