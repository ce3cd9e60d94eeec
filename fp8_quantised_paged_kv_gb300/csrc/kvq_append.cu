// kvq_append.cu -- quantise-on-append of new K/V tokens into the paged cache.
//
// The cache is kept as FP8 e4m3 instead of BF16, halving its size (blog post
// "Smaller, faster, safer: running Kimi and GLM at scale", page-1 mirror,
// section "量化KV缓存").  Each element becomes e4m3(x / scale[h]): the
// division is one IEEE fp32 round-to-nearest operation and the conversion
// rounds to nearest even and saturates at +-448 (cvt ... .satfinite).
//
// One row = one (token, K|V, KV head) vector of 128 elements; 16 threads per
// row, each loading 16 bytes (8 bf16) and storing 8 bytes (8 codes), so both
// the bf16 source and the paged destination are accessed fully coalesced.
#include "kvq_rowops.cuh"

namespace kvq {
namespace {

constexpr int kAppendThreads = 256;

template <bool kBf16Cache>
__global__ void __launch_bounds__(kAppendThreads) append_kernel(AppendArgs a)
{
    grid_launch_dependents();              // a dependent decode launch may begin now
    const int64_t row = static_cast<int64_t>(blockIdx.x) * (kAppendThreads / kThreadsPerRow) +
                        threadIdx.x / kThreadsPerRow;
    const int part = threadIdx.x % kThreadsPerRow;
    const int64_t rows = static_cast<int64_t>(a.num_tokens) * 2 * a.num_kv_heads;
    if (row >= rows)
        return;
    const int64_t t = row / (2 * a.num_kv_heads);
    const int rem = static_cast<int>(row % (2 * a.num_kv_heads));
    const bool is_v = rem >= a.num_kv_heads;
    const int h = is_v ? rem - a.num_kv_heads : rem;

    // every load is issued before the first decision, so the kernel waits on
    // one round trip to memory, not a chain of them
    const uint16_t *src = static_cast<const uint16_t *>(is_v ? a.v_new : a.k_new) +
                          (t * a.num_kv_heads + h) * kHeadDim + part * 8;
    const uint4 x = __ldg(reinterpret_cast<const uint4 *>(src));
    const int64_t slot = __ldg(a.slot_mapping + t);
    const bool aborted = a.abort_flags != nullptr && __ldg(a.abort_flags + t) != 0;
    const float scale = kBf16Cache ? 1.f : __ldg((is_v ? a.v_scale : a.k_scale) + h);
    if (aborted || slot < 0 || slot >= a.num_slots)
        return;
    const int64_t page = slot / a.page_size;
    const int64_t off = slot % a.page_size;
    const int64_t dst_row = (page * a.num_kv_heads + h) * a.page_size + off;

    void *cache = is_v ? a.v_cache : a.k_cache;
    void *dst = kBf16Cache ? static_cast<void *>(static_cast<uint16_t *>(cache) + dst_row * kHeadDim)
                           : static_cast<void *>(static_cast<uint8_t *>(cache) + dst_row * kHeadDim);
    store_row_part<kBf16Cache>(dst, part, x, scale);
}

} // namespace

cudaError_t launch_append(const AppendArgs &a, cudaStream_t stream)
{
    const int64_t rows = static_cast<int64_t>(a.num_tokens) * 2 * a.num_kv_heads;
    if (rows == 0)
        return cudaSuccess;
    const int64_t rows_per_block = kAppendThreads / kThreadsPerRow;
    const int64_t blocks = (rows + rows_per_block - 1) / rows_per_block;
    if (blocks > 0x7FFFFFFF)
        return cudaErrorInvalidValue;
    if (a.bf16_cache)
        append_kernel<true><<<static_cast<unsigned>(blocks), kAppendThreads, 0, stream>>>(a);
    else
        append_kernel<false><<<static_cast<unsigned>(blocks), kAppendThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

} // namespace kvq
