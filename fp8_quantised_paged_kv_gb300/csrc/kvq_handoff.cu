// kvq_handoff.cu -- handing prefill pages to the FP8 decode pool.
//
// Prefill is compute-bound and keeps its cache in BF16; only the decode pool
// stores FP8 (blog post "Smaller, faster, safer", page-1 mirror section
// "量化KV缓存"; page-2 mirror section "KV Cache 量化以提高并发量"; page-3
// mirror section "FP8 省的不仅是显存").  So pages that move from prefill to
// decode are quantised whole:
//   amax_kernel + scales_kernel   per-KV-head scale = amax / 448 over the
//                                 listed bf16 pages (1 if amax is 0)
//   quantize_pages_kernel         bf16 page src[i] -> e4m3 page dst[i],
//                                 element by element e4m3(x / scale[h]) --
//                                 the append rule on every slot
// All three are plain HBM streams: the amax pass reads 2 B per element, the
// quantise pass reads 2 B and writes 1 B per element.
#include "kvq_rowops.cuh"

namespace kvq {
namespace {

constexpr int kHandoffThreads = 256;

// One CTA per (listed page, KV head, K|V): max |x| of the ps x 128 tile,
// folded into amax_bits[kv][h] with an integer max on the float's bits
// (valid because every value folded is non-negative).
__global__ void __launch_bounds__(kHandoffThreads) amax_kernel(HandoffArgs a)
{
    const int i = blockIdx.x, h = blockIdx.y, kv = blockIdx.z;
    const int32_t page = a.src_pages[i];
    if (page < 0 || page >= a.src_num_pages)
        return;
    const uint16_t *src = static_cast<const uint16_t *>(kv ? a.v_src : a.k_src) +
                          (static_cast<int64_t>(page) * a.num_kv_heads + h) * a.page_size * kHeadDim;
    const int vecs = a.page_size * kHeadDim / 8;
    float m = 0.f;
    for (int v = threadIdx.x; v < vecs; v += kHandoffThreads) {
        const uint4 x = __ldg(reinterpret_cast<const uint4 *>(src) + v);
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 f = bf16x2_to_f32x2(w[j]);
            m = fmaxf(m, fmaxf(fabsf(f.x), fabsf(f.y)));
        }
    }
    for (int off = 16; off > 0; off >>= 1)
        m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
    __shared__ float red[kHandoffThreads / 32];
    if (threadIdx.x % 32 == 0)
        red[threadIdx.x / 32] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < kHandoffThreads / 32; ++w)
            m = fmaxf(m, red[w]);
        atomicMax(reinterpret_cast<unsigned int *>(kv ? a.v_scale_out : a.k_scale_out) + h,
                  __float_as_uint(m));
    }
}

// amax bits (in the output arrays) -> scale = amax / 448, or 1 when amax is 0.
__global__ void scales_kernel(HandoffArgs a)
{
    for (int i = threadIdx.x; i < 2 * a.num_kv_heads; i += blockDim.x) {
        float *out = i < a.num_kv_heads ? a.k_scale_out + i : a.v_scale_out + (i - a.num_kv_heads);
        const float amax = __uint_as_float(*reinterpret_cast<unsigned int *>(out));
        *out = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
    }
}

// 16 rows (of 128 elements) per CTA; rows enumerate (listed page, K|V, KV
// head, slot).  A listed pair whose source or destination page id is out of
// range is skipped.
__global__ void __launch_bounds__(kHandoffThreads) quantize_pages_kernel(HandoffArgs a)
{
    const int64_t row = static_cast<int64_t>(blockIdx.x) * (kHandoffThreads / kThreadsPerRow) +
                        threadIdx.x / kThreadsPerRow;
    const int part = threadIdx.x % kThreadsPerRow;
    const int64_t rows_per_page = 2LL * a.num_kv_heads * a.page_size;
    if (row >= rows_per_page * a.num_listed)
        return;
    const int64_t i = row / rows_per_page;
    const int64_t rem = row % rows_per_page;
    const int kv = static_cast<int>(rem / (static_cast<int64_t>(a.num_kv_heads) * a.page_size));
    const int h = static_cast<int>((rem / a.page_size) % a.num_kv_heads);
    const int slot = static_cast<int>(rem % a.page_size);
    const int32_t sp = __ldg(a.src_pages + i), dp = __ldg(a.dst_pages + i);
    if (sp < 0 || sp >= a.src_num_pages || dp < 0 || dp >= a.dst_num_pages)
        return;
    const int64_t src_row = (static_cast<int64_t>(sp) * a.num_kv_heads + h) * a.page_size + slot;
    const int64_t dst_row = (static_cast<int64_t>(dp) * a.num_kv_heads + h) * a.page_size + slot;
    const uint4 x = __ldg(reinterpret_cast<const uint4 *>(
        static_cast<const uint16_t *>(kv ? a.v_src : a.k_src) + src_row * kHeadDim + part * 8));
    const float scale = __ldg((kv ? a.v_scale : a.k_scale) + h);
    store_row_part<false>(static_cast<uint8_t *>(kv ? a.v_dst : a.k_dst) + dst_row * kHeadDim, part, x,
                          scale);
}

} // namespace

cudaError_t launch_amax_scales(const HandoffArgs &a, cudaStream_t stream)
{
    cudaError_t e = cudaMemsetAsync(a.k_scale_out, 0, sizeof(float) * a.num_kv_heads, stream);
    if (e == cudaSuccess)
        e = cudaMemsetAsync(a.v_scale_out, 0, sizeof(float) * a.num_kv_heads, stream);
    if (e != cudaSuccess)
        return e;
    if (a.num_listed > 0) {
        const dim3 grid(static_cast<unsigned>(a.num_listed), static_cast<unsigned>(a.num_kv_heads), 2);
        amax_kernel<<<grid, kHandoffThreads, 0, stream>>>(a);
        e = cudaGetLastError();
        if (e != cudaSuccess)
            return e;
    }
    scales_kernel<<<1, 128, 0, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_quantize_pages(const HandoffArgs &a, cudaStream_t stream)
{
    const int64_t rows = 2LL * a.num_kv_heads * a.page_size * a.num_listed;
    if (rows == 0)
        return cudaSuccess;
    const int64_t per_block = kHandoffThreads / kThreadsPerRow;
    const int64_t blocks = (rows + per_block - 1) / per_block;
    if (blocks > 0x7FFFFFFF)
        return cudaErrorInvalidValue;
    quantize_pages_kernel<<<static_cast<unsigned>(blocks), kHandoffThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

} // namespace kvq
