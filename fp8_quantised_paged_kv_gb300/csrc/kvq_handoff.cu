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
// quantise pass reads 2 B and writes 1 B per element.  Both run one wave of
// 256-thread CTAs (8 per SM for amax, 4 for quantise); a warp streams one
// (page, head) tile at a time with eight 16-byte loads in flight per lane.
// Each quotient is the correctly rounded one, as the append rule's IEEE
// division gives it, but from a multiplication by RN(1 / scale) and one
// correction step (quotient_rn): no division per element.
// The tile loads are streaming loads (evict first): they do not push out
// of L2 what is already there (dirty lines that would have to be written
// back meanwhile), which made the amax pass 13 % faster.
#include "kvq_rowops.cuh"

namespace kvq {
namespace {

constexpr int kHandoffThreads = 256;
constexpr int kHandoffWarps = kHandoffThreads / 32;
constexpr int kVecsPerLane = 8;          // 16-byte loads in flight per lane
constexpr int kCtasPerSmAmax = 8;        // 2,048 threads per SM
constexpr int kCtasPerSmQuant = 4;       // 1,024 threads per SM (64 registers each)

__device__ __forceinline__ float absmax8(uint4 x, float m)
{
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float2 f = bf16x2_to_f32x2(w[k]);
        m = fmaxf(m, fmaxf(fabsf(f.x), fabsf(f.y)));
    }
    return m;
}

// CTA (x = K|V x KV head, y): its warps take every (gridDim.y x 8)-th listed
// page, one page's (ps x 128) tile of the CTA's head at a time, eight 16-byte
// loads in flight per lane; the next page id is loaded while the current tile
// streams.  The CTA's max |x| is folded into amax_bits[kv][h] with an integer
// max on the float's bits (valid because every value folded is non-negative).
__global__ void __launch_bounds__(kHandoffThreads, kCtasPerSmAmax) amax_kernel(HandoffArgs a)
{
    const int kv = blockIdx.x / a.num_kv_heads, h = blockIdx.x % a.num_kv_heads;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int per_tile = a.page_size * kHeadDim / 8;             // 16-byte vectors per tile
    const int64_t step = static_cast<int64_t>(gridDim.y) * kHandoffWarps;
    const uint4 *base = reinterpret_cast<const uint4 *>(kv ? a.v_src : a.k_src);
    float m = 0.f;
    int64_t i = static_cast<int64_t>(blockIdx.y) * kHandoffWarps + warp;
    int32_t page = i < a.num_listed ? __ldg(a.src_pages + i) : -1;
    for (; i < a.num_listed; i += step) {
        const int32_t next = i + step < a.num_listed ? __ldg(a.src_pages + i + step) : -1;
        if (page >= 0 && page < a.src_num_pages) {
            const uint4 *tile = base + (static_cast<int64_t>(page) * a.num_kv_heads + h) * per_tile;
            for (int e0 = 0; e0 < per_tile; e0 += 32 * kVecsPerLane) {
                uint4 x[kVecsPerLane];
#pragma unroll
                for (int k = 0; k < kVecsPerLane; ++k) {
                    const int e = e0 + k * 32 + lane;
                    x[k] = e < per_tile ? __ldcs(tile + e) : make_uint4(0u, 0u, 0u, 0u);
                }
#pragma unroll
                for (int k = 0; k < kVecsPerLane; ++k)
                    m = absmax8(x[k], m);
            }
        }
        page = next;
    }
    for (int off = 16; off > 0; off >>= 1)
        m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
    __shared__ float red[kHandoffWarps];
    if (lane == 0)
        red[warp] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < kHandoffWarps; ++w)
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

// One warp's (page, head) tile: per_tile 16-byte bf16 vectors to 8-byte
// e4m3 vectors, eight loads in flight per lane.  kRcp: the quotients from
// quotient_rn; otherwise one IEEE division each (scales outside its range).
template <bool kRcp>
__device__ __forceinline__ void quantize_tile(const uint4 *__restrict__ src, uint2 *__restrict__ dst,
                                              int per_tile, int lane, const QuotientRcp &c)
{
    for (int e0 = 0; e0 < per_tile; e0 += 32 * kVecsPerLane) {
        uint4 x[kVecsPerLane];
#pragma unroll
        for (int k = 0; k < kVecsPerLane; ++k) {
            const int e = e0 + k * 32 + lane;
            x[k] = e < per_tile ? __ldcs(src + e) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int k = 0; k < kVecsPerLane; ++k) {
            const int e = e0 + k * 32 + lane;
            if (e < per_tile) {
                if constexpr (kRcp)
                    dst[e] = make_uint2(encode4_e4m3_rcp(x[k].x, x[k].y, c),
                                        encode4_e4m3_rcp(x[k].z, x[k].w, c));
                else
                    dst[e] = make_uint2(encode4_e4m3(x[k].x, x[k].y, c.scale),
                                        encode4_e4m3(x[k].z, x[k].w, c.scale));
            }
        }
    }
}

// One warp per (listed pair, K|V, KV head) tile at a time, grid-stride over
// the tiles; eight 16-byte loads (64 bf16 elements) in flight per lane; the
// next tile's page ids are loaded while the current one streams.  Every
// element becomes e4m3(x / scale[h]) by the append rule.  A listed pair whose
// source or destination page id is out of range is skipped.
__global__ void __launch_bounds__(kHandoffThreads, kCtasPerSmQuant) quantize_pages_kernel(HandoffArgs a)
{
    const int lane = threadIdx.x % 32;
    const int per_tile = a.page_size * kHeadDim / 8;
    const int64_t tiles = 2LL * a.num_kv_heads * a.num_listed;
    const int64_t step = static_cast<int64_t>(gridDim.x) * kHandoffWarps;
    int64_t t = static_cast<int64_t>(blockIdx.x) * kHandoffWarps + threadIdx.x / 32;
    auto ids = [&](int64_t tile) {
        const int64_t i = tile / (2LL * a.num_kv_heads);
        return make_int2(__ldg(a.src_pages + i), __ldg(a.dst_pages + i));
    };
    int2 cur = t < tiles ? ids(t) : make_int2(-1, -1);
    for (; t < tiles; t += step) {
        const int2 next = t + step < tiles ? ids(t + step) : make_int2(-1, -1);
        const int h = static_cast<int>(t % a.num_kv_heads);
        const int kv = static_cast<int>((t / a.num_kv_heads) % 2);
        if (cur.x >= 0 && cur.x < a.src_num_pages && cur.y >= 0 && cur.y < a.dst_num_pages) {
            const uint4 *src = reinterpret_cast<const uint4 *>(kv ? a.v_src : a.k_src) +
                               (static_cast<int64_t>(cur.x) * a.num_kv_heads + h) * per_tile;
            uint2 *dst = reinterpret_cast<uint2 *>(kv ? a.v_dst : a.k_dst) +
                         (static_cast<int64_t>(cur.y) * a.num_kv_heads + h) * per_tile;
            const float scale = __ldg((kv ? a.v_scale : a.k_scale) + h);
            QuotientRcp c;
            if (quotient_rcp_init(scale, c))
                quantize_tile<true>(src, dst, per_tile, lane, c);
            else
                quantize_tile<false>(src, dst, per_tile, lane, c);
        }
        cur = next;
    }
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
        // about kCtasPerSmAmax CTAs per SM in all (one wave), every CTA on one head
        const int heads2 = 2 * a.num_kv_heads;
        int64_t py = static_cast<int64_t>(device_sm_count()) * kCtasPerSmAmax / heads2;
        const int64_t most = (a.num_listed + kHandoffWarps - 1) / kHandoffWarps;
        py = py < 1 ? 1 : (py > most ? most : py);
        py = py > 65535 ? 65535 : py;
        const dim3 grid(static_cast<unsigned>(heads2), static_cast<unsigned>(py));
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
    const int64_t tiles = 2LL * a.num_kv_heads * a.num_listed;
    if (tiles == 0)
        return cudaSuccess;
    int64_t blocks = static_cast<int64_t>(device_sm_count()) * kCtasPerSmQuant;
    const int64_t need = (tiles + kHandoffWarps - 1) / kHandoffWarps;
    blocks = blocks < need ? blocks : need;
    quantize_pages_kernel<<<static_cast<unsigned>(blocks), kHandoffThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

} // namespace kvq
