// kvq_w4a16.cu -- INT4 weight-only product for decode, on the tensor cores.
//
// What it computes (blog post "Smaller, faster, safer: running Kimi and GLM
// at scale", page-1 mirror section "压缩模型权重"; page-2 mirror section
// "模型权重压缩以降低延迟"): decode streams the model's weights from HBM, so
// 4-bit weights move less data; they are expanded before the multiply.  The
// pages fix no format; the one taken here is symmetric signed 4-bit q with
// one bf16 scale per output column and group of 128 k, byte k/2 of row n of
// W holding q[n][k] (low nibble: even k):
//   y[m][n] = sum_k x[m][k] * q[n][k] * s[n][k / 128]
//
// A CTA owns 64 output columns and one of `splits` ranges of K.  Its four
// warps take turns over that range one 128-k group at a time; a group is one
// 2-D tensor copy (TMA, 64-byte swizzle) of 64 weight rows x 64 bytes into
// the warp's 4-stage ring, so three copies stay in flight while the warp
// works on the fourth.  Per group a lane expands the nibbles of two
// weight columns of each 16-column tile into exact f16 integers (nibble |
// 0x6400 is the f16 value 1024 + nibble) and multiplies them with x on the
// tensor cores (mma.sync m16n8k16, f16 in, fp32 accumulate).  The weight
// columns are the mma's M and the rows of x its N, so a batch of up to 8
// rows costs one n-tile and 9..16 rows two: decode's few rows do not pay
// for a 16-row tile.  Each group is folded into the result with the
// columns' scales in fp32.  A lane reads 32 contiguous k of x and of each
// weight column: k-slot pairs of the mma hold elements (e, e + 4) of each
// group of eight, the pairing that the nibble expansion produces.  The
// warps' partials meet in shared memory; the splits of a column tile form
// one thread-block cluster and merge through distributed shared memory.
#include <map>
#include <mutex>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kvq_internal.h"
#include "kvq_ptx.cuh"

namespace kvq {

// Sticky device error word of this kernel family (bit 0: a copy wait timed out).
__device__ unsigned int g_w4_error = 0;

namespace {

constexpr int kW4Warps = 4;
constexpr int kW4Threads = kW4Warps * 32;
constexpr int kW4CtasPerSm = 3;
constexpr int kW4Stages = 4;
constexpr int kW4StageBytes = kW4Cols * kW4CopyK / 2;          // 64 rows x 64 bytes: one group
constexpr int kW4WarpRing = kW4Stages * kW4StageBytes;
constexpr int kW4RingBytes = kW4Warps * kW4WarpRing;
constexpr int kW4MaxGroups = 64;                               // groups of one split: k_split <= 8192
constexpr int kW4ScStride = kW4MaxGroups + 2;                  // halves per column: rows 132 bytes apart
constexpr int kW4SmemBytes = 1024 /* alignment slack */ + kW4RingBytes + kW4Warps * kW4Stages * 8 +
                             kW4Cols * kW4ScStride * 2 /* scales */ + 16;
constexpr uint64_t kW4WaitLimitNs = 1000000000ull;
// A warp's partial [16 rows][64 columns] in its idle ring, rows 68 floats
// apart: the four row pairs a lane group stores land in different banks.
constexpr int kW4RedStride = kW4Cols + 4;
static_assert(16 * kW4RedStride * 4 <= kW4WarpRing, "a warp's partial fits in its idle ring");
static_assert(16 * kW4Cols * 4 <= kW4Cols * kW4ScStride * 2, "the CTA's partial fits over the scales");

// Byte offset of 16-byte chunk c of row `line` in a tile of 64-byte rows
// written by a tensor copy with 64-byte swizzle.
__device__ __forceinline__ uint32_t swz64(int line, int c)
{
    return static_cast<uint32_t>(line * 64 + ((c ^ ((line >> 1) & 3)) << 4));
}

// (a & b) ^ c
__device__ __forceinline__ uint32_t and_xor(uint32_t a, uint32_t b, uint32_t c)
{
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Four 8x8 b16 matrices from shared memory: lane l gives the address of row
// l % 8 of matrix l / 8 and receives, of each matrix, row l / 4, b16
// elements 2 (l % 4) and 2 (l % 4) + 1.
__device__ __forceinline__ uint4 ldmatrix_x4(uint32_t addr)
{
    uint4 r;
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "r"(addr));
    return r;
}

__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }
__device__ __forceinline__ __half2 bits_h2(uint32_t u) { return *reinterpret_cast<__half2 *>(&u); }

// Two bf16 (as f32) -> f16x2, low half first.
__device__ __forceinline__ uint32_t f16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ void store_y(void *y, int64_t idx, float v, bool fp32)
{
    if (fp32)
        static_cast<float *>(y)[idx] = v;
    else
        static_cast<__nv_bfloat16 *>(y)[idx] = __float2bfloat16_rn(v);
}

template <bool kCluster, int kNT>
__global__ void __launch_bounds__(kW4Threads, kW4CtasPerSm)
w4a16_kernel(const __grid_constant__ CUtensorMap w_map, const W4Args a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kW4RingBytes);
    uint16_t *sc_sm = reinterpret_cast<uint16_t *>(full + kW4Warps * kW4Stages);   // [64][kW4ScStride]
    __shared__ int s_failed;

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int gq = lane >> 2, tq = lane & 3;
    const int col0 = blockIdx.x * kW4Cols;
    const int k0 = blockIdx.y * a.k_split;
    const int kcount = a.k - k0 < a.k_split ? a.k - k0 : a.k_split;   // a multiple of 256
    const int nblocks = kcount / kW4CopyK;                            // copies, one group each
    const int groups = nblocks;
    const int gtot = a.k / 128;

    const uint64_t policy = l2_policy_evict_first();
    // copy `it` of warp w: block w + it * kW4Warps into stage it % kW4Stages of w's ring
    auto issue = [&](int w, int it) {
        const int blk = w + it * kW4Warps;
        const int st = it % kW4Stages;
        uint64_t *bar = full + w * kW4Stages + st;
        mbar_arrive_expect_tx(bar, kW4StageBytes);
        tma_load_2d(smem + w * kW4WarpRing + st * kW4StageBytes, &w_map, (k0 + blk * kW4CopyK) / 2, col0, bar,
                    policy);
    };
    // The first copies of every warp start before the scales are read, so
    // that the prologue overlaps the weight stream.
    if (threadIdx.x == 0) {
        prefetch_tensor_map(&w_map);
        s_failed = 0;
        for (int i = 0; i < kW4Warps * kW4Stages; ++i)
            mbar_init(&full[i], 1);
        fence_mbar_init();
        fence_proxy_async_smem();
        for (int it = 0; it < kW4Stages; ++it)
            for (int w = 0; w < kW4Warps; ++w)
                if (w + it * kW4Warps < nblocks)
                    issue(w, it);
    }
    // this CTA's scales, [column][group] with a padded row (consecutive
    // threads read consecutive groups of a column)
    for (int i = threadIdx.x; i < groups * kW4Cols; i += kW4Threads) {
        const int c = i / groups, g = i % groups;
        sc_sm[c * kW4ScStride + g] = __ldg(static_cast<const uint16_t *>(a.scales) +
                                           static_cast<int64_t>(col0 + c) * gtot + k0 / 128 + g);
    }
    __syncthreads();

    const int my_blocks = nblocks > warp ? (nblocks - warp + kW4Warps - 1) / kW4Warps : 0;
    uint8_t *ring = smem + warp * kW4WarpRing;
    uint64_t *my_full = full + warp * kW4Stages;

    const uint16_t *xb = static_cast<const uint16_t *>(a.x);
    const __half2 minus1032 = bits_h2(0xE408E408u);      // -1032
    const __half2 sixteenth = bits_h2(0x2C002C00u);      // 1/16
    const __half2 minus72 = bits_h2(0xD480D480u);        // -72

    // acc[mt][nt][.]: weight columns mt * 16 + gq (0, 1) and + 8 (2, 3) of
    // the tile, batch rows nt * 8 + 2 tq (0, 2) and + 1 (1, 3)
    float acc[4][kNT][4];
#pragma unroll
    for (int mt = 0; mt < 4; ++mt)
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt)
            acc[mt][nt][0] = acc[mt][nt][1] = acc[mt][nt][2] = acc[mt][nt][3] = 0.f;

    // x of one 128-k group for this lane: batch rows nt * 8 + gq, the eight k
    // kg + 32 j + 8 tq .. + 7 for j = 0..3 (the k the lane's weight words
    // cover).  Loaded one group ahead, so the load overlaps a group of work.
    uint4 xr[kNT][4];
    auto load_x = [&](int kg) {
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt) {
            const int row = nt * 8 + gq;
            const uint16_t *p = xb + static_cast<int64_t>(row) * a.k + kg + 8 * tq;
#pragma unroll
            for (int j = 0; j < 4; ++j)
                xr[nt][j] = row < a.rows ? __ldg(reinterpret_cast<const uint4 *>(p + 32 * j))
                                         : make_uint4(0u, 0u, 0u, 0u);
        }
    };
    if (my_blocks > 0)
        load_x(k0 + warp * kW4CopyK);

    // The weights of a word (eight nibbles, k = e0 .. e7) as two f16 pairs:
    // flipping a nibble's top bit turns two's complement q into q + 8; with
    // 0x64 above it a half is the f16 1024 + (q + 8).  Nibbles (0, 4) give
    // (e0, e4) that way; nibbles (1, 5) sit 4 bits higher and give
    // 1024 + 16 (q + 8) for (e1, e5).  Both become exact integers q.
    auto q_even = [&](uint32_t u) {
        return h2_bits(__hadd2(bits_h2(and_xor(u, 0x000F000Fu, 0x64086408u)), minus1032));
    };
    auto q_odd = [&](uint32_t u) {
        return h2_bits(__hfma2(bits_h2(and_xor(u, 0x00F000F0u, 0x64806480u)), sixteenth, minus72));
    };

    bool failed = false;
    int it = 0;
    for (; it < my_blocks; ++it) {
        const int st = it % kW4Stages;
        // every lane polls; the warp gives up as one if any lane did
        if (!__all_sync(0xFFFFFFFFu, mbar_wait_bounded(&my_full[st], (it / kW4Stages) & 1, kW4WaitLimitNs))) {
            failed = true;
            break;
        }
        const uint8_t *tile = ring + st * kW4StageBytes;
        const int blk = warp + it * kW4Warps;           // the group this copy holds
        {
            const int kg = k0 + blk * kW4CopyK;
            const int gl = blk;                         // group index within the split
            // x fragments (mma B, k x batch): k-step 2j pairs (e0, e4) and
            // (e1, e5) of word j, k-step 2j+1 (e2, e6) and (e3, e7)
            uint32_t bx[kNT][8][2];
#pragma unroll
            for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint4 x = xr[nt][j];
                    bx[nt][2 * j][0] = f16x2(bf16lo(x.x), bf16lo(x.z));
                    bx[nt][2 * j][1] = f16x2(bf16hi(x.x), bf16hi(x.z));
                    bx[nt][2 * j + 1][0] = f16x2(bf16lo(x.y), bf16lo(x.w));
                    bx[nt][2 * j + 1][1] = f16x2(bf16hi(x.y), bf16hi(x.w));
                }
            // the x of this warp's next group
            if (it + 1 < my_blocks)
                load_x(kg + kW4Warps * kW4CopyK);
#pragma unroll
            for (int mt = 0; mt < 4; ++mt) {            // 16-column tiles (mma A, columns x k)
                // words j of weight rows mt * 16 + gq and + 8: bytes 4 tq ..
                // 4 tq + 3 of 16-byte chunk j (k = kg + 32 j + 8 tq .. + 7);
                // ldmatrix reads each chunk's eight rows conflict-free
                const uint4 w0 = ldmatrix_x4(smem_addr(tile + swz64(mt * 16 + (lane & 7), lane >> 3)));
                const uint4 w1 = ldmatrix_x4(smem_addr(tile + swz64(mt * 16 + 8 + (lane & 7), lane >> 3)));
                const uint32_t u0[4] = {w0.x, w0.y, w0.z, w0.w};
                const uint32_t u1[4] = {w1.x, w1.y, w1.z, w1.w};
                float part[kNT][4];
#pragma unroll
                for (int nt = 0; nt < kNT; ++nt)
                    part[nt][0] = part[nt][1] = part[nt][2] = part[nt][3] = 0.f;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t a00 = q_even(u0[j]), a01 = q_even(u1[j]);
                    const uint32_t a02 = q_odd(u0[j]), a03 = q_odd(u1[j]);
                    const uint32_t a10 = q_even(u0[j] >> 8), a11 = q_even(u1[j] >> 8);
                    const uint32_t a12 = q_odd(u0[j] >> 8), a13 = q_odd(u1[j] >> 8);
#pragma unroll
                    for (int nt = 0; nt < kNT; ++nt) {
                        mma_f16(part[nt], a00, a01, a02, a03, bx[nt][2 * j][0], bx[nt][2 * j][1]);
                        mma_f16(part[nt], a10, a11, a12, a13, bx[nt][2 * j + 1][0], bx[nt][2 * j + 1][1]);
                    }
                }
                // rows gq and gq + 8 of the tile take their columns' scales
                const float s0 =
                    __uint_as_float(static_cast<uint32_t>(sc_sm[(mt * 16 + gq) * kW4ScStride + gl]) << 16);
                const float s1 =
                    __uint_as_float(static_cast<uint32_t>(sc_sm[(mt * 16 + gq + 8) * kW4ScStride + gl]) << 16);
#pragma unroll
                for (int nt = 0; nt < kNT; ++nt) {
                    acc[mt][nt][0] = fmaf(s0, part[nt][0], acc[mt][nt][0]);
                    acc[mt][nt][1] = fmaf(s0, part[nt][1], acc[mt][nt][1]);
                    acc[mt][nt][2] = fmaf(s1, part[nt][2], acc[mt][nt][2]);
                    acc[mt][nt][3] = fmaf(s1, part[nt][3], acc[mt][nt][3]);
                }
            }
        }
        __syncwarp();
        if (lane == 0 && it + kW4Stages < my_blocks) {
            fence_proxy_async_smem();
            issue(warp, it + kW4Stages);
        }
    }
    if (failed) {
        // drain every copy still in flight (the one given up on included)
        // with the full limit; bit 1 if that gives up too
        if (lane == 0) {
            atomicOr(&g_w4_error, 1u);
            s_failed = 1;
        }
        const int issued = my_blocks < it + kW4Stages ? my_blocks : it + kW4Stages;
        bool drained = true;
        for (int j = it; j < issued; ++j)
            drained &= mbar_wait_bounded(&my_full[j % kW4Stages], (j / kW4Stages) & 1, kW4WaitLimitNs);
        if (!drained && lane == 0)
            atomicOr(&g_w4_error, 2u);
    }

    // ---- the four warps' partials (each in its own idle ring), then the CTA's
    constexpr int kRowsT = 8 * kNT;                                  // batch rows the CTA holds
    float *red = reinterpret_cast<float *>(ring);                    // [kRowsT][kW4RedStride]
#pragma unroll
    for (int mt = 0; mt < 4; ++mt)
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt) {
            const int c = mt * 16 + gq, r = nt * 8 + 2 * tq;
            red[r * kW4RedStride + c] = acc[mt][nt][0];
            red[(r + 1) * kW4RedStride + c] = acc[mt][nt][1];
            red[r * kW4RedStride + c + 8] = acc[mt][nt][2];
            red[(r + 1) * kW4RedStride + c + 8] = acc[mt][nt][3];
        }
    __syncthreads();
    float *cta = reinterpret_cast<float *>(sc_sm);                   // [kRowsT][64], scales are done
    for (int o = threadIdx.x; o < kRowsT * kW4Cols; o += kW4Threads) {
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < kW4Warps; ++w)
            v += reinterpret_cast<const float *>(smem + w * kW4WarpRing)[(o / kW4Cols) * kW4RedStride + o % kW4Cols];
        if (s_failed)                               // a copy timed out: this tile gives zeros
            v = 0.f;
        if constexpr (kCluster) {
            cta[o] = v;
        } else if (o / kW4Cols < a.rows) {
            store_y(a.y, static_cast<int64_t>(o / kW4Cols) * a.n + col0 + o % kW4Cols, v, a.out_fp32);
        }
    }
    if constexpr (kCluster) {
        // splits of the column tile: CTA r sums outputs [r, r + n, ...) of every peer
        cluster_sync();
        const int n = a.splits;
        const int rank = static_cast<int>(cluster_ctarank());
        const uint32_t base = smem_addr(cta);
        for (int o = rank * kW4Threads + threadIdx.x; o < kRowsT * kW4Cols; o += n * kW4Threads) {
            if (o / kW4Cols >= a.rows)
                continue;
            float v = 0.f;
            for (int s = 0; s < n; ++s)
                v += ld_shared_cluster_f32(map_shared_rank(base + 4u * o, static_cast<uint32_t>(s)));
            store_y(a.y, static_cast<int64_t>(o / kW4Cols) * a.n + col0 + o % kW4Cols, v, a.out_fp32);
        }
        cluster_sync();
    }
}

template <bool kCluster, int kNT>
cudaError_t configure_w4(int dev)
{
    static int configured[64] = {0};
    if (dev >= 0 && dev < 64 && configured[dev])
        return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(w4a16_kernel<kCluster, kNT>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, kW4SmemBytes);
    if (e == cudaSuccess && dev >= 0 && dev < 64)
        configured[dev] = 1;
    return e;
}

cudaLaunchConfig_t w4_config(dim3 grid, int splits, cudaStream_t stream, cudaLaunchAttribute (&attr)[1])
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kW4Threads);
    cfg.dynamicSmemBytes = kW4SmemBytes;
    cfg.stream = stream;
    cfg.numAttrs = 0;
    if (splits > 1) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 1;
        attr[0].val.clusterDim.y = static_cast<unsigned>(splits);
        attr[0].val.clusterDim.z = 1;
        cfg.numAttrs = 1;
    }
    cfg.attrs = attr;
    return cfg;
}

template <bool kCluster, int kNT>
cudaError_t launch_variant(const cudaLaunchConfig_t &cfg, const CUtensorMap &w_map, const W4Args &a, int dev)
{
    const cudaError_t e = configure_w4<kCluster, kNT>(dev);
    if (e != cudaSuccess)
        return e;
    return cudaLaunchKernelEx(&cfg, w4a16_kernel<kCluster, kNT>, w_map, a);
}

} // namespace

cudaError_t launch_w4a16(const W4Args &a, const CUtensorMap &w_map, cudaStream_t stream)
{
    if (a.rows == 0 || a.n == 0)
        return cudaSuccess;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    const dim3 grid(static_cast<unsigned>(a.n / kW4Cols), static_cast<unsigned>(a.splits), 1);
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = w4_config(grid, a.splits, stream, attr);
    if (a.splits > 1 && a.rows <= 8)
        e = launch_variant<true, 1>(cfg, w_map, a, dev);
    else if (a.splits > 1)
        e = launch_variant<true, 2>(cfg, w_map, a, dev);
    else if (a.rows <= 8)
        e = launch_variant<false, 1>(cfg, w_map, a, dev);
    else
        e = launch_variant<false, 2>(cfg, w_map, a, dev);
    if (e != cudaSuccess)
        return e;
    return cudaGetLastError();
}

int w4a16_ctas_per_sm()
{
    static std::mutex mu;
    static std::map<int, int> cache;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return kW4CtasPerSm;
    }
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(dev);
    if (it != cache.end())
        return it->second;
    int n = 0;
    if (configure_w4<false, 2>(dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, w4a16_kernel<false, 2>, kW4Threads, kW4SmemBytes) !=
            cudaSuccess ||
        n <= 0) {
        cudaGetLastError();
        n = kW4CtasPerSm;
    }
    cache[dev] = n;
    return n;
}

int w4a16_cluster_capacity(int splits)
{
    if (splits < 2 || splits > kW4MaxSplits)
        return 0;
    static std::mutex mu;
    static std::map<std::pair<int, int>, int> cache;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    std::lock_guard<std::mutex> lock(mu);
    const auto key = std::make_pair(dev, splits);
    auto it = cache.find(key);
    if (it != cache.end())
        return it->second;
    int c = 0;
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = w4_config(dim3(1, static_cast<unsigned>(splits), 1), splits, nullptr, attr);
    if (configure_w4<true, 2>(dev) != cudaSuccess ||
        cudaOccupancyMaxActiveClusters(&c, w4a16_kernel<true, 2>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        c = 0;
    }
    cache[key] = c;
    return c;
}

cudaError_t read_w4_error(uint32_t *bits, bool clear)
{
    unsigned int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_w4_error, sizeof v);
    if (e != cudaSuccess)
        return e;
    if (bits)
        *bits = v;
    if (clear) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_w4_error, &zero, sizeof zero);
    }
    return e;
}

} // namespace kvq
