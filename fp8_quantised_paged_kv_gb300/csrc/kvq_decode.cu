// kvq_decode.cu -- single-token paged decode attention over an FP8 e4m3 (or
// BF16) KV cache, split along the context, plus the log-sum-exp combine.
//
// What it computes (blog post "Smaller, faster, safer: running Kimi and GLM
// at scale", page-1 mirror section "量化KV缓存"; page-3 mirror section
// "FP8 省的不仅是显存"): decode attention whose kernel converts the FP8
// values it reads.  For query head h of request r, KV head kvh = h / g:
//   out = sum_j exp(s_j - max s) V^_j / sum_j exp(s_j - max s),
//   s_j = softmax_scale * <q, K^_j>,  K^ = e4m3 value * k_scale[kvh].
//
// Split kernel (persistent, warp-specialised).  The context of every
// (request, KV head) is cut into splits of `split_tokens` tokens; a split is
// one work unit.  About two CTAs per SM stay resident and take units from a
// device counter until none are left.  In each CTA:
//   - one producer warp maps each unit to its pages (block-table rows read 32
//     entries per coalesced load) and streams 32-token chunks of K and V into
//     a ring of shared-memory stages with 2-D tensor bulk copies (TMA,
//     128-byte swizzle), tracked by full/empty mbarriers; it also copies the
//     unit's query rows into a small descriptor ring.  It runs ahead across
//     unit boundaries, so HBM keeps streaming while consumers finish a unit.
//   - four consumer warps take the chunks round-robin.  Per chunk, on the
//     tensor cores (mma.sync m16n8k16, f16 operands, fp32 accumulate):
//     S^T = K Q^T with the 32 tokens as M and the g <= 8 query heads of the
//     group as N, an fp32 online softmax, and O^T += V^T P^T.  e4m3 codes
//     become f16 in registers (exact); movmatrix turns the score fragment
//     into the PV operand.  At the end of a unit the four warps merge through
//     double-buffered shared scratch; a request that fits in one split gets
//     its output here, longer ones leave (lse, o) partials for the combine.
// Every K/V byte is read from HBM once and converted once for all g heads.
// Every wait is a bounded mbarrier wait: no named barrier, no unbounded spin.
#include <cfloat>

#include <cuda_bf16.h>

#include "kvq_internal.h"
#include "kvq_ptx.cuh"

namespace kvq {

// Sticky device error word (bit 0: a wait on a bulk copy or a pipeline
// barrier gave up after its time limit).
__device__ unsigned int g_device_error = 0;

namespace {

constexpr int kConsumerWarps = 4;
constexpr int kConsumerThreads = kConsumerWarps * 32;     // == kHeadDim: one dim per thread in the merge
constexpr int kThreads = kConsumerThreads + 32;           // + one producer warp
constexpr int kUnitSlots = 4;
constexpr uint64_t kWaitLimitNs = 1000000000ull;          // ~1 s per wait, then give up
constexpr int kCombineThreads = 128;
constexpr int kMaxSplits = 1024;
constexpr int kMaxBatch = 1024;                           // requests one launch can take

static_assert(kConsumerThreads == kHeadDim, "the merge gives each consumer thread one head dim");

template <bool kBf16Cache>
struct Tile {
    static constexpr int kRowBytes = kBf16Cache ? 256 : 128;      // one token of one head
    static constexpr int kBytes = kChunkTokens * kRowBytes;       // K (or V) part of a stage
    static constexpr int kStageBytes = 2 * kBytes;
    static constexpr int kStages = kBf16Cache ? 4 : 8;
    static constexpr int kRingBytes = kStages * kStageBytes;      // 64 KB
};

struct UnitDesc {
    int32_t b, kvh, split, nsplit;
    int64_t t0, t1;                  // token range of the unit
    float k_scale, v_scale;
    int32_t kind;                    // kUnitWork, kUnitZero, kUnitEnd
    int32_t pad;
};
constexpr int kUnitWork = 0, kUnitZero = 1, kUnitEnd = 2;

constexpr int kMergeFloats = kConsumerWarps * kMaxGroup * kHeadDim + 2 * kConsumerWarps * kMaxGroup;

// Shared-memory map (byte offsets from a 1024-byte-aligned base).
template <bool kBf16Cache>
struct Smem {
    using T = Tile<kBf16Cache>;
    static constexpr int kRing = 0;
    static constexpr int kMerge = kRing + T::kRingBytes;                    // 2 x (o[4][8][128], m[4][8], l[4][8])
    static constexpr int kQ = kMerge + 2 * kMergeFloats * 4;                // [slots][8][128] bf16
    static constexpr int kDesc = kQ + kUnitSlots * kMaxGroup * kHeadDim * 2;
    static constexpr int kBars = kDesc + kUnitSlots * static_cast<int>(sizeof(UnitDesc));
    static constexpr int kNumBars = 2 * T::kStages + 2 * kUnitSlots + 2;   // full, empty, unit full/empty, merge
    static constexpr int kStageBad = kBars + 8 * kNumBars;
    static constexpr int kPrefix = kStageBad + 4 * T::kStages;             // int32[kMaxBatch]
    static constexpr int kFlags = kPrefix + 4 * kMaxBatch;
    static constexpr int kBytes = kFlags + 16;
    static constexpr int kAlloc = kBytes + 1024;                            // alignment slack
};

// Byte offset of 16-byte chunk `c` of 128-byte line `line` in a tile written
// by a 128-byte-swizzled tensor copy into a 1024-byte-aligned buffer.
__device__ __forceinline__ uint32_t swz(int line, int c)
{
    return static_cast<uint32_t>(line * 128 + ((c ^ (line & 7)) << 4));
}

__device__ __forceinline__ uint4 lds128(const uint8_t *base, uint32_t off)
{
    return *reinterpret_cast<const uint4 *>(base + off);
}

__device__ __forceinline__ float warp_max_over_rows(float v)
{
    // lanes that share lane % 4 hold the same query heads
    v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, 4));
    v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, 8));
    v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, 16));
    return v;
}

__device__ __forceinline__ float warp_sum_over_rows(float v)
{
    v += __shfl_xor_sync(0xFFFFFFFFu, v, 4);
    v += __shfl_xor_sync(0xFFFFFFFFu, v, 8);
    v += __shfl_xor_sync(0xFFFFFFFFu, v, 16);
    return v;
}

__device__ __forceinline__ void store_out(void *out, int64_t idx, float v, bool fp32)
{
    if (fp32)
        static_cast<float *>(out)[idx] = v;
    else
        static_cast<__nv_bfloat16 *>(out)[idx] = __float2bfloat16_rn(v);
}

// 1-D bulk copy global -> shared (both 16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_load(void *smem_dst, const void *src, uint32_t bytes,
                                          uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_addr(smem_dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Warp-wide bounded wait.  Once any wait of this CTA has failed, later waits
// return at once (the results are then invalid and the error bit is set).
__device__ __forceinline__ void warp_wait(uint64_t *bar, uint32_t parity, volatile int *failed)
{
    if (!*failed && !mbar_wait_bounded(bar, parity, kWaitLimitNs)) {
        *failed = 1;
        atomicOr(&g_device_error, 1u);
    }
    __syncwarp();
}

// One 32-token chunk of K (ks) and V (vs) in shared memory: update the
// warp's online-softmax state (m_run, l_run) and O^T accumulators.  Lane
// (gq, tq) = (lane / 4, lane % 4) owns query heads 2tq, 2tq+1.
template <bool kBf16Cache, bool kPreciseP>
__device__ __forceinline__ void attend_chunk(const uint8_t *ks, const uint8_t *vs, int n_valid,
                                             const uint32_t (&qf)[8][2], float qk_scale,
                                             float (&m_run)[2], float (&l_run)[2],
                                             float (&o)[8][4], int gq, int tq)
{
    // ---- S^T = K Q^T for the two 16-token m-tiles
    float sc[2][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
        sc[mt][0] = sc[mt][1] = sc[mt][2] = sc[mt][3] = 0.f;
        const int r0 = mt * 16 + gq, r1 = r0 + 8;
        if constexpr (kBf16Cache) {
            uint32_t w0[16], w1[16];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int line0 = 2 * r0 + (tq >> 1), line1 = 2 * r1 + (tq >> 1);
                const uint4 x0 = lds128(ks, swz(line0, (tq & 1) * 4 + j));
                const uint4 x1 = lds128(ks, swz(line1, (tq & 1) * 4 + j));
                w0[4 * j] = x0.x; w0[4 * j + 1] = x0.y; w0[4 * j + 2] = x0.z; w0[4 * j + 3] = x0.w;
                w1[4 * j] = x1.x; w1[4 * j + 1] = x1.y; w1[4 * j + 2] = x1.z; w1[4 * j + 3] = x1.w;
            }
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                mma_bf16(sc[mt], w0[2 * kk], w1[2 * kk], w0[2 * kk + 1], w1[2 * kk + 1],
                         qf[kk][0], qf[kk][1]);
        } else {
            const uint4 x0a = lds128(ks, swz(r0, 2 * tq)), x0b = lds128(ks, swz(r0, 2 * tq + 1));
            const uint4 x1a = lds128(ks, swz(r1, 2 * tq)), x1b = lds128(ks, swz(r1, 2 * tq + 1));
            const uint32_t w0[8] = {x0a.x, x0a.y, x0a.z, x0a.w, x0b.x, x0b.y, x0b.z, x0b.w};
            const uint32_t w1[8] = {x1a.x, x1a.y, x1a.z, x1a.w, x1b.x, x1b.y, x1b.z, x1b.w};
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                mma_f16(sc[mt], lo16_e4m3x2_to_f16x2(w0[kk]), lo16_e4m3x2_to_f16x2(w1[kk]),
                        hi16_e4m3x2_to_f16x2(w0[kk]), hi16_e4m3x2_to_f16x2(w1[kk]),
                        qf[kk][0], qf[kk][1]);
        }
    }

    // ---- online softmax (log2 domain); lane holds heads 2tq, 2tq+1
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int row = mt * 16 + gq + ((i & 2) ? 8 : 0);
            float x = sc[mt][i] * qk_scale;
            x = row < n_valid ? x : -INFINITY;
            sc[mt][i] = x;
            mx[i & 1] = fmaxf(mx[i & 1], x);
        }
    }
    float alpha[2], base[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const float mnew = fmaxf(m_run[j], warp_max_over_rows(mx[j]));
        base[j] = mnew == -INFINITY ? 0.f : mnew;
        alpha[j] = fast_exp2(m_run[j] - base[j]);
        m_run[j] = mnew;
    }
    float psum[2] = {0.f, 0.f};
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float p = fast_exp2(sc[mt][i] - base[i & 1]);
            sc[mt][i] = p;
            psum[i & 1] += p;
        }
    }
#pragma unroll
    for (int j = 0; j < 2; ++j)
        l_run[j] = l_run[j] * alpha[j] + psum[j];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        o[i][0] *= alpha[0];
        o[i][1] *= alpha[1];
        o[i][2] *= alpha[0];
        o[i][3] *= alpha[1];
    }

    // ---- O^T += V^T P^T
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
        uint32_t x0, x1;
        if constexpr (kBf16Cache) {
            x0 = f32x2_to_bf16x2(sc[mt][0], sc[mt][1]);
            x1 = f32x2_to_bf16x2(sc[mt][2], sc[mt][3]);
        } else {
            x0 = f32x2_to_f16x2(sc[mt][0], sc[mt][1]);
            x1 = f32x2_to_f16x2(sc[mt][2], sc[mt][3]);
        }
        const uint32_t pb0 = movmatrix_trans(x0), pb1 = movmatrix_trans(x1);
        uint32_t pl0 = 0, pl1 = 0;
        if constexpr (kPreciseP) {
            // second term carries what the 16-bit rounding of P dropped
            const float2 h0 = kBf16Cache ? bf16x2_to_f32x2(x0) : f16x2_to_f32x2(x0);
            const float2 h1 = kBf16Cache ? bf16x2_to_f32x2(x1) : f16x2_to_f32x2(x1);
            const uint32_t y0 = kBf16Cache ? f32x2_to_bf16x2(sc[mt][0] - h0.x, sc[mt][1] - h0.y)
                                           : f32x2_to_f16x2(sc[mt][0] - h0.x, sc[mt][1] - h0.y);
            const uint32_t y1 = kBf16Cache ? f32x2_to_bf16x2(sc[mt][2] - h1.x, sc[mt][3] - h1.y)
                                           : f32x2_to_f16x2(sc[mt][2] - h1.x, sc[mt][3] - h1.y);
            pl0 = movmatrix_trans(y0);
            pl1 = movmatrix_trans(y1);
        }
        // V rows of token slots 2tq, 2tq+1, 2tq+8, 2tq+9 of this m-tile
        const int rv = mt * 16 + 2 * tq;
        const int rows[4] = {rv, rv + 1, rv + 8, rv + 9};
        if constexpr (kBf16Cache) {
            uint32_t R[4][8];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int line = 2 * rows[q] + (gq >> 2);
                const uint4 lo = lds128(vs, swz(line, (gq & 3) * 2));
                const uint4 hi = lds128(vs, swz(line, (gq & 3) * 2 + 1));
                const bool keep = rows[q] < n_valid;
                R[q][0] = keep ? lo.x : 0u; R[q][1] = keep ? lo.y : 0u;
                R[q][2] = keep ? lo.z : 0u; R[q][3] = keep ? lo.w : 0u;
                R[q][4] = keep ? hi.x : 0u; R[q][5] = keep ? hi.y : 0u;
                R[q][6] = keep ? hi.z : 0u; R[q][7] = keep ? hi.w : 0u;
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint32_t a0 = prmt(R[0][i], R[1][i], 0x5410);
                const uint32_t a1 = prmt(R[0][i], R[1][i], 0x7632);
                const uint32_t a2 = prmt(R[2][i], R[3][i], 0x5410);
                const uint32_t a3 = prmt(R[2][i], R[3][i], 0x7632);
                mma_bf16(o[i], a0, a1, a2, a3, pb0, pb1);
                if constexpr (kPreciseP)
                    mma_bf16(o[i], a0, a1, a2, a3, pl0, pl1);
            }
        } else {
            uint32_t R[4][4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint4 v = lds128(vs, swz(rows[q], gq));
                const bool keep = rows[q] < n_valid;
                R[q][0] = keep ? v.x : 0u; R[q][1] = keep ? v.y : 0u;
                R[q][2] = keep ? v.z : 0u; R[q][3] = keep ? v.w : 0u;
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint32_t sel = (i & 1) ? 0x7362u : 0x5140u;
                const uint32_t p01 = prmt(R[0][i >> 1], R[1][i >> 1], sel);
                const uint32_t p23 = prmt(R[2][i >> 1], R[3][i >> 1], sel);
                const uint32_t a0 = lo16_e4m3x2_to_f16x2(p01), a1 = hi16_e4m3x2_to_f16x2(p01);
                const uint32_t a2 = lo16_e4m3x2_to_f16x2(p23), a3 = hi16_e4m3x2_to_f16x2(p23);
                mma_f16(o[i], a0, a1, a2, a3, pb0, pb1);
                if constexpr (kPreciseP)
                    mma_f16(o[i], a0, a1, a2, a3, pl0, pl1);
            }
        }
    }
}

template <bool kBf16Cache, bool kPreciseP>
__global__ void __launch_bounds__(kThreads, 2)
decode_split_kernel(const __grid_constant__ CUtensorMap k_map,
                    const __grid_constant__ CUtensorMap v_map, const DecodeArgs a)
{
    using T = Tile<kBf16Cache>;
    using S = Smem<kBf16Cache>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *ring = smem + S::kRing;
    float *merge = reinterpret_cast<float *>(smem + S::kMerge);
    uint8_t *qbuf = smem + S::kQ;
    UnitDesc *desc = reinterpret_cast<UnitDesc *>(smem + S::kDesc);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + S::kBars);
    uint64_t *empty = full + T::kStages;
    uint64_t *unit_full = empty + T::kStages;
    uint64_t *unit_empty = unit_full + kUnitSlots;
    uint64_t *merge_bar = unit_empty + kUnitSlots;
    volatile int *stage_bad = reinterpret_cast<volatile int *>(smem + S::kStageBad);
    int32_t *prefix = reinterpret_cast<int32_t *>(smem + S::kPrefix);
    volatile int *failed = reinterpret_cast<volatile int *>(smem + S::kFlags);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int g = a.group, ps = a.page_size;

    if (threadIdx.x == 0) {
        *failed = 0;
        for (int i = 0; i < T::kStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < kUnitSlots; ++i) {
            mbar_init(&unit_full[i], 1);
            mbar_init(&unit_empty[i], kConsumerWarps);
            desc[i].kind = kUnitEnd;          // a slot never written reads as "stop"
        }
        mbar_init(&merge_bar[0], kConsumerWarps);
        mbar_init(&merge_bar[1], kConsumerWarps);
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        // ================================================================ producer
        if (lane == 0) {
            prefetch_tensor_map(&k_map);
            prefetch_tensor_map(&v_map);
        }
        // units of request b: one per (KV head, split), or one per KV head that
        // writes zeros when the request is aborted, empty or longer than its row
        const int64_t cap = static_cast<int64_t>(a.max_pages_per_seq) * ps;
        int running = 0;
        for (int base = 0; base < a.batch; base += 32) {
            const int b = base + lane;
            int n = 0;
            if (b < a.batch) {
                const int64_t len = a.seq_lens[b];
                const bool aborted = a.abort_flags != nullptr && a.abort_flags[b] != 0;
                const bool zero = aborted || len <= 0 || len > cap;
                const int ns = zero ? 1 : static_cast<int>((len + a.split_tokens - 1) / a.split_tokens);
                n = ns * a.num_kv_heads;
            }
            int x = n;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(0xFFFFFFFFu, x, off);
                if (lane >= off)
                    x += y;
            }
            if (b < a.batch)
                prefix[b] = running + x;        // inclusive prefix
            running += __shfl_sync(0xFFFFFFFFu, x, 31);
        }
        __syncwarp();
        const int total = running;
        const uint64_t policy = l2_policy_evict_first();
        const int box_tok = ps < kChunkTokens ? ps : kChunkTokens;
        const int parts = kChunkTokens / box_tok;                      // 2 at page size 16, else 1
        const uint32_t part_bytes = static_cast<uint32_t>(box_tok * T::kRowBytes);
        const int lines_per_tok = kBf16Cache ? 2 : 1;
        const int chunks_per_page = ps / kChunkTokens > 0 ? ps / kChunkTokens : 1;
        const uint32_t qbytes = static_cast<uint32_t>(g * kHeadDim * 2);

        uint32_t q = 0;          // chunk sequence number (same schedule as the consumers)
        uint32_t k = 0;          // unit sequence number
        int next = 0;
        if (lane == 0)
            next = static_cast<int>(atomicAdd(&a.counters[0], 1u));
        next = __shfl_sync(0xFFFFFFFFu, next, 0);
        while (true) {
            // warp-uniform decision (another warp may set the failed flag meanwhile)
            const int u = __shfl_sync(0xFFFFFFFFu, *failed ? total : next, 0);
            const int slot = static_cast<int>(k % kUnitSlots);
            if (k >= kUnitSlots)
                warp_wait(&unit_empty[slot], ((k / kUnitSlots) & 1) ^ 1, failed);
            if (u >= total) {
                if (lane == 0) {
                    desc[slot].kind = kUnitEnd;
                    mbar_arrive(&unit_full[slot]);
                }
                ++k;
                break;
            }
            if (lane == 0)
                next = static_cast<int>(atomicAdd(&a.counters[0], 1u));   // prefetch the next unit
            int lo = 0, hi = a.batch - 1;                                   // first b with prefix[b] > u
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (prefix[mid] > u)
                    hi = mid;
                else
                    lo = mid + 1;
            }
            const int b = lo;
            const int rem = u - (b > 0 ? prefix[b - 1] : 0);
            const int kvh = rem % a.num_kv_heads;
            const int split = rem / a.num_kv_heads;
            const int64_t t0 = static_cast<int64_t>(split) * a.split_tokens;
            const int first_page = static_cast<int>(t0 / ps);
            const int32_t *bt = a.block_table + static_cast<int64_t>(b) * a.max_pages_per_seq + first_page;
            // one round trip: length, abort flag, scales and the first 32 page ids
            const int64_t len = a.seq_lens[b];
            const bool aborted = a.abort_flags != nullptr && a.abort_flags[b] != 0;
            const float ksc = kBf16Cache ? 1.f : a.k_scale[kvh];
            const float vsc = kBf16Cache ? 1.f : a.v_scale[kvh];
            const int row_left = a.max_pages_per_seq - first_page;        // entries left in the row
            int32_t id = lane < row_left ? bt[lane] : 0;
            const bool zero = aborted || len <= 0 || len > cap;
            const int nsplit = zero ? 1 : static_cast<int>((len + a.split_tokens - 1) / a.split_tokens);
            const int64_t t1 = zero ? t0 : (len < t0 + a.split_tokens ? len : t0 + a.split_tokens);
            if (lane == 0) {
                UnitDesc &d = desc[slot];
                d.b = b;
                d.kvh = kvh;
                d.split = split;
                d.nsplit = nsplit;
                d.t0 = t0;
                d.t1 = t1;
                d.k_scale = ksc;
                d.v_scale = vsc;
                d.kind = zero ? kUnitZero : kUnitWork;
                if (zero || *failed) {
                    mbar_arrive(&unit_full[slot]);
                } else {
                    mbar_arrive_expect_tx(&unit_full[slot], qbytes);
                    bulk_load(qbuf + slot * kMaxGroup * kHeadDim * 2,
                              static_cast<const uint16_t *>(a.q) +
                                  (static_cast<int64_t>(b) * a.num_q_heads + kvh * g) * kHeadDim,
                              qbytes, &unit_full[slot]);
                }
            }
            ++k;
            next = __shfl_sync(0xFFFFFFFFu, next, 0);
            if (zero)
                continue;

            // stream the unit's chunks: chunk c covers tokens t0 + 32c ..
            const int n_pages = static_cast<int>((t1 - 1) / ps) - first_page + 1;
            const int n_chunks = static_cast<int>((t1 - t0 + kChunkTokens - 1) / kChunkTokens);
            int c = 0;
            for (int pb = 0; pb < n_pages; pb += 32) {
                if (pb > 0)
                    id = pb + lane < n_pages ? bt[pb + lane] : 0;
                // chunks whose pages lie in this batch of 32 pages
                const int c_end_batch = parts == 2 ? (pb + 32) / 2 : (pb + 32) * chunks_per_page;
                const int c_end = n_chunks < c_end_batch ? n_chunks : c_end_batch;
                for (; c < c_end; ++c) {
                    const int st = static_cast<int>(q % T::kStages);
                    const uint32_t use = q / T::kStages;
                    if (use > 0)
                        warp_wait(&empty[st], (use & 1) ^ 1, failed);
                    const int64_t tok = t0 + static_cast<int64_t>(c) * kChunkTokens;
                    int32_t ys[2] = {0, 0};
                    int np = 0;
                    bool bad = false;
#pragma unroll
                    for (int part = 0; part < 2; ++part) {
                        if (part < parts) {
                            const int64_t ptok = tok + part * box_tok;
                            const int lp = static_cast<int>(ptok / ps) - first_page - pb;  // 0 .. 31
                            const int32_t page = __shfl_sync(0xFFFFFFFFu, id, lp & 31);
                            if (ptok < t1) {
                                bad |= page < 0 || page >= a.num_pages;
                                const int64_t row =
                                    (static_cast<int64_t>(page) * a.num_kv_heads + kvh) * ps + ptok % ps;
                                ys[np++] = static_cast<int32_t>(row * lines_per_tok);
                            }
                        }
                    }
                    if (lane == 0) {
                        stage_bad[st] = bad ? 1 : 0;
                        uint8_t *kdst = ring + st * T::kStageBytes;
                        uint8_t *vdst = kdst + T::kBytes;
                        if (bad || *failed) {
                            mbar_arrive(&full[st]);
                        } else {
                            fence_proxy_async_smem();
                            mbar_arrive_expect_tx(&full[st], 2u * part_bytes * np);
                            for (int i = 0; i < np; ++i) {
                                tma_load_2d(kdst + i * part_bytes, &k_map, 0, ys[i], &full[st], policy);
                                tma_load_2d(vdst + i * part_bytes, &v_map, 0, ys[i], &full[st], policy);
                            }
                        }
                    }
                    __syncwarp();
                    ++q;
                }
            }
        }
        // every unit is handed out: the last CTA to get here resets the counters
        if (lane == 0) {
            __threadfence();
            const unsigned int done = atomicAdd(&a.counters[1], 1u);
            if (done == gridDim.x - 1) {
                atomicExch(&a.counters[0], 0u);
                atomicExch(&a.counters[1], 0u);
            }
        }
        if (*failed && lane == 0) {
            // wait (bounded) for copies still in flight before the CTA can exit
            for (uint32_t j = q > static_cast<uint32_t>(T::kStages) ? q - T::kStages : 0; j < q; ++j)
                mbar_wait_bounded(&full[j % T::kStages], (j / T::kStages) & 1, kWaitLimitNs);
            for (uint32_t j = k > static_cast<uint32_t>(kUnitSlots) ? k - kUnitSlots : 0; j < k; ++j)
                mbar_wait_bounded(&unit_full[j % kUnitSlots], (j / kUnitSlots) & 1, kWaitLimitNs);
        }
        return;
    }

    // ==================================================================== consumers
    const int gq = lane >> 2, tq = lane & 3;
    uint32_t q = 0, k = 0, m = 0;     // chunk, unit and merged-unit sequence numbers
    while (true) {
        const int slot = static_cast<int>(k % kUnitSlots);
        warp_wait(&unit_full[slot], (k / kUnitSlots) & 1, failed);
        const UnitDesc d = desc[slot];
        const int stop = (*failed != 0 || d.kind == kUnitEnd) ? 1 : 0;
        if (__shfl_sync(0xFFFFFFFFu, stop, 0))          // one decision for the whole warp
            break;
        const int hq0 = d.kvh * g;
        if (d.kind == kUnitZero) {
            if (warp == 0) {
                for (int i = lane; i < g * kHeadDim; i += 32)
                    store_out(a.out, (static_cast<int64_t>(d.b) * a.num_q_heads + hq0) * kHeadDim + i,
                              0.f, a.out_fp32);
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&unit_empty[slot]);
            ++k;
            continue;
        }

        // query fragments (mma B operand): lane (gq, tq) holds query head gq
        // of the group at dims 32*tq .. 32*tq+31; the k-slot pairs of k-step c
        // map to dims 32*tq + 4*c + {0,1} and {2,3}.
        uint32_t qf[8][2];
        {
            uint32_t w[16];
            if (gq < g) {
                const uint8_t *src = qbuf + slot * kMaxGroup * kHeadDim * 2 + (gq * kHeadDim + 32 * tq) * 2;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint4 v = *reinterpret_cast<const uint4 *>(src + 16 * i);
                    w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
                }
            } else {
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    w[i] = 0;
            }
#pragma unroll
            for (int c = 0; c < 8; ++c) {
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    if constexpr (kBf16Cache) {
                        qf[c][j] = w[2 * c + j];
                    } else {
                        const float2 f = bf16x2_to_f32x2(w[2 * c + j]);
                        qf[c][j] = f32x2_to_f16x2(f.x, f.y);
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&unit_empty[slot]);
        ++k;

        const float qk_scale = a.qk_scale_log2 * d.k_scale;
        const int n_chunks = static_cast<int>((d.t1 - d.t0 + kChunkTokens - 1) / kChunkTokens);
        float m_run[2] = {-INFINITY, -INFINITY};
        float l_run[2] = {0.f, 0.f};
        float o[8][4];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
        int bad = 0;

        // this warp's chunks: those whose sequence number is warp (mod 4)
        for (int c = static_cast<int>((warp + kConsumerWarps - q % kConsumerWarps) % kConsumerWarps);
             c < n_chunks; c += kConsumerWarps) {
            const uint32_t qc = q + static_cast<uint32_t>(c);
            const int st = static_cast<int>(qc % T::kStages);
            warp_wait(&full[st], (qc / T::kStages) & 1, failed);
            bad |= stage_bad[st];
            const uint8_t *ks = ring + st * T::kStageBytes;
            const int64_t left = d.t1 - (d.t0 + static_cast<int64_t>(c) * kChunkTokens);
            const int n_valid = left < kChunkTokens ? static_cast<int>(left) : kChunkTokens;
            attend_chunk<kBf16Cache, kPreciseP>(ks, ks + T::kBytes, n_valid, qf, qk_scale, m_run,
                                                l_run, o, gq, tq);
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&empty[st]);                 // stage free for the producer
        }
        q += static_cast<uint32_t>(n_chunks);

        // ---- merge the four warps' states through scratch buffer m % 2
        float *sm_o = merge + (m & 1) * kMergeFloats;                 // [4][8][128]
        float *sm_m = sm_o + kConsumerWarps * kMaxGroup * kHeadDim;   // [4][8]
        float *sm_l = sm_m + kConsumerWarps * kMaxGroup;               // [4][8]
#pragma unroll
        for (int j = 0; j < 2; ++j)
            l_run[j] = warp_sum_over_rows(l_run[j]);
        bad = __any_sync(0xFFFFFFFFu, bad != 0) ? 1 : 0;
        {
            float *ow = sm_o + warp * kMaxGroup * kHeadDim;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int dd = 16 * gq + 2 * i;
                *reinterpret_cast<float2 *>(ow + (2 * tq) * kHeadDim + dd) = make_float2(o[i][0], o[i][2]);
                *reinterpret_cast<float2 *>(ow + (2 * tq + 1) * kHeadDim + dd) = make_float2(o[i][1], o[i][3]);
            }
            if (gq == 0) {
                // a warp that met an invalid page poisons m, which drops the unit
                const float nan = __int_as_float(0x7FC00000);
                sm_m[warp * kMaxGroup + 2 * tq] = bad ? nan : m_run[0];
                sm_m[warp * kMaxGroup + 2 * tq + 1] = bad ? nan : m_run[1];
                sm_l[warp * kMaxGroup + 2 * tq] = l_run[0];
                sm_l[warp * kMaxGroup + 2 * tq + 1] = l_run[1];
            }
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&merge_bar[m & 1]);
        warp_wait(&merge_bar[m & 1], (m >> 1) & 1, failed);
        const int dd = threadIdx.x;                      // 0 .. 127
        for (int h = 0; h < g; ++h) {
            float mmax = -INFINITY;
            bool poisoned = false;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) {
                const float mw = sm_m[w * kMaxGroup + h];
                poisoned |= mw != mw;
                mmax = fmaxf(mmax, mw);
            }
            float lsum = 0.f, acc = 0.f;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) {
                const float mw = sm_m[w * kMaxGroup + h];
                const float f = mw == -INFINITY ? 0.f : fast_exp2(mw - mmax);
                lsum += sm_l[w * kMaxGroup + h] * f;
                acc += sm_o[(w * kMaxGroup + h) * kHeadDim + dd] * f;
            }
            const int64_t bh = static_cast<int64_t>(d.b) * a.num_q_heads + hq0 + h;
            if (d.nsplit == 1) {
                store_out(a.out, bh * kHeadDim + dd, poisoned ? 0.f : acc / lsum * d.v_scale,
                          a.out_fp32);
            } else {
                a.ws_o[(bh * a.max_splits + d.split) * kHeadDim + dd] =
                    poisoned ? 0.f : acc / lsum * d.v_scale;
                if (dd == 0)
                    a.ws_lse[bh * a.max_splits + d.split] =
                        poisoned ? __int_as_float(0x7FC00000) : mmax + __log2f(lsum);
            }
        }
        ++m;
    }
}

// One CTA per (query head, request): merge the split partials by their
// log-sum-exp weights.  Requests that fit in one split were finished by the
// split kernel and are skipped here.
__global__ void __launch_bounds__(kCombineThreads) decode_combine_kernel(const DecodeArgs a)
{
    __shared__ float s_w[kMaxSplits];
    __shared__ float s_red[kCombineThreads / 32];
    __shared__ int s_bad;
    const int h = blockIdx.x, b = blockIdx.y;
    const int64_t len = a.seq_lens[b];
    const bool aborted = a.abort_flags != nullptr && a.abort_flags[b] != 0;
    const int64_t cap = static_cast<int64_t>(a.max_pages_per_seq) * a.page_size;
    if (aborted || len <= 0 || len > cap)
        return;
    const int nsplit = static_cast<int>((len + a.split_tokens - 1) / a.split_tokens);
    if (nsplit <= 1)
        return;
    const int64_t bh = static_cast<int64_t>(b) * a.num_q_heads + h;
    const float *lse = a.ws_lse + bh * a.max_splits;
    const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
    if (tid == 0)
        s_bad = 0;
    __syncthreads();

    float mloc = -INFINITY;
    for (int s = tid; s < nsplit; s += kCombineThreads) {
        const float v = lse[s];
        if (v != v)
            s_bad = 1;
        s_w[s] = v;
        mloc = fmaxf(mloc, v);
    }
    for (int off = 16; off > 0; off >>= 1)
        mloc = fmaxf(mloc, __shfl_xor_sync(0xFFFFFFFFu, mloc, off));
    if (lane == 0)
        s_red[warp] = mloc;
    __syncthreads();
    float mmax = s_red[0];
    for (int w = 1; w < kCombineThreads / 32; ++w)
        mmax = fmaxf(mmax, s_red[w]);
    const bool bad = s_bad != 0;
    __syncthreads();

    float wsum = 0.f;
    for (int s = tid; s < nsplit; s += kCombineThreads) {
        const float w = bad ? 0.f : fast_exp2(s_w[s] - mmax);
        s_w[s] = w;
        wsum += w;
    }
    for (int off = 16; off > 0; off >>= 1)
        wsum += __shfl_xor_sync(0xFFFFFFFFu, wsum, off);
    if (lane == 0)
        s_red[warp] = wsum;
    __syncthreads();
    float total = 0.f;
    for (int w = 0; w < kCombineThreads / 32; ++w)
        total += s_red[w];

    for (int d = tid; d < kHeadDim; d += kCombineThreads) {
        float acc = 0.f;
        if (!bad) {
            const float *ob = a.ws_o + bh * a.max_splits * kHeadDim + d;
            for (int s = 0; s < nsplit; ++s)
                acc += s_w[s] * ob[static_cast<int64_t>(s) * kHeadDim];
            acc /= total;
        }
        store_out(a.out, bh * kHeadDim + d, acc, a.out_fp32);
    }
}

template <bool kBf16, bool kPrecise>
cudaError_t launch_split(const DecodeArgs &a, const CUtensorMap &k_map, const CUtensorMap &v_map,
                         cudaStream_t stream, int grid)
{
    using S = Smem<kBf16>;
    static int configured[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 64 && !configured[dev]) {
        e = cudaFuncSetAttribute(decode_split_kernel<kBf16, kPrecise>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, S::kAlloc);
        if (e != cudaSuccess)
            return e;
        configured[dev] = 1;
    }
    decode_split_kernel<kBf16, kPrecise><<<grid, kThreads, S::kAlloc, stream>>>(k_map, v_map, a);
    return cudaGetLastError();
}

} // namespace

int decode_max_batch() { return kMaxBatch; }

cudaError_t launch_decode_partial(const DecodeArgs &a, const CUtensorMap &k_map,
                                  const CUtensorMap &v_map, cudaStream_t stream, int grid)
{
    if (a.batch == 0)
        return cudaSuccess;
    if (a.bf16_cache)
        return a.out_fp32 ? launch_split<true, true>(a, k_map, v_map, stream, grid)
                          : launch_split<true, false>(a, k_map, v_map, stream, grid);
    return a.out_fp32 ? launch_split<false, true>(a, k_map, v_map, stream, grid)
                      : launch_split<false, false>(a, k_map, v_map, stream, grid);
}

cudaError_t launch_decode_combine(const DecodeArgs &a, cudaStream_t stream)
{
    if (a.batch == 0 || a.max_splits <= 1)
        return cudaSuccess;
    const dim3 grid(static_cast<unsigned>(a.num_q_heads), static_cast<unsigned>(a.batch));
    decode_combine_kernel<<<grid, kCombineThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t read_device_error(uint32_t *bits, bool clear)
{
    unsigned int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_device_error, sizeof v);
    if (e != cudaSuccess)
        return e;
    if (bits)
        *bits = v;
    if (clear) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof zero);
    }
    return e;
}

} // namespace kvq
