// kvq_decode_umma.cu -- multi-token paged decode attention over an FP8 (e4m3)
// cache on the 5th-generation tensor cores: tcgen05.mma with operands in
// shared memory and the score and output accumulators in tensor memory.
//
// What it computes (blog post "Smaller, faster, safer: running Kimi and GLM
// at scale", page-1 mirror section "量化KV缓存": the kernel reads FP8 and
// converts on the fly): for request b with L tokens, of which the last n are
// new (already in the cache), KV head kvh and query row r = i * g + h (new
// token i < n, head h < g of the group),
//   out[b][i][kvh g + h] = sum_{t < L - n + 1 + i} e^{s_t - m} V^_t / sum e^{s_t - m},
//   s_t = softmax_scale * <q, K^_t>,  K^ = code * k_scale[kvh], V^ = code * v_scale[kvh].
//
// One CTA per (split of the context, KV head, request) takes all n g <= 128
// query rows of the group, so every cache byte is read from HBM and
// converted from e4m3 to f16 once, whatever n is.  The CTA's warps have one
// job each and hand 64-token tiles to one another through mbarriers:
//   - warp 8 (producer): tensor copies (TMA, 128-byte swizzle) of the e4m3 K
//     and V rows of tile j into a 5-stage ring, one copy per lane;
//   - warps 4..7 (converters): e4m3 -> f16 (exact) into one of four operand
//     buffers, V rows past the split zeroed;
//   - warp 9, one lane: S_j = Q K_j^T (M 128 query-row slots, N 64 tokens,
//     K 128) into one of two score buffers in tensor memory;
//   - warp 10, one lane: once P_j is written, O += P_j V_j (M 128, N 128,
//     K 64).  A tcgen05.mma holds its issuing thread for about 125 cycles
//     at M 128 and N <= 128, while two issuing warps complete twice as many,
//     so the two streams go from two warps and overlap;
//     Q and P are the A operands, read from tensor memory, K and V the B
//     operands, read from shared memory;
//   - warps 0..3 (softmax, thread m = tensor-memory lane m): row m of Q
//     (f16) into tensor memory once, then per tile row m of S_j, the online
//     softmax in fp32, row m of P_j (f16) into tensor memory; at the end the
//     output.
// So tile j's scores are computed while the softmax works on tile j - 1,
// and the conversion of tile j + 1 overlaps both.
// The rows fill the 128 M slots in C = 128 / R' copies (R' the power of two
// >= max(n g, 8)); copy c takes the tokens [c R'/2, (c + 1) R'/2) of every
// tile (its P row is zero elsewhere), so the softmax work spreads over all
// four warps.  At the end each copy's (max, sum, O) is merged per row, and a
// request with several splits merges them through the workspace: the last
// split of a (request, KV head) to finish combines them (log-sum-exp) and
// resets the arrival counter.
//
// Online softmax: the running maximum is raised only when a tile's maximum
// exceeds it by more than 8 (log2 units); otherwise the stale maximum is
// kept and p = 2^(x - m) stays below 2^8, exact for the final normalisation
// because the sum and the output carry the same maximum.
#include <cfloat>

#include <cuda_bf16.h>

#include "kvq_internal.h"
#include "kvq_ptx.cuh"
#include "kvq_umma.cuh"

namespace kvq {

// Sticky error word of this kernel (read together with the other decode
// kernels' word).  Bit 0: a bulk-copy wait timed out.  Bit 1: the drain that
// follows also gave up.  Bit 2: a tensor-core completion wait timed out.
__device__ unsigned int g_umma_error = 0;

namespace {

constexpr int kSoftWarps = 4;                             // warps 0..3: one per tensor-memory lane quarter
constexpr int kConvWarp0 = kSoftWarps;                    // warps 4..7
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;                               // issues S = Q K^T
constexpr int kPvWarp = 10;                               // issues O += P V
constexpr int kUThreads = 352;
constexpr int kTile = 64;                                 // tokens per tile
constexpr int kStages = 5;                                // e4m3 ring
constexpr int kStageBytes = 2 * kTile * 128;              // K then V rows of one tile
constexpr int kOffRing = 0;
constexpr int kOffKV = kOffRing + kStages * kStageBytes;  // operand buffers: K f16 [64 tok][64 d] x 2, V alike
constexpr int kKVBytes = 32768;
constexpr int kKV = 4;                                    // operand buffers in flight
constexpr int kDataBytes = kOffKV + kKV * kKVBytes;
constexpr int kMergeStride = 132;                         // floats per row of the copies' merge buffer
constexpr int kMaxPageList = 8192 / 16 + 8;
// tensor-memory columns (lane m = M-row m): Q as f16 pairs, two score
// buffers, O, two P buffers as f16 pairs, and two for P's low parts (fp32
// output)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColQ = 0, kColS = 64, kColO = 192, kColP = 320, kColPlo = 384;
constexpr float kRaiseThreshold = 8.f;
constexpr int kCombineTable = 8192;                       // (row, split) weights the combine keeps in shared memory
constexpr int kNumBars = 2 * kStages + 2 * kKV + 3 * 2 + 3;   // see the barrier map in the kernel

__host__ __device__ constexpr int smem_bytes()
{
    return 1024 /* alignment slack */ + kDataBytes + kNumBars * 8 + 16 /* tmem slot */ + kMaxPageList * 4;
}
static_assert(128 * kMergeStride * 4 + 3 * 128 * 4 <= kDataBytes, "the merge buffer fits in the idle ring and buffers");
static_assert(smem_bytes() <= 232448, "one CTA fits an SM");
static_assert((128 + kCombineTable) * 4 <= kDataBytes, "the combine's weights fit in the idle ring and buffers");

constexpr uint32_t kIdescS = umma_idesc_f16(128, kTile, false);
constexpr uint32_t kIdescPV = umma_idesc_f16(128, 128, true);

__device__ __forceinline__ void store_row_value(void *out, int64_t idx, float v, bool fp32)
{
    if (fp32)
        static_cast<float *>(out)[idx] = v;
    else
        static_cast<__nv_bfloat16 *>(out)[idx] = __float2bfloat16_rn(v);
}

// Four consecutive values (idx a multiple of 4).
__device__ __forceinline__ void store_row_value4(void *out, int64_t idx, float4 v, bool fp32)
{
    if (fp32) {
        *reinterpret_cast<float4 *>(static_cast<float *>(out) + idx) = v;
    } else {
        uint2 h;
        h.x = f32x2_to_bf16x2(v.x, v.y);
        h.y = f32x2_to_bf16x2(v.z, v.w);
        *reinterpret_cast<uint2 *>(static_cast<__nv_bfloat16 *>(out) + idx) = h;
    }
}

// Exponent e putting the largest |q| of a row (bf16 bits, sign cleared) in
// [2^14, 2^15) (capped at 100; a zero row keeps 0): the row is multiplied by
// 2^e before it becomes f16 and its scores by 2^-e, so no element overflows
// f16 and every element within 2^28 of the row's largest keeps its bits.
__device__ __forceinline__ int q_row_exponent(uint32_t mx)
{
    if (mx == 0)
        return 0;
    const int field = static_cast<int>(mx >> 7);
    const int e_floor = field != 0 ? field - 127 : (31 - __clz(static_cast<int>(mx))) - 133;
    const int e = 14 - e_floor;
    return e > 100 ? 100 : e;
}

// Global row (in [B][n][Hq]) of local row r of (request b, KV head kvh).
__device__ __forceinline__ int64_t row_id(const DecodeArgs &a, int b, int kvh, int r)
{
    return (static_cast<int64_t>(b) * a.n_query + r / a.group) * a.num_q_heads + kvh * a.group + r % a.group;
}

// Wait for phase `parity` of `bar`, suspended in hardware between looks
// (at most 200 us at a time).  Gives up when another warp has given up (the
// CTA's abort flag), or after limit_ns (0: at once, without looking), in
// which case it raises the abort flag and sets `bit` in the error word.
__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, uint64_t limit_ns,
                                              volatile int *abort_flag, unsigned bit)
{
    if (limit_ns != 0) {
        if (mbar_try_wait(bar, parity))                    // already complete: no clock read
            return true;
        const uint64_t start = global_timer_ns();
        for (uint32_t i = 0; i < (1u << 24); ++i) {
            if (mbar_try_wait_sleep(bar, parity, 200000u))
                return true;
            if (*abort_flag)
                return false;
            if (global_timer_ns() - start > limit_ns)
                break;
        }
    }
    *abort_flag = 1;
    atomicOr(&g_umma_error, bit);
    return false;
}

// kTpc: tokens of a tile each copy of the rows takes: 32 for up to 64 rows
// (two copies fill the 128 M slots), 64 for 65 .. 128 rows (one copy).
template <bool kPrecise, int kTpc>
__global__ void __launch_bounds__(kUThreads, 1)
decode_mt_umma_kernel(const __grid_constant__ CUtensorMap k_map, const __grid_constant__ CUtensorMap v_map,
                      const DecodeArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    // barriers: copy landed / stage free (per ring stage); operands converted,
    // scores ready, P written, O += P V done (per operand / score buffer);
    // Q staged; each issuing lane's final drain (S, then O += P V); scores
    // read (per score buffer)
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + kDataBytes);
    uint64_t *full_e = bars, *empty_e = bars + kStages;
    uint64_t *conv_full = bars + 2 * kStages, *pv_done = conv_full + kKV;   // per operand buffer
    uint64_t *s_full = pv_done + kKV, *p_full = s_full + 2;                // per score / P buffer
    uint64_t *q_ready = p_full + 2, *mma_drain = q_ready + 1, *pv_drain = mma_drain + 1;
    uint64_t *s_free = pv_drain + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + kNumBars);
    int32_t *page_list = reinterpret_cast<int32_t *>(tmem_slot + 4);
    __shared__ int s_abort;
    __shared__ int s_landed;                               // tiles whose copies a converter saw land
    __shared__ int s_last;

    const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = a.group, R = a.n_query * g, ps = a.page_size;
    const int ps_shift = __ffs(ps) - 1;                  // ps is 16, 32, 64 or 128
    constexpr int Rp = 2 * kTpc;                           // M slots per copy of the rows
    const int first_page = static_cast<int>(static_cast<int64_t>(split) * a.split_tokens / ps);
    const int span_left = a.max_pages_per_seq - first_page;
    const int span = a.split_tokens / ps < span_left ? a.split_tokens / ps : span_left;
    const int32_t *bt = a.block_table + static_cast<int64_t>(b) * a.max_pages_per_seq + first_page;

    // Launched as a programmatic dependent of the previous kernel on the
    // stream: nothing is read from global memory before the wait returns.
    if (tid == 0) {
        prefetch_tensor_map(&k_map);
        prefetch_tensor_map(&v_map);
    }
    grid_dependency_wait();

    constexpr int kIdsPerThread = (kMaxPageList + kUThreads - 1) / kUThreads;
    int32_t ids[kIdsPerThread];
#pragma unroll
    for (int k = 0; k < kIdsPerThread; ++k) {
        const int i = tid + k * kUThreads;
        ids[k] = i < span ? __ldg(bt + i) : -1;
    }
    const int64_t len = a.seq_lens[b];
    const bool aborted_req = a.abort_flags != nullptr && a.abort_flags[b] != 0;
    const int64_t cap = static_cast<int64_t>(a.max_pages_per_seq) * ps;
    const bool zero_request = aborted_req || len <= 0 || len > cap;
    const int nsplit = zero_request ? 1 : static_cast<int>((len + a.split_tokens - 1) / a.split_tokens);
    if (split >= nsplit)
        return;
    if (zero_request) {                                    // split 0 writes the zeros
        for (int i = tid; i < R * kHeadDim; i += kUThreads)
            store_row_value(a.out, row_id(a, b, kvh, i / kHeadDim) * kHeadDim + i % kHeadDim, 0.f, a.out_fp32);
        return;
    }

    const int64_t t0 = static_cast<int64_t>(split) * a.split_tokens;
    const int64_t t1 = min(len, t0 + a.split_tokens);
    const int n_pages = static_cast<int>((t1 - 1) / ps) - first_page + 1;
    bool bad = false;
#pragma unroll
    for (int k = 0; k < kIdsPerThread; ++k) {
        const int i = tid + k * kUThreads;
        if (i < n_pages) {
            bad |= (ids[k] < 0 || ids[k] >= a.num_pages);
            page_list[i] = ids[k];
        }
    }
    if (tid == 0) {
        s_abort = 0;
        s_landed = 0;
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&full_e[i], 1);
            mbar_init(&empty_e[i], 4);
        }
        for (int i = 0; i < kKV; ++i) {
            mbar_init(&conv_full[i], 4);
            mbar_init(&pv_done[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&s_free[i], 4);
            mbar_init(&p_full[i], 4);
        }
        mbar_init(q_ready, 4);
        mbar_init(mma_drain, 1);
        mbar_init(pv_drain, 1);
        fence_mbar_init();
    }
    bad = __syncthreads_or(bad);

    auto publish_invalid = [&]() {                         // the request's rows get zeros
        if (nsplit == 1) {
            for (int i = tid; i < R * kHeadDim; i += kUThreads)
                store_row_value(a.out, row_id(a, b, kvh, i / kHeadDim) * kHeadDim + i % kHeadDim, 0.f,
                                a.out_fp32);
        } else if (tid < R) {
            a.ws_lse[row_id(a, b, kvh, tid) * a.max_splits + split] = __uint_as_float(0x7FC00000u);
        }
    };

    const int n_tiles = static_cast<int>((t1 - t0 + kTile - 1) / kTile);
    volatile int *abort_flag = &s_abort;
    // softmax thread m's row: copy m / Rp of local row m % Rp
    const int m = tid;
    const int copy = m / Rp, r = m % Rp;
    const bool row_valid = tid < 128 && r < R;
    float m_used = -INFINITY, l_sum = 0.f;
    int issued = 0;                                        // producer lane 0: tiles whose copies it issued

    if (bad) {
        publish_invalid();
    } else {
        if (warp == 0)
            tmem_alloc(tmem_slot, kTmemCols);
        tmem_fence_before_sync();
        __syncthreads();
        tmem_fence_after_sync();
        const uint32_t tmem = *tmem_slot;

        if (warp == kProducerWarp) {
            // ------------------------------------------------ producer
            const int box_tok = ps < kChunkTokens ? ps : kChunkTokens;
            const int parts = kTile / box_tok;             // 2 or 4 copies per tensor
            const uint64_t policy = l2_policy_evict_first();
            for (int j = 0; j < n_tiles; ++j) {
                const int st = j % kStages;
                if (j >= kStages &&
                    !__all_sync(0xFFFFFFFFu, wait_or_abort(&empty_e[st], ((j / kStages) - 1) & 1,
                                                           kCopyWaitLimitNs, abort_flag, 4u)))
                    break;
                const int64_t tok = t0 + static_cast<int64_t>(j) * kTile;
                const int64_t left = t1 - tok;
                const int np = static_cast<int>(left >= kTile ? parts : (left + box_tok - 1) / box_tok);
                if (lane == 0)
                    mbar_arrive_expect_tx(&full_e[st], static_cast<uint32_t>(2 * np * box_tok * 128));
                __syncwarp();
                if (lane < 2 * np) {                       // lanes 0 .. np - 1: K parts, np .. 2 np - 1: V parts
                    const bool is_v = lane >= np;
                    const int part = is_v ? lane - np : lane;
                    const int64_t ptok = tok + part * box_tok;
                    const int32_t page = page_list[static_cast<int>(ptok >> ps_shift) - first_page];
                    const int32_t y = static_cast<int32_t>((static_cast<int64_t>(page) * a.num_kv_heads + kvh) * ps +
                                                           (ptok & (ps - 1)));
                    uint8_t *dst = sm + kOffRing + st * kStageBytes + (is_v ? kTile * 128 : 0) +
                                   part * box_tok * 128;
                    tma_load_2d(dst, lane < np ? static_cast<const void *>(&k_map) : static_cast<const void *>(&v_map),
                                0, y, &full_e[st], policy);
                }
                issued = j + 1;
            }
        } else if (warp >= kConvWarp0 && warp < kConvWarp0 + 4) {
            // ------------------------------------------------ converters
            const int ct = tid - 32 * kConvWarp0;          // 0 .. 127
            const int c = ct & 7;                          // 16-byte chunk (16 dims) of an e4m3 row
            for (int j = 0; j < n_tiles; ++j) {
                const int st = j % kStages, kb = j % kKV;
                // every lane polls; the warp goes on or gives up as one
                if (!__all_sync(0xFFFFFFFFu, wait_or_abort(&full_e[st], (j / kStages) & 1, a.copy_wait_ns,
                                                           abort_flag, 1u)))
                    break;
                if (lane == 0)
                    atomicMax(&s_landed, j + 1);
                // operand buffer kb is free once O += P V of tile j - kKV is done
                if (j >= kKV && !__all_sync(0xFFFFFFFFu, wait_or_abort(&pv_done[kb], ((j - kKV) / kKV) & 1,
                                                                       kCopyWaitLimitNs, abort_flag, 4u)))
                    break;
                const uint8_t *kr = sm + kOffRing + st * kStageBytes;
                const uint8_t *vr = kr + kTile * 128;
                uint8_t *kd = sm + kOffKV + kb * kKVBytes;
                uint8_t *vd = kd + 16384;
                const int64_t tok0 = t0 + static_cast<int64_t>(j) * kTile;
                uint4 xk[4], xv[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {              // every load of the tile first
                    const int t = (ct >> 3) + 16 * k;
                    const uint32_t src = static_cast<uint32_t>(t * 128 + ((c ^ (t & 7)) << 4));
                    xk[k] = *reinterpret_cast<const uint4 *>(kr + src);
                    xv[k] = *reinterpret_cast<const uint4 *>(vr + src);
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int t = (ct >> 3) + 16 * k;
                    if (tok0 + t >= t1)                    // past the split: V rows must be zero
                        xv[k] = make_uint4(0u, 0u, 0u, 0u);
                    const uint32_t base = static_cast<uint32_t>((c >> 2) * 8192);
                    const uint32_t o0 = base + sw128_chunk(t, 2 * (c & 3));
                    const uint32_t o1 = base + sw128_chunk(t, 2 * (c & 3) + 1);
                    // the two slices share banks: lanes with c >= 4 store their
                    // two 16-byte chunks in the other order, so a store's 8
                    // lanes hit 8 bank groups (the words are picked before
                    // they are converted)
                    const bool swap = c >= 4;
                    const uint32_t oa = swap ? o1 : o0, ob = swap ? o0 : o1;
                    const uint32_t ka0 = swap ? xk[k].z : xk[k].x, ka1 = swap ? xk[k].w : xk[k].y;
                    const uint32_t kb0 = swap ? xk[k].x : xk[k].z, kb1 = swap ? xk[k].y : xk[k].w;
                    const uint32_t va0 = swap ? xv[k].z : xv[k].x, va1 = swap ? xv[k].w : xv[k].y;
                    const uint32_t vb0 = swap ? xv[k].x : xv[k].z, vb1 = swap ? xv[k].y : xv[k].w;
                    *reinterpret_cast<uint4 *>(kd + oa) =
                        make_uint4(lo16_e4m3x2_to_f16x2(ka0), hi16_e4m3x2_to_f16x2(ka0),
                                   lo16_e4m3x2_to_f16x2(ka1), hi16_e4m3x2_to_f16x2(ka1));
                    *reinterpret_cast<uint4 *>(kd + ob) =
                        make_uint4(lo16_e4m3x2_to_f16x2(kb0), hi16_e4m3x2_to_f16x2(kb0),
                                   lo16_e4m3x2_to_f16x2(kb1), hi16_e4m3x2_to_f16x2(kb1));
                    *reinterpret_cast<uint4 *>(vd + oa) =
                        make_uint4(lo16_e4m3x2_to_f16x2(va0), hi16_e4m3x2_to_f16x2(va0),
                                   lo16_e4m3x2_to_f16x2(va1), hi16_e4m3x2_to_f16x2(va1));
                    *reinterpret_cast<uint4 *>(vd + ob) =
                        make_uint4(lo16_e4m3x2_to_f16x2(vb0), hi16_e4m3x2_to_f16x2(vb0),
                                   lo16_e4m3x2_to_f16x2(vb1), hi16_e4m3x2_to_f16x2(vb1));
                }
                fence_proxy_async_smem();                  // the writes, for the tensor core;
                __syncwarp();                              // the ring reads, for the next copy
                if (lane == 0) {
                    mbar_arrive(&conv_full[kb]);
                    mbar_arrive(&empty_e[st]);
                }
            }
        } else if (warp == kMmaWarp) {
            // ------------------------------------------------ S = Q K^T issue
            // A tcgen05.mma occupies its issuing thread for about 125 cycles
            // at these shapes, while two issuing warps complete twice as
            // many: the two streams (S here, O += P V in warp kPvWarp) go
            // from two warps and run side by side.
            if (lane == 0) {
                // descriptor of the first operand buffer's K; a k step or
                // another buffer adds its byte offset / 16 to the start field
                const uint64_t dk = umma_desc(smem_addr(sm + kOffKV), 0, 1024);
                bool ok = wait_or_abort(q_ready, 0, kCopyWaitLimitNs, abort_flag, 4u);
                if (ok)
                    tmem_fence_after_sync();
                for (int js = 0; ok && js < n_tiles; ++js) {
                    // score buffer js & 1 is free once the softmax has read
                    // the scores of tile js - 2
                    if (js >= 2 && !wait_or_abort(&s_free[js & 1], ((js - 2) >> 1) & 1, kCopyWaitLimitNs,
                                                  abort_flag, 4u))
                        break;
                    if (!wait_or_abort(&conv_full[js % kKV], (js / kKV) & 1, kCopyWaitLimitNs, abort_flag, 4u))
                        break;
                    tmem_fence_after_sync();
                    const uint64_t dkb = dk + static_cast<uint64_t>(((js % kKV) * kKVBytes) >> 4);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)         // Q: 8 columns (16 dims) per k step
                        umma_f16_ts(tmem + kColS + 64u * (js & 1), tmem + kColQ + 8u * kk,
                                    dkb + static_cast<uint64_t>(((kk >> 2) * 8192 + (kk & 3) * 32) >> 4), kIdescS,
                                    kk > 0);
                    umma_commit(&s_full[js & 1]);
                }
                // nothing this lane issued may still run when the CTA moves on
                umma_commit(mma_drain);
                if (!mbar_wait_bounded(mma_drain, 0, kCopyWaitLimitNs))
                    atomicOr(&g_umma_error, 4u);
            }
            __syncwarp();
        } else if (warp == kPvWarp) {
            // ------------------------------------------------ O += P V issue
            if (lane == 0) {
                const uint64_t dv = umma_desc(smem_addr(sm + kOffKV + 16384), 8192, 1024);
                for (int jp = 0; jp < n_tiles; ++jp) {
                    // P of tile jp written (so its scores, hence its K and V
                    // operands, are complete too)
                    if (!wait_or_abort(&p_full[jp & 1], (jp >> 1) & 1, kCopyWaitLimitNs, abort_flag, 4u))
                        break;
                    const int pb = jp & 1, kb = jp % kKV;
                    tmem_fence_after_sync();
                    const uint64_t dvb = dv + static_cast<uint64_t>((kb * kKVBytes) >> 4);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)         // P: 8 columns (16 tokens) per k step
                        umma_f16_ts(tmem + kColO, tmem + kColP + 32u * pb + 8u * kk,
                                    dvb + static_cast<uint64_t>(kk * 128), kIdescPV, jp > 0 || kk > 0);
                    if constexpr (kPrecise) {
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            umma_f16_ts(tmem + kColO, tmem + kColPlo + 32u * pb + 8u * kk,
                                        dvb + static_cast<uint64_t>(kk * 128), kIdescPV, true);
                    }
                    umma_commit(&pv_done[kb]);
                }
                umma_commit(pv_drain);
                if (!mbar_wait_bounded(pv_drain, 0, kCopyWaitLimitNs))
                    atomicOr(&g_umma_error, 4u);
            }
            __syncwarp();
        } else {
            // ------------------------------------------------ softmax (warps 0..3)
            float mul = 0.f;                               // score multiplier (log2 domain)
            int64_t lim = t0;                              // positions below lim are visible
            {
                uint32_t w[64];
                if (row_valid) {
                    const uint4 *src = reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(a.q) +
                                                                       row_id(a, b, kvh, r) * kHeadDim);
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const uint4 v = __ldg(src + i);
                        w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 64; ++i)
                        w[i] = 0;
                }
                uint32_t mx = 0;
#pragma unroll
                for (int i = 0; i < 64; ++i)
                    mx = max(mx, max(w[i] & 0x7FFFu, (w[i] >> 16) & 0x7FFFu));
                const int e = q_row_exponent(mx);
                const float q_mul = __int_as_float((127 + e) << 23);
                // row m of Q as f16 pairs (dims 2c, 2c + 1 in column c)
                const uint32_t lane_q = static_cast<uint32_t>(32 * warp) << 16;
#pragma unroll
                for (int c0 = 0; c0 < 64; c0 += 16) {
                    uint32_t h[16];
#pragma unroll
                    for (int t = 0; t < 16; ++t) {
                        const float2 f = bf16x2_to_f32x2(w[c0 + t]);
                        h[t] = f32x2_to_f16x2(f.x * q_mul, f.y * q_mul);
                    }
                    tmem_st16(tmem + lane_q + kColQ + c0, h);
                }
                mul = a.qk_scale_log2 * a.k_scale[kvh] * __int_as_float((127 - e) << 23);
                if (row_valid) {
                    const int64_t vis = len - a.n_query + 1 + r / g;
                    lim = vis < t1 ? vis : t1;
                }
                tmem_fence_before_sync();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(q_ready);
            }
            const uint32_t lane_base = static_cast<uint32_t>(32 * warp) << 16;
            const int my0 = copy * kTpc;                   // this thread's tokens in a tile (its warp's)
            // Row m of P is this thread's alone: its columns outside the
            // copy's tokens are zeroed once here and never written again.
            {
                uint32_t zero[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    zero[i] = 0u;
#pragma unroll
                for (int c0 = 0; c0 < 64; c0 += 16) {
                    tmem_st16(tmem + lane_base + kColP + c0, zero);
                    if constexpr (kPrecise)
                        tmem_st16(tmem + lane_base + kColPlo + c0, zero);
                }
            }
            for (int j = 0; j < n_tiles; ++j) {
                const int sb = j & 1;                      // score and P buffer
                if (!__all_sync(0xFFFFFFFFu,
                                wait_or_abort(&s_full[sb], (j >> 1) & 1, kCopyWaitLimitNs, abort_flag, 4u)))
                    break;
                tmem_fence_after_sync();
                // this row's visible tokens of the tile: [my0, hi)
                const int64_t vl = lim - (t0 + static_cast<int64_t>(j) * kTile);
                const int hi = vl <= my0 ? my0 : (vl >= my0 + kTpc ? my0 + kTpc : static_cast<int>(vl));
                const uint32_t scol = tmem + lane_base + kColS + 64u * sb + static_cast<uint32_t>(my0);
                float p[kTpc];
                const uint64_t mul2 = f2_pack(mul, mul);
                if (__all_sync(0xFFFFFFFFu, hi == my0 + kTpc)) {   // every column visible: no masks
#pragma unroll
                    for (int q = 0; q < kTpc / 16; ++q) {
                        uint32_t sv[16];
                        tmem_ld16(scol + 16u * q, sv);
#pragma unroll
                        for (int i = 0; i < 16; i += 2)
                            f2_unpack(f2_mul(f2_pack(__uint_as_float(sv[i]), __uint_as_float(sv[i + 1])), mul2),
                                      p[16 * q + i], p[16 * q + i + 1]);
                    }
                } else {
#pragma unroll
                    for (int q = 0; q < kTpc / 16; ++q) {
                        uint32_t sv[16];
                        tmem_ld16(scol + 16u * q, sv);
#pragma unroll
                        for (int i = 0; i < 16; i += 2) {
                            float x0, x1;
                            f2_unpack(f2_mul(f2_pack(__uint_as_float(sv[i]), __uint_as_float(sv[i + 1])), mul2),
                                      x0, x1);
                            p[16 * q + i] = my0 + 16 * q + i < hi ? x0 : -INFINITY;
                            p[16 * q + i + 1] = my0 + 16 * q + i + 1 < hi ? x1 : -INFINITY;
                        }
                    }
                }
                // the scores are in registers: the buffer can take tile j + 2
                tmem_fence_before_sync();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&s_free[sb]);
                float mxa[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int i = 0; i < kTpc; ++i)
                    mxa[i & 3] = fmaxf(mxa[i & 3], p[i]);
                const float mx = fmaxf(fmaxf(mxa[0], mxa[1]), fmaxf(mxa[2], mxa[3]));
                const bool raise = mx > m_used + kRaiseThreshold;  // raise the running maximum
                const float alpha = raise ? (m_used == -INFINITY ? 0.f : fast_exp2(m_used - mx)) : 1.f;
                // O holds earlier tiles of row m: rescale it once O += P V of
                // tile j - 1 is done (warp-wide loads and stores: the other
                // lanes multiply by 1)
                const bool rescale = raise && m_used != -INFINITY && j > 0;
                if (__any_sync(0xFFFFFFFFu, rescale)) {
                    if (!__all_sync(0xFFFFFFFFu, wait_or_abort(&pv_done[(j - 1) % kKV], ((j - 1) / kKV) & 1,
                                                               kCopyWaitLimitNs, abort_flag, 4u)))
                        break;
                    tmem_fence_after_sync();
                    const float f = rescale ? alpha : 1.f;
#pragma unroll 1
                    for (int cc = 0; cc < 8; ++cc) {
                        uint32_t o[16];
                        const uint32_t addr = tmem + lane_base + kColO + 16 * cc;
                        tmem_ld16(addr, o);
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            o[i] = __float_as_uint(__uint_as_float(o[i]) * f);
                        tmem_st16(addr, o);
                    }
                }
                if (raise) {
                    l_sum *= alpha;
                    m_used = mx;
                }
                const float base = m_used == -INFINITY ? 0.f : m_used;
                const uint64_t nb2 = f2_pack(-base, -base);
                uint64_t sa2[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
#pragma unroll
                for (int i = 0; i < kTpc; i += 2) {
                    float x0, x1;
                    f2_unpack(f2_add(f2_pack(p[i], p[i + 1]), nb2), x0, x1);
                    p[i] = fast_exp2(x0);
                    p[i + 1] = fast_exp2(x1);
                    sa2[(i >> 1) & 1] = f2_add(sa2[(i >> 1) & 1], f2_pack(p[i], p[i + 1]));
                }
                float s0, s1, s2, s3;
                f2_unpack(sa2[0], s0, s1);
                f2_unpack(sa2[1], s2, s3);
                l_sum += (s0 + s1) + (s2 + s3);
                // P buffer sb is free once O += P V of tile j - 2 is done
                if (j >= 2 && !__all_sync(0xFFFFFFFFu, wait_or_abort(&pv_done[(j - 2) % kKV], ((j - 2) / kKV) & 1,
                                                                     kCopyWaitLimitNs, abort_flag, 4u)))
                    break;
                // row m of P over the copy's tokens, as f16 pairs
                const uint32_t pcol = tmem + lane_base + kColP + 32u * sb + static_cast<uint32_t>(my0 / 2);
                const uint32_t lcol = tmem + lane_base + kColPlo + 32u * sb + static_cast<uint32_t>(my0 / 2);
#pragma unroll
                for (int q = 0; q < kTpc / 16; ++q) {
                    uint32_t h[8];
#pragma unroll
                    for (int t = 0; t < 8; ++t)
                        h[t] = f32x2_to_f16x2(p[16 * q + 2 * t], p[16 * q + 2 * t + 1]);
                    tmem_st8(pcol + 8u * q, h);
                    if constexpr (kPrecise) {              // what the f16 rounding of P dropped
                        uint32_t l[8];
#pragma unroll
                        for (int t = 0; t < 8; ++t) {
                            const float2 hf = f16x2_to_f32x2(h[t]);
                            l[t] = f32x2_to_f16x2(p[16 * q + 2 * t] - hf.x, p[16 * q + 2 * t + 1] - hf.y);
                        }
                        tmem_st8(lcol + 8u * q, l);
                    }
                }
                tmem_fence_before_sync();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&p_full[sb]);
            }
            // the last tile's O += P V
            if (!*abort_flag)
                wait_or_abort(&pv_done[(n_tiles - 1) % kKV], ((n_tiles - 1) / kKV) & 1, kCopyWaitLimitNs,
                              abort_flag, 4u);
            __syncwarp();
            tmem_fence_after_sync();
        }

        tmem_fence_before_sync();
        __syncthreads();                                   // every role has finished or given up
        tmem_fence_after_sync();
        const bool failed = s_abort != 0;
        if (failed) {
            // Drain the copies still in flight (issued, not seen landed) with
            // the full limit, so that none lands in shared memory after the
            // CTA has moved on.  Tile t's copy is phase t / kStages of stage
            // t % kStages.
            if (warp == kProducerWarp && lane == 0) {
                bool drained = true;
                for (int t = s_landed; t < issued; ++t)
                    drained &= mbar_wait_bounded(&full_e[t % kStages], (t / kStages) & 1, kCopyWaitLimitNs);
                if (!drained)
                    atomicOr(&g_umma_error, 2u);
            }
            publish_invalid();
        }

        // ------------------------------------------ merge the copies of each row
        float *buf = reinterpret_cast<float *>(sm);                      // [128][kMergeStride]
        float *sm_m = buf + 128 * kMergeStride;
        float *sm_l = sm_m + 128;
        float *sm_lse = sm_l + 128;
        if (!failed && tid < 128) {
            sm_m[m] = m_used;
            sm_l[m] = l_sum;
            named_barrier_sync(1, 128);
            float wgt = 0.f;
            if (row_valid) {
                const int C = 128 / Rp;
                float M = -INFINITY;
                for (int c2 = 0; c2 < C; ++c2)
                    M = fmaxf(M, sm_m[Rp * c2 + r]);
                float L = 0.f;
                for (int c2 = 0; c2 < C; ++c2) {
                    const float mc = sm_m[Rp * c2 + r];
                    if (mc != -INFINITY)
                        L += fast_exp2(mc - M) * sm_l[Rp * c2 + r];
                }
                if (m_used != -INFINITY && L > 0.f)
                    wgt = fast_exp2(m_used - M) * a.v_scale[kvh] / L;
                if (copy == 0)
                    sm_lse[r] = L > 0.f ? M + __log2f(L) : -INFINITY;
            }
            // row m of O, weighted, into the merge buffer (a copy that saw no
            // token writes zeros)
            __syncwarp();
            const uint32_t lane_base = static_cast<uint32_t>(32 * warp) << 16;
#pragma unroll
            for (int cc = 0; cc < 8; ++cc) {
                uint32_t o[16];
                tmem_ld16(tmem + lane_base + kColO + 16 * cc, o);
#pragma unroll
                for (int i = 0; i < 16; i += 4) {
                    const float4 v = wgt != 0.f
                                         ? make_float4(__uint_as_float(o[i]) * wgt, __uint_as_float(o[i + 1]) * wgt,
                                                       __uint_as_float(o[i + 2]) * wgt, __uint_as_float(o[i + 3]) * wgt)
                                         : make_float4(0.f, 0.f, 0.f, 0.f);
                    *reinterpret_cast<float4 *>(buf + m * kMergeStride + 16 * cc + i) = v;
                }
            }
            tmem_fence_before_sync();
            named_barrier_sync(1, 128);
            // the copies' sum of each (row, 4 dims) item
            const int C = 128 / Rp;
            for (int it = tid; it < R * 32; it += 128) {
                const int rr = it >> 5, d4 = 4 * (it & 31);
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int c2 = 0; c2 < C; ++c2) {
                    const float4 x = *reinterpret_cast<const float4 *>(buf + (Rp * c2 + rr) * kMergeStride + d4);
                    v.x += x.x; v.y += x.y; v.z += x.z; v.w += x.w;
                }
                const int64_t id = row_id(a, b, kvh, rr);
                if (nsplit == 1)
                    store_row_value4(a.out, id * kHeadDim + d4, v, a.out_fp32);
                else
                    *reinterpret_cast<float4 *>(a.ws_o + (id * a.max_splits + split) * kHeadDim + d4) = v;
            }
            if (nsplit > 1 && tid < R)
                a.ws_lse[row_id(a, b, kvh, tid) * a.max_splits + split] = sm_lse[tid];
        }
        tmem_fence_before_sync();
        __syncthreads();
        if (warp == 0) {
            tmem_fence_after_sync();
            tmem_dealloc(tmem, kTmemCols);
        }
    }
    if (nsplit == 1 || tid >= 128)
        return;

    // ---------------------------------------------- combine of the splits
    // (warps 0..3).  The barrier orders every thread's partial before thread
    // 0's release; the last split's acquire, then its barrier, orders the
    // peers' partials before its loads.
    named_barrier_sync(1, 128);
    unsigned int *counter = a.counters + static_cast<int64_t>(b) * gridDim.y + kvh;
    if (tid == 0)
        s_last = atom_add_acq_rel_gpu(counter, 1u) == static_cast<unsigned int>(nsplit - 1);
    named_barrier_sync(1, 128);
    if (!s_last)
        return;
    // per row: the largest lse and the sum of the weights 2^(lse_s - max)
    // (0: a split was invalid, or none saw a token); with room, every
    // (row, split) weight over that sum in a table
    float *sm_S = reinterpret_cast<float *>(sm);            // [128]
    float *sm_w = sm_S + 128;                               // [R][nsplit] when it fits
    const bool table = R * nsplit <= kCombineTable;
    if (tid < R) {
        const int64_t base = row_id(a, b, kvh, tid) * a.max_splits;
        float M = -INFINITY;
        bool bad_row = false;
        for (int s2 = 0; s2 < nsplit; ++s2) {
            const float v = __ldcg(a.ws_lse + base + s2);
            bad_row |= v != v;
            M = fmaxf(M, v);
        }
        float S = 0.f;
        if (!bad_row && M != -INFINITY)
            for (int s2 = 0; s2 < nsplit; ++s2) {
                const float v = __ldcg(a.ws_lse + base + s2);
                if (v != -INFINITY)
                    S += fast_exp2(v - M);
            }
        S = bad_row ? 0.f : S;
        sm_S[tid] = S;
        if (table)
            for (int s2 = 0; s2 < nsplit; ++s2) {
                const float v = __ldcg(a.ws_lse + base + s2);
                sm_w[tid * nsplit + s2] = S > 0.f && v != -INFINITY ? fast_exp2(v - M) / S : 0.f;
            }
        else
            sm_w[tid] = M;                                  // the max, for weights computed on the fly
    }
    named_barrier_sync(1, 128);
    for (int it = tid; it < R * 32; it += 128) {
        const int rr = it >> 5, d4 = 4 * (it & 31);
        const int64_t id = row_id(a, b, kvh, rr);
        const float S = sm_S[rr];
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (S > 0.f) {
            const int64_t base = id * a.max_splits;
#pragma unroll 4
            for (int s2 = 0; s2 < nsplit; ++s2) {
                float w;
                if (table) {
                    w = sm_w[rr * nsplit + s2];
                } else {
                    const float v = __ldcg(a.ws_lse + base + s2);
                    w = v != -INFINITY ? fast_exp2(v - sm_w[rr]) / S : 0.f;
                }
                if (w != 0.f) {
                    const float4 x = __ldcg(reinterpret_cast<const float4 *>(a.ws_o + (base + s2) * kHeadDim + d4));
                    acc.x += w * x.x; acc.y += w * x.y; acc.z += w * x.z; acc.w += w * x.w;
                }
            }
        }
        store_row_value4(a.out, id * kHeadDim + d4, acc, a.out_fp32);
    }
    if (tid == 0)
        *counter = 0;                                      // ready for the next call
}

template <bool kPrecise, int kTpc>
cudaError_t configure_umma(int dev)
{
    static int configured[64] = {0};
    if (dev >= 0 && dev < 64 && configured[dev])
        return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(decode_mt_umma_kernel<kPrecise, kTpc>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes());
    if (e == cudaSuccess && dev >= 0 && dev < 64)
        configured[dev] = 1;
    return e;
}

template <bool kPrecise, int kTpc>
cudaError_t launch_umma(const DecodeArgs &a, const CUtensorMap &k_map, const CUtensorMap &v_map,
                        cudaStream_t stream)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    e = configure_umma<kPrecise, kTpc>(dev);
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(a.max_splits), static_cast<unsigned>(a.num_kv_heads),
                       static_cast<unsigned>(a.batch));
    cfg.blockDim = dim3(kUThreads);
    cfg.dynamicSmemBytes = smem_bytes();
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, decode_mt_umma_kernel<kPrecise, kTpc>, k_map, v_map, a);
    if (e != cudaSuccess)
        return e;
    return cudaGetLastError();
}

} // namespace

cudaError_t launch_decode_umma(const DecodeArgs &a, const CUtensorMap &k_map, const CUtensorMap &v_map,
                               cudaStream_t stream)
{
    if (a.batch == 0)
        return cudaSuccess;
    const int rows = a.n_query * a.group;
    if (rows < 33 || rows > 128)
        return cudaErrorInvalidValue;                      // the planner sends 64 .. 128 rows here
    if (rows > 64)
        return a.out_fp32 ? launch_umma<true, 64>(a, k_map, v_map, stream)
                          : launch_umma<false, 64>(a, k_map, v_map, stream);
    return a.out_fp32 ? launch_umma<true, 32>(a, k_map, v_map, stream)
                      : launch_umma<false, 32>(a, k_map, v_map, stream);
}

int decode_umma_ctas_per_sm()
{
    return 1;                                              // its shared memory takes most of an SM
}

cudaError_t read_umma_error(uint32_t *bits, bool clear)
{
    unsigned int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_umma_error, sizeof v);
    if (e != cudaSuccess)
        return e;
    if (bits)
        *bits = v;
    if (clear) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_umma_error, &zero, sizeof zero);
    }
    return e;
}

} // namespace kvq
