// kvq_decode.cu -- single-token paged decode attention over an FP8 e4m3 (or
// BF16) KV cache, split along the context, with the log-sum-exp combine of
// the splits fused into the same launch.
//
// What it computes (blog post "Smaller, faster, safer: running Kimi and GLM
// at scale", page-1 mirror section "量化KV缓存"; page-3 mirror section
// "FP8 省的不仅是显存"): decode attention whose kernel converts the FP8
// values it reads.  For query head h of request r, KV head kvh = h / g:
//   out = sum_j exp(s_j - max s) V^_j / sum_j exp(s_j - max s),
//   s_j = softmax_scale * <q, K^_j>,  K^ = e4m3 value * k_scale[kvh].
//
// One CTA per (split, KV head, request) covers every query head of the
// group, so each cache byte is fetched from HBM and converted once.  Four
// warps; each warp owns every 4th 32-token chunk of the split and a private
// 2-stage ring of shared-memory tiles filled by 2-D tensor bulk copies (TMA,
// 128-byte swizzle) that an mbarrier per stage tracks, a chunk's copies
// issued from several lanes at once; three CTAs fit on an SM, so twelve
// independent copy streams keep HBM busy.  Per chunk the warp
// runs, on the tensor cores (mma.sync m16n8k16, f16 in, fp32 accumulate),
// S^T = K Q^T with tokens as M and the g <= 8 query heads as N, an fp32
// online softmax, and O^T += V^T P^T.  e4m3 codes become f16 in registers
// (exact); movmatrix turns the score fragment into the PV operand.  The four
// warps merge in shared memory.  A request that fits in one split gets its
// output here.  Otherwise the splits merge (the combine) in one of two forms:
// when every (request, KV head)'s splits can be resident at once as one
// thread-block cluster, through distributed shared memory after a cluster
// barrier; else each split publishes (lse, o) to the workspace and the last
// split of the (request, KV head) to finish merges them all, counted by a
// per-(request, KV head) arrival counter that it resets to zero.
#include <cfloat>
#include <map>
#include <mutex>
#include <tuple>
#include <type_traits>

#include <cuda_bf16.h>

#include "kvq_internal.h"
#include "kvq_ptx.cuh"
#include "kvq_rowops.cuh"

namespace kvq {

// Sticky device error word.  Bit 0: a bulk-copy wait timed out.  Bit 1: the
// drain that follows also gave up, so a copy may still land in the shared
// memory the CTA leaves behind.
__device__ unsigned int g_device_error = 0;

#ifdef KVQ_PHASE_STAMPS
// Instrumented build only (-DKVQ_PHASE_STAMPS, a library of its own): thread
// 0 of every CTA of a decode launch records %globaltimer at fixed points;
// the host reads them back after the launch (nothing is cleared in between,
// so no extra operation separates the launch from the one before it: a point
// a CTA did not reach keeps an older time than its entry).  Points:
// 0 entry, 1 the programmatic-launch wait returned, 2 warp 0's first chunk
// landed, 3 every warp done streaming, 4 in-CTA merge done, 5 the combine's
// first synchronisation passed (cluster barrier or arrival counter),
// 6 exit of a CTA that streamed.
constexpr int kStampCtas = 8192;
constexpr int kStampPoints = 8;
__device__ unsigned long long g_phase_stamps[kStampCtas * kStampPoints];
__device__ __forceinline__ void phase_stamp(int point)
{
    if (threadIdx.x == 0) {
        const unsigned cta = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
        if (cta < kStampCtas)
            g_phase_stamps[cta * kStampPoints + point] = global_timer_ns();
    }
}
#define KVQ_STAMP(p) phase_stamp(p)
#else
#define KVQ_STAMP(p) ((void)0)
#endif

namespace {

constexpr int kWarps = 4;
constexpr int kCtasPerSm = 3;
constexpr int kThreads = kWarps * 32;
constexpr int kMaxPageList = 8192 / 16 + 8;       // page ids of one split (<= 8192 tokens)
// Published lse of a split that has no result: both are NaN, so the combine
// zeroes the request either way; the payload tells a failed tag check (the
// request is aborted and its new token not written) from a copy timeout.
constexpr uint32_t kLseInvalid = 0x7FC00000u;
constexpr uint32_t kLseStale = 0x7FC0A5A5u;

template <bool kBf16Cache>
struct Tile {
    static constexpr int kRowBytes = kBf16Cache ? 256 : 128;      // one token of one head
    static constexpr int kBytes = kChunkTokens * kRowBytes;       // K (or V) part of a stage
    static constexpr int kStages = 2;
    static constexpr int kStageBytes = 2 * kBytes;
    static constexpr int kRingBytes = kWarps * kStages * kStageBytes;
    static constexpr int kSmemBytes = 1024 /* alignment slack */ + kRingBytes +
                                      kWarps * kStages * 8 /* barriers */ + kMaxPageList * 4 +
                                      2 * kMaxPageList * 4 /* tags of the split's pages */ +
                                      512 /* the new token's K and V row */ + 16;
};

// Byte offset of 16-byte chunk `c` of 128-byte line `line` in a tile written
// by a 128-byte-swizzled tensor copy into a 1024-byte-aligned buffer.
__device__ __forceinline__ uint32_t swz(int line, int c)
{
    return static_cast<uint32_t>(line * 128 + ((c ^ (line & 7)) << 4));
}

// The exponent e that puts a row's largest magnitude, given as the bf16 bits
// `mx` of |q| (sign cleared), in [2^14, 2^15): e = 14 - floor(log2 |q|max),
// at most 100 (a row below 2^-86 is scaled up less; its scores are that much
// closer to 0 anyway), so that 2^e and 2^-e are normal fp32 numbers (e is at
// least -113 for finite bf16).  A row of zeros keeps e = 0.
__device__ __forceinline__ int row_pow2_exponent(uint32_t mx)
{
    if (mx == 0)
        return 0;
    const int field = static_cast<int>(mx >> 7);           // biased exponent (no sign bit)
    const int e_floor = field != 0 ? field - 127 : (31 - __clz(static_cast<int>(mx))) - 133;
    const int e = 14 - e_floor;
    return e > 100 ? 100 : e;
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


// The query rows one CTA serves.  The rows of (request b, KV head kvh) are
// (token i, head h) for the request's n_query new tokens and the g query
// heads of the group, row i * g + h; a CTA takes rows row0 .. row0 + nrows - 1
// (at most rows_per_cta(kMulti)).  With one query token (kMulti false, the
// kernel compiled for that case) the rows are the group's heads, one mma
// n-tile of 8, and one CTA takes them all; the multi-token kernel gives each
// warp two n-tiles (16 rows), so every chunk's conversions serve 16 rows.
template <bool kMulti>
struct Rows {
    int b, kvh, row0, nrows;
    int64_t slot;                            // this (request, KV head, row block)'s arrival counter

    // Row of q and out ([B][n_query][Hq][D], in units of head_dim) of local row r.
    __device__ __forceinline__ int64_t id(const DecodeArgs &a, int r) const
    {
        if constexpr (!kMulti)
            return static_cast<int64_t>(b) * a.num_q_heads + kvh * a.group + r;
        const int rr = row0 + r;
        return (static_cast<int64_t>(b) * a.n_query + rr / a.group) * a.num_q_heads + kvh * a.group +
               rr % a.group;
    }
};

// The warps' merge area holds one row of 128 floats per (warp, head).  Row
// stride and a skew of 2 words per 32 dims make the fragment stores (a lane
// writes dims 16*(lane/4) + 2i, +1 of heads 2*(lane%4), +1) hit 16 distinct
// bank pairs per half-warp, and keep the row reads (thread d) conflict-free.
constexpr int kMergeStride = 146;                 // >= 128 + 6, == 2 (mod 16)
__device__ __forceinline__ int merge_col(int d) { return d + 2 * (d >> 5); }

// Shared-memory offset (in floats) of the combine scratch: just past the
// warps' merge area, inside the ring (idle by then).
// Query rows of one CTA: one mma n-tile (8) for a single query token, two
// (16) for the multi-token kernel.
__host__ __device__ constexpr int rows_per_cta(bool multi) { return multi ? 2 * kMaxGroup : kMaxGroup; }


// Shared-memory offset (in floats) of the cluster partial: just past the
// warps' merge area, inside the ring (idle by then).  The workspace combine's
// scratch starts at offset 0: it runs after the CTA's own partial has left
// the merge area for global memory.
__host__ __device__ constexpr int scratch_offset(bool multi)
{
    return (kWarps * rows_per_cta(multi) * kMergeStride + 3 * kWarps * rows_per_cta(multi) +
            2 * rows_per_cta(multi) + 3) / 4 * 4;
}
constexpr int kScratchOffset = scratch_offset(false);
static_assert((kMaxGroup + kMaxGroup * kMaxSplitsTotal) * 4 <= Tile<false>::kRingBytes,
              "the workspace combine's scratch fits in the idle ring");
static_assert((2 * kMaxGroup + 2 * kMaxGroup * kMultiMaxSplitsPerRequest) * 4 <= Tile<false>::kRingBytes,
              "the multi-token workspace combine's scratch fits in the idle ring");
static_assert((kScratchOffset + kMaxGroup + kMaxGroup * kHeadDim) * 4 <= Tile<false>::kRingBytes,
              "the cluster combine's partial fits in the idle ring");
static_assert((scratch_offset(true) + 2 * kMaxGroup + 2 * kMaxGroup * kHeadDim) * 4 <= Tile<false>::kRingBytes,
              "the multi-token cluster partial fits in the idle ring");

// Count this split's arrival for (request b, KV head kvh).  The last split
// to arrive merges the partials of all nsplit splits of the group:
//   M = max_s lse_s,  out = sum_s 2^(lse_s - M) o_s / sum_s 2^(lse_s - M),
// for every query head of the group at once, writes the output (zeros for
// a head if any split was invalid) and resets the counter.
// kvq_decode_step, once per (request, KV head), by the CTA that knows the
// verdict of all the request's splits: KV head 0 writes the abort flag, and
// a request that passed gets its new token written for this KV head (the
// codes kvq_append writes).  A split holding the token has already patched
// them into its own tile, and no other CTA of this launch reads that row.
__device__ void finish_step(const DecodeArgs &a, int b, int kvh, bool stale)
{
    if (kvh == 0 && threadIdx.x == 0)
        a.abort_out[b] = stale ? 1 : 0;
    if (stale || threadIdx.x >= 32)
        return;
    const int lane = threadIdx.x;
    const int64_t tpos = static_cast<int64_t>(a.seq_lens[b]) - 1;     // > 0: the request was not empty
    const int32_t page = a.block_table[static_cast<int64_t>(b) * a.max_pages_per_seq + tpos / a.page_size];
    if (page < 0 || page >= a.num_pages)                                 // excluded by the check
        return;
    const int64_t row = (static_cast<int64_t>(page) * a.num_kv_heads + kvh) * a.page_size + tpos % a.page_size;
    const int64_t src = (static_cast<int64_t>(b) * a.num_kv_heads + kvh) * kHeadDim + 4 * lane;
    const uint2 xk = *reinterpret_cast<const uint2 *>(static_cast<const uint16_t *>(a.k_new) + src);
    const uint2 xv = *reinterpret_cast<const uint2 *>(static_cast<const uint16_t *>(a.v_new) + src);
    if (a.bf16_cache) {
        *reinterpret_cast<uint2 *>(static_cast<uint8_t *>(a.k_cache) + row * 256 + 8 * lane) = xk;
        *reinterpret_cast<uint2 *>(static_cast<uint8_t *>(a.v_cache) + row * 256 + 8 * lane) = xv;
    } else {
        *reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(a.k_cache) + row * 128 + 4 * lane) =
            encode4_e4m3(xk.x, xk.y, a.k_scale[kvh]);
        *reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(a.v_cache) + row * 128 + 4 * lane) =
            encode4_e4m3(xv.x, xv.y, a.v_scale[kvh]);
    }
}

template <bool kMulti>
__device__ void publish_and_combine(const DecodeArgs &a, const Rows<kMulti> &R, int nsplit, float *scratch)
{
    __shared__ int s_last;
    // The block barrier orders every thread's partial before thread 0's
    // release; the last split's acquire, then its barrier, orders all the
    // peers' partials before its loads (the counter is the only
    // synchronisation between the splits).
    __syncthreads();
    unsigned int *counter = a.counters + R.slot;
    if (threadIdx.x == 0)
        s_last = atom_add_acq_rel_gpu(counter, 1u) == static_cast<unsigned int>(nsplit - 1);
    __syncthreads();
    KVQ_STAMP(5);
    if (!s_last)
        return;
    constexpr int kRowsT = rows_per_cta(kMulti);
    const int g = R.nrows, n = nsplit;
    float *s_tot = scratch;                  // [kRowsT] sum of weights (0: drop the row)
    float *s_w = scratch + kRowsT;           // [g][n]: lse, then weights
    for (int i = threadIdx.x; i < g * n; i += kThreads)
        s_w[i] = __ldcg(a.ws_lse + R.id(a, i / n) * a.max_splits + i % n);
    __syncthreads();
    // one warp per head: max, validity, weights, their sum
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    for (int h = warp; h < g; h += kWarps) {
        float *w = s_w + h * n;
        float m = -INFINITY;
        bool bad = false;
        for (int s = lane; s < n; s += 32) {
            bad |= w[s] != w[s];
            m = fmaxf(m, w[s]);
        }
        bad = __any_sync(0xFFFFFFFFu, bad);
        for (int off = 16; off > 0; off >>= 1)
            m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
        float sum = 0.f;
        for (int s = lane; s < n; s += 32) {         // a split that saw no token: lse -inf, weight 0
            const float e = (bad || w[s] == -INFINITY) ? 0.f : fast_exp2(w[s] - m);
            w[s] = e;
            sum += e;
        }
        for (int off = 16; off > 0; off >>= 1)
            sum += __shfl_xor_sync(0xFFFFFFFFu, sum, off);
        if (lane == 0)
            s_tot[h] = bad ? 0.f : sum;
    }
    __syncthreads();
    // thread t: the (row, 4 dims) pairs t, t + 128, ... of the rows x 32;
    // kRound splits per round, every 16-byte load of a round issued before
    // any is used, so a round costs one trip to L2
    constexpr int kPairs = kRowsT * (kHeadDim / 4) / kThreads;          // 2, or 4 with 16 rows
    constexpr int kRound = kMulti ? 4 : 8;
    static_assert(kRowsT * (kHeadDim / 4) == kPairs * kThreads, "whole (row, 4 dims) pairs per thread");
    int hp[kPairs];
#pragma unroll
    for (int q = 0; q < kPairs; ++q)
        hp[q] = static_cast<int>(threadIdx.x + q * kThreads) / 32;
    const int cp = 4 * (threadIdx.x % 32);
    float4 acc[kPairs];
#pragma unroll
    for (int q = 0; q < kPairs; ++q)
        acc[q] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < n; s0 += kRound) {
        float4 v[kPairs][kRound];
#pragma unroll
        for (int q = 0; q < kPairs; ++q)
#pragma unroll
            for (int j = 0; j < kRound; ++j)
                v[q][j] = (hp[q] < g && s0 + j < n)
                              ? __ldcg(reinterpret_cast<const float4 *>(
                                    a.ws_o + (R.id(a, hp[q]) * a.max_splits + s0 + j) * kHeadDim + cp))
                              : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int q = 0; q < kPairs; ++q)
#pragma unroll
            for (int j = 0; j < kRound; ++j)
                if (hp[q] < g && s0 + j < n) {
                    const float wt = s_w[hp[q] * n + s0 + j];
                    acc[q].x += wt * v[q][j].x;
                    acc[q].y += wt * v[q][j].y;
                    acc[q].z += wt * v[q][j].z;
                    acc[q].w += wt * v[q][j].w;
                }
    }
#pragma unroll
    for (int q = 0; q < kPairs; ++q)
        if (hp[q] < g) {
            const int64_t o0 = R.id(a, hp[q]) * kHeadDim + cp;
            store_out(a.out, o0, s_tot[hp[q]] > 0.f ? acc[q].x / s_tot[hp[q]] : 0.f, a.out_fp32);
            store_out(a.out, o0 + 1, s_tot[hp[q]] > 0.f ? acc[q].y / s_tot[hp[q]] : 0.f, a.out_fp32);
            store_out(a.out, o0 + 2, s_tot[hp[q]] > 0.f ? acc[q].z / s_tot[hp[q]] : 0.f, a.out_fp32);
            store_out(a.out, o0 + 3, s_tot[hp[q]] > 0.f ? acc[q].w / s_tot[hp[q]] : 0.f, a.out_fp32);
        }
    if (a.expected_tags != nullptr) {        // kvq_decode_step: the request's verdict
        __shared__ int s_stale_any;
        if (threadIdx.x == 0) {
            int any = 0;
            for (int sp = 0; sp < n; ++sp)
                any |= __float_as_uint(__ldcg(a.ws_lse + R.id(a, 0) * a.max_splits + sp)) == kLseStale;
            s_stale_any = any;
        }
        __syncthreads();
        finish_step(a, R.b, R.kvh, s_stale_any != 0);
    }
    if (threadIdx.x == 0)
        *counter = 0;                        // ready for the next call
}

// A split that cannot produce a result (invalid page id, or a copy that
// timed out): a single-split request gets zeros; otherwise the split
// publishes an invalid (NaN) lse so the combine zeroes the request.
template <bool kMulti>
__device__ void drop_split(const DecodeArgs &a, const Rows<kMulti> &R, int split, int nsplit, float *smem,
                           uint32_t lse_bits = kLseInvalid)
{
    if (nsplit == 1) {
        for (int i = threadIdx.x; i < R.nrows * kHeadDim; i += kThreads)
            store_out(a.out, R.id(a, i / kHeadDim) * kHeadDim + i % kHeadDim, 0.f, a.out_fp32);
        if (a.expected_tags != nullptr)
            finish_step(a, R.b, R.kvh, lse_bits == kLseStale);
        return;
    }
    if (threadIdx.x < R.nrows)
        a.ws_lse[R.id(a, threadIdx.x) * a.max_splits + split] = __uint_as_float(lse_bits);
    publish_and_combine(a, R, nsplit, kMulti ? smem : smem + kScratchOffset);
}

// What a split contributes to the cluster form of the combine.
// Cluster-wide barrier with a relaxed arrive: it orders no memory access,
// only the threads' progress (the wait still acquires).
__device__ __forceinline__ void cluster_sync_relaxed_arrive()
{
    asm volatile("barrier.cluster.arrive.relaxed.aligned;\n\t"
                 "barrier.cluster.wait.aligned;" ::: "memory");
}

enum PartialStatus { kPartialOk = 0, kPartialEmpty = 1, kPartialInvalid = 2, kPartialStale = 3 };

// Cluster form of the combine, used when the splits of each (request, KV
// head) are the CTAs of one thread-block cluster (every split resident at
// once).  Each CTA leaves its partial in its own shared memory at `part`:
// [rows] lse (log2 domain), then [rows][128] normalised o (rows =
// rows_per_cta(kMulti)); an empty
// split (no tokens) publishes lse = -inf (weight 0), an invalid one NaN (its
// heads get zeros).  After a cluster barrier CTA r merges the query heads
// h = r, r + n, ... of the group from every peer's partial, read through
// distributed shared memory:
//   M = max_s lse_s,  out = sum_s 2^(lse_s - M) o_s / sum_s 2^(lse_s - M).
// A second barrier keeps every CTA's shared memory alive until its peers
// have read it.  It needs no release: a thread reaches it only after the
// values it loaded from its peers have been consumed by its output stores,
// and a release there would make every CTA wait for those global stores.
// Every CTA of the cluster calls this exactly once, with the same
// `finisher`: for kvq_decode_step the rank that reads every peer's verdict,
// else -1.  Returns, on the finisher, whether any split of the
// request failed its tag check (false elsewhere).
template <bool kMulti>
__device__ bool cluster_finish(const DecodeArgs &a, const Rows<kMulti> &R, PartialStatus status, float *part,
                               int finisher)
{
    __shared__ int s_any_stale;
    constexpr int kRowsT = rows_per_cta(kMulti);
    if (status != kPartialOk && threadIdx.x < kRowsT)
        part[threadIdx.x] = status == kPartialEmpty ? -INFINITY
                            : __uint_as_float(status == kPartialStale ? kLseStale : kLseInvalid);
    cluster_sync();
    KVQ_STAMP(5);
    const int g = R.nrows, n = a.max_splits;
    const int rank = static_cast<int>(cluster_ctarank());
    const uint32_t base = smem_addr(part);
    if (rank == finisher && threadIdx.x == 0) {            // every peer's head-0 lse carries its verdict
        int stale = 0;
        for (int sp = 0; sp < n; ++sp)
            stale |= __float_as_uint(ld_shared_cluster_f32(map_shared_rank(base, static_cast<uint32_t>(sp)))) ==
                     kLseStale;
        s_any_stale = stale;
    }
    // thread t takes dims 4 (t % 32) .. + 3 of head h0 + t / 32 (16-byte
    // loads from each peer), 4 of this CTA's heads per pass
    for (int h0 = rank; h0 < g; h0 += kThreads / 32 * n) {
        const int h = h0 + (threadIdx.x / 32) * n;
        if (h >= g)
            continue;
        const int d = 4 * (threadIdx.x % 32);
        float lse[kMaxCluster];
        float4 ov[kMaxCluster];
#pragma unroll
        for (int s = 0; s < kMaxCluster; ++s) {
            lse[s] = -INFINITY;
            ov[s] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (s < n) {
                const uint32_t peer = map_shared_rank(base, static_cast<uint32_t>(s));
                lse[s] = ld_shared_cluster_f32(peer + 4u * h);
                ov[s] = ld_shared_cluster_v4(peer + 4u * (kRowsT + h * kHeadDim + d));
            }
        }
        float m = -INFINITY;
        bool bad = false;
#pragma unroll
        for (int s = 0; s < kMaxCluster; ++s) {
            bad |= lse[s] != lse[s];
            m = fmaxf(m, lse[s]);
        }
        float sum = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int s = 0; s < kMaxCluster; ++s) {
            if (lse[s] != -INFINITY) {
                const float w = fast_exp2(lse[s] - m);
                sum += w;
                acc.x += w * ov[s].x;
                acc.y += w * ov[s].y;
                acc.z += w * ov[s].z;
                acc.w += w * ov[s].w;
            }
        }
        const bool zero = bad || !(sum > 0.f);
        const int64_t o0 = R.id(a, h) * kHeadDim + d;
        store_out(a.out, o0, zero ? 0.f : acc.x / sum, a.out_fp32);
        store_out(a.out, o0 + 1, zero ? 0.f : acc.y / sum, a.out_fp32);
        store_out(a.out, o0 + 2, zero ? 0.f : acc.z / sum, a.out_fp32);
        store_out(a.out, o0 + 3, zero ? 0.f : acc.w / sum, a.out_fp32);
    }
    __syncthreads();                         // orders s_any_stale within the CTA
    cluster_sync_relaxed_arrive();           // peers' reads of this CTA's partial are done
    return rank == finisher && s_any_stale != 0;
}

template <bool kBf16Cache, bool kPreciseP, bool kCluster, bool kMulti>
__global__ void __launch_bounds__(kThreads, kMulti ? 2 : kCtasPerSm)
decode_split_kernel(const __grid_constant__ CUtensorMap k_map,
                    const __grid_constant__ CUtensorMap v_map, const DecodeArgs a)
{
    using T = Tile<kBf16Cache>;
    KVQ_STAMP(0);
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + T::kRingBytes);
    int32_t *page_list = reinterpret_cast<int32_t *>(full + kWarps * T::kStages);
    uint32_t *tag_live = reinterpret_cast<uint32_t *>(page_list + kMaxPageList);   // kvq_decode_step:
    uint32_t *tag_want = tag_live + kMaxPageList;                                  // the split's tags
    uint8_t *new_tok = reinterpret_cast<uint8_t *>(tag_want + kMaxPageList);       // [K row][V row]
    __shared__ int s_failed;
    __shared__ int s_stale;                                // kvq_decode_step: a page of this split failed

    const int split = blockIdx.x, b = blockIdx.z;
    // with several query tokens, blockIdx.y = KV head x row blocks of 8 rows
    const int kvh = kMulti ? static_cast<int>(blockIdx.y) / a.row_blocks : static_cast<int>(blockIdx.y);
    const int rb = kMulti ? static_cast<int>(blockIdx.y) % a.row_blocks : 0;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int gq = lane >> 2, tq = lane & 3;
    const int g = a.group, ps = a.page_size;
    const int ps_shift = __ffs(ps) - 1;                  // ps is 16, 32, 64 or 128
    Rows<kMulti> R;
    R.b = b;
    R.kvh = kvh;
    R.row0 = rb * rows_per_cta(kMulti);
    R.nrows = kMulti ? min(rows_per_cta(true), a.n_query * g - R.row0) : g;
    R.slot = static_cast<int64_t>(b) * gridDim.y + blockIdx.y;

    const int first_page = static_cast<int>(static_cast<int64_t>(split) * a.split_tokens / ps);
    const int span_left = a.max_pages_per_seq - first_page;
    const int span = a.split_tokens / ps < span_left ? a.split_tokens / ps : span_left;
    const int32_t *bt = a.block_table + static_cast<int64_t>(b) * a.max_pages_per_seq + first_page;
    const int lines_per_tok = kBf16Cache ? 2 : 1;

    // Launched as a programmatic dependent of the previous kernel on the
    // stream (in a decode step: the tag check): the CTA can be resident and
    // have its tensor maps fetched while that kernel runs, and it reads no
    // global memory until the wait has returned, that is until the previous
    // kernel has completed and its writes are visible.  (Asking L2 for the
    // split's first pages before the wait made the step slower: those
    // requests compete with the check for the memory system.)
    if (threadIdx.x == 0) {
        prefetch_tensor_map(&k_map);
        prefetch_tensor_map(&v_map);
    }
    grid_dependency_wait();
    KVQ_STAMP(1);

    // The block-table entries this split can use depend only on the split
    // index, so they are loaded together with the request's length.
    constexpr int kIdsPerThread = (kMaxPageList + kThreads - 1) / kThreads;
    int32_t ids[kIdsPerThread];
#pragma unroll
    for (int k = 0; k < kIdsPerThread; ++k) {
        const int i = threadIdx.x + k * kThreads;
        ids[k] = i < span ? __ldg(bt + i) : -1;
    }
    const int64_t len = a.seq_lens[b];
    // kvq_decode_step: each split checks the tags of its own pages (together
    // the request's used entries) while it streams them, and publishes a
    // failure with its partial; the CTA that sees every split's partial
    // writes the flag and, if the request passed, its new token
    // (finish_here, or finish_step in the workspace form).  A request
    // without tokens to check is decided here.
    const bool step_check = a.expected_tags != nullptr;
    const bool reporter = step_check && split == 0 && kvh == 0 && threadIdx.x == 0;
    const bool aborted = !step_check && a.abort_flags != nullptr && a.abort_flags[b] != 0;
    const int64_t cap = static_cast<int64_t>(a.max_pages_per_seq) * ps;
    const bool zero_request = aborted || len <= 0 || len > cap;
    if (reporter && zero_request)                          // the check's verdict without a look:
        a.abort_out[b] = len > cap ? 1 : 0;                // too long fails, empty passes
    const int nsplit = zero_request ? 1 : static_cast<int>((len + a.split_tokens - 1) / a.split_tokens);
    float *part = reinterpret_cast<float *>(smem) + scratch_offset(kMulti);   // cluster partial
    // kvq_decode_step: the split that finishes the step of a request with
    // tokens in the cluster form and when there is one split -- the last
    // split, which holds the new token (the workspace form's combine
    // finishes in whichever split arrives last)
    const int finisher = step_check && !zero_request ? nsplit - 1 : -1;
    if constexpr (kCluster) {
        if (zero_request || split >= nsplit) {             // no tokens: weight 0
            cluster_finish(a, R, kPartialEmpty, part, finisher);
            return;
        }
    }
    if (split >= nsplit)
        return;

    if (zero_request) {                                    // split 0 writes the zeros
        for (int i = threadIdx.x; i < R.nrows * kHeadDim; i += kThreads)
            store_out(a.out, R.id(a, i / kHeadDim) * kHeadDim + i % kHeadDim, 0.f, a.out_fp32);
        return;
    }

    const int64_t t0 = static_cast<int64_t>(split) * a.split_tokens;
    const int64_t t1 = min(len, t0 + a.split_tokens);
    // page ids of this split (t0 is a multiple of the page size)
    const int n_pages = static_cast<int>((t1 - 1) / ps) - first_page + 1;
    bool bad = false;
#pragma unroll
    for (int k = 0; k < kIdsPerThread; ++k) {
        const int i = threadIdx.x + k * kThreads;
        if (i < n_pages) {
            bad |= (ids[k] < 0 || ids[k] >= a.num_pages);
            page_list[i] = ids[k];
        }
    }
    if (threadIdx.x == 0) {
        s_failed = 0;
        s_stale = 0;
        for (int i = 0; i < kWarps * T::kStages; ++i)
            mbar_init(&full[i], 1);
        fence_mbar_init();
    }
    bad = __syncthreads_or(bad);

    // Fused append (kvq_decode_attn_append): the split holding token len - 1
    // writes that token's codes for KV head kvh into the cache now (when its
    // page id is valid, as kvq_append would) and patches them into its tile
    // when the chunk's copy lands, so its own attention uses them without
    // reading them back.
    int it_new = -1;
    using NewRow = std::conditional_t<kBf16Cache, uint2, uint32_t>;   // a lane's part of the row
    NewRow new_k{}, new_v{};
    int64_t new_row = -1;                                  // cache row of the new token
    if (a.k_new != nullptr && split == nsplit - 1) {
        const int64_t tpos = len - 1;
        const int c_last = static_cast<int>((tpos - t0) / kChunkTokens);
        const int32_t page = page_list[static_cast<int>(tpos / ps) - first_page];
        if (warp == c_last % kWarps && page >= 0 && page < a.num_pages) {
            it_new = c_last / kWarps;
            const int64_t src = (static_cast<int64_t>(b) * a.num_kv_heads + kvh) * kHeadDim + 4 * lane;
            const uint2 xk = *reinterpret_cast<const uint2 *>(static_cast<const uint16_t *>(a.k_new) + src);
            const uint2 xv = *reinterpret_cast<const uint2 *>(static_cast<const uint16_t *>(a.v_new) + src);
            new_row = (static_cast<int64_t>(page) * a.num_kv_heads + kvh) * ps + tpos % ps;
            if constexpr (kBf16Cache) {
                new_k = xk;
                new_v = xv;
            } else {
                new_k = encode4_e4m3(xk.x, xk.y, a.k_scale[kvh]);
                new_v = encode4_e4m3(xv.x, xv.y, a.v_scale[kvh]);
            }
            if (step_check) {                              // kept for the end of the step
                reinterpret_cast<NewRow *>(new_tok)[lane] = new_k;
                reinterpret_cast<NewRow *>(new_tok + T::kRowBytes)[lane] = new_v;
            }
        }
    }
    // kvq_decode_step, on the split that holds the new token (the request's
    // last split) once the request's verdict is known: KV head 0 reports
    // it, and a request that passed gets the staged row written.
    auto finish_here = [&](bool stale) {
        if (kvh == 0 && threadIdx.x == 0)
            a.abort_out[b] = stale ? 1 : 0;
        const int64_t tpos = len - 1;
        const int32_t page = page_list[static_cast<int>(tpos / ps) - first_page];
        if (stale || threadIdx.x >= 32 || page < 0 || page >= a.num_pages)
            return;
        const int64_t row = (static_cast<int64_t>(page) * a.num_kv_heads + kvh) * ps + tpos % ps;
        const int ln = threadIdx.x;
        *reinterpret_cast<NewRow *>(static_cast<uint8_t *>(a.k_cache) + row * T::kRowBytes + sizeof(NewRow) * ln) =
            reinterpret_cast<const NewRow *>(new_tok)[ln];
        *reinterpret_cast<NewRow *>(static_cast<uint8_t *>(a.v_cache) + row * T::kRowBytes + sizeof(NewRow) * ln) =
            reinterpret_cast<const NewRow *>(new_tok + T::kRowBytes)[ln];
    };
    auto write_new = [&]() {
        if (new_row < 0)
            return;
        if constexpr (kBf16Cache) {
            *reinterpret_cast<uint2 *>(static_cast<uint8_t *>(a.k_cache) + new_row * 256 + 8 * lane) = new_k;
            *reinterpret_cast<uint2 *>(static_cast<uint8_t *>(a.v_cache) + new_row * 256 + 8 * lane) = new_v;
        } else {
            *reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(a.k_cache) + new_row * 128 + 4 * lane) = new_k;
            *reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(a.v_cache) + new_row * 128 + 4 * lane) = new_v;
        }
    };
    if (!step_check)                                       // kvq_decode_step: finish_step writes it
        write_new();

    if (bad) {                                             // for kvq_decode_step a failed check
        if constexpr (kCluster) {
            cluster_finish(a, R, step_check ? kPartialStale : kPartialInvalid, part, finisher);
            if (split == finisher)                         // this split failed: so did the request
                finish_here(true);
        } else
            drop_split(a, R, split, nsplit, reinterpret_cast<float *>(smem),
                       step_check ? kLseStale : kLseInvalid);
        return;
    }

    // ---------------------------------------------------------------- setup
    const int n_chunks = static_cast<int>((t1 - t0 + kChunkTokens - 1) / kChunkTokens);
    const int my_chunks = n_chunks > warp ? (n_chunks - warp + kWarps - 1) / kWarps : 0;
    uint8_t *ring = smem + warp * T::kStages * T::kStageBytes;
    uint64_t *my_full = full + warp * T::kStages;
    const int box_tok = ps < kChunkTokens ? ps : kChunkTokens;
    const int parts = kChunkTokens / box_tok;                       // 1 or 2 copies per tensor
    const uint32_t part_bytes = static_cast<uint32_t>(box_tok * T::kRowBytes);
    // evict-first unless other row blocks of the split read the same pages
    const uint64_t policy = kMulti && a.row_blocks > 1 ? l2_policy_evict_normal() : l2_policy_evict_first();


    // Issue the copies of this warp's local chunk `it`: the whole warp, one
    // copy per lane (lanes 0 .. np - 1 the K parts, np .. 2 np - 1 the V
    // parts), which issues them about twice as fast as one lane in turn.
    auto issue = [&](int it) {
        const int c = warp + it * kWarps;
        const int64_t tok = t0 + static_cast<int64_t>(c) * kChunkTokens;
        const int st = it % T::kStages;
        const int64_t left = t1 - tok;
        const int np = left >= kChunkTokens ? parts : static_cast<int>((left + box_tok - 1) / box_tok);
        if (lane == 0)
            mbar_arrive_expect_tx(&my_full[st], 2u * part_bytes * np);
        __syncwarp();
        if (lane < 2 * np) {
            const int part = lane < np ? lane : lane - np;
            const int64_t ptok = tok + part * box_tok;
            const int32_t page = page_list[static_cast<int>(ptok >> ps_shift) - first_page];
            const int64_t row = (static_cast<int64_t>(page) * a.num_kv_heads + kvh) * ps + (ptok & (ps - 1));
            uint8_t *dst = ring + st * T::kStageBytes + (lane < np ? 0 : T::kBytes) + part * part_bytes;
            tma_load_2d(dst, lane < np ? static_cast<const void *>(&k_map) : static_cast<const void *>(&v_map), 0,
                        static_cast<int32_t>(row * lines_per_tok), &my_full[st], policy);
        }
    };

    const int pro = my_chunks < T::kStages ? my_chunks : T::kStages;
    for (int it = 0; it < pro; ++it)
        issue(it);

    if (step_check) {
        // kvq_decode_step: this split's share of the tag check, its own pages
        // (whose ids are in range here).  The live and expected tags come in
        // by asynchronous copies behind the first bulk copies and are compared
        // once the split has attended: a failure only changes what it
        // publishes.  Thread t copies (and later compares) entries t, t + 128, ...
        const uint32_t *want = a.expected_tags + static_cast<int64_t>(b) * a.max_pages_per_seq + first_page;
#pragma unroll
        for (int k = 0; k < kIdsPerThread; ++k) {
            const int i = threadIdx.x + k * kThreads;
            if (i < n_pages) {
                cp_async_4(tag_live + i, a.page_tags + page_list[i]);
                cp_async_4(tag_want + i, want + i);
            }
        }
        cp_async_commit();
    }

    // Query fragments (mma B operand): lane (gq, tq) holds query row gq of
    // this CTA (with one query token: head gq of the group) at dims 32*tq ..
    // 32*tq+31; k-slot pairs of k-step c map to dims 32*tq + 4*c + {0,1} and
    // {2,3}.
    //
    // FP8 cache: the product runs in f16, whose range is narrower than
    // bf16's.  Each q row is first multiplied by 2^e_h, the power of two that
    // puts its largest magnitude in [2^14, 2^15) (exact: only the exponent
    // changes), so no element overflows and every element within 2^28 of the
    // row's largest keeps all its bits; the score multiplier of head h then
    // carries 2^-e_h.
    constexpr int kNT = rows_per_cta(kMulti) / kMaxGroup;   // mma n-tiles of query rows per warp
    constexpr int kRowsT = rows_per_cta(kMulti);
    uint32_t qf[kNT][8][2];
    int q_exp[kNT];                                        // e of row nt * 8 + gq
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt) {
        q_exp[nt] = 0;
        uint32_t w[16];
        if (nt * kMaxGroup + gq < R.nrows) {
            const uint4 *src = reinterpret_cast<const uint4 *>(
                static_cast<const uint16_t *>(a.q) + (R.id(a, nt * kMaxGroup + gq) * kHeadDim + 32 * tq));
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint4 v = __ldg(src + i);
                w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
            }
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i)
                w[i] = 0;
        }
        float q_mul = 1.f;
        if constexpr (!kBf16Cache) {
            uint32_t mx = 0;                               // largest |q| of the row, as bf16 bits
#pragma unroll
            for (int i = 0; i < 16; ++i)
                mx = max(mx, max(w[i] & 0x7FFFu, (w[i] >> 16) & 0x7FFFu));
            mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
            mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
            q_exp[nt] = row_pow2_exponent(mx);
            q_mul = __int_as_float((127 + q_exp[nt]) << 23);
        }
#pragma unroll
        for (int c = 0; c < 8; ++c) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                if constexpr (kBf16Cache) {
                    qf[nt][c][j] = w[2 * c + j];
                } else {
                    const float2 f = bf16x2_to_f32x2(w[2 * c + j]);
                    qf[nt][c][j] = f32x2_to_f16x2(f.x * q_mul, f.y * q_mul);
                }
            }
        }
    }

    const float kscale = kBf16Cache ? 1.f : a.k_scale[kvh];
    const float vscale = kBf16Cache ? 1.f : a.v_scale[kvh];
    // score multiplier (log2 domain) of the two query heads 2tq, 2tq + 1
    // whose scores this lane holds: the softmax scale, the K scale and the
    // undoing of their q rows' power-of-two scaling
    float qk_col[kNT][2];
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int e = __shfl_sync(0xFFFFFFFFu, q_exp[nt], 4 * (2 * tq + j));
            qk_col[nt][j] = a.qk_scale_log2 * kscale * __int_as_float((127 - e) << 23);
        }
    // Causal limit of those two rows: query token i sees the positions below
    // len - n_query + 1 + i (with one query token: all of them), kept as a
    // count from the split's start, at most one chunk past its end.  Below
    // full_end every row of the CTA sees every token.
    [[maybe_unused]] int vis_col[kNT][2] = {};
    int64_t full_end = t1;
    if constexpr (kMulti) {
        const int64_t vis0 = len - a.n_query + 1;
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int64_t v = vis0 + (R.row0 + nt * kMaxGroup + 2 * tq + j) / g - t0;
                vis_col[nt][j] = static_cast<int>(
                    v < -1 ? -1 : (v > a.split_tokens + kChunkTokens ? a.split_tokens + kChunkTokens : v));
            }
        full_end = min(t1, vis0 + R.row0 / g);
    }

    float m_run[kNT][2], l_run[kNT][2];
    float o[kNT][8][4];
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt) {
        m_run[nt][0] = m_run[nt][1] = -INFINITY;
        l_run[nt][0] = l_run[nt][1] = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i)
            o[nt][i][0] = o[nt][i][1] = o[nt][i][2] = o[nt][i][3] = 0.f;
    }

    bool failed = false;
    int it = 0;
    for (; it < my_chunks; ++it) {
        const int st = it % T::kStages;
        // every lane polls; the warp gives up as one if any lane did
        if (!__all_sync(0xFFFFFFFFu, mbar_wait_bounded(&my_full[st], (it / T::kStages) & 1, a.copy_wait_ns))) {
            failed = true;
            break;
        }
        if (it == 0 && warp == 0)
            KVQ_STAMP(2);
        const uint8_t *ks = ring + st * T::kStageBytes;
        const uint8_t *vs = ks + T::kBytes;
        const int c = warp + it * kWarps;
        const int64_t tok = t0 + static_cast<int64_t>(c) * kChunkTokens;
        if (it == it_new) {                  // fused append: the new token's row
            const int r = static_cast<int>(len - 1 - tok);
            uint8_t *kt = ring + st * T::kStageBytes;
            uint8_t *vt = kt + T::kBytes;
            if constexpr (kBf16Cache) {
                const uint32_t off = swz(2 * r + (lane >> 4), (lane & 15) >> 1) + 8 * (lane & 1);
                *reinterpret_cast<uint2 *>(kt + off) = new_k;
                *reinterpret_cast<uint2 *>(vt + off) = new_v;
            } else {
                const uint32_t off = swz(r, lane >> 2) + 4 * (lane & 3);
                *reinterpret_cast<uint32_t *>(kt + off) = new_k;
                *reinterpret_cast<uint32_t *>(vt + off) = new_v;
            }
            __syncwarp();
        }
        const int64_t left = t1 - tok;
        const int n_valid = left < kChunkTokens ? static_cast<int>(left) : kChunkTokens;   // V rows
        int s_valid[kNT][2];                             // tokens of the chunk each score column sees
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
            for (int j = 0; j < 2; ++j)
                s_valid[nt][j] = kMulti ? min(n_valid, vis_col[nt][j] - c * kChunkTokens) : n_valid;

        // The chunk's arithmetic; a full chunk (every token valid, the
        // common case) is compiled without the masking of tail tokens.
        auto chunk = [&](auto full) {
            constexpr bool kFull = decltype(full)::value;
            // ---- S^T = K Q^T for the two 16-token m-tiles; each K fragment,
            // converted once, feeds every n-tile of query rows
            float sc[kNT][2][4];
    #pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
    #pragma unroll
                for (int nt = 0; nt < kNT; ++nt)
                    sc[nt][mt][0] = sc[nt][mt][1] = sc[nt][mt][2] = sc[nt][mt][3] = 0.f;
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
    #pragma unroll
                        for (int nt = 0; nt < kNT; ++nt)
                            mma_bf16(sc[nt][mt], w0[2 * kk], w1[2 * kk], w0[2 * kk + 1], w1[2 * kk + 1],
                                     qf[nt][kk][0], qf[nt][kk][1]);
                } else {
                    const uint4 x0a = lds128(ks, swz(r0, 2 * tq)), x0b = lds128(ks, swz(r0, 2 * tq + 1));
                    const uint4 x1a = lds128(ks, swz(r1, 2 * tq)), x1b = lds128(ks, swz(r1, 2 * tq + 1));
                    const uint32_t w0[8] = {x0a.x, x0a.y, x0a.z, x0a.w, x0b.x, x0b.y, x0b.z, x0b.w};
                    const uint32_t w1[8] = {x1a.x, x1a.y, x1a.z, x1a.w, x1b.x, x1b.y, x1b.z, x1b.w};
    #pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t k0 = lo16_e4m3x2_to_f16x2(w0[kk]), k1 = lo16_e4m3x2_to_f16x2(w1[kk]);
                        const uint32_t k2 = hi16_e4m3x2_to_f16x2(w0[kk]), k3 = hi16_e4m3x2_to_f16x2(w1[kk]);
    #pragma unroll
                        for (int nt = 0; nt < kNT; ++nt)
                            mma_f16(sc[nt][mt], k0, k1, k2, k3, qf[nt][kk][0], qf[nt][kk][1]);
                    }
                }
            }

            // ---- online softmax (log2 domain); lane holds rows nt*8 + 2tq, +1
            float alpha[kNT][2];
    #pragma unroll
            for (int nt = 0; nt < kNT; ++nt) {
                float mx[2] = {-INFINITY, -INFINITY};
    #pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
    #pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int row = mt * 16 + gq + ((i & 2) ? 8 : 0);
                        float x = sc[nt][mt][i] * qk_col[nt][i & 1];
                        x = (kFull || row < s_valid[nt][i & 1]) ? x : -INFINITY;
                        sc[nt][mt][i] = x;
                        mx[i & 1] = fmaxf(mx[i & 1], x);
                    }
                }
                float base[2];
    #pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const float mnew = fmaxf(m_run[nt][j], warp_max_over_rows(mx[j]));
                    base[j] = mnew == -INFINITY ? 0.f : mnew;
                    alpha[nt][j] = fast_exp2(m_run[nt][j] - base[j]);
                    m_run[nt][j] = mnew;
                }
                float psum[2] = {0.f, 0.f};
    #pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
    #pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float p = fast_exp2(sc[nt][mt][i] - base[i & 1]);
                        sc[nt][mt][i] = p;
                        psum[i & 1] += p;
                    }
                }
    #pragma unroll
                for (int j = 0; j < 2; ++j)
                    l_run[nt][j] = l_run[nt][j] * alpha[nt][j] + psum[j];
    #pragma unroll
                for (int i = 0; i < 8; ++i) {
                    o[nt][i][0] *= alpha[nt][0];
                    o[nt][i][1] *= alpha[nt][1];
                    o[nt][i][2] *= alpha[nt][0];
                    o[nt][i][3] *= alpha[nt][1];
                }
            }

            // ---- O^T += V^T P^T; each V fragment, converted once, feeds
            // every n-tile
    #pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
                uint32_t pb0[kNT], pb1[kNT];
                [[maybe_unused]] uint32_t pl0[kNT], pl1[kNT];
    #pragma unroll
                for (int nt = 0; nt < kNT; ++nt) {
                    uint32_t x0, x1;
                    if constexpr (kBf16Cache) {
                        x0 = f32x2_to_bf16x2(sc[nt][mt][0], sc[nt][mt][1]);
                        x1 = f32x2_to_bf16x2(sc[nt][mt][2], sc[nt][mt][3]);
                    } else {
                        x0 = f32x2_to_f16x2(sc[nt][mt][0], sc[nt][mt][1]);
                        x1 = f32x2_to_f16x2(sc[nt][mt][2], sc[nt][mt][3]);
                    }
                    pb0[nt] = movmatrix_trans(x0);
                    pb1[nt] = movmatrix_trans(x1);
                    if constexpr (kPreciseP) {
                        // second term carries what the 16-bit rounding of P dropped
                        const float2 h0 = kBf16Cache ? bf16x2_to_f32x2(x0) : f16x2_to_f32x2(x0);
                        const float2 h1 = kBf16Cache ? bf16x2_to_f32x2(x1) : f16x2_to_f32x2(x1);
                        const float *p = sc[nt][mt];
                        const uint32_t y0 = kBf16Cache ? f32x2_to_bf16x2(p[0] - h0.x, p[1] - h0.y)
                                                       : f32x2_to_f16x2(p[0] - h0.x, p[1] - h0.y);
                        const uint32_t y1 = kBf16Cache ? f32x2_to_bf16x2(p[2] - h1.x, p[3] - h1.y)
                                                       : f32x2_to_f16x2(p[2] - h1.x, p[3] - h1.y);
                        pl0[nt] = movmatrix_trans(y0);
                        pl1[nt] = movmatrix_trans(y1);
                    }
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
                        const bool keep = kFull || rows[q] < n_valid;
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
    #pragma unroll
                        for (int nt = 0; nt < kNT; ++nt) {
                            mma_bf16(o[nt][i], a0, a1, a2, a3, pb0[nt], pb1[nt]);
                            if constexpr (kPreciseP)
                                mma_bf16(o[nt][i], a0, a1, a2, a3, pl0[nt], pl1[nt]);
                        }
                    }
                } else {
                    uint32_t R[4][4];
    #pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint4 v = lds128(vs, swz(rows[q], gq));
                        const bool keep = kFull || rows[q] < n_valid;
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
    #pragma unroll
                        for (int nt = 0; nt < kNT; ++nt) {
                            mma_f16(o[nt][i], a0, a1, a2, a3, pb0[nt], pb1[nt]);
                            if constexpr (kPreciseP)
                                mma_f16(o[nt][i], a0, a1, a2, a3, pl0[nt], pl1[nt]);
                        }
                    }
                }
            }
        };
        if (tok + kChunkTokens <= full_end)
            chunk(std::true_type{});
        else
            chunk(std::false_type{});

        // ---- refill this stage with the chunk kStages ahead
        __syncwarp();
        if (it + T::kStages < my_chunks) {
            fence_proxy_async_smem();
            issue(it + T::kStages);
        }
    }

    if (failed) {
        // Drain the copies this warp still has in flight -- the one it gave
        // up on and those issued after it -- with the full limit, so none
        // lands in shared memory after the CTA has moved on.  A drain that
        // gives up too is reported as bit 1.
        if (lane == 0) {
            atomicOr(&g_device_error, 1u);
            s_failed = 1;
        }
        const int issued = my_chunks < it + T::kStages ? my_chunks : it + T::kStages;
        bool drained = true;
        for (int j = it; j < issued; ++j)
            drained &= mbar_wait_bounded(&my_full[j % T::kStages], (j / T::kStages) & 1, kCopyWaitLimitNs);
        if (!drained && lane == 0)
            atomicOr(&g_device_error, 2u);
    }
    if (step_check) {                                      // this thread's tag entries
        cp_async_wait_all();
        bool stale = false;
#pragma unroll
        for (int k = 0; k < kIdsPerThread; ++k) {
            const int i = threadIdx.x + k * kThreads;
            if (i < n_pages)
                stale |= tag_live[i] != tag_want[i];
        }
        if (stale)
            s_stale = 1;
    }
    __syncthreads();
    KVQ_STAMP(3);
    if (s_stale || s_failed) {                             // a failed check outranks a timeout
        if constexpr (kCluster) {
            const bool stale = cluster_finish(a, R, s_stale ? kPartialStale : kPartialInvalid, part, finisher);
            if (split == finisher)
                finish_here(stale);
        } else
            drop_split(a, R, split, nsplit, reinterpret_cast<float *>(smem),
                       s_stale ? kLseStale : kLseInvalid);
        return;
    }

    // ---- merge the four warps' states in shared memory (ring is free now)
    float *sm_o = reinterpret_cast<float *>(smem);                     // [kWarps][kRowsT][128]
    float *sm_m = sm_o + kWarps * kRowsT * kMergeStride;              // [kWarps][kRowsT]
    float *sm_l = sm_m + kWarps * kRowsT;                             // [kWarps][kRowsT]
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j)
            l_run[nt][j] = warp_sum_over_rows(l_run[nt][j]);
    {
        float *ow = sm_o + warp * kRowsT * kMergeStride;
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt) {
            const int r = nt * kMaxGroup + 2 * tq;                  // rows r, r + 1 of this lane
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int c = merge_col(16 * gq + 2 * i);
                *reinterpret_cast<float2 *>(ow + r * kMergeStride + c) = make_float2(o[nt][i][0], o[nt][i][2]);
                *reinterpret_cast<float2 *>(ow + (r + 1) * kMergeStride + c) =
                    make_float2(o[nt][i][1], o[nt][i][3]);
            }
            if (gq == 0) {
                sm_m[warp * kRowsT + r] = m_run[nt][0];
                sm_m[warp * kRowsT + r + 1] = m_run[nt][1];
                sm_l[warp * kRowsT + r] = l_run[nt][0];
                sm_l[warp * kRowsT + r + 1] = l_run[nt][1];
            }
        }
    }
    __syncthreads();

    // per-row merge factors of the four warps, computed once (thread h)
    float *sm_f = sm_l + kWarps * kRowsT;                             // [kRowsT][kWarps] weights
    float *sm_t = sm_f + kRowsT * kWarps;                             // [kRowsT] 1 / sum, [kRowsT] lse
    if (threadIdx.x < R.nrows) {
        const int h = threadIdx.x;
        float mmax = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w)
            mmax = fmaxf(mmax, sm_m[w * kRowsT + h]);
        float lsum = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float mw = sm_m[w * kRowsT + h];
            const float f = mw == -INFINITY ? 0.f : fast_exp2(mw - mmax);
            sm_f[h * kWarps + w] = f;
            lsum += sm_l[w * kRowsT + h] * f;
        }
        // a row that saw no token of this split (causal limit): weight 0
        sm_t[h] = lsum > 0.f ? vscale / lsum : 0.f;
        sm_t[kRowsT + h] = lsum > 0.f ? mmax + __log2f(lsum) : -INFINITY;
    }
    __syncthreads();
    for (int d = threadIdx.x; d < kHeadDim; d += kThreads)
#pragma unroll
    for (int h = 0; h < kRowsT; ++h) {
        if (h >= R.nrows)
            break;
        float acc = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w)
            acc += sm_o[(w * kRowsT + h) * kMergeStride + merge_col(d)] * sm_f[h * kWarps + w];
        const float val = acc * sm_t[h];
        const int64_t bh = R.id(a, h);
        if constexpr (kCluster) {
            part[kRowsT + h * kHeadDim + d] = val;
            if (d == 0)
                part[h] = sm_t[kRowsT + h];
        } else if (nsplit == 1) {
            store_out(a.out, bh * kHeadDim + d, val, a.out_fp32);
        } else {
            a.ws_o[(bh * a.max_splits + split) * kHeadDim + d] = val;
            if (d == 0)
                a.ws_lse[bh * a.max_splits + split] = sm_t[kRowsT + h];
        }
    }
    KVQ_STAMP(4);
    if constexpr (kCluster) {
        const bool stale = cluster_finish(a, R, kPartialOk, part, finisher);
        if (split == finisher)
            finish_here(stale);
    } else if (nsplit > 1) {
        publish_and_combine(a, R, nsplit, reinterpret_cast<float *>(smem) + (kMulti ? 0 : kScratchOffset));
    } else if (step_check) {                               // one split: its own verdict
        finish_here(false);
    }
    KVQ_STAMP(6);
}

template <bool kBf16, bool kPrecise, bool kCluster, bool kMulti = false>
cudaError_t configure(int dev)
{
    static int configured[64] = {0};
    if (dev >= 0 && dev < 64 && configured[dev])
        return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(decode_split_kernel<kBf16, kPrecise, kCluster, kMulti>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Tile<kBf16>::kSmemBytes);
    if (e == cudaSuccess && dev >= 0 && dev < 64)
        configured[dev] = 1;
    return e;
}

template <bool kBf16, bool kPrecise, bool kCluster>
cudaLaunchConfig_t launch_config(const DecodeArgs &a, dim3 grid, cudaStream_t stream,
                                 cudaLaunchAttribute (&attr)[2])
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = Tile<kBf16>::kSmemBytes;
    cfg.stream = stream;
    // programmatic dependent launch: the grid may start while the previous
    // kernel on the stream finishes; the kernel waits before its first read
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.numAttrs = 1;
    if (kCluster) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = static_cast<unsigned>(a.max_splits);
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
    }
    cfg.attrs = attr;
    return cfg;
}

template <bool kBf16, bool kPrecise, bool kCluster, bool kMulti>
cudaError_t launch_split(const DecodeArgs &a, const CUtensorMap &k_map, const CUtensorMap &v_map,
                         cudaStream_t stream)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    e = configure<kBf16, kPrecise, kCluster, kMulti>(dev);
    if (e != cudaSuccess)
        return e;
    const dim3 grid(static_cast<unsigned>(a.max_splits),
                    static_cast<unsigned>(a.num_kv_heads * a.row_blocks), static_cast<unsigned>(a.batch));
    cudaLaunchAttribute attr[2];
    const cudaLaunchConfig_t cfg = launch_config<kBf16, kPrecise, kCluster>(a, grid, stream, attr);
    e = cudaLaunchKernelEx(&cfg, decode_split_kernel<kBf16, kPrecise, kCluster, kMulti>, k_map, v_map, a);
    if (e != cudaSuccess)
        return e;
    return cudaGetLastError();
}

template <bool kCluster, bool kMulti>
cudaError_t launch_variant(const DecodeArgs &a, const CUtensorMap &k_map, const CUtensorMap &v_map,
                           cudaStream_t stream)
{
    if (a.bf16_cache)
        return a.out_fp32 ? launch_split<true, true, kCluster, kMulti>(a, k_map, v_map, stream)
                          : launch_split<true, false, kCluster, kMulti>(a, k_map, v_map, stream);
    return a.out_fp32 ? launch_split<false, true, kCluster, kMulti>(a, k_map, v_map, stream)
                      : launch_split<false, false, kCluster, kMulti>(a, k_map, v_map, stream);
}

template <bool kBf16, bool kMulti>
int cluster_capacity_query(int n)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || configure<kBf16, false, true, kMulti>(dev) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    DecodeArgs a = {};
    a.max_splits = n;
    cudaLaunchAttribute attr[2];
    const cudaLaunchConfig_t cfg =
        launch_config<kBf16, false, true>(a, dim3(static_cast<unsigned>(n), 1, 1), nullptr, attr);
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, decode_split_kernel<kBf16, false, true, kMulti>, &cfg) !=
        cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return clusters;
}

} // namespace

cudaError_t launch_decode(const DecodeArgs &a, const CUtensorMap &k_map, const CUtensorMap &v_map,
                          cudaStream_t stream)
{
    if (a.batch == 0)
        return cudaSuccess;

    if (a.n_query > 1)                      // several query tokens: the causal, row-blocked build
        return a.cluster ? launch_variant<true, true>(a, k_map, v_map, stream)
                         : launch_variant<false, true>(a, k_map, v_map, stream);
    return a.cluster ? launch_variant<true, false>(a, k_map, v_map, stream)
                     : launch_variant<false, false>(a, k_map, v_map, stream);
}

int decode_cluster_capacity(int n, bool bf16_cache, bool multi)
{
    if (n < 2 || n > kMaxCluster)
        return 0;
    static std::mutex mu;
    static std::map<std::tuple<int, int, bool, bool>, int> cache;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    std::lock_guard<std::mutex> lock(mu);
    const auto key = std::make_tuple(dev, n, bf16_cache, multi);
    auto it = cache.find(key);
    if (it != cache.end())
        return it->second;
    const int c = multi ? (bf16_cache ? cluster_capacity_query<true, true>(n) : cluster_capacity_query<false, true>(n))
                        : (bf16_cache ? cluster_capacity_query<true, false>(n)
                                      : cluster_capacity_query<false, false>(n));
    cache[key] = c;
    return c;
}

int decode_ctas_per_sm(bool bf16_cache, bool multi)
{
    // resident CTAs per SM as the shared-memory footprint and the launch
    // bounds allow (no device)
    const int by_smem = bf16_cache ? 233472 / (Tile<true>::kSmemBytes + 1024)
                                   : 233472 / (Tile<false>::kSmemBytes + 1024);
    const int bound = multi ? 2 : kCtasPerSm;
    const int fallback = by_smem < bound ? (by_smem > 0 ? by_smem : 1) : bound;
    static std::mutex mu;
    static std::map<std::tuple<int, bool, bool>, int> cache;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return fallback;
    }
    std::lock_guard<std::mutex> lock(mu);
    const auto key = std::make_tuple(dev, bf16_cache, multi);
    auto it = cache.find(key);
    if (it != cache.end())
        return it->second;
    int n = 0;
    cudaError_t e = cudaSuccess;
    if (multi) {
        e = bf16_cache ? configure<true, false, false, true>(dev) : configure<false, false, false, true>(dev);
        if (e == cudaSuccess)
            e = bf16_cache ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                                 &n, decode_split_kernel<true, false, false, true>, kThreads, Tile<true>::kSmemBytes)
                           : cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                                 &n, decode_split_kernel<false, false, false, true>, kThreads, Tile<false>::kSmemBytes);
    } else {
        e = bf16_cache ? configure<true, false, false>(dev) : configure<false, false, false>(dev);
        if (e == cudaSuccess)
            e = bf16_cache ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                                 &n, decode_split_kernel<true, false, false, false>, kThreads, Tile<true>::kSmemBytes)
                           : cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                                 &n, decode_split_kernel<false, false, false, false>, kThreads, Tile<false>::kSmemBytes);
    }
    if (e != cudaSuccess || n <= 0) {
        cudaGetLastError();
        n = fallback;
    }
    cache[key] = n;
    return n;
}

#ifdef KVQ_PHASE_STAMPS
cudaError_t read_decode_stamps(unsigned long long *host, size_t count)
{
    const size_t n = count < static_cast<size_t>(kStampCtas * kStampPoints) ? count
                                                                            : kStampCtas * kStampPoints;
    return cudaMemcpyFromSymbol(host, g_phase_stamps, n * sizeof(unsigned long long));
}
#endif

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
