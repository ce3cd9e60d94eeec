// kvq_abi.cu -- the extern "C" boundary declared in include/kvq.h: host-side
// argument checks, split planning, tensor-map encoding and kernel launches.
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>

#include "../../include/kvq.h"
#include "kvq_internal.h"

namespace kvq {

int device_sm_count()
{
    constexpr int kHostFallbackSms = 152;
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();                     // leave no error for a later launch check
        return kHostFallbackSms;
    }
    if (dev >= 0 && dev < 64) {
        const int c = cache[dev].load(std::memory_order_relaxed);
        if (c > 0)
            return c;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        n = kHostFallbackSms;
    }
    if (dev >= 0 && dev < 64)
        cache[dev].store(n, std::memory_order_relaxed);
    return n;
}

namespace {
std::atomic<uint64_t> g_copy_wait_ns{kCopyWaitLimitNs};
} // namespace

uint64_t decode_copy_wait_ns() { return g_copy_wait_ns.load(std::memory_order_relaxed); }

} // namespace kvq

namespace {

using kvq::kChunkTokens;
using kvq::kHeadDim;

constexpr int kMaxSplitTokens = 8192;
constexpr int kMinAutoSplitTokens = 128;   // one 32-token chunk per warp

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

kvq_status check_desc(const kvq_cache_desc *d)
{
    if (d == nullptr)
        return KVQ_ERR_INVALID_ARG;
    if (d->num_pages <= 0 || d->page_size <= 0 || d->num_kv_heads <= 0 || d->head_dim <= 0)
        return KVQ_ERR_INVALID_ARG;
    if (d->cache_dtype != KVQ_CACHE_FP8_E4M3 && d->cache_dtype != KVQ_CACHE_BF16)
        return KVQ_ERR_INVALID_ARG;
    if (d->head_dim != kHeadDim)
        return KVQ_ERR_UNSUPPORTED;
    if (d->page_size != 16 && d->page_size != 32 && d->page_size != 64 && d->page_size != 128)
        return KVQ_ERR_UNSUPPORTED;
    // tensor-copy row coordinates are 32-bit: rows of 128 bytes in one cache
    const int64_t lines = static_cast<int64_t>(d->num_pages) * d->num_kv_heads * d->page_size *
                          (d->cache_dtype == KVQ_CACHE_BF16 ? 2 : 1);
    if (lines > 0x7FFFFFFFLL)
        return KVQ_ERR_UNSUPPORTED;
    return KVQ_OK;
}

struct Plan {
    int32_t split_tokens, max_splits, row_blocks;
    int32_t cluster;              // 0, or the cluster size (= max_splits) of the cluster combine
    size_t counter_bytes, lse_bytes, o_bytes;
};

// Automatic split count per (request, KV head).  Large jobs use the largest
// split (8,192 tokens): there are many waves of CTAs anyway.  Small jobs pick
// the count whose CTAs best fill whole waves of the resident CTA slots (SMs x
// CTAs per SM), preferring fewer waves, with splits of at least 128 tokens
// (one 32-token chunk per warp: a short job finishes sooner in more, shorter
// splits).
int64_t auto_splits(int64_t pairs, int64_t max_ctx, int64_t slots)
{
    // Long jobs: splits of up to 8,192 tokens.  The plan knows only the
    // longest context; when that gives between 4 and 8 waves, requests
    // shorter than it (a mixed batch) leave the last waves ragged, and
    // splits half as long fill them better (ragged64: 359 us against 372 us;
    // long4, at 8 waves and more, is 5 % slower with the shorter splits).
    const int64_t big = (max_ctx + kMaxSplitTokens - 1) / kMaxSplitTokens;
    if (pairs * big >= 8 * slots)
        return big;
    if (pairs * big >= 4 * slots)
        return 2 * big;
    int64_t most = max_ctx / kMinAutoSplitTokens;
    if (most < 1)
        most = 1;
    if (most > kvq::kMaxSplitsTotal)
        most = kvq::kMaxSplitsTotal;
    int64_t best = 1;
    double best_score = -1.0;
    for (int64_t n = 1; n <= most; ++n) {
        const int64_t ctas = pairs * n;
        const int64_t waves = (ctas + slots - 1) / slots;
        if (waves > 4)
            break;
        const double fill = static_cast<double>(ctas) / static_cast<double>(waves * slots);
        const double score = fill - 0.1 * static_cast<double>(waves);
        if (score > best_score + 1e-9) {
            best_score = score;
            best = n;
        }
    }
    return best;
}

// Split count for a job that can run in one wave, or 0 if none can.  Among
// the counts whose CTAs are all resident at once -- every (request, KV
// head) as one resident cluster of its splits, or as plain CTAs -- it takes
// the smallest estimate of
//   fixed cost + smooth max(all bytes / HBM rate, one split's bytes / the
//   rate one CTA's copy pipeline sustains) + the combine's tail,
// the constants measured on GB300: a CTA streams about 20 GB/s (FP8; 40 for
// the BF16 tile, whose copies are twice as large), the combine costs about
// 2.5 us through distributed shared memory and 9 us through the workspace.
// (16 requests x 8,193 tokens: 3 splits in clusters, 58.5 us, where the
// multi-wave rule took 7 through the workspace, 79.6 us; 32 x 4,097: one
// split, 62.0 us against 73.5 us.)
int64_t single_wave_splits(int64_t pairs, int64_t max_ctx, int64_t unit, int64_t slots, bool bf16,
                           bool multi)
{
    const double bytes_per_tok = bf16 ? 512.0 : 256.0;       // K + V of one token of one KV head
    const double cta_rate = bf16 ? 40e9 : 20e9;               // bytes per second per CTA
    const double hbm_rate = 6.3e12;
    const double total_us = static_cast<double>(pairs) * static_cast<double>(max_ctx) * bytes_per_tok / hbm_rate * 1e6;
    int64_t most = max_ctx / kMinAutoSplitTokens;
    if (most < 1)
        most = 1;
    if (most > kvq::kMaxSplitsTotal)
        most = kvq::kMaxSplitsTotal;
    int64_t best = 0, last = 0;
    double best_us = 1e30;
    for (int64_t n = 1; n <= most; ++n) {
        int64_t split = (max_ctx + n - 1) / n;
        split = (split + unit - 1) / unit * unit;
        if (split > kMaxSplitTokens)
            continue;
        const int64_t splits = (max_ctx + split - 1) / split;
        if (splits == last)
            continue;                                           // the same plan as a smaller n
        last = splits;
        const bool cluster = splits >= 2 && splits <= kvq::kMaxCluster &&
                             pairs <= kvq::decode_cluster_capacity(static_cast<int>(splits), bf16, multi);
        if (!cluster && pairs * splits > slots)
            continue;                                           // more than one wave
        const double split_us = static_cast<double>(split) * bytes_per_tok / cta_rate * 1e6;
        const double stream_us = std::pow(std::pow(total_us, 4.0) + std::pow(split_us, 4.0), 0.25);
        const double combine_us = splits == 1 ? 0.0 : cluster ? 2.5 : 9.0;
        const double est = 11.0 + stream_us + combine_us;
        if (est < best_us - 1e-9) {
            best_us = est;
            best = splits;
        }
    }
    return best;
}

// The most new query tokens per request a multi-token call takes.
constexpr int kMaxQueryTokens = 16;

kvq_status make_plan(const kvq_cache_desc *d, int32_t batch, int32_t num_q_heads,
                     int32_t max_pages, int32_t num_splits, Plan *p, int32_t n_query = 1)
{
    kvq_status st = check_desc(d);
    if (st != KVQ_OK)
        return st;
    if (batch < 0 || num_q_heads <= 0 || max_pages <= 0 || num_splits < 0 || n_query < 1)
        return KVQ_ERR_INVALID_ARG;
    if (n_query > kMaxQueryTokens)
        return KVQ_ERR_UNSUPPORTED;
    if (batch > 65535)
        return KVQ_ERR_UNSUPPORTED;
    if (num_q_heads % d->num_kv_heads != 0)
        return KVQ_ERR_INVALID_ARG;
    const int g = num_q_heads / d->num_kv_heads;
    if (g > kvq::kMaxGroup)
        return KVQ_ERR_UNSUPPORTED;
    const int64_t max_ctx = static_cast<int64_t>(max_pages) * d->page_size;
    const bool bf16 = d->cache_dtype == KVQ_CACHE_BF16;
    const bool multi = n_query > 1;
    // Many query rows over an FP8 cache: the tensor-memory kernel, one CTA
    // per (split, request, KV head) for all n g rows, splits in whole
    // 64-token tiles, combined through the workspace.
    const bool umma = kvq::use_umma(bf16, n_query, g);
    const int64_t min_unit = umma ? kvq::kUmmaTileTokens : kChunkTokens;
    const int64_t unit = d->page_size > min_unit ? d->page_size : min_unit;
    // CTAs per split: one per (request, KV head), or in the BF16 multi-token
    // build one per (request, KV head, block of 16 query rows)
    const int64_t row_blocks = multi && !umma
                                   ? (static_cast<int64_t>(n_query) * g + kvq::kMultiRowsPerCta - 1) /
                                         kvq::kMultiRowsPerCta
                                   : 1;
    const int64_t pairs = static_cast<int64_t>(batch) * d->num_kv_heads * row_blocks;
    p->row_blocks = static_cast<int32_t>(row_blocks);
    if (static_cast<int64_t>(d->num_kv_heads) * row_blocks > 65535)
        return KVQ_ERR_UNSUPPORTED;                  // the grid's second dimension
    int64_t want;
    bool single_wave = false;
    if (num_splits > 0) {
        want = num_splits;
    } else if (umma) {
        // One wave: as many splits as keep every CTA resident at once, each
        // at least kMinAutoSplitTokens long; a job that needs more than one
        // wave even with the longest splits takes those.
        const int64_t slots = static_cast<int64_t>(kvq::device_sm_count()) * kvq::decode_umma_ctas_per_sm();
        const int64_t jobs = static_cast<int64_t>(batch > 0 ? batch : 1) * d->num_kv_heads;
        const int64_t big = (max_ctx + kMaxSplitTokens - 1) / kMaxSplitTokens;
        if (jobs * big >= slots) {
            want = big;
        } else {
            want = slots / jobs;
            const int64_t most = max_ctx / kMinAutoSplitTokens;
            if (want > most)
                want = most;
            if (want < big)
                want = big;
        }
        single_wave = true;                          // no cluster form
    } else {
        const int64_t slots =
            static_cast<int64_t>(kvq::device_sm_count()) * kvq::decode_ctas_per_sm(bf16, multi);
        const int64_t jobs = static_cast<int64_t>(batch > 0 ? batch : 1) * d->num_kv_heads * row_blocks;
        const int64_t big = (max_ctx + kMaxSplitTokens - 1) / kMaxSplitTokens;
        want = jobs * big < 4 * slots ? single_wave_splits(jobs, max_ctx, unit, slots, bf16, multi) : 0;
        single_wave = want > 0;
        if (!single_wave)
            want = auto_splits(jobs, max_ctx, slots);
    }
    if (want < 1)
        want = 1;
    if (num_splits == 0 && !single_wave && want >= 2 && batch > 0) {
        // A job whose splits could all be resident as clusters merges them
        // through distributed shared memory, a much shorter tail than the
        // workspace combine; that is worth giving up up to half the splits.
        int64_t c = want < kvq::kMaxCluster ? want : kvq::kMaxCluster;
        while (c >= 2 && pairs > kvq::decode_cluster_capacity(static_cast<int>(c), bf16, multi))
            --c;
        if (c >= 2 && 2 * c >= want)
            want = c;
    }
    int64_t split = (max_ctx + want - 1) / want;
    split = (split + unit - 1) / unit * unit;
    if (split > kMaxSplitTokens)
        split = kMaxSplitTokens;
    int64_t splits = (max_ctx + split - 1) / split;
    if (splits > (multi ? kvq::kMultiMaxSplitsPerRequest : kvq::kMaxSplitsTotal))
        return KVQ_ERR_UNSUPPORTED;
    p->split_tokens = static_cast<int32_t>(split);
    p->max_splits = static_cast<int32_t>(splits);
    // When every (request, KV head) fits in one resident cluster of `splits`
    // CTAs, the splits merge through distributed shared memory instead of
    // the workspace.
    p->cluster = 0;
    if (!umma && splits >= 2 && batch > 0 &&
        pairs <= kvq::decode_cluster_capacity(static_cast<int>(splits), bf16, multi))
        p->cluster = static_cast<int32_t>(splits);
    p->counter_bytes = (static_cast<size_t>(pairs) * 4 + 255) / 256 * 256;
    if (p->counter_bytes == 0)
        p->counter_bytes = 256;
    if (splits > 1 && p->cluster == 0) {
        const size_t n = static_cast<size_t>(batch) * n_query * num_q_heads * splits;
        p->lse_bytes = (n * sizeof(float) + 255) / 256 * 256;
        p->o_bytes = n * kHeadDim * sizeof(float);
    } else {
        p->lse_bytes = p->o_bytes = 0;
    }
    return KVQ_OK;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point, so the
// library does not link libcuda directly.
using EncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                              const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                              const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encode_fn()
{
    static EncodeFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeFn>(p);
    });
    return fn;
}

bool make_cache_map(CUtensorMap *map, const kvq_cache_desc *d, const void *cache)
{
    EncodeFn fn = encode_fn();
    if (fn == nullptr)
        return false;
    const bool bf16 = d->cache_dtype == KVQ_CACHE_BF16;
    const cuuint64_t rows = static_cast<cuuint64_t>(d->num_pages) * d->num_kv_heads *
                            d->page_size * (bf16 ? 2 : 1);
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(bf16 ? 64 : 128), rows};
    const cuuint64_t strides[1] = {128};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(bf16 ? 64 : 128),
                               static_cast<cuuint32_t>(kvq::tma_box_rows(d->page_size, bf16))};
    const cuuint32_t estr[2] = {1, 1};
    std::memset(map, 0, sizeof *map);
    const CUresult r = fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8,
                          2, const_cast<void *>(cache), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

kvq_status to_status(cudaError_t e) { return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA; }

struct DecodeCall {
    kvq::DecodeArgs args;
    Plan plan;
};

kvq_status prepare_decode(const kvq_cache_desc *desc, const void *q, int32_t batch,
                          int32_t num_q_heads, const void *k_cache, const void *v_cache,
                          const float *k_scale, const float *v_scale, const int32_t *block_table,
                          int32_t max_pages_per_seq, const int32_t *seq_lens, float softmax_scale,
                          const uint8_t *abort_flags, void *out, int32_t out_dtype,
                          void *workspace, size_t workspace_bytes, int32_t num_splits,
                          DecodeCall *call, int32_t n_query = 1)
{
    kvq_status st = make_plan(desc, batch, num_q_heads, max_pages_per_seq, num_splits, &call->plan,
                              n_query);
    if (st != KVQ_OK)
        return st;
    if (out_dtype != KVQ_OUT_BF16 && out_dtype != KVQ_OUT_FP32)
        return KVQ_ERR_INVALID_ARG;
    if (!std::isfinite(softmax_scale))
        return KVQ_ERR_INVALID_ARG;
    const bool bf16 = desc->cache_dtype == KVQ_CACHE_BF16;
    if (batch > 0) {
        if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !out)
            return KVQ_ERR_INVALID_ARG;
        if (!bf16 && (!k_scale || !v_scale))
            return KVQ_ERR_INVALID_ARG;
        if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
            return KVQ_ERR_INVALID_ARG;
    }
    if (batch > 65535)
        return KVQ_ERR_UNSUPPORTED;
    const size_t need = call->plan.counter_bytes + call->plan.lse_bytes + call->plan.o_bytes;
    if (workspace == nullptr || workspace_bytes < need)
        return KVQ_ERR_WORKSPACE;
    if (!aligned16(workspace))
        return KVQ_ERR_INVALID_ARG;
    kvq::DecodeArgs &a = call->args;
    a = kvq::DecodeArgs{};
    a.q = q;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    a.block_table = block_table;
    a.seq_lens = seq_lens;
    a.abort_flags = abort_flags;
    a.out = out;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    a.counters = reinterpret_cast<unsigned int *>(ws);
    a.ws_lse = call->plan.lse_bytes ? reinterpret_cast<float *>(ws + call->plan.counter_bytes) : nullptr;
    a.ws_o = call->plan.o_bytes
                 ? reinterpret_cast<float *>(ws + call->plan.counter_bytes + call->plan.lse_bytes)
                 : nullptr;
    a.batch = batch;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = desc->num_kv_heads;
    a.group = num_q_heads / desc->num_kv_heads;
    a.page_size = desc->page_size;
    a.num_pages = desc->num_pages;
    a.max_pages_per_seq = max_pages_per_seq;
    a.split_tokens = call->plan.split_tokens;
    a.max_splits = call->plan.max_splits;
    a.cluster = call->plan.cluster;
    a.n_query = n_query;
    a.row_blocks = call->plan.row_blocks;
    a.qk_scale_log2 = softmax_scale * 1.4426950408889634f;
    a.copy_wait_ns = kvq::decode_copy_wait_ns();
    a.out_fp32 = out_dtype == KVQ_OUT_FP32;
    a.bf16_cache = bf16;
    return KVQ_OK;
}

} // namespace

extern "C" {

const char *kvq_status_string(kvq_status s)
{
    switch (s) {
    case KVQ_OK: return "ok";
    case KVQ_ERR_INVALID_ARG: return "invalid argument";
    case KVQ_ERR_UNSUPPORTED: return "unsupported shape";
    case KVQ_ERR_WORKSPACE: return "workspace too small";
    case KVQ_ERR_CUDA: return "CUDA error";
    }
    return "unknown status";
}

kvq_status kvq_append(const kvq_cache_desc *desc, const void *k_new, const void *v_new,
                      const int64_t *slot_mapping, int32_t num_tokens, const float *k_scale,
                      const float *v_scale, const uint8_t *abort_flags, void *k_cache,
                      void *v_cache, kvq_stream_t stream)
{
    kvq_status st = check_desc(desc);
    if (st != KVQ_OK)
        return st;
    if (num_tokens < 0)
        return KVQ_ERR_INVALID_ARG;
    if (num_tokens == 0)
        return KVQ_OK;
    const bool bf16 = desc->cache_dtype == KVQ_CACHE_BF16;
    if (!k_new || !v_new || !slot_mapping || !k_cache || !v_cache)
        return KVQ_ERR_INVALID_ARG;
    if (!bf16 && (!k_scale || !v_scale))
        return KVQ_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache))
        return KVQ_ERR_INVALID_ARG;
    kvq::AppendArgs a;
    a.k_new = k_new;
    a.v_new = v_new;
    a.slot_mapping = slot_mapping;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    a.abort_flags = abort_flags;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.num_tokens = num_tokens;
    a.num_kv_heads = desc->num_kv_heads;
    a.page_size = desc->page_size;
    a.num_slots = static_cast<int64_t>(desc->num_pages) * desc->page_size;
    a.bf16_cache = bf16;
    return to_status(kvq::launch_append(a, reinterpret_cast<cudaStream_t>(stream)));
}

kvq_status kvq_tag_check(const int32_t *block_table, const uint32_t *expected_tags,
                         const int32_t *seq_lens, int32_t batch, int32_t max_pages_per_seq,
                         int32_t page_size, const uint32_t *page_tags, int32_t num_pages,
                         uint8_t *abort_flags, kvq_stream_t stream)
{
    if (batch < 0 || max_pages_per_seq <= 0 || page_size <= 0 || num_pages <= 0)
        return KVQ_ERR_INVALID_ARG;
    if (batch == 0)
        return KVQ_OK;
    if (!block_table || !expected_tags || !seq_lens || !page_tags || !abort_flags)
        return KVQ_ERR_INVALID_ARG;
    kvq::TagCheckArgs a;
    a.block_table = block_table;
    a.expected_tags = expected_tags;
    a.seq_lens = seq_lens;
    a.page_tags = page_tags;
    a.abort_flags = abort_flags;
    a.batch = batch;
    a.max_pages_per_seq = max_pages_per_seq;
    a.page_size = page_size;
    a.num_pages = num_pages;
    return to_status(kvq::launch_tag_check(a, reinterpret_cast<cudaStream_t>(stream)));
}

kvq_status kvq_tag_check_append(const kvq_cache_desc *desc, const int32_t *block_table,
                                const uint32_t *expected_tags, const int32_t *seq_lens,
                                int32_t batch, int32_t max_pages_per_seq,
                                const uint32_t *page_tags, const void *k_new, const void *v_new,
                                const int64_t *slot_mapping, const float *k_scale,
                                const float *v_scale, void *k_cache, void *v_cache,
                                uint8_t *abort_flags, kvq_stream_t stream)
{
    kvq_status st = check_desc(desc);
    if (st != KVQ_OK)
        return st;
    if (batch < 0 || max_pages_per_seq <= 0)
        return KVQ_ERR_INVALID_ARG;
    if (batch == 0)
        return KVQ_OK;
    const bool bf16 = desc->cache_dtype == KVQ_CACHE_BF16;
    if (!block_table || !expected_tags || !seq_lens || !page_tags || !abort_flags || !k_new ||
        !v_new || !slot_mapping || !k_cache || !v_cache)
        return KVQ_ERR_INVALID_ARG;
    if (!bf16 && (!k_scale || !v_scale))
        return KVQ_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache))
        return KVQ_ERR_INVALID_ARG;
    if (desc->num_kv_heads > 64)
        return KVQ_ERR_UNSUPPORTED;
    kvq::TagCheckArgs t;
    t.block_table = block_table;
    t.expected_tags = expected_tags;
    t.seq_lens = seq_lens;
    t.page_tags = page_tags;
    t.abort_flags = abort_flags;
    t.batch = batch;
    t.max_pages_per_seq = max_pages_per_seq;
    t.page_size = desc->page_size;
    t.num_pages = desc->num_pages;
    kvq::AppendArgs a;
    a.k_new = k_new;
    a.v_new = v_new;
    a.slot_mapping = slot_mapping;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    a.abort_flags = nullptr;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.num_tokens = batch;
    a.num_kv_heads = desc->num_kv_heads;
    a.page_size = desc->page_size;
    a.num_slots = static_cast<int64_t>(desc->num_pages) * desc->page_size;
    a.bf16_cache = bf16;
    return to_status(kvq::launch_tag_check_append(t, a, reinterpret_cast<cudaStream_t>(stream)));
}

kvq_status kvq_amax_scales(const kvq_cache_desc *desc, const void *k_cache, const void *v_cache,
                           const int32_t *pages, int32_t num_listed, float *k_scale,
                           float *v_scale, kvq_stream_t stream)
{
    kvq_status st = check_desc(desc);
    if (st != KVQ_OK)
        return st;
    if (desc->cache_dtype != KVQ_CACHE_BF16)
        return KVQ_ERR_INVALID_ARG;
    if (num_listed < 0 || !k_scale || !v_scale || (num_listed > 0 && (!k_cache || !v_cache || !pages)))
        return KVQ_ERR_INVALID_ARG;
    if (num_listed > 0 && (!aligned16(k_cache) || !aligned16(v_cache)))
        return KVQ_ERR_INVALID_ARG;
    kvq::HandoffArgs a = {};
    a.k_src = k_cache;
    a.v_src = v_cache;
    a.src_pages = pages;
    a.k_scale_out = k_scale;
    a.v_scale_out = v_scale;
    a.num_listed = num_listed;
    a.num_kv_heads = desc->num_kv_heads;
    a.page_size = desc->page_size;
    a.src_num_pages = desc->num_pages;
    return to_status(kvq::launch_amax_scales(a, reinterpret_cast<cudaStream_t>(stream)));
}

kvq_status kvq_quantize_pages(const kvq_cache_desc *src_desc, const void *k_src, const void *v_src,
                              const int32_t *src_pages, const kvq_cache_desc *dst_desc, void *k_dst,
                              void *v_dst, const int32_t *dst_pages, int32_t num_listed,
                              const float *k_scale, const float *v_scale, kvq_stream_t stream)
{
    kvq_status st = check_desc(src_desc);
    if (st == KVQ_OK)
        st = check_desc(dst_desc);
    if (st != KVQ_OK)
        return st;
    if (src_desc->cache_dtype != KVQ_CACHE_BF16 || dst_desc->cache_dtype != KVQ_CACHE_FP8_E4M3 ||
        src_desc->page_size != dst_desc->page_size || src_desc->num_kv_heads != dst_desc->num_kv_heads)
        return KVQ_ERR_INVALID_ARG;
    if (num_listed < 0)
        return KVQ_ERR_INVALID_ARG;
    if (num_listed == 0)
        return KVQ_OK;
    if (!k_src || !v_src || !src_pages || !k_dst || !v_dst || !dst_pages || !k_scale || !v_scale)
        return KVQ_ERR_INVALID_ARG;
    if (!aligned16(k_src) || !aligned16(v_src) || !aligned16(k_dst) || !aligned16(v_dst))
        return KVQ_ERR_INVALID_ARG;
    kvq::HandoffArgs a = {};
    a.k_src = k_src;
    a.v_src = v_src;
    a.src_pages = src_pages;
    a.k_dst = k_dst;
    a.v_dst = v_dst;
    a.dst_pages = dst_pages;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    a.num_listed = num_listed;
    a.num_kv_heads = src_desc->num_kv_heads;
    a.page_size = src_desc->page_size;
    a.src_num_pages = src_desc->num_pages;
    a.dst_num_pages = dst_desc->num_pages;
    return to_status(kvq::launch_quantize_pages(a, reinterpret_cast<cudaStream_t>(stream)));
}

kvq_status kvq_decode_plan(const kvq_cache_desc *desc, int32_t batch, int32_t num_q_heads,
                           int32_t max_pages_per_seq, int32_t num_splits, int32_t *split_tokens,
                           int32_t *max_splits, size_t *workspace_bytes)
{
    Plan p;
    kvq_status st = make_plan(desc, batch, num_q_heads, max_pages_per_seq, num_splits, &p);
    if (st != KVQ_OK)
        return st;
    if (split_tokens)
        *split_tokens = p.split_tokens;
    if (max_splits)
        *max_splits = p.max_splits;
    if (workspace_bytes)
        *workspace_bytes = p.counter_bytes + p.lse_bytes + p.o_bytes;
    return KVQ_OK;
}

kvq_status kvq_decode_attn(const kvq_cache_desc *desc, const void *q, int32_t batch,
                           int32_t num_q_heads, const void *k_cache, const void *v_cache,
                           const float *k_scale, const float *v_scale, const int32_t *block_table,
                           int32_t max_pages_per_seq, const int32_t *seq_lens, float softmax_scale,
                           const uint8_t *abort_flags, void *out, int32_t out_dtype,
                           void *workspace, size_t workspace_bytes, int32_t num_splits,
                           kvq_stream_t stream)
{
    DecodeCall call;
    kvq_status st = prepare_decode(desc, q, batch, num_q_heads, k_cache, v_cache, k_scale, v_scale,
                                   block_table, max_pages_per_seq, seq_lens, softmax_scale,
                                   abort_flags, out, out_dtype, workspace, workspace_bytes,
                                   num_splits, &call);
    if (st != KVQ_OK || batch == 0)
        return st;
    CUtensorMap km, vm;
    if (!make_cache_map(&km, desc, k_cache) || !make_cache_map(&vm, desc, v_cache))
        return KVQ_ERR_CUDA;
    return to_status(kvq::launch_decode(call.args, km, vm, reinterpret_cast<cudaStream_t>(stream)));
}

kvq_status kvq_decode_plan_mt(const kvq_cache_desc *desc, int32_t batch, int32_t num_query_tokens,
                              int32_t num_q_heads, int32_t max_pages_per_seq, int32_t num_splits,
                              int32_t *split_tokens, int32_t *max_splits, size_t *workspace_bytes)
{
    Plan p;
    kvq_status st = make_plan(desc, batch, num_q_heads, max_pages_per_seq, num_splits, &p,
                              num_query_tokens);
    if (st != KVQ_OK)
        return st;
    if (split_tokens)
        *split_tokens = p.split_tokens;
    if (max_splits)
        *max_splits = p.max_splits;
    if (workspace_bytes)
        *workspace_bytes = p.counter_bytes + p.lse_bytes + p.o_bytes;
    return KVQ_OK;
}

kvq_status kvq_decode_attn_mt(const kvq_cache_desc *desc, const void *q, int32_t batch,
                              int32_t num_query_tokens, int32_t num_q_heads, const void *k_cache,
                              const void *v_cache, const float *k_scale, const float *v_scale,
                              const int32_t *block_table, int32_t max_pages_per_seq,
                              const int32_t *seq_lens, float softmax_scale,
                              const uint8_t *abort_flags, void *out, int32_t out_dtype,
                              void *workspace, size_t workspace_bytes, int32_t num_splits,
                              kvq_stream_t stream)
{
    DecodeCall call;
    kvq_status st = prepare_decode(desc, q, batch, num_q_heads, k_cache, v_cache, k_scale, v_scale,
                                   block_table, max_pages_per_seq, seq_lens, softmax_scale,
                                   abort_flags, out, out_dtype, workspace, workspace_bytes,
                                   num_splits, &call, num_query_tokens);
    if (st != KVQ_OK || batch == 0)
        return st;
    CUtensorMap km, vm;
    if (!make_cache_map(&km, desc, k_cache) || !make_cache_map(&vm, desc, v_cache))
        return KVQ_ERR_CUDA;
    if (kvq::use_umma(desc->cache_dtype == KVQ_CACHE_BF16, num_query_tokens, call.args.group))
        return to_status(kvq::launch_decode_umma(call.args, km, vm, reinterpret_cast<cudaStream_t>(stream)));
    return to_status(kvq::launch_decode(call.args, km, vm, reinterpret_cast<cudaStream_t>(stream)));
}

kvq_status kvq_decode_attn_append(const kvq_cache_desc *desc, const void *q, int32_t batch,
                                  int32_t num_q_heads, void *k_cache, void *v_cache,
                                  const float *k_scale, const float *v_scale,
                                  const int32_t *block_table, int32_t max_pages_per_seq,
                                  const int32_t *seq_lens, float softmax_scale,
                                  const uint8_t *abort_flags, const void *k_new, const void *v_new,
                                  void *out, int32_t out_dtype, void *workspace,
                                  size_t workspace_bytes, int32_t num_splits, kvq_stream_t stream)
{
    DecodeCall call;
    kvq_status st = prepare_decode(desc, q, batch, num_q_heads, k_cache, v_cache, k_scale, v_scale,
                                   block_table, max_pages_per_seq, seq_lens, softmax_scale,
                                   abort_flags, out, out_dtype, workspace, workspace_bytes,
                                   num_splits, &call);
    if (st != KVQ_OK || batch == 0)
        return st;
    if (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new))
        return KVQ_ERR_INVALID_ARG;
    call.args.k_new = k_new;
    call.args.v_new = v_new;
    call.args.k_cache = k_cache;
    call.args.v_cache = v_cache;
    CUtensorMap km, vm;
    if (!make_cache_map(&km, desc, k_cache) || !make_cache_map(&vm, desc, v_cache))
        return KVQ_ERR_CUDA;
    return to_status(kvq::launch_decode(call.args, km, vm, reinterpret_cast<cudaStream_t>(stream)));
}

kvq_status kvq_decode_step(const kvq_cache_desc *desc, const void *q, int32_t batch, int32_t num_q_heads,
                           void *k_cache, void *v_cache, const float *k_scale, const float *v_scale,
                           const int32_t *block_table, int32_t max_pages_per_seq, const int32_t *seq_lens,
                           const uint32_t *expected_tags, const uint32_t *page_tags, uint8_t *abort_flags,
                           float softmax_scale, const void *k_new, const void *v_new, void *out,
                           int32_t out_dtype, void *workspace, size_t workspace_bytes, int32_t num_splits,
                           kvq_stream_t stream)
{
    DecodeCall call;
    kvq_status st = prepare_decode(desc, q, batch, num_q_heads, k_cache, v_cache, k_scale, v_scale,
                                   block_table, max_pages_per_seq, seq_lens, softmax_scale, nullptr, out,
                                   out_dtype, workspace, workspace_bytes, num_splits, &call);
    if (st != KVQ_OK || batch == 0)
        return st;
    if (!expected_tags || !page_tags || !abort_flags)
        return KVQ_ERR_INVALID_ARG;
    if (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new))
        return KVQ_ERR_INVALID_ARG;
    call.args.k_new = k_new;
    call.args.v_new = v_new;
    call.args.k_cache = k_cache;
    call.args.v_cache = v_cache;
    call.args.expected_tags = expected_tags;
    call.args.page_tags = page_tags;
    call.args.abort_out = abort_flags;
    CUtensorMap km, vm;
    if (!make_cache_map(&km, desc, k_cache) || !make_cache_map(&vm, desc, v_cache))
        return KVQ_ERR_CUDA;
    return to_status(kvq::launch_decode(call.args, km, vm, reinterpret_cast<cudaStream_t>(stream)));
}

kvq_status kvq_diag_set_copy_wait_ns(int64_t ns)
{
    const uint64_t v = ns < 0 || static_cast<uint64_t>(ns) > kvq::kCopyWaitLimitNs
                           ? kvq::kCopyWaitLimitNs
                           : static_cast<uint64_t>(ns);
    kvq::g_copy_wait_ns.store(v, std::memory_order_relaxed);
    return KVQ_OK;
}

#ifdef KVQ_PHASE_STAMPS
// Instrumented build only (no declaration in the public header): copy the
// phase stamps of the last launch to host memory.  which = 0: decode kernel,
// [CTA][8]; 1: tag check + append kernel, [CTA][2]; 2: tag check kernel,
// [CTA][2].
KVQ_API kvq_status kvq_phase_stamps(int32_t which, unsigned long long *host, size_t count)
{
    if (host == nullptr)
        return KVQ_ERR_INVALID_ARG;
    return to_status(which == 0 ? kvq::read_decode_stamps(host, count)
                     : which == 1 ? kvq::read_check_stamps(host, count)
                                  : kvq::read_tag_stamps(host, count));
}
#endif

kvq_status kvq_device_error(uint32_t *bits, int32_t clear)
{
    uint32_t a = 0, b = 0, c = 0;
    cudaError_t e = kvq::read_device_error(&a, clear != 0);
    if (e == cudaSuccess)
        e = kvq::read_w4_error(&b, clear != 0);
    if (e == cudaSuccess)
        e = kvq::read_umma_error(&c, clear != 0);
    if (bits)
        *bits = a | b | c;
    return to_status(e);
}

kvq_status kvq_w4a16_plan(int32_t m, int32_t n, int32_t k, int32_t num_splits, int32_t *splits)
{
    if (m < 0 || n < 0 || k <= 0 || num_splits < 0)
        return KVQ_ERR_INVALID_ARG;
    if (k % kvq::kW4BlockK != 0 || n % kvq::kW4Cols != 0)
        return KVQ_ERR_UNSUPPORTED;
    // K is cut into at most kW4MaxSplits ranges of at most 8,192 k (the scales
    // of one range are staged in shared memory) that are whole 256-k blocks.
    auto usable = [&](int s) { return s >= 1 && s <= kvq::kW4MaxSplits && k % (s * kvq::kW4BlockK) == 0 &&
                                      k / s <= 8192; };
    int dev = 0;
    const bool have_device = cudaGetDevice(&dev) == cudaSuccess;
    if (!have_device)
        cudaGetLastError();
    auto runnable = [&](int s) { return s == 1 || !have_device || kvq::w4a16_cluster_capacity(s) >= 1; };
    int best = 0;
    if (num_splits > 0) {
        if (!usable(num_splits) || !runnable(num_splits))
            return KVQ_ERR_UNSUPPORTED;
        best = num_splits;
    } else {
        // the count whose CTAs best fill whole waves of the resident CTA
        // slots, preferring fewer waves and at least four 256-k blocks per
        // warp (a warp's copies then overlap its arithmetic)
        const int64_t tiles = n / kvq::kW4Cols;
        const int64_t slots = static_cast<int64_t>(kvq::device_sm_count()) * kvq::w4a16_ctas_per_sm();
        double best_score = -1e9;
        for (int s = 1; s <= kvq::kW4MaxSplits; ++s) {
            if (!usable(s) || !runnable(s))
                continue;
            const int64_t ctas = tiles * s;
            const int64_t waves = (ctas + slots - 1) / slots;
            const double fill = waves == 0 ? 0.0
                                           : static_cast<double>(ctas) / static_cast<double>(waves * slots);
            const int64_t blocks_per_warp = k / s / kvq::kW4BlockK / 4;
            const double score = fill - 0.1 * static_cast<double>(waves) - (blocks_per_warp < 4 ? 0.5 : 0.0);
            if (score > best_score + 1e-9) {
                best_score = score;
                best = s;
            }
        }
    }
    if (best == 0)
        return KVQ_ERR_UNSUPPORTED;
    if (splits)
        *splits = best;
    return KVQ_OK;
}

kvq_status kvq_w4a16_gemm(const void *x, const uint8_t *w, const void *scales, int32_t m, int32_t n,
                          int32_t k, void *y, int32_t out_dtype, int32_t num_splits, kvq_stream_t stream)
{
    int32_t splits = 0;
    kvq_status st = kvq_w4a16_plan(m, n, k, num_splits, &splits);
    if (st != KVQ_OK)
        return st;
    if (out_dtype != KVQ_OUT_BF16 && out_dtype != KVQ_OUT_FP32)
        return KVQ_ERR_INVALID_ARG;
    if (m == 0 || n == 0)
        return KVQ_OK;
    if (!x || !w || !scales || !y || !aligned16(x) || !aligned16(w) || !aligned16(y))
        return KVQ_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(scales) & 1u) != 0)
        return KVQ_ERR_INVALID_ARG;
    EncodeFn fn = encode_fn();
    if (fn == nullptr)
        return KVQ_ERR_CUDA;
    CUtensorMap map;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(k / 2), static_cast<cuuint64_t>(n)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(k / 2)};
    const cuuint32_t box[2] = {kvq::kW4CopyK / 2, static_cast<cuuint32_t>(kvq::kW4Cols)};
    const cuuint32_t estr[2] = {1, 1};
    std::memset(&map, 0, sizeof map);
    if (fn(&map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(w), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return KVQ_ERR_CUDA;
    const size_t out_elem = out_dtype == KVQ_OUT_FP32 ? 4 : 2;
    for (int32_t r0 = 0; r0 < m; r0 += 16) {             // 16 rows of x per launch
        kvq::W4Args a = {};
        a.x = static_cast<const uint8_t *>(x) + static_cast<size_t>(r0) * k * 2;
        a.scales = scales;
        a.y = static_cast<uint8_t *>(y) + static_cast<size_t>(r0) * n * out_elem;
        a.rows = m - r0 < 16 ? m - r0 : 16;
        a.n = n;
        a.k = k;
        a.splits = splits;
        a.k_split = k / splits;
        a.out_fp32 = out_dtype == KVQ_OUT_FP32;
        const cudaError_t e = kvq::launch_w4a16(a, map, reinterpret_cast<cudaStream_t>(stream));
        if (e != cudaSuccess)
            return KVQ_ERR_CUDA;
    }
    return KVQ_OK;
}

} // extern "C"
