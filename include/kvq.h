/*
 * kvq.h -- C ABI of the FP8 paged-KV decode path for GB300 (sm_103a).
 *
 * Three operations, each one hand-written CUDA kernel family:
 *
 *   kvq_tag_check    per-page integrity tags: the separate batched check that
 *                    runs before decode reads the cache and aborts a request
 *                    whose pages changed owner.  Source: blog post "Smaller,
 *                    faster, safer: running Kimi and GLM at scale" (page-2
 *                    mirror, section "KV Cache 完整性检查"; page-3 mirror,
 *                    section "一个不能出错的共享缓存").
 *   kvq_append       quantise-on-append: each new token's BF16 K and V
 *                    stored as FP8 e4m3 (or kept as BF16) in its paged slot.
 *                    Source: page-1 mirror, section "量化KV缓存" (the cache
 *                    is stored as FP8 e4m3 instead of BF16, halving its size).
 *   kvq_decode_attn  single-token paged attention over the cache, converting
 *                    FP8 values on read, split across CTAs along the context
 *                    and merged with a log-sum-exp combine.  Source: page-1
 *                    mirror, section "量化KV缓存" (the FP8 attention kernel
 *                    converts the values it reads); page-3 mirror, section
 *                    "FP8 省的不仅是显存".
 *
 * Argument dimensions follow the KV-size formula of the page-4 article
 * (section "显存为什么会成为长上下文推理的瓶颈"): requests x tokens x
 * layers x KV heads x head_dim x {K, V} x bytes per element.  One call
 * handles one layer; a multi-layer model calls once per layer with that
 * layer's caches and scales (page ids and tags are shared by all layers).
 *
 * Common rules
 *   - Every pointer argument is a DEVICE pointer unless stated otherwise and
 *     must be 16-byte aligned.  The caller owns every buffer, including the
 *     decode workspace; the library allocates no device memory.
 *   - Every call is asynchronous on `stream` (NULL = the legacy default
 *     stream).  Argument checks are made on the host before anything is
 *     launched and are returned synchronously; a failed launch returns
 *     KVQ_ERR_CUDA.
 *   - Bad DATA never traps: an out-of-range slot is skipped by append; a page
 *     id outside [0, num_pages) or a request longer than its block-table row
 *     aborts the request in the tag check and makes decode write zeros for
 *     it without reading any page.
 *   - Cache layout (page-major): cache[num_pages][num_kv_heads][page_size]
 *     [head_dim], 1 byte per element (e4m3 codes) or 2 (bf16).  Each
 *     (page, KV head) tile is one contiguous run of page_size * head_dim
 *     elements.  A token at logical position j of request r lives in page
 *     block_table[r][j / page_size], slot j % page_size.
 *   - Supported: head_dim 128; page_size 16, 32, 64 or 128; query heads per
 *     KV head (g = num_q_heads / num_kv_heads) 1 to 8; up to 65535 requests
 *     per decode call.  Others return KVQ_ERR_UNSUPPORTED.
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define KVQ_API __attribute__((visibility("default")))
#else
#define KVQ_API
#endif

struct CUstream_st;
/* The same handle as cudaStream_t / CUstream. */
typedef struct CUstream_st *kvq_stream_t;

typedef enum {
    KVQ_OK = 0,
    KVQ_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misaligned pointer */
    KVQ_ERR_UNSUPPORTED = 2,   /* shape outside the supported set above */
    KVQ_ERR_WORKSPACE = 3,     /* decode workspace smaller than kvq_decode_plan says */
    KVQ_ERR_CUDA = 4           /* a CUDA runtime call or launch failed */
} kvq_status;

typedef enum { KVQ_CACHE_FP8_E4M3 = 0, KVQ_CACHE_BF16 = 1 } kvq_cache_dtype;
typedef enum { KVQ_OUT_BF16 = 0, KVQ_OUT_FP32 = 1 } kvq_out_dtype;

/* Shape of one layer's K cache (the V cache has the same shape). */
typedef struct {
    int32_t num_pages;     /* physical pages N in the pool */
    int32_t page_size;     /* tokens per page */
    int32_t num_kv_heads;  /* Hkv */
    int32_t head_dim;      /* D */
    int32_t cache_dtype;   /* kvq_cache_dtype */
} kvq_cache_desc;

/*
 * kvq_append -- write T new tokens' K and V into their cache slots.
 *
 *   k_new, v_new   bf16 [T][Hkv][D], token-major.
 *   slot_mapping   int64 [T]; token t goes to page slot_mapping[t] / page_size,
 *                  slot slot_mapping[t] % page_size.  A slot < 0 or >= N *
 *                  page_size skips the token (no write, no error).
 *   k_scale, v_scale  fp32 [Hkv], this layer's per-KV-head scales (K and V
 *                  separate).  FP8 cache: code = e4m3(x / scale), the
 *                  division one IEEE fp32 round-to-nearest operation, the
 *                  conversion round-to-nearest-even and saturating at
 *                  +-448 (a NaN input stays NaN).  Ignored (may be NULL) for
 *                  the bf16 cache, which stores x unchanged.
 *   abort_flags    uint8 [T] or NULL: a non-zero flag skips token t (in a
 *                  decode step token t belongs to request t).
 *   k_cache, v_cache  the caches described by *desc; only the addressed
 *                  slots are written.
 * Two tokens mapped to the same slot race; the caller must not do that.
 */
KVQ_API kvq_status kvq_append(const kvq_cache_desc *desc, const void *k_new, const void *v_new,
                      const int64_t *slot_mapping, int32_t num_tokens,
                      const float *k_scale, const float *v_scale,
                      const uint8_t *abort_flags, void *k_cache, void *v_cache,
                      kvq_stream_t stream);

/*
 * kvq_tag_check -- the separate batched integrity pass, run before decode
 * reads the cache.
 *
 *   block_table    int32 [B][max_pages_per_seq], physical page of each of a
 *                  request's logical pages.
 *   expected_tags  uint32 [B][max_pages_per_seq], the tag each request
 *                  recorded for each of its pages when it was given the page.
 *   seq_lens       int32 [B], tokens of each request (entries beyond
 *                  ceil(seq_lens[r] / page_size) are ignored).
 *   page_tags      uint32 [num_pages], the live tag of every physical page
 *                  (the allocator changes it whenever the page is reassigned).
 *   abort_flags    uint8 [B], OUTPUT: 1 if any used entry names a page
 *                  outside [0, num_pages), a page whose live tag differs from
 *                  the expected one, or if the request needs more entries than
 *                  its row has; else 0.  Every flag is written.
 * Pass the flags to kvq_append and kvq_decode_attn of the same step.  A
 * deployment that does not want the check skips this call and passes NULL
 * flags (the no-op tracker of the page-3 article: zero cost).
 */
KVQ_API kvq_status kvq_tag_check(const int32_t *block_table, const uint32_t *expected_tags,
                         const int32_t *seq_lens, int32_t batch, int32_t max_pages_per_seq,
                         int32_t page_size, const uint32_t *page_tags, int32_t num_pages,
                         uint8_t *abort_flags, kvq_stream_t stream);

/*
 * kvq_tag_check_append -- kvq_tag_check followed by kvq_append, fused into
 * one launch for a decode step in which request r appends exactly one new
 * token, token r (the page-3 article's check-before-read, then the page-1
 * article's quantise-on-append).  For every request: the tag check of
 * kvq_tag_check writes abort_flags[r]; then, only if the request passed,
 * token r is written as kvq_append would write it.
 *
 *   desc, k_new, v_new, slot_mapping, k_scale, v_scale, k_cache, v_cache
 *                  as in kvq_append with num_tokens = batch;
 *   block_table, expected_tags, seq_lens, batch, max_pages_per_seq,
 *   page_tags, abort_flags   as in kvq_tag_check (page_size and num_pages
 *                  come from desc).
 * Same results as the two calls in sequence.  Supports up to 64 KV heads.
 */
KVQ_API kvq_status kvq_tag_check_append(const kvq_cache_desc *desc, const int32_t *block_table,
                                        const uint32_t *expected_tags, const int32_t *seq_lens,
                                        int32_t batch, int32_t max_pages_per_seq,
                                        const uint32_t *page_tags, const void *k_new,
                                        const void *v_new, const int64_t *slot_mapping,
                                        const float *k_scale, const float *v_scale,
                                        void *k_cache, void *v_cache, uint8_t *abort_flags,
                                        kvq_stream_t stream);

/*
 * Prefill -> decode handoff.  Prefill is compute-bound and keeps its cache in
 * BF16; the decode pool stores FP8 (page-1 article, section "量化KV缓存";
 * page-2 summary, section "KV Cache 量化以提高并发量").  Pages that move
 * from a prefill (bf16) cache to a decode (e4m3) cache are quantised whole.
 *
 * kvq_amax_scales -- per-KV-head scales of a set of bf16 pages:
 *   k_scale[h] = amax_h / 448 (one IEEE fp32 division), amax_h = max |x|
 *   over head h of every listed page of k_cache (1 when amax_h is 0); same
 *   for V.  desc describes the bf16 caches; pages int32 [num_listed];
 *   k_scale, v_scale fp32 [Hkv] OUTPUT (device).  Listed ids outside
 *   [0, num_pages) are ignored.
 */
KVQ_API kvq_status kvq_amax_scales(const kvq_cache_desc *desc, const void *k_cache,
                                   const void *v_cache, const int32_t *pages, int32_t num_listed,
                                   float *k_scale, float *v_scale, kvq_stream_t stream);

/*
 * kvq_quantize_pages -- bf16 page src_pages[i] of (k_src, v_src) becomes
 * e4m3 page dst_pages[i] of (k_dst, v_dst): every element e4m3(x / scale[h])
 * by the kvq_append rule (the correctly rounded fp32 quotient, round to
 * nearest even, saturate at +-448), so the codes equal kvq_append's bit for
 * bit.  For scales in [2^-90, 2^100] the kernel reaches that quotient without
 * a division (reciprocal, then one fused multiply-add correction); other
 * scales divide.  src_desc must be a bf16 cache and dst_desc an e4m3 cache with the
 * same page size and KV-head count.  A pair with an out-of-range source or
 * destination id is skipped; destination pages listed twice race.
 */
KVQ_API kvq_status kvq_quantize_pages(const kvq_cache_desc *src_desc, const void *k_src,
                                      const void *v_src, const int32_t *src_pages,
                                      const kvq_cache_desc *dst_desc, void *k_dst, void *v_dst,
                                      const int32_t *dst_pages, int32_t num_listed,
                                      const float *k_scale, const float *v_scale,
                                      kvq_stream_t stream);

/*
 * kvq_decode_plan -- HOST-only query: how kvq_decode_attn (and the calls
 * that run the same kernel: kvq_decode_attn_append, kvq_decode_step,
 * kvq_decode_attn_static_ws) will split the context and how many workspace
 * bytes it needs.
 *
 *   num_splits     requested splits per (request, KV head); 0 = automatic
 *                  (sized from the device's SM count and the batch).  A split
 *                  never exceeds 8,192 tokens, so long contexts get at least
 *                  ceil(context / 8192) splits.
 *   *split_tokens  OUT: tokens per split (a multiple of 32).
 *   *max_splits    OUT: splits of the longest possible request,
 *                  ceil(max_pages_per_seq * page_size / *split_tokens).
 *   *workspace_bytes OUT: bytes of workspace kvq_decode_attn needs: the
 *                  arrival counters (4 bytes per request and KV head, padded
 *                  to 256) plus, when a request can span more than one split
 *                  and the splits merge through the workspace, the per-split
 *                  partial results.
 * Any OUT pointer may be NULL.
 */
KVQ_API kvq_status kvq_decode_plan(const kvq_cache_desc *desc, int32_t batch, int32_t num_q_heads,
                           int32_t max_pages_per_seq, int32_t num_splits,
                           int32_t *split_tokens, int32_t *max_splits,
                           size_t *workspace_bytes);

/*
 * kvq_decode_attn -- single-token attention for B requests over the paged
 * cache, computed as:
 *   for query head h of request r (KV head kvh = h / g):
 *     s_j = softmax_scale * <q[r][h], K^_j>,   j = 0 .. seq_lens[r] - 1
 *     out[r][h] = sum_j exp(s_j - max s) V^_j / sum_j exp(s_j - max s)
 *   with K^ = e4m3 value * k_scale[kvh] (bf16 cache: the bf16 value), same
 *   for V.
 *
 *   q              bf16 [B][Hq][D], any finite values.  On the FP8 path the
 *                  product runs in f16: each q row is first multiplied by the
 *                  power of two that puts its largest magnitude in [2^14,
 *                  2^15) (exact) and the score multiplier divides it out, so
 *                  nothing overflows; an element more than 2^28 times smaller
 *                  than its row's largest loses low bits (error below 2^-39 of
 *                  that largest magnitude).
 *   k_cache, v_cache, desc  as in kvq_append.
 *   k_scale, v_scale  fp32 [Hkv] (ignored, may be NULL, for the bf16 cache).
 *   block_table, max_pages_per_seq, seq_lens  as in kvq_tag_check.
 *   abort_flags    uint8 [B] or NULL; a set flag gives zeros and no reads.
 *   out            [B][Hq][D], bf16 or fp32 per out_dtype.  Requests that are
 *                  aborted, empty (seq_len <= 0), longer than their table row
 *                  or that name a page outside [0, num_pages) get zeros.
 *   workspace      device scratch of at least the kvq_decode_plan size for
 *                  the same arguments.  It starts with one uint32 arrival
 *                  counter per (request, KV head), padded to 256 bytes: they
 *                  must be zero before the first call that uses the buffer,
 *                  and every call leaves them zero again.  The rest holds the
 *                  per-split partial results (lse, o) of one call.  Two calls
 *                  in flight at once must not share a workspace.
 *   num_splits     as in kvq_decode_plan.
 * One kernel launch: every (split, KV head, request) is one CTA.  The
 * splits' partials are merged by their log-sum-exp weights (the combine)
 * inside the launch: when the splits of every (request, KV head) fit on the
 * GPU at once as one thread-block cluster each, through distributed shared
 * memory; otherwise the last split of a (request, KV head) to finish merges
 * them from the workspace before it exits.
 */
KVQ_API kvq_status kvq_decode_attn(const kvq_cache_desc *desc, const void *q, int32_t batch,
                           int32_t num_q_heads, const void *k_cache, const void *v_cache,
                           const float *k_scale, const float *v_scale,
                           const int32_t *block_table, int32_t max_pages_per_seq,
                           const int32_t *seq_lens, float softmax_scale,
                           const uint8_t *abort_flags, void *out, int32_t out_dtype,
                           void *workspace, size_t workspace_bytes, int32_t num_splits,
                           kvq_stream_t stream);

/*
 * kvq_decode_plan_mt / kvq_decode_attn_mt -- decode attention with several
 * new query tokens per request (verifying speculative drafts).  The source
 * pages describe one new token per step; this extends kvq_decode_attn's
 * definition: the n = num_query_tokens new tokens are the request's last n
 * positions, already in the cache (kvq_append), and query token i attends
 * causally to positions 0 .. seq_lens[r] - n + i:
 *   for query token i, query head h of request r (KV head kvh = h / g):
 *     s_j = softmax_scale * <q[r][i][h], K^_j>,   j = 0 .. seq_lens[r] - n + i
 *     out[r][i][h] = sum_j exp(s_j - max s) V^_j / sum_j exp(s_j - max s)
 *
 *   q              bf16 [B][n][Hq][D] (row r * n + i of a [B * n][Hq][D] array).
 *   out            [B][n][Hq][D], bf16 or fp32 per out_dtype.  A query with no
 *                  position to attend to (seq_lens[r] < n - i) gets zeros, as
 *                  does every query of a request kvq_decode_attn would zero.
 *   num_query_tokens  n, 1 to 16 (KVQ_ERR_UNSUPPORTED above); n = 1 is
 *                  kvq_decode_attn.
 *   Every other argument as in kvq_decode_plan / kvq_decode_attn; the
 *   workspace size comes from kvq_decode_plan_mt with the same n.
 * One launch.  With an FP8 cache and n * g >= 64 query rows (token, head) per
 * KV head, one CTA per (split, request, KV head) serves every row on the
 * 5th-generation tensor cores (tcgen05: Q, P and the accumulators in tensor
 * memory, K and V converted once to f16 in shared memory); its splits merge
 * through the workspace and are whole 64-token tiles.  Otherwise a CTA
 * serves up to 16 query rows, and ceil(n * g / 16) CTAs stream the same pages
 * (each reads them; the copies share them through L2).
 */
KVQ_API kvq_status kvq_decode_plan_mt(const kvq_cache_desc *desc, int32_t batch,
                                      int32_t num_query_tokens, int32_t num_q_heads,
                                      int32_t max_pages_per_seq, int32_t num_splits,
                                      int32_t *split_tokens, int32_t *max_splits,
                                      size_t *workspace_bytes);
KVQ_API kvq_status kvq_decode_attn_mt(const kvq_cache_desc *desc, const void *q, int32_t batch,
                                      int32_t num_query_tokens, int32_t num_q_heads,
                                      const void *k_cache, const void *v_cache,
                                      const float *k_scale, const float *v_scale,
                                      const int32_t *block_table, int32_t max_pages_per_seq,
                                      const int32_t *seq_lens, float softmax_scale,
                                      const uint8_t *abort_flags, void *out, int32_t out_dtype,
                                      void *workspace, size_t workspace_bytes, int32_t num_splits,
                                      kvq_stream_t stream);

/*
 * kvq_decode_attn_append -- kvq_append of each request's new token followed
 * by kvq_decode_attn, in one launch.  Request r's new token is the last one
 * it attends to: position seq_lens[r] - 1, written at
 *   slot = block_table[r][(seq_lens[r] - 1) / page_size] * page_size
 *          + (seq_lens[r] - 1) % page_size,
 * with the codes kvq_append would write (blog post "Smaller, faster, safer",
 * page-1 mirror section "量化KV缓存": quantise on append; FP8 attention that
 * converts what it reads).
 *
 *   k_new, v_new   bf16 [B][Hkv][D], 16-byte aligned: row r is request r's
 *                  new token.
 *   k_cache, v_cache  written (one row per request and KV head) and read.
 *   Every other argument as in kvq_decode_attn.
 * Results equal kvq_append(k_new, v_new, slots as above, abort_flags) then
 * kvq_decode_attn with the same arguments, bit for bit.  A request that is
 * aborted, empty, longer than its table row or that names a page outside
 * [0, num_pages) gets zeros and no write.  Only request r's own last page
 * is written, so the rows of different requests must not share a page
 * position.
 */
KVQ_API kvq_status kvq_decode_attn_append(const kvq_cache_desc *desc, const void *q, int32_t batch,
                                  int32_t num_q_heads, void *k_cache, void *v_cache,
                                  const float *k_scale, const float *v_scale,
                                  const int32_t *block_table, int32_t max_pages_per_seq,
                                  const int32_t *seq_lens, float softmax_scale,
                                  const uint8_t *abort_flags, const void *k_new, const void *v_new,
                                  void *out, int32_t out_dtype, void *workspace,
                                  size_t workspace_bytes, int32_t num_splits, kvq_stream_t stream);

/*
 * kvq_decode_step -- one decode step in one launch: the tag check of every
 * request (page-3 article: check before the cache is read; page-2 summary,
 * section "KV Cache 完整性检查"), then, for each request that passed, the
 * append of its new token and paged decode attention over the FP8 (or BF16)
 * cache (page-1 article, section "量化KV缓存").
 *
 *   expected_tags  uint32 [B][max_pages_per_seq]: the tag request r expects
 *                  for each of its pages, as in kvq_tag_check.
 *   page_tags      uint32 [desc->num_pages]: the live tag of every page.
 *   abort_flags    uint8 [B] OUTPUT: 1 where the check failed, else 0 --
 *                  the flags kvq_tag_check writes.
 *   Every other argument as in kvq_decode_attn_append (the abort_flags
 *   input of that call is this call's output).
 * Results equal kvq_tag_check followed by kvq_decode_attn_append with its
 * flags, bit for bit: flags, cache writes and outputs.  Each split of the
 * attention checks the entries of its own pages while it streams them; the
 * CTA that combines a request's splits (per KV head) learns the verdict,
 * and only then is the flag written (by KV head 0) and, if the request
 * passed, its new token.  A failed request gets zeros and no write.  Null
 * expected_tags, page_tags or abort_flags is KVQ_ERR_INVALID_ARG;
 * everything else is checked as in kvq_decode_attn_append.
 */
KVQ_API kvq_status kvq_decode_step(const kvq_cache_desc *desc, const void *q, int32_t batch,
                                   int32_t num_q_heads, void *k_cache, void *v_cache,
                                   const float *k_scale, const float *v_scale,
                                   const int32_t *block_table, int32_t max_pages_per_seq,
                                   const int32_t *seq_lens, const uint32_t *expected_tags,
                                   const uint32_t *page_tags, uint8_t *abort_flags,
                                   float softmax_scale, const void *k_new, const void *v_new,
                                   void *out, int32_t out_dtype, void *workspace,
                                   size_t workspace_bytes, int32_t num_splits, kvq_stream_t stream);

/*
 * kvq_w4a16_plan / kvq_w4a16_gemm -- INT4 weight-only product for decode
 * (blog post "Smaller, faster, safer", page-1 mirror section "压缩模型权重":
 * weights compressed from FP8 to 4-bit integers for decode, which streams
 * the weights; page-2 mirror section "模型权重压缩以降低延迟"):
 *   y[m][n] = sum_k x[m][k] * q[n][k] * s[n][k / 128]
 * The pages fix no format; this library's:
 *   w              uint8 [N][K/2]: byte k/2 of row n holds q[n][k], a signed
 *                  (two's complement) 4-bit integer in [-8, 7], in its low
 *                  nibble for even k and its high nibble for odd k.
 *   scales         bf16 [N][K/128] (2-byte aligned): one per output column
 *                  and group of 128 consecutive k.
 *   x              bf16 [M][K], 16-byte aligned.  On the tensor cores x and
 *                  the expanded weights are f16: x is exact for |x| in
 *                  [2^-14, 65504] and is not range-scaled (unlike q in
 *                  kvq_decode_attn): |x| above 65504 overflows, below 2^-14
 *                  loses low bits; q is an exact f16 integer and the scales
 *                  apply in fp32.
 *   y              [M][N], bf16 or fp32 per out_dtype, 16-byte aligned.
 *   Shapes: K a positive multiple of 256 and at most 65,536; N a multiple of
 *   64 (KVQ_ERR_UNSUPPORTED otherwise); any M >= 0 (16 rows per launch: a
 *   batch of more than 16 rows reads the weights once per 16 rows).
 *   num_splits     ranges K is cut into (1..8, each a whole number of 256-k
 *                  blocks, at most 8,192 k); 0 = automatic.
 * kvq_w4a16_plan (HOST only) returns the split count kvq_w4a16_gemm uses.
 * A copy wait that gives up sets bit 0 of kvq_device_error and gives zeros
 * for that launch's tile of 64 columns.
 */
KVQ_API kvq_status kvq_w4a16_plan(int32_t m, int32_t n, int32_t k, int32_t num_splits, int32_t *splits);
KVQ_API kvq_status kvq_w4a16_gemm(const void *x, const uint8_t *w, const void *scales, int32_t m,
                                  int32_t n, int32_t k, void *y, int32_t out_dtype, int32_t num_splits,
                                  kvq_stream_t stream);

/* ------------------------------------------------------------------------
 * Calibration and test hooks.  Not part of the decode path: a deployment
 * never needs them.
 * ------------------------------------------------------------------------ */

/*
 * kvq_read_probe -- calibration, not part of the decode path: read `bytes`
 * of device memory at `src` once, with a plain streaming kernel (16-byte
 * loads, 8 CTAs x 256 threads per SM, each CTA one contiguous slice), and
 * XOR every 32-bit word into *sink (device, uint32; the caller zeroes it first).  Timed like the
 * decode kernels, it says how fast one launch reads that many bytes on this
 * GPU.  src and bytes must be multiples of 16 (KVQ_ERR_INVALID_ARG
 * otherwise); bytes == 0 does nothing.
 */
KVQ_API kvq_status kvq_read_probe(const void *src, size_t bytes, uint32_t *sink, kvq_stream_t stream);

/*
 * kvq_decode_attn_static_ws -- kvq_decode_attn for callers that cannot
 * allocate device memory while they decode (an engine that has already
 * handed all of its device memory to its own pool, or C code that holds no
 * allocator).  The source pages have no counterpart to this entry point.
 *
 * Same arguments and results as kvq_decode_attn, without the workspace: the
 * scratch is one array of KVQ_STATIC_WS_BYTES (16 MiB) compiled into the
 * library, which every GPU that loads the library holds until the process
 * exits.  The call allocates nothing.
 *   - A call whose kvq_decode_plan workspace size exceeds KVQ_STATIC_WS_BYTES
 *     returns KVQ_ERR_WORKSPACE before touching the GPU; pass a smaller
 *     num_splits, or use kvq_decode_attn with a workspace of your own.
 *   - The first call on a device looks up the array's device address on the
 *     current device (once per device); make that first call before any
 *     stream capture.  The address is kept for the life of the process: after
 *     cudaDeviceReset (or anything else that destroys the device's primary
 *     context) restart the process before calling this again.
 *   - All calls share the one array and it keeps the last call's contents;
 *     each call clears the part that must start at zero (the arrival
 *     counters) on its stream before the kernel runs.  Calls that overlap on
 *     the GPU (other streams, other threads) race on the array: serialise
 *     them.
 */
#define KVQ_STATIC_WS_BYTES (16u << 20)
KVQ_API kvq_status kvq_decode_attn_static_ws(const kvq_cache_desc *desc, const void *q,
                                             int32_t batch, int32_t num_q_heads,
                                             const void *k_cache, const void *v_cache,
                                             const float *k_scale, const float *v_scale,
                                             const int32_t *block_table,
                                             int32_t max_pages_per_seq, const int32_t *seq_lens,
                                             float softmax_scale, const uint8_t *abort_flags,
                                             void *out, int32_t out_dtype, int32_t num_splits,
                                             kvq_stream_t stream);

/*
 * kvq_diag_set_copy_wait_ns -- test hook, process-wide: the time limit the
 * decode kernel (kvq_decode_attn and every call that runs its kernel) gives a
 * warp's wait on each of its bulk copies, for launches made after this call.
 * ns < 0 or above the default restores the default (about one second); 0
 * makes every warp give up at its first wait, without looking.  Whatever the
 * setting, a warp that gave up then waits for its copies still in flight
 * with the default limit, so a shortened limit runs the failure path
 * (kvq_device_error bit 0, zeros for every (request, KV head) a failed CTA
 * served) without leaving a copy unaccounted for.  Not thread-safe against
 * launches on other threads.
 */
KVQ_API kvq_status kvq_diag_set_copy_wait_ns(int64_t ns);

/*
 * kvq_device_error -- HOST call, synchronous: reads (into *bits, host
 * memory) and, if `clear` is non-zero, resets the sticky device error word
 * of the current device.
 *   Bit 0: a bulk-copy wait in the decode kernel or the INT4 kernel gave up
 *          after its time limit; the warp then waited for its copies still in
 *          flight and the CTA returned without its results (the requests it
 *          served, or the INT4 tile, get zeros).
 *   Bit 1: that wait for the copies in flight gave up as well, so a copy may
 *          still land in shared memory that a later CTA uses: results of the
 *          launches made since are undefined; synchronise the device, check
 *          the bits and rerun them.
 *   Bit 2: in the tensor-core multi-token kernel, a wait for a tensor-core
 *          step or for another warp's hand-off gave up after its time limit;
 *          every warp of the CTA gave up with it, the copies in flight were
 *          waited for, and the requests it served get zeros.
 * 0 means no such event since the last clear.
 */
KVQ_API kvq_status kvq_device_error(uint32_t *bits, int32_t clear);

/* Static, human-readable name of a status code. */
KVQ_API const char *kvq_status_string(kvq_status status);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H */
