// kvq_internal.h -- launch interfaces shared by the C ABI (kvq_abi.cu) and
// the kernel translation units.  Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace kvq {

constexpr int kHeadDim = 128;
constexpr int kChunkTokens = 32;     // tokens one warp consumes per pipeline stage
constexpr int kMaxGroup = 8;         // query heads per KV head on one mma n-tile
constexpr int kMaxCluster = 8;       // splits merged inside one thread-block cluster
constexpr int kMaxSplitsTotal = 1024;  // splits of one (request, KV head)

struct AppendArgs {
    const void *k_new, *v_new;       // bf16 [T][Hkv][D]
    const int64_t *slot_mapping;     // [T]
    const float *k_scale, *v_scale;  // [Hkv]
    const uint8_t *abort_flags;      // [T] or null
    void *k_cache, *v_cache;
    int32_t num_tokens, num_kv_heads, page_size;
    int64_t num_slots;               // num_pages * page_size
    bool bf16_cache;
};
cudaError_t launch_append(const AppendArgs &a, cudaStream_t stream);

struct TagCheckArgs {
    const int32_t *block_table;
    const uint32_t *expected_tags;
    const int32_t *seq_lens;
    const uint32_t *page_tags;
    uint8_t *abort_flags;
    int32_t batch, max_pages_per_seq, page_size, num_pages;
};
cudaError_t launch_tag_check(const TagCheckArgs &a, cudaStream_t stream);

// Prefill -> decode handoff of whole pages (bf16 source, e4m3 destination).
struct HandoffArgs {
    const void *k_src, *v_src;              // bf16 caches [src_num_pages][Hkv][ps][D]
    const int32_t *src_pages;               // [num_listed]
    void *k_dst, *v_dst;                    // e4m3 caches [dst_num_pages][Hkv][ps][D]
    const int32_t *dst_pages;               // [num_listed]
    const float *k_scale, *v_scale;         // [Hkv] (quantise)
    float *k_scale_out, *v_scale_out;       // [Hkv] (amax -> scale)
    int32_t num_listed, num_kv_heads, page_size, src_num_pages, dst_num_pages;
};
cudaError_t launch_amax_scales(const HandoffArgs &a, cudaStream_t stream);
cudaError_t launch_quantize_pages(const HandoffArgs &a, cudaStream_t stream);

// Tag check of every request, then the append of token r for request r
// unless it was aborted (decode step: one new token per request).
cudaError_t launch_tag_check_append(const TagCheckArgs &t, const AppendArgs &a, cudaStream_t stream);

// INT4 weight-only product y[m][n] = sum_k x[m][k] q[n][k] s[n][k / 128] for
// up to 16 rows of x per launch.  The weights are read through a 2-D tensor
// map over W viewed as [N rows][K / 2 bytes].
struct W4Args {
    const void *x;                   // bf16 [rows][k] (this launch's rows)
    const void *scales;              // bf16 [n][k / 128]
    void *y;                         // [rows][n], bf16 or fp32
    int32_t rows, n, k;              // rows <= 16; k % 256 == 0; n % 64 == 0
    int32_t splits, k_split;         // K is cut into `splits` ranges of k_split
    bool out_fp32;
};
constexpr int kW4Cols = 64;          // output columns per CTA
constexpr int kW4BlockK = 256;       // granularity of K and of its split ranges
constexpr int kW4CopyK = 128;        // k per tensor copy: 64 bytes of every column, one scale group
constexpr int kW4MaxSplits = 8;      // splits of K (one thread-block cluster)
cudaError_t launch_w4a16(const W4Args &a, const CUtensorMap &w_map, cudaStream_t stream);
// Resident CTAs of the INT4 kernel per SM, and resident clusters of `splits`.
int w4a16_ctas_per_sm();
int w4a16_cluster_capacity(int splits);
cudaError_t read_w4_error(uint32_t *bits, bool clear);

// Workspace layout (bytes from the workspace base):
//   [0, counter_bytes)       uint32 arrivals[B][Hkv][row_blocks]: splits of each
//                            (request, KV head, row block) that have published;
//                            zero before the first call, and every call leaves
//                            them zero
//   [counter_bytes, +lse)    fp32 lse[B][n_query][Hq][S]  (log2 domain, NaN =
//                            invalid split, -inf = a split that saw no token)
//   [.., +o)                 fp32 o[B][n_query][Hq][S][D]  (each split's normalised output)
struct DecodeArgs {
    const void *q;                   // bf16 [B][Hq][D]
    const float *k_scale, *v_scale;  // [Hkv] (unused for bf16 cache)
    const int32_t *block_table;      // [B][max_pages]
    const int32_t *seq_lens;         // [B]
    const uint8_t *abort_flags;      // [B] or null
    void *out;                       // [B][Hq][D]
    unsigned int *counters;
    float *ws_lse;
    float *ws_o;
    int32_t batch, num_q_heads, num_kv_heads, group, page_size, num_pages;
    int32_t max_pages_per_seq, split_tokens, max_splits;
    const void *k_new, *v_new;       // fused append: bf16 [B][Hkv][D] new token, else null
    void *k_cache, *v_cache;         // fused append: the caches the token is written to
    int32_t cluster;                 // 0: combine through memory; else the splits of a
                                     // (request, KV head) form one cluster of max_splits CTAs
    const uint32_t *expected_tags;   // in-launch tag check (kvq_decode_step): [B][max_pages],
    const uint32_t *page_tags;       // [num_pages] and the flags written, [B]; else null and
    uint8_t *abort_out;              // abort_flags (if any) is read instead
    int32_t n_query;                 // new query tokens per request (q, out: [B][n_query][Hq][D])
    int32_t row_blocks;              // CTAs per (split, request, KV head): ceil(n_query * g / 8)
    float qk_scale_log2;             // softmax_scale * log2(e)
    uint64_t copy_wait_ns;           // a consumer's limit on one copy wait (0: give up at once)
    bool out_fp32, bf16_cache;
};

// Default limit of a wait on a bulk copy in the decode kernel: about one
// second.  The drain that follows a timeout always waits this long.
constexpr uint64_t kCopyWaitLimitNs = 1000000000ull;
// The limit decode launches use for a consumer's copy waits: the default
// unless the diagnostics entry point changed it.
uint64_t decode_copy_wait_ns();

// Split kernel with the combine fused into its epilogue.  The tensor maps
// describe the K and V caches as 2-D [rows][128 bytes] tensors with 128-byte
// swizzle.
cudaError_t launch_decode(const DecodeArgs &a, const CUtensorMap &k_map, const CUtensorMap &v_map,
                          cudaStream_t stream);
// Resident decode CTAs per SM for the cache type (occupancy of the kernel;
// multi: the multi-token build, 16 query rows per CTA).
int decode_ctas_per_sm(bool bf16_cache, bool multi = false);
// How many clusters of n split CTAs can be resident at once on the current
// device (0 if clusters of n cannot be used).
int decode_cluster_capacity(int n, bool bf16_cache, bool multi = false);
// Query rows one CTA of the multi-token build serves, and the most splits of
// one of its requests.
constexpr int kMultiRowsPerCta = 16;
constexpr int kMultiMaxSplitsPerRequest = 512;

// Multi-token decode over an FP8 cache on the 5th-generation tensor cores
// (tcgen05, accumulators and the A operands in tensor memory): one CTA per
// (split, KV head, request) takes all n_query * g <= 128 query rows; the
// splits merge through the workspace (never a cluster).  Split sizes are
// multiples of kUmmaTileTokens.
constexpr int kUmmaTileTokens = 64;
// Query rows per KV head (n_query * g) from which multi-token decode over an
// FP8 cache takes that kernel; fewer rows take the mma.sync build, which
// converts K and V per 16 rows but has no tensor-memory pipeline to fill.
constexpr int kUmmaMinRows = 64;
inline bool use_umma(bool bf16_cache, int n_query, int group)
{
    return !bf16_cache && n_query > 1 && n_query * group >= kUmmaMinRows;
}
cudaError_t launch_decode_umma(const DecodeArgs &a, const CUtensorMap &k_map, const CUtensorMap &v_map,
                               cudaStream_t stream);
// Resident CTAs per SM of that kernel (bf16 output; at most 2: tensor memory).
int decode_umma_ctas_per_sm();
cudaError_t read_umma_error(uint32_t *bits, bool clear);

// Box height (in 128-byte rows) of one bulk copy for a page size.
inline int tma_box_rows(int page_size, bool bf16_cache)
{
    int tok = page_size < kChunkTokens ? page_size : kChunkTokens;
    return bf16_cache ? 2 * tok : tok;
}

cudaError_t read_device_error(uint32_t *bits, bool clear);

#ifdef KVQ_PHASE_STAMPS
// Instrumented build only: the %globaltimer stamps of the last decode launch
// ([CTA][8] points) and of the last tag-check + append launch ([CTA][2]).
cudaError_t read_decode_stamps(unsigned long long *host, size_t count);
cudaError_t read_check_stamps(unsigned long long *host, size_t count);
cudaError_t read_tag_stamps(unsigned long long *host, size_t count);   // tag check alone, [CTA][2]
#endif

// SMs of the current device, queried once per device.  A host with no usable
// device (the planner's host-only queries) plans for a 152-SM GB300.
int device_sm_count();

} // namespace kvq
