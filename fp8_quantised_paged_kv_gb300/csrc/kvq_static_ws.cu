// kvq_static_ws.cu -- kvq_decode_attn with its scratch built into the library.
//
// Some callers cannot call cudaMalloc when they decode: an engine that has
// handed every byte of device memory to its own pool before serving starts,
// or plain C code that links this library but owns no allocator at all.
// kvq_decode_attn_static_ws gives them the same attention with no workspace
// argument: the scratch is one fixed-size array compiled into this file, and
// every GPU that loads the library keeps it until the process exits.
#include <mutex>

#include "../../include/kvq.h"
#include "kvq_internal.h"

namespace {

constexpr size_t kStaticScratchBytes = static_cast<size_t>(KVQ_STATIC_WS_BYTES);
constexpr int kMaxDevices = 64;

// The scratch itself.  In host code this name is only a stand-in for the
// device array: its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

void *g_scratch_address[kMaxDevices] = {};
std::mutex g_scratch_mutex;

// Device address of the scratch on the current device, looked up once per
// device (with that device current) and remembered.
kvq_status scratch_address(void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return KVQ_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_address[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr)
            return KVQ_ERR_CUDA;
        g_scratch_address[dev] = p;
    }
    *out = g_scratch_address[dev];
    return KVQ_OK;
}

} // namespace

extern "C" {

kvq_status kvq_decode_attn_static_ws(const kvq_cache_desc *desc, const void *q, int32_t batch,
                                     int32_t num_q_heads, const void *k_cache, const void *v_cache,
                                     const float *k_scale, const float *v_scale,
                                     const int32_t *block_table, int32_t max_pages_per_seq,
                                     const int32_t *seq_lens, float softmax_scale,
                                     const uint8_t *abort_flags, void *out, int32_t out_dtype,
                                     int32_t num_splits, kvq_stream_t stream)
{
    size_t need = 0;
    kvq_status st = kvq_decode_plan(desc, batch, num_q_heads, max_pages_per_seq, num_splits,
                                    nullptr, nullptr, &need);
    if (st != KVQ_OK)
        return st;
    if (need > kStaticScratchBytes)
        return KVQ_ERR_WORKSPACE;        // the plan needs more than the built-in scratch holds
    if (batch == 0)
        return KVQ_OK;
    void *scratch = nullptr;
    st = scratch_address(&scratch);
    if (st != KVQ_OK)
        return st;
    // The scratch keeps whatever the previous call left.  Its arrival
    // counters (4 bytes per request and KV head, first in the layout) must
    // start at zero, so clear them on the caller's stream first.
    const size_t counter_bytes =
        (static_cast<size_t>(batch) * static_cast<size_t>(desc->num_kv_heads) * 4 + 255) / 256 * 256;
    if (cudaMemsetAsync(scratch, 0, counter_bytes, reinterpret_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
        return KVQ_ERR_CUDA;
    return kvq_decode_attn(desc, q, batch, num_q_heads, k_cache, v_cache, k_scale, v_scale,
                           block_table, max_pages_per_seq, seq_lens, softmax_scale, abort_flags,
                           out, out_dtype, scratch, kStaticScratchBytes, num_splits, stream);
}

} // extern "C"
