// kvq_probe.cu -- a read-only bandwidth probe for calibration.
//
// Not part of the decode path.  It reads a buffer once, the way a plain
// streaming kernel would: 8 CTAs of 256 threads per SM, CTA c reading the
// c-th contiguous slice of the buffer with four 16-byte loads in flight per
// thread.  Of the shapes tried (grid-stride or per-CTA slices; 2, 4 or 8
// loads in flight; 2 to 16 CTAs per SM), slices read 134 MB fastest,
// 28.7-29.0 us against 30.5 us for the grid-stride form.  Every word is
// folded into one XOR that the caller can check.  Timed under the same
// protocol as the decode kernels, it says how fast one launch can read the
// same number of bytes on the same GPU.
#include <cstdint>

#include <cuda_runtime.h>

#include "kvq.h"

namespace {

constexpr int kProbeThreads = 256;
constexpr int kProbeCtasPerSm = 8;

__global__ void __launch_bounds__(kProbeThreads) read_probe_kernel(const uint4 *__restrict__ src, int64_t n16,
                                                                   unsigned int *sink)
{
    const int64_t per = (n16 + gridDim.x - 1) / gridDim.x;            // this CTA's slice
    const int64_t beg = static_cast<int64_t>(blockIdx.x) * per;
    const int64_t end = beg + per < n16 ? beg + per : n16;
    const int nt = blockDim.x;
    int64_t i = beg + threadIdx.x;
    uint32_t acc = 0;
    for (; i + 3 * nt < end; i += 4 * nt) {
        const uint4 a = __ldcs(src + i), b = __ldcs(src + i + nt);
        const uint4 c = __ldcs(src + i + 2 * nt), d = __ldcs(src + i + 3 * nt);
        acc ^= a.x ^ a.y ^ a.z ^ a.w ^ b.x ^ b.y ^ b.z ^ b.w ^ c.x ^ c.y ^ c.z ^ c.w ^ d.x ^ d.y ^ d.z ^ d.w;
    }
    for (; i < end; i += nt) {
        const uint4 a = __ldcs(src + i);
        acc ^= a.x ^ a.y ^ a.z ^ a.w;
    }
    // one atomic per CTA: per-warp atomics on the one word cost the probe
    // ~3 us of contention at the end
    __shared__ uint32_t s_warp[kProbeThreads / 32];
    for (int off = 16; off > 0; off >>= 1)
        acc ^= __shfl_xor_sync(0xFFFFFFFFu, acc, off);
    if (threadIdx.x % 32 == 0)
        s_warp[threadIdx.x / 32] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t v = 0;
        for (int w = 0; w < kProbeThreads / 32; ++w)
            v ^= s_warp[w];
        if (v != 0)
            atomicXor(sink, v);
    }
}

} // namespace

extern "C" {

KVQ_API kvq_status kvq_read_probe(const void *src, size_t bytes, uint32_t *sink, kvq_stream_t stream)
{
    if (bytes == 0)
        return KVQ_OK;
    if (!src || !sink || (reinterpret_cast<uintptr_t>(src) & 15u) != 0 || (bytes & 15u) != 0)
        return KVQ_ERR_INVALID_ARG;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        return KVQ_ERR_CUDA;
    read_probe_kernel<<<static_cast<unsigned>(sms * kProbeCtasPerSm), kProbeThreads, 0,
                        reinterpret_cast<cudaStream_t>(stream)>>>(static_cast<const uint4 *>(src),
                                                                  static_cast<int64_t>(bytes / 16),
                                                                  reinterpret_cast<unsigned int *>(sink));
    return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

} // extern "C"
