// kvq_probe.cu -- a read-only bandwidth probe for calibration.
//
// Not part of the decode path.  It reads a buffer once, the way a plain
// streaming kernel would: 8 CTAs of 256 threads per SM, each thread keeping
// four 16-byte loads in flight per pass of a grid-stride loop (the shape
// that streamed fastest among the grid and block sizes tried).  Every word
// is folded into one XOR that the caller can check.  Timed under the same
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
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    uint32_t acc = 0;
    for (; i + 3 * stride < n16; i += 4 * stride) {
        const uint4 a = __ldcs(src + i), b = __ldcs(src + i + stride);
        const uint4 c = __ldcs(src + i + 2 * stride), d = __ldcs(src + i + 3 * stride);
        acc ^= a.x ^ a.y ^ a.z ^ a.w ^ b.x ^ b.y ^ b.z ^ b.w ^ c.x ^ c.y ^ c.z ^ c.w ^ d.x ^ d.y ^ d.z ^ d.w;
    }
    for (; i < n16; i += stride) {
        const uint4 a = __ldcs(src + i);
        acc ^= a.x ^ a.y ^ a.z ^ a.w;
    }
    for (int off = 16; off > 0; off >>= 1)
        acc ^= __shfl_xor_sync(0xFFFFFFFFu, acc, off);
    if (threadIdx.x % 32 == 0 && acc != 0)
        atomicXor(sink, acc);
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
