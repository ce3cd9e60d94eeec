// kvq_rowops.cuh -- the per-request tag check and the per-row quantise-store
// shared by the tag-check, append and fused step-prologue kernels.
#pragma once

#include "kvq_internal.h"
#include "kvq_ptx.cuh"

namespace kvq {

constexpr int kThreadsPerRow = kHeadDim / 8;   // 16 threads x 8 elements per 128-element row

// Tag check of request r by the whole block (blockDim.x threads, kUnroll
// entries per thread per pass, every block-table and expected-tag load of a
// pass issued before the live-tag gathers).  Returns the block-wide verdict:
// true if any used entry names a page outside [0, num_pages) or a page whose
// live tag differs from the expected one, or if the request needs more
// entries than its row holds.  Every thread of the block must call it.
template <int kUnroll>
__device__ __forceinline__ bool tag_check_request(const int32_t *block_table,
                                                  const uint32_t *expected_tags,
                                                  const int32_t *seq_lens, const uint32_t *page_tags,
                                                  int32_t max_pages_per_seq, int32_t page_size,
                                                  int32_t num_pages, int64_t r)
{
    const int32_t *bt = block_table + r * max_pages_per_seq;
    const uint32_t *exp = expected_tags + r * max_pages_per_seq;
    const int nt = blockDim.x;
    const int64_t pass = static_cast<int64_t>(nt) * kUnroll;
    // The first pass's table and expected-tag loads go out together with the
    // length load (entries of the row past the used ones are read and then
    // ignored), so the check costs two rounds of dependent loads, not three.
    int32_t p[kUnroll];
    uint32_t want[kUnroll];
#pragma unroll
    for (int k = 0; k < kUnroll; ++k) {
        const int64_t i = k * nt + threadIdx.x;
        p[k] = i < max_pages_per_seq ? __ldg(bt + i) : 0;
        want[k] = i < max_pages_per_seq ? __ldg(exp + i) : 0u;
    }
    const int64_t len = seq_lens[r] > 0 ? seq_lens[r] : 0;
    int64_t used = (len + page_size - 1) / page_size;
    bool bad = false;
    if (used > max_pages_per_seq) {
        bad = true;
        used = max_pages_per_seq;
    }
    for (int64_t base = 0; base < used; base += pass) {
        uint32_t live[kUnroll];
        if (base > 0) {
#pragma unroll
            for (int k = 0; k < kUnroll; ++k) {
                const int64_t i = base + k * nt + threadIdx.x;
                p[k] = i < used ? __ldg(bt + i) : 0;
                want[k] = i < used ? __ldg(exp + i) : 0u;
            }
        }
#pragma unroll
        for (int k = 0; k < kUnroll; ++k) {
            const int64_t i = base + k * nt + threadIdx.x;
            const bool in_range = i < used && p[k] >= 0 && p[k] < num_pages;
            live[k] = in_range ? __ldg(page_tags + p[k]) : 0u;
        }
#pragma unroll
        for (int k = 0; k < kUnroll; ++k) {
            const int64_t i = base + k * nt + threadIdx.x;
            if (i < used && (p[k] < 0 || p[k] >= num_pages || live[k] != want[k]))
                bad = true;
        }
    }
    return __syncthreads_or(bad) != 0;
}

// Four bf16 elements (two words) -> four e4m3 codes e4m3(x / scale), one
// IEEE fp32 division each, rounding to nearest even, saturating at +-448;
// element 0 in the low byte.
__device__ __forceinline__ uint32_t encode4_e4m3(uint32_t w0, uint32_t w1, float scale)
{
    const float2 p0 = bf16x2_to_f32x2(w0);
    const float2 p1 = bf16x2_to_f32x2(w1);
    const uint16_t c01 = f32x2_to_e4m3x2(__fdiv_rn(p0.x, scale), __fdiv_rn(p0.y, scale));
    const uint16_t c23 = f32x2_to_e4m3x2(__fdiv_rn(p1.x, scale), __fdiv_rn(p1.y, scale));
    return static_cast<uint32_t>(c01) | (static_cast<uint32_t>(c23) << 16);
}

// The correctly rounded fp32 quotient x / scale without a division, for
// scales in [2^-90, 2^100].  With rcp = RN(1 / scale), q0 = RN(x * rcp) and
// the exact remainder r = scale * q0 - x (one fma), RN(q0 - r * rcp) is
// RN(x / scale): the correction step of P. Markstein, "Computation of
// elementary functions on the IBM RISC System/6000 processor", IBM J. Res.
// Dev. 34(1), 1990, checked here exhaustively over every bf16 significand of
// x against every fp32 significand of the scale.  x is first clamped to
// +-1024 * scale, NaN kept: a clamped quotient is +-1024, which saturates like
// the true one, and no intermediate overflows.  Within the scale range every
// intermediate that decides an e4m3 code (|x / scale| >= 2^-12) is normal or
// exact, and the remainder's sign rule keeps -0 as -0.
struct QuotientRcp {
    float scale, rcp, lim;
};

// The per-scale constants; false outside the scale range above, where the
// caller divides instead.
__device__ __forceinline__ bool quotient_rcp_init(float scale, QuotientRcp &c)
{
    c.scale = scale;
    c.rcp = __frcp_rn(scale);
    c.lim = 1024.0f * scale;
    return scale >= 0x1p-90f && scale <= 0x1p100f;
}

__device__ __forceinline__ float quotient_rn(float x, const QuotientRcp &c)
{
    float xc;
    asm("min.NaN.f32 %0, %1, %2;" : "=f"(xc) : "f"(x), "f"(c.lim));
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(xc) : "f"(xc), "f"(-c.lim));
    const float q0 = __fmul_rn(xc, c.rcp);
    const float r = __fmaf_rn(c.scale, q0, -xc);
    return __fmaf_rn(r, -c.rcp, q0);
}

// encode4_e4m3 with the quotients from quotient_rn (the same codes).
__device__ __forceinline__ uint32_t encode4_e4m3_rcp(uint32_t w0, uint32_t w1, const QuotientRcp &c)
{
    const float2 p0 = bf16x2_to_f32x2(w0);
    const float2 p1 = bf16x2_to_f32x2(w1);
    const uint16_t c01 = f32x2_to_e4m3x2(quotient_rn(p0.x, c), quotient_rn(p0.y, c));
    const uint16_t c23 = f32x2_to_e4m3x2(quotient_rn(p1.x, c), quotient_rn(p1.y, c));
    return static_cast<uint32_t>(c01) | (static_cast<uint32_t>(c23) << 16);
}

// Eight consecutive elements of one K or V row: bf16 x (16 bytes) becomes
// eight e4m3 codes e4m3(x / scale) -- one IEEE fp32 division each, rounding
// to nearest even, saturating at +-448 -- stored as 8 bytes at dst; or, for
// the bf16 cache, the 16 bytes unchanged.
template <bool kBf16Cache>
__device__ __forceinline__ void store_row_part(void *dst_row, int part, uint4 x, float scale)
{
    if constexpr (kBf16Cache) {
        *reinterpret_cast<uint4 *>(static_cast<uint16_t *>(dst_row) + part * 8) = x;
    } else {
        *reinterpret_cast<uint2 *>(static_cast<uint8_t *>(dst_row) + part * 8) =
            make_uint2(encode4_e4m3(x.x, x.y, scale), encode4_e4m3(x.z, x.w, scale));
    }
}

} // namespace kvq
