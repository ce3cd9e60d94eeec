// kvq_umma.cuh -- inline-PTX wrappers for the 5th-generation tensor cores
// (tcgen05: tensor-memory allocation, single-thread MMA issue with operands
// in shared memory, completion through an mbarrier, tensor-memory loads and
// stores).  sm_100a / sm_103a only.
//
// Operand layout used throughout: a tile of 16-bit values with 64 elements
// (128 bytes) per row, rows 128 bytes apart, groups of 8 rows 1024 bytes
// apart, and 16-byte chunk c of row r stored at chunk position c ^ (r % 8)
// (the 128-byte swizzle; the tile starts on a 1024-byte boundary).  As a
// K-major operand the rows are M (or N) and the 64 elements are K; as an
// MN-major operand the rows are K and the 64 elements are N, with further
// 64-element slices of N `lbo` bytes apart.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "kvq_ptx.cuh"

namespace kvq {

// Byte offset of 16-bit element (row r, column k < 64) in a swizzled tile.
__device__ __forceinline__ uint32_t sw128_off(int r, int k)
{
    return static_cast<uint32_t>(r * 128 + ((((k >> 3) ^ (r & 7))) << 4) + (k & 7) * 2);
}

// Byte offset of 16-byte chunk c (elements 8c .. 8c + 7) of row r.
__device__ __forceinline__ uint32_t sw128_chunk(int r, int c)
{
    return static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) << 4));
}

// Shared-memory matrix descriptor: start address, leading-dimension byte
// offset (the distance between 64-element slices of an MN-major operand;
// unused for K-major), stride byte offset (between groups of 8 rows),
// descriptor version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t umma_desc(uint32_t smem_byte_addr, uint32_t lbo, uint32_t sbo)
{
    uint64_t d = static_cast<uint64_t>((smem_byte_addr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

// Instruction descriptor of kind::f16 with f16 A and B and an fp32
// accumulator: M x N, A K-major, B K-major or (b_mn) MN-major.
__host__ __device__ constexpr uint32_t umma_idesc_f16(int m, int n, bool b_mn)
{
    return (1u << 4) | (b_mn ? (1u << 16) : 0u) | (static_cast<uint32_t>(n >> 3) << 17) |
           (static_cast<uint32_t>(m >> 4) << 24);
}

// D (tensor memory) = A B (+ D if accumulate), issued by one thread.
__device__ __forceinline__ void umma_f16(uint32_t tmem_d, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         bool accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n"
                 ::"r"(tmem_d), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u)
                 : "memory");
}

// D (tensor memory) = A B (+ D), A from tensor memory (lane m = row m;
// 32-bit column c holds k = 2c in its low half and 2c + 1 in its high half),
// B from shared memory.
__device__ __forceinline__ void umma_f16_ts(uint32_t tmem_d, uint32_t tmem_a, uint64_t b_desc, uint32_t idesc,
                                            bool accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n"
                 ::"r"(tmem_d), "r"(tmem_a), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u)
                 : "memory");
}

// Arrive once on `bar` when every tensor-core operation this thread issued
// before has completed.
__device__ __forceinline__ void umma_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 ::"r"(smem_addr(bar)) : "memory");
}

// Allocation by one whole warp; the tensor-memory address lands in *slot.
__device__ __forceinline__ void tmem_alloc(uint32_t *slot, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(smem_addr(slot)), "r"(ncols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// One look at phase `parity` of `bar` that may suspend the thread in
// hardware for up to `hint_ns` while the phase is incomplete: a waiting warp
// takes no issue slots from the warps that work beside it.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t *bar, uint32_t parity, uint32_t hint_ns)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(smem_addr(bar)), "r"(parity), "r"(hint_ns)
                 : "memory");
    return ok != 0;
}

// Plain arrival on an mbarrier (release semantics at CTA scope).
__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Named barrier `id` for `count` threads (whole warps).
__device__ __forceinline__ void named_barrier_sync(uint32_t id, uint32_t count)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ void tmem_fence_before_sync()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tmem_fence_after_sync()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 16 consecutive 32-bit columns of this thread's lane (the warp reads lanes
// 32 (warp % 4) .. + 31; taddr carries that lane base and the first column).
// The wait for the load is part of the same statement, so no use of the
// registers can be scheduled before the data has arrived.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 "
                 "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
                 "tcgen05.wait::ld.sync.aligned;"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                   "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
                   "=r"(r[14]), "=r"(r[15])
                 : "r"(taddr)
                 : "memory");
}

// 8 columns; the store's wait is part of the same statement.
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};\n\t"
                 "tcgen05.wait::st.sync.aligned;"
                 ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
                   "r"(r[7])
                 : "memory");
}

// The store's wait is part of the same statement.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 "
                 "[%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};\n\t"
                 "tcgen05.wait::st.sync.aligned;"
                 ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
                   "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
                   "r"(r[15])
                 : "memory");
}


// Packed fp32 pairs (sm_100 family): two IEEE round-to-nearest operations per instruction.
__device__ __forceinline__ uint64_t f2_pack(float a, float b)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float &a, float &b)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b)
{
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b)
{
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

} // namespace kvq
