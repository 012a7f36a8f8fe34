// kda_tc.cuh -- sm_103a tensor-core helpers: tcgen05 (UMMA, TMEM), mbarrier, shared-memory
// matrix descriptors and the warp-level mma.sync used for the 16x16 in-chunk products.
//
// Operand layouts used by this library (bf16, "K-major" = the reduction dimension contiguous):
//   SW128  : rows of 64 elements (128 B); 8-row atoms of 1024 B; within an atom the 16-byte chunk
//            index is XORed with (row % 8).  A K extent of 128 is two such blocks ("K-blocks")
//            stored one after the other.  Descriptor: SBO = 1024 B, layout type SWIZZLE_128B.
//            The k-th group of 16 elements inside a K-block is addressed by advancing the
//            descriptor's start address by 32 B (the hardware applies the XOR on the final address).
//   NONE   : rows of 16 elements as two 8x8 "core matrices" (8 rows x 16 B, 128 B contiguous);
//            the K-direction core-matrix stride (LBO) is 128 B and the 8-row-group stride (SBO)
//            is 256 B.
// Accumulators are fp32 in tensor memory: for M = 128 and one CTA, row m of D is TMEM lane m and
// column n is TMEM column (base + n).  A warp can read only the 32 lanes of its quarter (warp % 4).
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace kda {
namespace tc {

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// ---------------------------------------------------------------- layouts (byte offsets)

// SW128 K-major tile with R rows; element (r, k), k < 128.
__host__ __device__ __forceinline__ uint32_t sw128_off(int r, int k, int R)
{
    const int kb = k >> 6, kk = k & 63;
    return (uint32_t)(kb * R * 128 + (r >> 3) * 1024 + (r & 7) * 128 + (((kk >> 3) ^ (r & 7)) << 4) + (kk & 7) * 2);
}

// Byte offset of the 16-byte chunk holding elements (r, 8*ch .. 8*ch+7) of an SW128 tile.
__host__ __device__ __forceinline__ uint32_t sw128_chunk_off(int r, int ch, int R)
{
    const int kb = ch >> 3, cc = ch & 7;
    return (uint32_t)(kb * R * 128 + (r >> 3) * 1024 + (r & 7) * 128 + ((cc ^ (r & 7)) << 4));
}

// NONE K-major tile with 16 columns; element (r, k), k < 16.
__host__ __device__ __forceinline__ uint32_t none_off(int r, int k)
{
    return (uint32_t)((r >> 3) * 256 + (k >> 3) * 128 + (r & 7) * 16 + (k & 7) * 2);
}

// ---------------------------------------------------------------- descriptors

__device__ __forceinline__ uint64_t desc_sw128(uint32_t addr)
{
    uint64_t d = 0;
    d |= (uint64_t)((addr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;            // leading byte offset: unused for swizzled K-major
    d |= (uint64_t)(1024 >> 4) << 32;  // stride byte offset: one 8-row atom
    d |= (uint64_t)1 << 46;            // descriptor version for this architecture
    d |= (uint64_t)2 << 61;            // SWIZZLE_128B
    return d;
}

__device__ __forceinline__ uint64_t desc_none(uint32_t addr)
{
    uint64_t d = 0;
    d |= (uint64_t)((addr & 0x3FFFFu) >> 4);
    d |= (uint64_t)(128 >> 4) << 16;   // K-direction core-matrix stride
    d |= (uint64_t)(256 >> 4) << 32;   // 8-row-group stride
    d |= (uint64_t)1 << 46;
    return d;                          // layout type 0: no swizzle
}

// No-swizzle K-major operand with a K-direction core-matrix stride of `lbo` bytes and an
// 8-row-group stride of `sbo` bytes (rows of 32 elements: lbo = 128, sbo = 512).
__device__ __forceinline__ uint64_t desc_none_strided(uint32_t addr, uint32_t lbo, uint32_t sbo)
{
    uint64_t d = 0;
    d |= (uint64_t)((addr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    return d;
}

// kind::f16 instruction descriptor: bf16 A and B (K-major), fp32 accumulator, M x N.
__host__ __device__ __forceinline__ uint32_t idesc_bf16(int M, int N)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// ---------------------------------------------------------------- tcgen05

__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)), "r"(ncols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols));
}

// D[tmem] (+)= A[smem] * B[smem]^T, issued by one thread.
__device__ __forceinline__ void umma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]^T, issued by one thread.  A (M = 128 rows) sits in tensor memory
// with row m in lane m and its 16-bit K elements packed in pairs (even k in the low half) along
// the columns: one K = 16 step occupies 8 columns.
__device__ __forceinline__ void umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on an mbarrier once all previously issued tcgen05 operations of this thread complete.
__device__ __forceinline__ void umma_commit(uint64_t* bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// Generic-proxy shared-memory writes become visible to the tensor core (async proxy).
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

#define KDA_TMEM_LD16(taddr, v)                                                                                   \
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, " \
                 "[%16];"                                                                                         \
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),     \
                   "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]),           \
                   "=r"(v[15])                                                                                    \
                 : "r"(taddr))

#define KDA_TMEM_LD8(taddr, v)                                                                                  \
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"                         \
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]) \
                 : "r"(taddr))

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Store 32-bit registers to this warp's 32 lanes of tensor memory, consecutive columns.
#define KDA_TMEM_ST8(taddr, v)                                                                       \
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), \
                 "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])  \
                 : "memory")

#define KDA_TMEM_ST16(taddr, v)                                                                             \
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14," \
                 "%15,%16};" ::"r"(taddr),                                                                   \
                 "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),      \
                 "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])  \
                 : "memory")

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

// Bounded wait for the phase with the given parity; returns false if the limit was reached.
// Each try parks the thread in hardware until the phase completes or `hint_ns` elapses, so a
// waiting thread issues a handful of instructions instead of spinning; at most max_iters tries.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t max_iters, uint32_t hint_ns = 20000u)
{
    uint32_t done = 0;
    for (uint32_t it = 0; it < max_iters && !done; ++it) {
        asm volatile(
            "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\tselp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
            : "memory");
    }
    return done != 0;
}

// Plain arrival (release semantics at CTA scope).
__device__ __forceinline__ void mbar_arrive(uint64_t* bar)
{
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Arrive on the barrier and add `bytes` to the transaction count it waits for.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

// ---------------------------------------------------------------- TMA (tensor map in kernel parameters)

// 3-D tiled bulk copy global -> shared, completion counted on `bar` in bytes.
__device__ __forceinline__ void tma_load_3d(void* dst, const void* tmap, int c0, int c1, int c2, uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cta.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
            smem_u32(dst)),
        "l"(tmap), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
        : "memory");
}

// ---------------------------------------------------------------- plain bulk copies (TMA engine, no tensor map)

// Contiguous global -> shared copy of `bytes` (multiple of 16, both addresses 16-byte aligned),
// completion counted on `bar` in bytes.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

// ---------------------------------------------------------------- warp-level MMA (16x8x16, bf16 -> fp32)

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

}  // namespace tc
}  // namespace kda
