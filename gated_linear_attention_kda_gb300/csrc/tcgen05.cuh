// tcgen05.cuh -- inline-PTX wrappers for the 5th-generation tensor core
// (tcgen05.*: tensor memory allocation, MMA, commit, TMEM load/store) and
// the shared-memory matrix / instruction descriptors, sm_103a.
//
// Descriptor conventions (checked on hardware against host references):
//  * K-major, no swizzle: 8-row x 16-byte core matrices; LBO = byte stride
//    between core matrices adjacent in K, SBO = stride between core matrices
//    adjacent in M/N.
//  * K-major, 128-byte swizzle: rows of 128 B, 8-row atoms (1024 B, 1024-B
//    aligned); SBO = 1024; K steps inside an atom advance the start address.
//  * MN-major, 128-byte swizzle: 64 (16-bit) MN elements per 128-B row, 8 K
//    rows per atom; LBO = stride between MN atoms, SBO = stride between K
//    atoms.
//  * A operand in tensor memory: lane = row, 32-bit columns along K (two
//    16-bit elements per column, one tf32 element per column).
#pragma once
#include <cstdint>

namespace kda {
namespace tc {

__device__ __forceinline__ void alloc(uint32_t dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// generic-proxy shared-memory writes -> visible to the tensor core (async proxy)
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Arrive on `bar` once every tcgen05 operation this thread issued so far has completed.
__device__ __forceinline__ void commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint32_t swizzle)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFF) >> 4);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFF) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFF) << 32;
    d |= static_cast<uint64_t>(1) << 46;  // descriptor version
    d |= static_cast<uint64_t>(swizzle & 7) << 61;
    return d;
}
constexpr uint32_t SWZ_NONE = 0, SWZ_128B = 2;

// Instruction descriptor for kind::f16 / kind::tf32 with fp32 accumulation.
// fmt: 0 = f16, 1 = bf16, 2 = tf32; a_mn / b_mn: operand stored MN-major.
__host__ __device__ constexpr uint32_t idesc(uint32_t fmt, uint32_t M, uint32_t N, uint32_t a_mn, uint32_t b_mn)
{
    return (1u << 4) | (fmt << 7) | (fmt << 10) | (a_mn << 15) | (b_mn << 16) | ((N >> 3) << 17) | ((M >> 4) << 24);
}
constexpr uint32_t F16 = 0, BF16 = 1, TF32 = 2;

// D[tmem] (+)= A[smem desc] * B[smem desc]
__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t id, uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
                 "l"(a), "l"(b), "r"(id), "r"(accumulate)
                 : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem desc]
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t id, uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
                 "r"(a_tmem), "l"(b), "r"(id), "r"(accumulate)
                 : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem desc], kind::tf32 (A holds fp32 words)
__device__ __forceinline__ void mma_ts_tf32(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t id, uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
                 "r"(a_tmem), "l"(b), "r"(id), "r"(accumulate)
                 : "memory");
}

// Warp-wide issue forms: executed by all 32 lanes of a warp together (convergent), the warp
// elects one lane -- always the lowest, so the same lane every time -- which issues the MMA or the
// commit. Operands computed by the whole warp stay warp-uniform, so no lane-0 branch is needed.
__device__ __forceinline__ void mma_ss_w(uint32_t d, uint64_t a, uint64_t b, uint32_t id, uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred e, p;\n\t.reg .b32 r;\n\telect.sync r|e, 0xffffffff;\n\t"
                 "setp.ne.u32 p, %4, 0;\n\t"
                 "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
                 "l"(a), "l"(b), "r"(id), "r"(accumulate)
                 : "memory");
}
__device__ __forceinline__ void mma_ts_w(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t id, uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred e, p;\n\t.reg .b32 r;\n\telect.sync r|e, 0xffffffff;\n\t"
                 "setp.ne.u32 p, %4, 0;\n\t"
                 "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
                 "r"(a_tmem), "l"(b), "r"(id), "r"(accumulate)
                 : "memory");
}
__device__ __forceinline__ void mma_ts_tf32_w(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t id, uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred e, p;\n\t.reg .b32 r;\n\telect.sync r|e, 0xffffffff;\n\t"
                 "setp.ne.u32 p, %4, 0;\n\t"
                 "@e tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
                 "r"(a_tmem), "l"(b), "r"(id), "r"(accumulate)
                 : "memory");
}
__device__ __forceinline__ void commit_w(uint32_t bar)
{
    asm volatile("{\n\t.reg .pred e;\n\t.reg .b32 r;\n\telect.sync r|e, 0xffffffff;\n\t"
                 "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
                 : "memory");
}

// 32 lanes (this warp's quarter) x 32 consecutive 32-bit columns
__device__ __forceinline__ void ld32(uint32_t taddr, uint32_t (&r)[32])
{
    tmem_check(taddr, 32);
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                 "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
                   "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
                   "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
                   "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
                 : "r"(taddr)
                 : "memory");
}
__device__ __forceinline__ void st32(uint32_t taddr, const uint32_t (&r)[32])
{
    tmem_check(taddr, 32);
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                 "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
                 "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
                 "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
                 "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
                 : "memory");
}
__device__ __forceinline__ void st16(uint32_t taddr, const uint32_t (&r)[16])
{
    tmem_check(taddr, 16);
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                 "%16};" ::"r"(taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
                 "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
                 : "memory");
}
__device__ __forceinline__ void st8(uint32_t taddr, const uint32_t (&r)[8])
{
    tmem_check(taddr, 8);
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]),
                 "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}
__device__ __forceinline__ void wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

}  // namespace tc
}  // namespace kda
