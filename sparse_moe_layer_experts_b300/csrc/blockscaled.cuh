// Block-scaled tensor-core pieces shared by the NVFP4 / MXFP8 grouped GEMMs:
// bulk copies of scale atoms, scale copies into tensor memory, instruction
// descriptors and the block-scaled MMAs (tcgen05 kind::mxf4nvf4 and
// kind::mxf8f6f4, one CTA).
#pragma once

#include "common.cuh"

namespace beam {

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                         uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// Shared-memory descriptor of a 32-row x 16-byte scale atom slice without
// swizzle: core matrices of 8 rows x 16 bytes, 128 bytes apart.
__device__ __forceinline__ uint64_t smem_desc_atom(uint32_t saddr)
{
    uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)(128u >> 4) << 16;
    d |= (uint64_t)(128u >> 4) << 32;
    d |= (uint64_t)1 << 46;
    return d;
}

// 32 rows x 128 bits from shared memory into 4 TMEM columns, replicated to
// all four 32-lane quarters.
__device__ __forceinline__ void tmem_cp_atom(uint32_t taddr, uint32_t saddr)
{
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr),
                 "l"(smem_desc_atom(saddr))
                 : "memory");
}

// Instruction descriptor: E2M1 x E2M1 (format 1 each), UE4M3 scales, both
// K-major, FP32 accumulator.
__device__ __forceinline__ uint32_t idesc_nvf4(uint32_t m, uint32_t n)
{
    return (1u << 7) | (1u << 10) | ((n >> 3) << 17) | ((m >> 4) << 24);
}

__device__ __forceinline__ void mma_nvf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                         uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, "
        "[%5], [%6], p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
        : "memory");
}

// MXFP8: E4M3 x E4M3 (format 0), UE8M0 scales (bit 23), both K-major, FP32
// accumulator; the scale-factor ids (bits 29-30 for A, 4-5 for B) are OR-ed
// in per MMA.
__device__ __forceinline__ uint32_t idesc_mx8(uint32_t m, uint32_t n)
{
    return (1u << 23) | ((n >> 3) << 17) | ((m >> 4) << 24);
}

__device__ __forceinline__ void mma_mx8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                        uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                        uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, "
        "[%5], [%6], p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
        : "memory");
}

// 32 lanes x 32 bit, 16 consecutive columns per thread, from registers into
// tensor memory (this warp's lane quarter).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void tmem_st_wait()
{
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ float silu_mul_f(float g, float u)
{
    return __fdividef(g, 1.0f + __expf(-g)) * u;
}

}  // namespace beam
