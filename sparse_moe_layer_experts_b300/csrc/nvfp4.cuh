// NVFP4 numerics: E2M1 values with one E4M3 scale per 16 elements and an
// FP32 scale per matrix.  The Beam pages name the format only ("most
// parameters in 4 bits" for Blackwell: "Reflection Beam 1.0", section on
// hardware requirements); the recipe below is a reading:
//   gs = amax|W| / (6*448) per matrix (1 for an all-zero matrix)
//   sf = e4m3_rn_satfinite((amax16 / 6) / gs)
//   q  = e2m1_rn_satfinite(v / (sf * gs)),   0 when sf == 0
// Activations use the same blocks with gs = 1.  q * sf always fits an FP16
// exactly (at most 6 significant bits, magnitude in [2^-10, 2688]).
#pragma once

#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

namespace beam {

__device__ __forceinline__ uint32_t e4m3_code(float v)
{
    return (uint32_t)__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3);
}

__device__ __forceinline__ float e4m3_value(uint32_t c)
{
    __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)c, __NV_E4M3);
    return __half2float(__half(h));
}

// Block scale of 16 values whose largest magnitude is bmax, for global
// scale gs: returns the E4M3 code; *sfv its value.
__device__ __forceinline__ uint32_t nvfp4_block_scale(float bmax, float gs, float *sfv)
{
    const uint32_t c = e4m3_code(__fdiv_rn(__fdiv_rn(bmax, 6.0f), gs));
    *sfv = e4m3_value(c);
    return c;
}

// v / s rounded to nearest FP32 for an E4M3 scale value s > 0, given
// r = RN(1/s): one correction step after the reciprocal product (Markstein's
// method: q0 = RN(v r); the FMA gives the exact remainder v - s q0; q =
// RN(q0 + rem r)).  Over all 126 positive E4M3 values s it equals the
// correctly rounded quotient wherever that quotient decides an E2M1 code
// (every FP32 v within 64 ulps of a code boundary, checked exhaustively in
// exact arithmetic), so codes taken from it match codes from v / s.
__device__ __forceinline__ float div_by_scale(float v, float s, float r)
{
    const float q0 = __fmul_rn(v, r);
    const float rem = __fmaf_rn(-q0, s, v);
    return __fmaf_rn(rem, r, q0);
}

// Eight E2M1 codes, element i in bits 4i..4i+3 (sign in the top bit of each
// code): the hardware conversion rounds to the nearest of 0, 0.5, 1, 1.5, 2,
// 3, 4, 6 with ties to the even code and saturates at 6.
__device__ __forceinline__ uint32_t e2m1x8(const float *q)
{
    uint32_t out;
    asm("{\n\t.reg .b8 c0, c1, c2, c3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 c0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 c1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 c2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 c3, %8, %7;\n\t"
        "mov.b32 %0, {c0, c1, c2, c3};\n\t}"
        : "=r"(out)
        : "f"(q[0]), "f"(q[1]), "f"(q[2]), "f"(q[3]), "f"(q[4]), "f"(q[5]), "f"(q[6]),
          "f"(q[7]));
    return out;
}

// Quantise 16 values with global scale 1: 8 code bytes (even element in the
// low nibble) as two words, and the E4M3 scale code.
__device__ __forceinline__ uint32_t nvfp4_quant16(const float (&v)[16], uint32_t *lo, uint32_t *hi)
{
    float bmax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i)
        bmax = fmaxf(bmax, fabsf(v[i]));
    float sfv;
    const uint32_t sc = nvfp4_block_scale(bmax, 1.0f, &sfv);
    if (sfv == 0.0f) {
        *lo = 0u;
        *hi = 0u;
        return sc;
    }
    const float r = __frcp_rn(sfv);
    float q[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
        q[i] = div_by_scale(v[i], sfv, r);
    *lo = e2m1x8(q);
    *hi = e2m1x8(q + 8);
    return sc;
}

// MXFP8 (OCP microscaling, E4M3 elements): shared exponent of a 32-block
// with largest magnitude amax: floor(log2(amax)) - 8 clamped to [-127, 127],
// -127 for an all-zero block.  The scale byte is E + 127.
__device__ __forceinline__ int mx_shared_exp(float amax)
{
    if (!(amax > 0.0f))
        return -127;
    int ex;
    frexpf(amax, &ex);  // amax = m * 2^ex, m in [0.5, 1)
    return max(-127, min(127, ex - 1 - 8));
}

// 2^-e for a shared exponent e in [-127, 119] (the range mx_shared_exp
// gives for finite FP32 blocks): a normal FP32 power of two
__device__ __forceinline__ float mx_inv_scale(int e)
{
    return __int_as_float((127 - e) << 23);
}

// Four E4M3 codes of v * 2^-e (an exact power-of-two scaling, correctly
// rounded where it leaves the normal range), round to nearest even,
// saturating; element i in byte i.
__device__ __forceinline__ uint32_t mx_code4(const float *v, float inv)
{
    const __nv_fp8x2_storage_t a = __nv_cvt_float2_to_fp8x2(
        make_float2(__fmul_rn(v[0], inv), __fmul_rn(v[1], inv)), __NV_SATFINITE, __NV_E4M3);
    const __nv_fp8x2_storage_t b = __nv_cvt_float2_to_fp8x2(
        make_float2(__fmul_rn(v[2], inv), __fmul_rn(v[3], inv)), __NV_SATFINITE, __NV_E4M3);
    return (uint32_t)a | ((uint32_t)b << 16);
}

// Token chunks: an expert's n rows are split into nc near-equal chunks,
// chunk c holding rows [floor(c*n/nc), floor((c+1)*n/nc)) (the N tiles of
// the grouped GEMMs).  Returns the chunk of row i (0-based inside the
// expert), the largest c with floor(c*n/nc) <= i, and *j, the row's position
// in it.
__device__ __forceinline__ int nvfp4_chunk_of_row(int i, int n, int nc, int *j)
{
    const int c = (int)((((long long)i + 1) * nc - 1) / n);
    *j = i - (int)(((long long)c * n) / nc);
    return c;
}

// Byte offset, inside one 512-byte scale atom (128 rows x 4 scales), of the
// 4 scales of row j: row j = m0 + 32*m1 sits at 16*m0 + 4*m1, the order in
// which tcgen05.cp 32x128b.warpx4 hands the rows to the tensor core.
__device__ __forceinline__ int nvfp4_atom_offset(int j)
{
    return 16 * (j & 31) + 4 * (j >> 5);
}

}  // namespace beam
