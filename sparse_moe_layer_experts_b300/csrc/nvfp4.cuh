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

// Nearest E2M1 code (ties to the even mantissa bit, saturating at 6, sign
// kept in bit 3).  Thresholds are the midpoints of 0, .5, 1, 1.5, 2, 3, 4, 6.
__device__ __forceinline__ uint32_t e2m1_code(float v)
{
    const float a = fabsf(v);
    uint32_t c;
    if (a <= 0.25f)
        c = 0;
    else if (a < 0.75f)
        c = 1;
    else if (a <= 1.25f)
        c = 2;
    else if (a < 1.75f)
        c = 3;
    else if (a <= 2.5f)
        c = 4;
    else if (a < 3.5f)
        c = 5;
    else if (a <= 5.0f)
        c = 6;
    else
        c = 7;
    return c | (signbit(v) ? 8u : 0u);
}

__device__ __forceinline__ float e2m1_value(uint32_t c)
{
    // magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6 built as FP32 bit patterns:
    // exponent 126 + (m >> 1), mantissa bit (m & 1) for m >= 2
    const uint32_t m = c & 7u;
    const uint32_t bits =
        (m == 0u) ? 0u : ((126u + (m >> 1)) << 23) | ((m >= 2u ? (m & 1u) : 0u) << 22);
    return __uint_as_float(bits | ((c & 8u) << 28));
}

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

// E2M1 code of one value of a block with scale value sfv (global scale 1):
// 0 when the block scale is 0.
__device__ __forceinline__ uint32_t nvfp4_code(float v, float sfv)
{
    return sfv == 0.0f ? 0u : e2m1_code(__fdiv_rn(v, sfv));
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
    uint32_t a = 0, b = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        a |= nvfp4_code(v[i], sfv) << (4 * i);
        b |= nvfp4_code(v[i + 8], sfv) << (4 * i);
    }
    *lo = a;
    *hi = b;
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

// E4M3 code of v / 2^e (exact scaling), round to nearest even, saturating
__device__ __forceinline__ uint32_t mx_code(float v, int e)
{
    return (uint32_t)__nv_cvt_float_to_fp8(ldexpf(v, -e), __NV_SATFINITE, __NV_E4M3);
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
