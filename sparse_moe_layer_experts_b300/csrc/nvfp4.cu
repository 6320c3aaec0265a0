// NVFP4 weight quantisation (offline preparation of the expert weights).
//
// Layouts written (see beam_moe_quantize_nvfp4 in the header):
//   packed   [n_mat, rows, cols/2]  two E2M1 codes per byte, even element in
//                                   the low nibble
//   block_sf [n_mat, rows/128, cols/64, 512]  the E4M3 scale of elements
//            [16b, 16b+16) of row r sits in tile (r/128, b/4) at byte
//            16*(r%32) + 4*((r%128)/32) + b%4: the 512 scales one 128x64 GEMM
//            tile needs are contiguous, in the row order in which the tensor
//            core's scale copy (tcgen05.cp 32x128b.warpx4) takes them
//   global   [n_mat] FP32
#include "common.cuh"
#include "internal.h"
#include "nvfp4.cuh"

namespace beam {

namespace {

// One CTA per matrix: amax over rows*cols bf16 values, then the global scale.
__global__ void __launch_bounds__(1024)
nvfp4_global_scale_kernel(const uint16_t *__restrict__ w, int64_t per_mat, float *__restrict__ gs)
{
    __shared__ float red[32];
    const uint16_t *wm = w + (size_t)blockIdx.x * per_mat;
    float m = 0.0f;
    for (int64_t i = (int64_t)threadIdx.x * 8; i < per_mat; i += 1024 * 8) {
        const uint4 q = *reinterpret_cast<const uint4 *>(wm + i);
        const uint32_t v[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            m = fmaxf(m, fabsf(bf16_bits_to_f32(v[p] & 0xFFFFu)));
            m = fmaxf(m, fabsf(bf16_bits_to_f32(v[p] >> 16)));
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
    if ((threadIdx.x & 31) == 0)
        red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x < 32) {
        m = red[threadIdx.x];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
        if (threadIdx.x == 0)
            gs[blockIdx.x] = (m > 0.0f) ? __fdiv_rn(m, 6.0f * 448.0f) : 1.0f;
    }
}

// One thread per 16-element block.
__global__ void __launch_bounds__(256)
nvfp4_quantize_kernel(const uint16_t *__restrict__ w, int64_t n_blocks, int rows, int cols,
                      const float *__restrict__ gs, uint8_t *__restrict__ packed,
                      uint8_t *__restrict__ block_sf)
{
    const int64_t b = (int64_t)blockIdx.x * 256 + threadIdx.x;
    if (b >= n_blocks)
        return;
    const int bpr = cols / 16;
    const int64_t per_mat = (int64_t)rows * bpr;
    const int64_t mat = b / per_mat;
    const int64_t rem = b - mat * per_mat;
    const int r = (int)(rem / bpr), cb = (int)(rem % bpr);
    const int64_t elem = (mat * rows + r) * (int64_t)cols + (int64_t)cb * 16;

    const uint4 q0 = *reinterpret_cast<const uint4 *>(w + elem);
    const uint4 q1 = *reinterpret_cast<const uint4 *>(w + elem + 8);
    const uint32_t raw[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
    float v[16];
    float bmax = 0.0f;
#pragma unroll
    for (int p = 0; p < 8; ++p) {
        v[2 * p] = bf16_bits_to_f32(raw[p] & 0xFFFFu);
        v[2 * p + 1] = bf16_bits_to_f32(raw[p] >> 16);
    }
#pragma unroll
    for (int i = 0; i < 16; ++i)
        bmax = fmaxf(bmax, fabsf(v[i]));
    const float g = gs[mat];
    float sfv;
    const uint32_t sc = nvfp4_block_scale(bmax, g, &sfv);
    const float den = __fmul_rn(sfv, g);
    uint32_t lo = 0, hi = 0;
    if (sfv != 0.0f) {
        float q[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
            q[i] = __fdiv_rn(v[i], den);
        lo = e2m1x8(q);
        hi = e2m1x8(q + 8);
    }
    *reinterpret_cast<uint2 *>(packed + elem / 2) = make_uint2(lo, hi);
    const int64_t tile = (mat * (rows / 128) + r / 128) * (cols / 64) + cb / 4;
    block_sf[tile * 512 + nvfp4_atom_offset(r % 128) + (cb % 4)] = (uint8_t)sc;
}

// MXFP8: one thread per 32-element block (codes E4M3, scale byte E + 127 in
// the tile of 128 rows x 128 columns at the atom offset of row r % 128).
__global__ void __launch_bounds__(256)
mxfp8_quantize_kernel(const uint16_t *__restrict__ w, int64_t n_blocks, int rows, int cols,
                      uint8_t *__restrict__ codes, uint8_t *__restrict__ block_sf)
{
    const int64_t b = (int64_t)blockIdx.x * 256 + threadIdx.x;
    if (b >= n_blocks)
        return;
    const int bpr = cols / 32;
    const int64_t per_mat = (int64_t)rows * bpr;
    const int64_t mat = b / per_mat;
    const int64_t rem = b - mat * per_mat;
    const int r = (int)(rem / bpr), cb = (int)(rem % bpr);
    const int64_t elem = (mat * rows + r) * (int64_t)cols + (int64_t)cb * 32;
    float v[32];
    float amax = 0.0f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint4 u = *reinterpret_cast<const uint4 *>(w + elem + 8 * q);
        const uint32_t raw[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            v[8 * q + 2 * p] = bf16_bits_to_f32(raw[p] & 0xFFFFu);
            v[8 * q + 2 * p + 1] = bf16_bits_to_f32(raw[p] >> 16);
        }
    }
#pragma unroll
    for (int i = 0; i < 32; ++i)
        amax = fmaxf(amax, fabsf(v[i]));
    const int e = mx_shared_exp(amax);
    const float inv = mx_inv_scale(e);
    uint32_t out[8];
#pragma unroll
    for (int q = 0; q < 8; ++q)
        out[q] = mx_code4(v + 4 * q, inv);
    uint4 *dst = reinterpret_cast<uint4 *>(codes + elem);
    dst[0] = make_uint4(out[0], out[1], out[2], out[3]);
    dst[1] = make_uint4(out[4], out[5], out[6], out[7]);
    const int64_t tile = (mat * (rows / 128) + r / 128) * (cols / 128) + cb / 4;
    block_sf[tile * 512 + nvfp4_atom_offset(r % 128) + (cb % 4)] = (uint8_t)(e + 127);
}

}  // namespace

// Activation rows (FP32, global scale 1), the rule the layer applies to x
// and h: NVFP4 one thread per 16-block, MXFP8 one thread per 32-block;
// scales row-major [rows, cols/16] (E4M3) or [rows, cols/32] (E8M0).
__global__ void __launch_bounds__(256)
quantize_act_nvfp4_kernel(const float *__restrict__ x, int64_t n_blocks, uint8_t *__restrict__ codes,
                          uint8_t *__restrict__ sf)
{
    const int64_t b = (int64_t)blockIdx.x * 256 + threadIdx.x;
    if (b >= n_blocks)
        return;
    const float4 *src = reinterpret_cast<const float4 *>(x) + 4 * b;
    float v[16];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float4 f = src[q];
        v[4 * q] = f.x;
        v[4 * q + 1] = f.y;
        v[4 * q + 2] = f.z;
        v[4 * q + 3] = f.w;
    }
    uint32_t lo, hi;
    sf[b] = (uint8_t)nvfp4_quant16(v, &lo, &hi);
    reinterpret_cast<uint2 *>(codes)[b] = make_uint2(lo, hi);
}

__global__ void __launch_bounds__(256)
quantize_act_mxfp8_kernel(const float *__restrict__ x, int64_t n_blocks, uint8_t *__restrict__ codes,
                          uint8_t *__restrict__ sf)
{
    const int64_t b = (int64_t)blockIdx.x * 256 + threadIdx.x;
    if (b >= n_blocks)
        return;
    const float4 *src = reinterpret_cast<const float4 *>(x) + 8 * b;
    float v[32];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const float4 f = src[q];
        v[4 * q] = f.x;
        v[4 * q + 1] = f.y;
        v[4 * q + 2] = f.z;
        v[4 * q + 3] = f.w;
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i)
        amax = fmaxf(amax, fabsf(v[i]));
    const int e = mx_shared_exp(amax);
    const float inv = mx_inv_scale(e);
    uint32_t out[8];
#pragma unroll
    for (int q = 0; q < 8; ++q)
        out[q] = mx_code4(v + 4 * q, inv);
    uint4 *dst = reinterpret_cast<uint4 *>(codes) + 2 * b;
    dst[0] = make_uint4(out[0], out[1], out[2], out[3]);
    dst[1] = make_uint4(out[4], out[5], out[6], out[7]);
    sf[b] = (uint8_t)(e + 127);
}

cudaError_t launch_quantize_act(bool mx8, const float *x, int64_t rows, int cols, uint8_t *codes,
                                uint8_t *sf, cudaStream_t s)
{
    const int64_t n_blocks = rows * (int64_t)(cols / (mx8 ? 32 : 16));
    const unsigned grid = (unsigned)((n_blocks + 255) / 256);
    stage_begin(kNumStages, s);
    if (mx8)
        quantize_act_mxfp8_kernel<<<grid, 256, 0, s>>>(x, n_blocks, codes, sf);
    else
        quantize_act_nvfp4_kernel<<<grid, 256, 0, s>>>(x, n_blocks, codes, sf);
    stage_end(kNumStages, s);
    return cudaGetLastError();
}

cudaError_t launch_quantize_mxfp8(const uint16_t *w, int64_t n_mat, int rows, int cols,
                                  uint8_t *codes, uint8_t *block_sf, cudaStream_t s)
{
    const int64_t n_blocks = n_mat * rows * (int64_t)(cols / 32);
    stage_begin(kNumStages, s);
    mxfp8_quantize_kernel<<<(unsigned)((n_blocks + 255) / 256), 256, 0, s>>>(w, n_blocks, rows, cols,
                                                                             codes, block_sf);
    stage_end(kNumStages, s);
    return cudaGetLastError();
}

cudaError_t launch_quantize_nvfp4(const uint16_t *w, int64_t n_mat, int rows, int cols,
                                  uint8_t *packed, uint8_t *block_sf, float *global_sf,
                                  cudaStream_t s)
{
    stage_begin(kNumStages, s);
    nvfp4_global_scale_kernel<<<(unsigned)n_mat, 1024, 0, s>>>(w, (int64_t)rows * cols, global_sf);
    stage_end(kNumStages, s);
    const int64_t n_blocks = n_mat * rows * (int64_t)(cols / 16);
    stage_begin(kNumStages, s);
    nvfp4_quantize_kernel<<<(unsigned)((n_blocks + 255) / 256), 256, 0, s>>>(
        w, n_blocks, rows, cols, global_sf, packed, block_sf);
    stage_end(kNumStages, s);
    return cudaGetLastError();
}

}  // namespace beam
