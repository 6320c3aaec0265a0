// Expert dispatch of the Beam MoE layer: histogram of the routed (token,
// slot) pairs, exclusive offsets, the expert-grouped permutation of token
// rows, and the deterministic weighted combine back to token order.
//
// The order of rows inside an expert's segment is token-ascending (the pages
// do not fix it; this order makes the permutation unique and reproducible).
// The combine sums the K expert outputs of a token in slot order k = 0..K-1
// ("Reflection Beam 1.0" (agentlenshq.com), section "Mixture of Experts":
// expert outputs are combined with the normalised router weights).
#include "common.cuh"
#include "internal.h"
#include "nvfp4.cuh"

namespace beam {

namespace {

// Exclusive scan over the E (<= 256) values held one per thread.
__device__ int block_exclusive_scan_256(int v, int *tmp, int *total)
{
    const int tid = threadIdx.x;
    tmp[tid] = v;
    __syncthreads();
    for (int off = 1; off < 256; off <<= 1) {
        const int add = (tid >= off) ? tmp[tid - off] : 0;
        __syncthreads();
        tmp[tid] += add;
        __syncthreads();
    }
    const int incl = tmp[tid];
    *total = tmp[255];
    __syncthreads();
    return incl - v;
}

// Expert e's row count `run` (thread e) -> counts, offsets (exclusive
// scan, offsets[E] = total) and chunk_start (exclusive scan of the chunks of
// chunk_rows rows per expert).  All 256 threads call it.
__device__ void scan_experts(int run, int E, int chunk_rows, int32_t *__restrict__ counts,
                             int32_t *__restrict__ offsets, int32_t *__restrict__ chunk_start,
                             int *tmp)
{
    const int e = threadIdx.x;
    if (e < E)
        counts[e] = run;
    int total = 0;
    const int off = block_exclusive_scan_256(e < E ? run : 0, tmp, &total);
    if (e < E)
        offsets[e] = off;
    if (e == 0)
        offsets[E] = total;
    const int nchunk = (e < E) ? (run + chunk_rows - 1) / chunk_rows : 0;
    int total_chunks = 0;
    const int cs = block_exclusive_scan_256(nchunk, tmp, &total_chunks);
    if (e < E)
        chunk_start[e] = cs;
    if (e == 0)
        chunk_start[E] = total_chunks;
}

// CTA = 8 warps = 256 tokens.  mask[w][e] has bit l set when token
// (warp w, lane l) routes to expert e; a pair's rank inside its expert and
// CTA is the number of earlier tokens (lower warp, or lower lane in the same
// warp) with that expert.
__global__ void __launch_bounds__(256)
hist_kernel(const int32_t *__restrict__ ids, int T, int K, int E, int32_t *__restrict__ local_rank,
            int32_t *__restrict__ cta_counts, int *status, int chunk_rows,
            int32_t *__restrict__ cta_base, int32_t *__restrict__ counts,
            int32_t *__restrict__ offsets, int32_t *__restrict__ chunk_start)
{
    __shared__ uint32_t mask[8][256];
    __shared__ int32_t prefix[8][256];
    __shared__ int tmp[256];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    for (int i = tid; i < 8 * 256; i += 256)
        (&mask[0][0])[i] = 0u;
    __syncthreads();
    const int t = blockIdx.x * kHistTokens + tid;
    if (t < T) {
        for (int k = 0; k < K; ++k) {
            const int e = ids[(size_t)t * K + k];
            if (e < 0 || e >= E) {
                atomicOr(status, kStatusDevice);
                continue;
            }
            atomicOr(&mask[warp][e], 1u << lane);
        }
    }
    __syncthreads();
    int run = 0;
    if (tid < E) {
        for (int w = 0; w < 8; ++w) {
            prefix[w][tid] = run;
            run += __popc(mask[w][tid]);
        }
        cta_counts[(size_t)blockIdx.x * E + tid] = run;
    }
    if (gridDim.x == 1) {
        // one histogram CTA (T <= 256 tokens): it also does the scan
        if (tid < E)
            cta_base[tid] = 0;
        scan_experts(run, E, chunk_rows, counts, offsets, chunk_start, tmp);
    }
    __syncthreads();
    if (t < T) {
        const uint32_t below = (1u << lane) - 1u;
        for (int k = 0; k < K; ++k) {
            const int e = ids[(size_t)t * K + k];
            int r = 0;
            if (e >= 0 && e < E)
                r = prefix[warp][e] + __popc(mask[warp][e] & below);
            local_rank[(size_t)t * K + k] = r;
        }
    }
}

// One CTA of 256 threads, thread e owns expert e.
__global__ void __launch_bounds__(256)
scan_kernel(const int32_t *__restrict__ cta_counts, int n_cta, int E, int chunk_rows,
            int32_t *__restrict__ cta_base, int32_t *__restrict__ counts,
            int32_t *__restrict__ offsets, int32_t *__restrict__ chunk_start)
{
    __shared__ int tmp[256];
    const int e = threadIdx.x;
    int run = 0;
    if (e < E) {
        for (int c = 0; c < n_cta; ++c) {
            const int v = cta_counts[(size_t)c * E + e];
            cta_base[(size_t)c * E + e] = run;
            run += v;
        }
    }
    scan_experts(run, E, chunk_rows, counts, offsets, chunk_start, tmp);
}

// CTA per token: place the token's K rows, then read the token's activations
// once (16-byte vectors) and write them to all K rows.  With QUANT (NVFP4
// layers) each 16-element block is quantised to NVFP4 (global scale 1) once:
// its 8 code bytes go to every row, its E4M3 scale into the row's token-chunk
// scale atom (chunks of <= 128 rows), and row_pos records the row's place
// (chunk * 256 + position) for the kernels that quantise h.
template <bool QUANT>
__global__ void __launch_bounds__(256)
permute_kernel(const uint16_t *__restrict__ x, const int32_t *__restrict__ ids,
               const int32_t *__restrict__ local_rank, const int32_t *__restrict__ cta_base,
               const int32_t *__restrict__ offsets, const int32_t *__restrict__ chunk_start,
               int T, int K, int E, int H, int32_t *__restrict__ row_of,
               int32_t *__restrict__ row_src, int32_t *__restrict__ row_pos,
               void *__restrict__ x_perm, uint8_t *__restrict__ x_sf)
{
    __shared__ int rows[32];
    __shared__ int pos[32];
    const int t = blockIdx.x;
    const int cta = t / kHistTokens;
    if (threadIdx.x < K) {
        const int k = threadIdx.x;
        int e = ids[(size_t)t * K + k];
        e = (e < 0 || e >= E) ? 0 : e;
        const int rank = cta_base[(size_t)cta * E + e] + local_rank[(size_t)t * K + k];
        const int row = offsets[e] + rank;
        rows[k] = row;
        row_of[(size_t)t * K + k] = row;
        row_src[row] = t;
        if constexpr (QUANT) {
            const int n = offsets[e + 1] - offsets[e];
            int j;
            const int c = nvfp4_chunk_of_row(rank, n, chunk_start[e + 1] - chunk_start[e], &j);
            pos[k] = (chunk_start[e] + c) * 128 + j;
            row_pos[row] = (chunk_start[e] + c) * 256 + j;
        }
    }
    __syncthreads();
    const uint4 *src = reinterpret_cast<const uint4 *>(x + (size_t)t * H);
    if constexpr (!QUANT) {
        uint16_t *xp = static_cast<uint16_t *>(x_perm);
        for (int i = threadIdx.x; i < H / 8; i += 256) {
            const uint4 v = src[i];
            for (int k = 0; k < K; ++k)
                reinterpret_cast<uint4 *>(xp + (size_t)rows[k] * H)[i] = v;
        }
    } else {
        // NVFP4: codes [rows, H/2] and the scales in token-chunk atoms
        // [chunk, H/64, 512]; each 4 lanes (one 64-block) merge their scale
        // bytes into one word
        uint8_t *xq = static_cast<uint8_t *>(x_perm);
        const int nblk = H / 16;
        const int lane = threadIdx.x & 31;
        for (int blk0 = threadIdx.x & ~31; blk0 < nblk; blk0 += 256) {
            const int blk = blk0 + lane;
            const unsigned live = __ballot_sync(0xFFFFFFFFu, blk < nblk);
            if (blk >= nblk)
                break;
            const uint4 q0 = src[2 * blk], q1 = src[2 * blk + 1];
            const uint32_t raw[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
            float v[16];
#pragma unroll
            for (int p = 0; p < 8; ++p) {
                v[2 * p] = bf16_bits_to_f32(raw[p] & 0xFFFFu);
                v[2 * p + 1] = bf16_bits_to_f32(raw[p] >> 16);
            }
            uint32_t lo, hi;
            uint32_t word = nvfp4_quant16(v, &lo, &hi) << (8 * (blk & 3));
            word |= __shfl_xor_sync(live, word, 1);
            word |= __shfl_xor_sync(live, word, 2);
            for (int k = 0; k < K; ++k) {
                *reinterpret_cast<uint2 *>(xq + (size_t)rows[k] * (H / 2) + 8 * blk) =
                    make_uint2(lo, hi);
                if ((blk & 3) == 0) {
                    const int ps = pos[k];
                    *reinterpret_cast<uint32_t *>(
                        x_sf + ((size_t)(ps >> 7) * (H / 64) + (blk >> 2)) * 512 +
                        nvfp4_atom_offset(ps & 127)) = word;
                }
            }
        }
    }
}

// NVFP4 activation quantisation of an FP32 matrix [rows, cols] (global scale
// 1): codes [rows, cols/2], and the scales at the row's row_pos
// (chunk * 256 + j) in token-chunk atoms [chunk, cols/64, 512] (chunks of
// <= 128 rows).  One thread per 16-block.
__global__ void __launch_bounds__(256)
quantize_rows_kernel(const float *__restrict__ in, int64_t n_blocks, int cols,
                     const int32_t *__restrict__ row_pos, uint8_t *__restrict__ codes,
                     uint8_t *__restrict__ sf)
{
    const int64_t b = (int64_t)blockIdx.x * 256 + threadIdx.x;
    const unsigned live = __ballot_sync(0xFFFFFFFFu, b < n_blocks);
    if (b >= n_blocks)
        return;
    const float4 *src = reinterpret_cast<const float4 *>(in) + 4 * b;
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
    const int bpr = cols / 16;
    const int blk = (int)(b % bpr);
    uint32_t word = nvfp4_quant16(v, &lo, &hi) << (8 * (blk & 3));
    word |= __shfl_xor_sync(live, word, 1);
    word |= __shfl_xor_sync(live, word, 2);
    reinterpret_cast<uint2 *>(codes)[b] = make_uint2(lo, hi);
    if ((blk & 3) == 0) {
        const int ps = row_pos[b / bpr];
        const size_t unit = (size_t)(ps >> 8) * (cols / 64) + (blk >> 2);
        *reinterpret_cast<uint32_t *>(sf + unit * 512 + nvfp4_atom_offset(ps & 255)) = word;
    }
}

__global__ void __launch_bounds__(256)
rows_kernel(const int32_t *__restrict__ ids, const int32_t *__restrict__ local_rank,
            const int32_t *__restrict__ cta_base, const int32_t *__restrict__ offsets, int T, int K,
            int E, int32_t *__restrict__ row_of)
{
    const size_t i = (size_t)blockIdx.x * 256 + threadIdx.x;
    if (i >= (size_t)T * K)
        return;
    const int t = (int)(i / K);
    int e = ids[i];
    e = (e < 0 || e >= E) ? 0 : e;
    row_of[i] = offsets[e] + cta_base[(size_t)(t / kHistTokens) * E + e] + local_rank[i];
}

// acc[0..7] += w[k] * y[row k][8i .. 8i+8) for k = 0 .. K-1 in ascending
// order (an FP32 FMA chain per element).  The rows' 16-byte vectors are
// loaded eight at a time before their FMAs, so a thread waits for one L2
// round trip per eight rows instead of one per row.
__device__ __forceinline__ void combine_vec8(const uint16_t *__restrict__ y, const float *ws,
                                             const int *rs, int K, int H, int i, float (&acc)[8])
{
    for (int k0 = 0; k0 < K; k0 += 8) {
        uint4 q[8];
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
            if (k0 + kk < K)
                q[kk] = reinterpret_cast<const uint4 *>(y + (size_t)rs[k0 + kk] * H)[i];
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            if (k0 + kk < K) {
                const float wk = ws[k0 + kk];
                const uint32_t v[4] = {q[kk].x, q[kk].y, q[kk].z, q[kk].w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    acc[2 * j] = __fmaf_rn(wk, bf16_bits_to_f32(v[j] & 0xFFFFu), acc[2 * j]);
                    acc[2 * j + 1] = __fmaf_rn(wk, bf16_bits_to_f32(v[j] >> 16), acc[2 * j + 1]);
                }
            }
        }
    }
}

// out[t,:] = bf16( sum_{k=0..K-1} w[t,k] * y[row_of[t,k], :] ), FP32 FMA chain
// in ascending k over the bf16 expert outputs y.
__global__ void __launch_bounds__(256)
combine_kernel(const uint16_t *__restrict__ y, const float *__restrict__ w,
               const int32_t *__restrict__ row_of, int T, int K, int H, uint16_t *__restrict__ out)
{
    __shared__ float ws[32];
    __shared__ int rs[32];
    const int t = blockIdx.x;
    if (threadIdx.x < K) {
        ws[threadIdx.x] = w[(size_t)t * K + threadIdx.x];
        rs[threadIdx.x] = row_of[(size_t)t * K + threadIdx.x];
    }
    __syncthreads();
    const int nvec = H / 8;
    for (int i = threadIdx.x; i < nvec; i += 256) {
        float acc[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            acc[j] = 0.0f;
        combine_vec8(y, ws, rs, K, H, i, acc);
        uint4 o;
        o.x = pack_bf16x2(acc[0], acc[1]);
        o.y = pack_bf16x2(acc[2], acc[3]);
        o.z = pack_bf16x2(acc[4], acc[5]);
        o.w = pack_bf16x2(acc[6], acc[7]);
        reinterpret_cast<uint4 *>(out + (size_t)t * H)[i] = o;
    }
}


// ---- MXFP8 activations: E4M3 codes, one shared power-of-two scale per
// 32 elements (a 32-block is 4 lanes x 8 elements; the lanes take its max
// with shuffles), scales in token-chunk atoms [chunk, cols/128, 512] at the
// row's place j in its chunk: byte atom_offset(j) + (32-block % 4).

// 8 values of lane group member -> 8 code bytes; *e the block's exponent
__device__ __forceinline__ uint2 mx_quant8(const float (&v)[8], unsigned live, int *e)
{
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i)
        amax = fmaxf(amax, fabsf(v[i]));
    amax = fmaxf(amax, __shfl_xor_sync(live, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(live, amax, 2));
    *e = mx_shared_exp(amax);
    const float inv = mx_inv_scale(*e);
    return make_uint2(mx_code4(v, inv), mx_code4(v + 4, inv));
}

// CTA per token: place its K rows (as permute_kernel), then quantise x once
// and write the codes to every row and the scales to every row's chunk atom.
__global__ void __launch_bounds__(256)
permute_mx8_kernel(const uint16_t *__restrict__ x, const int32_t *__restrict__ ids,
                   const int32_t *__restrict__ local_rank, const int32_t *__restrict__ cta_base,
                   const int32_t *__restrict__ offsets, const int32_t *__restrict__ chunk_start,
                   int T, int K, int E, int H, int32_t *__restrict__ row_of,
                   int32_t *__restrict__ row_src, int32_t *__restrict__ row_pos,
                   uint8_t *__restrict__ xq, uint8_t *__restrict__ x_sf)
{
    __shared__ int rows[32];
    __shared__ int pos[32];
    const int t = blockIdx.x;
    const int cta = t / kHistTokens;
    if (threadIdx.x < K) {
        const int k = threadIdx.x;
        int e = ids[(size_t)t * K + k];
        e = (e < 0 || e >= E) ? 0 : e;
        const int rank = cta_base[(size_t)cta * E + e] + local_rank[(size_t)t * K + k];
        const int row = offsets[e] + rank;
        rows[k] = row;
        row_of[(size_t)t * K + k] = row;
        row_src[row] = t;
        int j;
        const int c = nvfp4_chunk_of_row(rank, offsets[e + 1] - offsets[e],
                                         chunk_start[e + 1] - chunk_start[e], &j);
        pos[k] = (chunk_start[e] + c) * 256 + j;
        row_pos[row] = pos[k];
    }
    __syncthreads();
    const uint4 *src = reinterpret_cast<const uint4 *>(x + (size_t)t * H);
    const int nvec = H / 8;
    const int lane = threadIdx.x & 31;
    for (int v0 = threadIdx.x & ~31; v0 < nvec; v0 += 256) {
        const int vi = v0 + lane;
        const unsigned live = __ballot_sync(0xFFFFFFFFu, vi < nvec);
        if (vi >= nvec)
            break;
        const uint4 q = src[vi];
        const uint32_t raw[4] = {q.x, q.y, q.z, q.w};
        float v[8];
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            v[2 * p] = bf16_bits_to_f32(raw[p] & 0xFFFFu);
            v[2 * p + 1] = bf16_bits_to_f32(raw[p] >> 16);
        }
        int e;
        const uint2 codes = mx_quant8(v, live, &e);
        for (int k = 0; k < K; ++k) {
            *reinterpret_cast<uint2 *>(xq + (size_t)rows[k] * H + 8 * vi) = codes;
            if ((vi & 3) == 0) {
                const int ps = pos[k];
                x_sf[((size_t)(ps >> 8) * (H / 128) + (vi >> 4)) * 512 +
                     nvfp4_atom_offset(ps & 255) + ((vi >> 2) & 3)] = (uint8_t)(e + 127);
            }
        }
    }
}

// MXFP8 h: thread per 8 values of the FP32 matrix [rows, cols]
__global__ void __launch_bounds__(256)
quantize_rows_mx8_kernel(const float *__restrict__ in, int64_t n_vec, int cols,
                         const int32_t *__restrict__ row_pos, uint8_t *__restrict__ codes,
                         uint8_t *__restrict__ sf)
{
    const int64_t b = (int64_t)blockIdx.x * 256 + threadIdx.x;
    const unsigned live = __ballot_sync(0xFFFFFFFFu, b < n_vec);
    if (b >= n_vec)
        return;
    const float4 f0 = reinterpret_cast<const float4 *>(in)[2 * b];
    const float4 f1 = reinterpret_cast<const float4 *>(in)[2 * b + 1];
    const float v[8] = {f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
    int e;
    reinterpret_cast<uint2 *>(codes)[b] = mx_quant8(v, live, &e);
    const int vpr = cols / 8;
    const int vi = (int)(b % vpr);
    if ((vi & 3) == 0) {
        const int ps = row_pos[b / vpr];
        sf[((size_t)(ps >> 8) * (cols / 128) + (vi >> 4)) * 512 + nvfp4_atom_offset(ps & 255) +
           ((vi >> 2) & 3)] = (uint8_t)(e + 127);
    }
}

// ---- fused MoE block ("Reflection Beam 1.0", section "Residual stream":
// sublayers are normalised before and after, in FP32; step k keeps the
// stream with sqrt((k-1)/k) and adds the sublayer output with 1/sqrt(k)).
// RMSNorm with a per-channel gain: the sum of squares is accumulated in FP64
// and rounded to FP32 once as a mean, r = 1/sqrt(mean + eps) in FP32.  Per
// thread the squares are summed as float-float pairs (FP64 arithmetic is
// slow on this part): a bf16 value's square is exact in FP32, an FP32
// value's square is p + e with e = fma(v, v, -p), and each addition keeps
// its rounding error (two-sum); hi + lo is exact in FP64, where the CTA's
// partial sums are added.

// hi + lo += p + e, with the rounding error of hi + p kept in lo
__device__ __forceinline__ void ff_acc(float &hi, float &lo, float p, float e)
{
    const float s = __fadd_rn(hi, p);
    const float bp = __fsub_rn(s, hi);
    const float err = __fadd_rn(__fsub_rn(hi, __fsub_rn(s, bp)), __fsub_rn(p, bp));
    hi = s;
    lo = __fadd_rn(lo, __fadd_rn(err, e));
}

// FP64 sum over the 256 threads of a CTA; every thread gets the total.
__device__ double block_sum_f64(double v, double *red)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
    const int w = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0)
        red[w] = v;
    __syncthreads();
    double t = 0.0;
#pragma unroll
    for (int i = 0; i < 8; ++i)
        t += red[i];
    __syncthreads();
    return t;
}

__device__ __forceinline__ float rms_inv_f32(double ss, int H, float eps)
{
    const float mean = __double2float_rn(ss / (double)H);
    return __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(mean, eps)));
}

// CTA per token: x = bf16((s * r) * gamma), the MoE layer's input.
__global__ void __launch_bounds__(256)
rmsnorm_bf16_kernel(const uint16_t *__restrict__ s, const float *__restrict__ gamma, float eps,
                    int H, uint16_t *__restrict__ x)
{
    __shared__ double red[8];
    const int t = blockIdx.x;
    const uint4 *row = reinterpret_cast<const uint4 *>(s + (size_t)t * H);
    const int nvec = H / 8;
    float hi = 0.0f, lo = 0.0f;
    for (int i = threadIdx.x; i < nvec; i += 256) {
        const uint4 q = row[i];
        const uint32_t v[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float a = bf16_bits_to_f32(v[j] & 0xFFFFu), b = bf16_bits_to_f32(v[j] >> 16);
            ff_acc(hi, lo, __fmul_rn(a, a), 0.0f);  // exact squares of bf16 values
            ff_acc(hi, lo, __fmul_rn(b, b), 0.0f);
        }
    }
    const float r = rms_inv_f32(block_sum_f64((double)hi + (double)lo, red), H, eps);
    for (int i = threadIdx.x; i < nvec; i += 256) {
        const uint4 q = row[i];
        const uint32_t v[4] = {q.x, q.y, q.z, q.w};
        const float4 g0 = reinterpret_cast<const float4 *>(gamma)[2 * i];
        const float4 g1 = reinterpret_cast<const float4 *>(gamma)[2 * i + 1];
        const float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float lo = __fmul_rn(__fmul_rn(bf16_bits_to_f32(v[j] & 0xFFFFu), r), g[2 * j]);
            const float hi = __fmul_rn(__fmul_rn(bf16_bits_to_f32(v[j] >> 16), r), g[2 * j + 1]);
            o[j] = pack_bf16x2(lo, hi);
        }
        reinterpret_cast<uint4 *>(x + (size_t)t * H)[i] = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

// CTA per token: o = sum_k w_k y_k (FP32, slot order, as combine_kernel),
// kept in registers (H <= 256 * 8 * kBlockMaxVec); z = (o * r) * gamma;
// s_out = bf16(a * s_in + b * z).  Each element is read and written by the
// same thread, so s_out may be s_in.
constexpr int kBlockMaxVec = 4;

__global__ void __launch_bounds__(256)
combine_block_kernel(const uint16_t *__restrict__ y, const float *__restrict__ w,
                     const int32_t *__restrict__ row_of, int K, int H, const uint16_t *s_in,
                     const float *__restrict__ gamma, float eps, float a, float b, uint16_t *s_out)
{
    __shared__ float ws[32];
    __shared__ int rs[32];
    __shared__ double red[8];
    const int t = blockIdx.x;
    if (threadIdx.x < K) {
        ws[threadIdx.x] = w[(size_t)t * K + threadIdx.x];
        rs[threadIdx.x] = row_of[(size_t)t * K + threadIdx.x];
    }
    __syncthreads();
    const int nvec = H / 8;
    float o[kBlockMaxVec][8];
    float hi = 0.0f, lo = 0.0f;
#pragma unroll
    for (int c = 0; c < kBlockMaxVec; ++c) {
        const int i = threadIdx.x + c * 256;
#pragma unroll
        for (int j = 0; j < 8; ++j)
            o[c][j] = 0.0f;
        if (i < nvec) {
            combine_vec8(y, ws, rs, K, H, i, o[c]);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float p = __fmul_rn(o[c][j], o[c][j]);
                ff_acc(hi, lo, p, __fmaf_rn(o[c][j], o[c][j], -p));
            }
        }
    }
    const float r = rms_inv_f32(block_sum_f64((double)hi + (double)lo, red), H, eps);
#pragma unroll
    for (int c = 0; c < kBlockMaxVec; ++c) {
        const int i = threadIdx.x + c * 256;
        if (i < nvec) {
            const uint4 q = reinterpret_cast<const uint4 *>(s_in + (size_t)t * H)[i];
            const uint32_t v[4] = {q.x, q.y, q.z, q.w};
            const float4 g0 = reinterpret_cast<const float4 *>(gamma)[2 * i];
            const float4 g1 = reinterpret_cast<const float4 *>(gamma)[2 * i + 1];
            const float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
            uint32_t res[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float z0 = __fmul_rn(__fmul_rn(o[c][2 * j], r), g[2 * j]);
                const float z1 = __fmul_rn(__fmul_rn(o[c][2 * j + 1], r), g[2 * j + 1]);
                const float s0 = __fadd_rn(__fmul_rn(a, bf16_bits_to_f32(v[j] & 0xFFFFu)),
                                           __fmul_rn(b, z0));
                const float s1 = __fadd_rn(__fmul_rn(a, bf16_bits_to_f32(v[j] >> 16)),
                                           __fmul_rn(b, z1));
                res[j] = pack_bf16x2(s0, s1);
            }
            reinterpret_cast<uint4 *>(s_out + (size_t)t * H)[i] =
                make_uint4(res[0], res[1], res[2], res[3]);
        }
    }
}

// Dense layers: the whole batch is one segment, offsets {0, T}, cut into
// ceil(T / chunk_rows) token chunks; also resets the call's status word.
__global__ void dense_setup_kernel(int T, int chunk_rows, int32_t *__restrict__ offsets,
                                   int32_t *__restrict__ chunk_start, int *__restrict__ status)
{
    if (threadIdx.x == 0) {
        offsets[0] = 0;
        offsets[1] = T;
        chunk_start[0] = 0;
        chunk_start[1] = (T + chunk_rows - 1) / chunk_rows;
        *status = 0;
    }
}
}  // namespace

cudaError_t launch_hist_scan(const int32_t *ids, int T, int K, int E, int chunk_rows,
                             int32_t *local_rank, int32_t *cta_counts, int32_t *cta_base,
                             int32_t *counts, int32_t *offsets, int32_t *chunk_start, int *status,
                             cudaStream_t s)
{
    const int n_cta = (T + kHistTokens - 1) / kHistTokens;
    stage_begin(kStHist, s);
    hist_kernel<<<n_cta, 256, 0, s>>>(ids, T, K, E, local_rank, cta_counts, status, chunk_rows,
                                      cta_base, counts, offsets, chunk_start);
    stage_end(kStHist, s);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || n_cta == 1)  // one CTA did the scan as well
        return e;
    stage_begin(kStScan, s);
    scan_kernel<<<1, 256, 0, s>>>(cta_counts, n_cta, E, chunk_rows, cta_base, counts, offsets,
                                  chunk_start);
    stage_end(kStScan, s);
    return cudaGetLastError();
}

cudaError_t launch_permute(const uint16_t *x, const int32_t *ids, const int32_t *local_rank,
                           const int32_t *cta_base, const int32_t *offsets, int T, int K, int E,
                           int H, int32_t *row_of, int32_t *row_src, void *x_perm,
                           cudaStream_t s)
{
    stage_begin(kStPermute, s);
    permute_kernel<false><<<T, 256, 0, s>>>(x, ids, local_rank, cta_base, offsets, nullptr, T, K,
                                            E, H, row_of, row_src, nullptr, x_perm, nullptr);
    stage_end(kStPermute, s);
    return cudaGetLastError();
}

cudaError_t launch_permute_nvfp4(const uint16_t *x, const int32_t *ids, const int32_t *local_rank,
                                 const int32_t *cta_base, const int32_t *offsets,
                                 const int32_t *chunk_start, int T, int K, int E, int H,
                                 int32_t *row_of, int32_t *row_src, int32_t *row_pos,
                                 uint8_t *x_codes, uint8_t *x_sf, cudaStream_t s)
{
    stage_begin(kStPermute, s);
    permute_kernel<true><<<T, 256, 0, s>>>(x, ids, local_rank, cta_base, offsets, chunk_start, T,
                                           K, E, H, row_of, row_src, row_pos, x_codes, x_sf);
    stage_end(kStPermute, s);
    return cudaGetLastError();
}

cudaError_t launch_rows(const int32_t *ids, const int32_t *local_rank, const int32_t *cta_base,
                        const int32_t *offsets, int T, int K, int E, int32_t *row_of,
                        cudaStream_t s)
{
    const size_t n = (size_t)T * K;
    stage_begin(kStPermute, s);
    rows_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(ids, local_rank, cta_base, offsets, T,
                                                             K, E, row_of);
    stage_end(kStPermute, s);
    return cudaGetLastError();
}

cudaError_t launch_quantize_rows(const float *in, int64_t rows, int cols, const int32_t *row_pos,
                                 uint8_t *codes, uint8_t *sf, cudaStream_t s)
{
    const int64_t n_blocks = rows * (int64_t)(cols / 16);
    const unsigned grid = (unsigned)((n_blocks + 255) / 256);
    stage_begin(kStQuantH, s);
    quantize_rows_kernel<<<grid, 256, 0, s>>>(in, n_blocks, cols, row_pos, codes, sf);
    stage_end(kStQuantH, s);
    return cudaGetLastError();
}

cudaError_t launch_combine(const uint16_t *y, const float *w, const int32_t *row_of, int T, int K,
                           int H, uint16_t *out, cudaStream_t s)
{
    stage_begin(kStCombine, s);
    combine_kernel<<<T, 256, 0, s>>>(y, w, row_of, T, K, H, out);
    stage_end(kStCombine, s);
    return cudaGetLastError();
}

cudaError_t launch_dense_setup(int T, int chunk_rows, int32_t *offsets, int32_t *chunk_start,
                               int *status, cudaStream_t s)
{
    stage_begin(kStScan, s);
    dense_setup_kernel<<<1, 32, 0, s>>>(T, chunk_rows, offsets, chunk_start, status);
    stage_end(kStScan, s);
    return cudaGetLastError();
}

cudaError_t launch_rmsnorm_bf16(const uint16_t *s_in, const float *gamma, float eps, int T, int H,
                               uint16_t *x, cudaStream_t st)
{
    stage_begin(kStNorm, st);
    rmsnorm_bf16_kernel<<<T, 256, 0, st>>>(s_in, gamma, eps, H, x);
    stage_end(kStNorm, st);
    return cudaGetLastError();
}

cudaError_t launch_combine_block(const uint16_t *y, const float *w, const int32_t *row_of, int T,
                                 int K, int H, const uint16_t *s_in, const float *gamma, float eps,
                                 float a, float b, uint16_t *s_out, cudaStream_t st)
{
    if (H > 256 * 8 * kBlockMaxVec)
        return cudaErrorInvalidValue;
    stage_begin(kStCombine, st);
    combine_block_kernel<<<T, 256, 0, st>>>(y, w, row_of, K, H, s_in, gamma, eps, a, b, s_out);
    stage_end(kStCombine, st);
    return cudaGetLastError();
}

cudaError_t launch_permute_mx8(const uint16_t *x, const int32_t *ids, const int32_t *local_rank,
                               const int32_t *cta_base, const int32_t *offsets,
                               const int32_t *chunk_start, int T, int K, int E, int H,
                               int32_t *row_of, int32_t *row_src, int32_t *row_pos,
                               uint8_t *x_codes, uint8_t *x_sf, cudaStream_t st)
{
    stage_begin(kStPermute, st);
    permute_mx8_kernel<<<T, 256, 0, st>>>(x, ids, local_rank, cta_base, offsets, chunk_start, T, K,
                                          E, H, row_of, row_src, row_pos, x_codes, x_sf);
    stage_end(kStPermute, st);
    return cudaGetLastError();
}

cudaError_t launch_quantize_rows_mx8(const float *in, int64_t rows, int cols, const int32_t *row_pos,
                                     uint8_t *codes, uint8_t *sf, cudaStream_t st)
{
    const int64_t n_vec = rows * (int64_t)(cols / 8);
    stage_begin(kStQuantH, st);
    quantize_rows_mx8_kernel<<<(unsigned)((n_vec + 255) / 256), 256, 0, st>>>(in, n_vec, cols,
                                                                             row_pos, codes, sf);
    stage_end(kStQuantH, st);
    return cudaGetLastError();
}

}  // namespace beam
