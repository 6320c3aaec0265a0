// Router of the Beam MoE layer: FP32 logits, sigmoid scores and the
// group-limited top-k selection with normalised, scaled weights.
//
// Method: "Reflection Beam 1.0: 501B open MoE model" (agentlenshq.com),
// section "Mixture of Experts: 256 experts, 8 routed per token"; the router is
// computed in FP32 (same page, section "Residual stream", last paragraph).
//
// Readings where the pages are silent: each logit is the FP32 fused
// multiply-add chain over h = 0..H-1 starting from +0; sigmoid(l) = 1/(1+E)
// with E = exp(-l) rounded once to FP32; ties go to the lower index; slots are
// ordered by score descending, index ascending; S = FP32 sum of the selected
// scores in slot order; w = (s/S)*scale with an IEEE divide and multiply.
#include "common.cuh"
#include "internal.h"

#include <math.h>

namespace beam {

namespace {

// Register-tiled FP32 GEMM with a fixed per-output accumulation order:
// every accumulator walks h = 0..H-1 in order, so the result does not depend
// on the tiling.  CTA tile TM tokens x TE experts, thread tile RT x RE,
// K chunk KC staged in shared memory.
template <int TM, int TE, int RT, int RE, int KC>
__global__ void __launch_bounds__(256)
router_scores_kernel(const uint16_t *__restrict__ x, const float *__restrict__ wr, int T, int H,
                     int E, float *__restrict__ scores, int *status)
{
    // first kernel of every call: reset the call's device status word
    if (status && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0)
        *status = 0;
    constexpr int NTX = TE / RE;
    constexpr int NTY = TM / RT;
    static_assert(NTX * NTY == 256, "256 threads");
    static_assert(KC % 8 == 0 && TE % 4 == 0 && RE % 4 == 0, "vector widths");
    __shared__ __align__(16) float xs[KC][TM + 4];
    __shared__ __align__(16) float ws[KC][TE];

    const int tid = threadIdx.x;
    const int tx = tid % NTX, ty = tid / NTX;
    const int t0 = blockIdx.x * TM, e0 = blockIdx.y * TE;

    float acc[RT][RE];
#pragma unroll
    for (int i = 0; i < RT; ++i)
#pragma unroll
        for (int j = 0; j < RE; ++j)
            acc[i][j] = 0.0f;

    for (int k0 = 0; k0 < H; k0 += KC) {
        // x chunk: TM rows x KC bf16, 8 per 16-byte vector, stored transposed
        for (int v = tid; v < TM * (KC / 8); v += 256) {
            const int r = v / (KC / 8), c8 = (v % (KC / 8)) * 8;
            const int t = t0 + r;
            uint4 q = make_uint4(0, 0, 0, 0);
            if (t < T)
                q = *reinterpret_cast<const uint4 *>(x + (size_t)t * H + k0 + c8);
            const uint32_t w4[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                xs[c8 + 2 * p][r] = bf16_bits_to_f32(w4[p] & 0xFFFFu);
                xs[c8 + 2 * p + 1][r] = bf16_bits_to_f32(w4[p] >> 16);
            }
        }
        // router weight chunk: KC rows x TE fp32
        for (int v = tid; v < KC * (TE / 4); v += 256) {
            const int r = v / (TE / 4), c4 = (v % (TE / 4)) * 4;
            float4 q = make_float4(0.f, 0.f, 0.f, 0.f);
            if (e0 + c4 < E)
                q = *reinterpret_cast<const float4 *>(wr + (size_t)(k0 + r) * E + e0 + c4);
            *reinterpret_cast<float4 *>(&ws[r][c4]) = q;
        }
        __syncthreads();
#pragma unroll 4
        for (int k = 0; k < KC; ++k) {
            float a[RT], b[RE];
#pragma unroll
            for (int i = 0; i < RT; ++i)
                a[i] = xs[k][ty * RT + i];
#pragma unroll
            for (int j = 0; j < RE; j += 4) {
                const float4 q = *reinterpret_cast<const float4 *>(&ws[k][tx * RE + j]);
                b[j] = q.x;
                b[j + 1] = q.y;
                b[j + 2] = q.z;
                b[j + 3] = q.w;
            }
#pragma unroll
            for (int i = 0; i < RT; ++i)
#pragma unroll
                for (int j = 0; j < RE; ++j)
                    acc[i][j] = __fmaf_rn(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }

#pragma unroll
    for (int i = 0; i < RT; ++i) {
        const int t = t0 + ty * RT + i;
        if (t >= T)
            continue;
#pragma unroll
        for (int j = 0; j < RE; ++j) {
            const int e = e0 + tx * RE + j;
            if (e >= E)
                continue;
            const float ex = static_cast<float>(exp(-static_cast<double>(acc[i][j])));
            const float den = __fadd_rn(1.0f, ex);
            scores[(size_t)t * E + e] = __fdiv_rn(1.0f, den);
        }
    }
}

// One warp per token.  Lane l holds the scores of experts l, l+32, ...
__global__ void __launch_bounds__(256)
select_kernel(const float *__restrict__ scores, int T, int E, int G, int TG, int K, float scale,
              int32_t *__restrict__ ids, float *__restrict__ wts, int *status)
{
    __shared__ float row_s[8][256];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + warp;
    if (t >= T)
        return;
    const unsigned full = 0xFFFFFFFFu;
    const float *s = scores + (size_t)t * E;
    const int gsize = E / G;

    float v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int e = lane + 32 * j;
        v[j] = (e < E) ? s[e] : -INFINITY;
        if (e < E)
            row_s[warp][e] = v[j];
    }
    __syncwarp();

    // group score: the two largest scores of the group, summed in FP32
    float gs = -INFINITY;
    if (lane < G) {
        float m1 = -INFINITY, m2 = -INFINITY;
        for (int j = 0; j < gsize; ++j) {
            const float q = row_s[warp][lane * gsize + j];
            if (q > m1) {
                m2 = m1;
                m1 = q;
            } else if (q > m2) {
                m2 = q;
            }
        }
        gs = (gsize == 1) ? m1 : __fadd_rn(m1, m2);
    }
    // rank of my group under (score desc, index asc)
    int rank = 0;
    for (int g = 0; g < G; ++g) {
        const float o = __shfl_sync(full, gs, g);
        if (g != lane && (o > gs || (o == gs && g < lane)))
            ++rank;
    }
    const unsigned kept = __ballot_sync(full, lane < G && rank < TG);

    // top-K among the kept groups' experts by repeated warp arg-max
    unsigned taken = 0;
    int my_e = -1;
    float my_v = 0.0f;
    for (int k = 0; k < K; ++k) {
        float bv = -INFINITY;
        int be = 0x7FFFFFFF;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int e = lane + 32 * j;
            if (e < E && ((kept >> (e / gsize)) & 1u) && !((taken >> j) & 1u) &&
                (v[j] > bv || (v[j] == bv && e < be))) {
                bv = v[j];
                be = e;
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float ov = __shfl_xor_sync(full, bv, off);
            const int oe = __shfl_xor_sync(full, be, off);
            if (ov > bv || (ov == bv && oe < be)) {
                bv = ov;
                be = oe;
            }
        }
        if (be == 0x7FFFFFFF) {  // no candidate left (non-finite scores)
            if (lane == 0)
                atomicOr(status, kStatusDevice);
            be = 0;
            bv = 0.0f;
        } else if ((be & 31) == lane) {
            taken |= 1u << (be >> 5);
        }
        if (lane == k) {
            my_e = be;
            my_v = bv;
        }
    }
    float S = 0.0f;
    for (int k = 0; k < K; ++k)
        S = __fadd_rn(S, __shfl_sync(full, my_v, k));
    if (lane < K) {
        ids[(size_t)t * K + lane] = my_e;
        wts[(size_t)t * K + lane] = __fmul_rn(__fdiv_rn(my_v, S), scale);
    }
}

}  // namespace

cudaError_t launch_router_scores(const uint16_t *x, const float *wr, int T, int H, int E,
                                 float *scores, int *status, cudaStream_t s)
{
    stage_begin(kStRouter, s);
    if (T >= 512) {
        constexpr int TM = 64, TE = 128;
        dim3 grid((T + TM - 1) / TM, (E + TE - 1) / TE);
        router_scores_kernel<TM, TE, 4, 8, 32><<<grid, 256, 0, s>>>(x, wr, T, H, E, scores, status);
    } else {
        constexpr int TM = 16, TE = 64;
        dim3 grid((T + TM - 1) / TM, (E + TE - 1) / TE);
        router_scores_kernel<TM, TE, 1, 4, 32><<<grid, 256, 0, s>>>(x, wr, T, H, E, scores, status);
    }
    stage_end(kStRouter, s);
    return cudaGetLastError();
}

cudaError_t launch_select(const float *scores, int T, int E, int G, int TG, int K, float scale,
                          int32_t *ids, float *w, int *status, cudaStream_t s)
{
    stage_begin(kStSelect, s);
    select_kernel<<<(T + 7) / 8, 256, 0, s>>>(scores, T, E, G, TG, K, scale, ids, w, status);
    stage_end(kStSelect, s);
    return cudaGetLastError();
}

}  // namespace beam
