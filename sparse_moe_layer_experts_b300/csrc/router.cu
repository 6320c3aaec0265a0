// Router of the Beam MoE layer: FP32 logits, sigmoid scores and the
// group-limited top-k selection with normalised, scaled weights.
//
// Method: "Reflection Beam 1.0: 501B open MoE model" (agentlenshq.com),
// section "Mixture of Experts: 256 experts, 8 routed per token"; the router is
// computed in FP32 (same page, section "Residual stream", last paragraph).
//
// Readings where the pages are silent: each logit is the FP32 fused
// multiply-add chain over h = 0..H-1 starting from +0; sigmoid(l) = 1/(1+E)
// with E = exp(-l) rounded once to FP32 (the value fp32(exp((double)-l)));
// ties go to the lower index; slots are
// ordered by score descending, index ascending; S = FP32 sum of the selected
// scores in slot order; w = (s/S)*scale with an IEEE divide and multiply.
#include "common.cuh"
#include "internal.h"
#include "router_math.cuh"

#include <math.h>

namespace beam {

namespace {

using router_math::router_sigmoid;

__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gsrc, bool valid)
{
    const uint32_t d = smem_u32(smem_dst);
    const int n = valid ? 16 : 0;  // 0 source bytes: the 16 bytes are zero-filled
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(gsrc), "r"(n)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit()
{
    asm volatile("cp.async.commit_group;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Batches below the tensor-core threshold: each output's 5,120-long FMA chain
// is the critical path and there are few outputs (T x E), so the work is
// spread thin: a CTA of two warps owns 8 tokens x 8 experts, and thread
// (w, tt, ep) runs the one chain of token t0 + tt and expert e0 + 2ep + w
// (T=32: 128 CTAs, 8,192 threads, one chain each, the two warps of a CTA on
// two of the SM's four schedulers; T=255: 1,024 CTAs, five per SM).  Per 8
// hidden values a thread issues one 128-bit load of x, eight 32-bit weight
// loads, 8 unpacks and 8 FMAs: about 4 instructions per hidden value at
// about 2 cycles each (ncu at T=32), twice the 4-cycle latency of the chain's
// FMA.  K chunks of 64 flow through a 12-stage cp.async ring filled by both
// warps (the ring runs microseconds ahead of the loads' latency).
constexpr int kSTM = 8, kSTE = 8, kSKC = 64, kSNS = 12, kSXP = kSKC + 8, kSThreads = 64;

__global__ void __launch_bounds__(kSThreads)
router_scores_small(const uint16_t *__restrict__ x, const float *__restrict__ wr, int T, int H,
                    int E, float *__restrict__ scores, int *status)
{
    if (status && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0)
        *status = 0;
    __shared__ __align__(16) uint16_t xs[kSNS][kSTM][kSXP];
    __shared__ __align__(16) float ws[kSNS][kSKC][kSTE];
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int tt = lane >> 2, el = 2 * (lane & 3) + w;  // token and expert within the tile
    const int t0 = blockIdx.x * kSTM, e0 = blockIdx.y * kSTE;
    const int nk = H / kSKC;

    auto load = [&](int st, int k0) {
        // x: 8 rows x 8 chunks of 16 B (one per thread); w: 64 rows x two
        // 16-B chunks of 4 experts (two per thread)
        {
            const int r = tid >> 3, q = tid & 7;
            const bool ok = t0 + r < T;
            cp_async16(&xs[st][r][q * 8], x + (size_t)(ok ? t0 + r : 0) * H + k0 + q * 8, ok);
        }
#pragma unroll
        for (int c = tid; c < kSKC * 2; c += kSThreads) {
            const int r = c >> 1, h4 = (c & 1) * 4;
            const bool ok = e0 + h4 < E;
            cp_async16(&ws[st][r][h4], wr + (size_t)(k0 + r) * E + (ok ? e0 + h4 : 0), ok);
        }
    };
    static_assert(kSTM * (kSKC / 8) == kSThreads, "one 16-byte x chunk per thread");

#pragma unroll
    for (int s = 0; s < kSNS - 1; ++s) {
        if (s < nk)
            load(s, s * kSKC);
        cp_async_commit();
    }
    float acc = 0.0f;
    for (int kc = 0; kc < nk; ++kc) {
        cp_async_wait<kSNS - 2>();
        // every thread's copies of chunk kc have landed, and every thread has
        // finished chunk kc - 1, whose stage the next load overwrites
        __syncthreads();
        if (kc + kSNS - 1 < nk)
            load((kc + kSNS - 1) % kSNS, (kc + kSNS - 1) * kSKC);
        cp_async_commit();
        const int st = kc % kSNS;
#pragma unroll
        for (int k8 = 0; k8 < kSKC; k8 += 8) {
            const uint4 xv = *reinterpret_cast<const uint4 *>(&xs[st][tt][k8]);
            const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float xf = (i & 1) ? __uint_as_float(xw[i >> 1] & 0xFFFF0000u)
                                         : __uint_as_float(xw[i >> 1] << 16);
                acc = __fmaf_rn(xf, ws[st][k8 + i][el], acc);
            }
        }
    }
    const int t = t0 + tt, e = e0 + el;
    if (t < T && e < E)
        scores[(size_t)t * E + e] = router_sigmoid(acc);
}

// Key of a float under the warp's max/min reductions: larger float, larger
// key.  0 means "no candidate"; a NaN is never a candidate.
__device__ __forceinline__ unsigned order_key(float f)
{
    if (f != f)
        return 0u;
    const unsigned u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_value(unsigned k)
{
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// One round of the warp arg-max under (value desc, index asc) over the
// candidate bits `cand` of this lane's experts lane + 32j, whose order keys
// are key[j].  Returns the key of the best value (0 if none is left) and its
// expert in *be; the lane holding it clears its bit.
__device__ __forceinline__ unsigned warp_argmax(const unsigned (&key)[8], unsigned &cand, int lane,
                                                int *be_out)
{
    const unsigned full = 0xFFFFFFFFu;
    unsigned bk = 0u;
    int be = 0x7FFFFFFF;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const unsigned k = ((cand >> j) & 1u) ? key[j] : 0u;
        if (k > bk) {  // j ascending: the first of equal keys has the lowest index
            bk = k;
            be = lane + 32 * j;
        }
    }
    const unsigned best = __reduce_max_sync(full, bk);
    be = (int)__reduce_min_sync(full, (bk == best && best != 0u) ? (unsigned)be : 0xFFFFFFFFu);
    if (best != 0u && (be & 31) == lane)
        cand &= ~(1u << (be >> 5));
    *be_out = best != 0u ? be : 0;
    return best;
}

// One warp per token.  Lane l holds the values of experts l, l+32, ...
// Three sources of the router's scores:
//  - nsplit == 0: the FMA-chain router wrote the FP32 scores;
//  - nsplit > 0, write_scores: the tensor-core router's partial logits
//    [nsplit][T][E] are added in order p = 0..nsplit-1 (FP32), the sigmoid
//    applied to every one and the scores written (`partials` may be
//    `scores` when nsplit == 1: each element is read and written by the
//    same lane);
//  - nsplit > 0, !write_scores: the same logits, but the sigmoid is
//    evaluated only where the selection needs it.  sigmoid is monotone
//    (non-decreasing in FP32), so a group's two largest scores are the
//    sigmoids of its two largest logits, and the top-K experts by (score
//    desc, index asc) are the top-K by (logit desc, index asc) re-ranked by
//    (score, index) -- unless the next candidate's score equals the K-th
//    (a plateau of the FP32 sigmoid, or tied logits), in which case every
//    candidate's score is evaluated and the plain selection runs.
// Both tensor-core modes therefore select exactly what the scores select.
__global__ void __launch_bounds__(256)
select_kernel(float *scores, const float *partials, int nsplit, int write_scores, int T, int E,
              int G, int TG, int K, float scale, int32_t *__restrict__ ids,
              float *__restrict__ wts, int *status)
{
    __shared__ float row_s[8][256];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + warp;
    if (t >= T)
        return;
    const unsigned full = 0xFFFFFFFFu;
    float *s = scores + (size_t)t * E;
    const int gsize = E / G;
    const bool lazy = nsplit > 0 && !write_scores;

    // v: scores, or logits in the lazy mode.  Each pass over j issues its
    // eight loads together (one round trip per partial, not per element).
    float v[8];
    const float *src = nsplit > 0 ? partials + (size_t)t * E : s;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int e = lane + 32 * j;
        v[j] = (e < E) ? src[e] : -INFINITY;
    }
    for (int p = 1; p < nsplit; ++p) {
        const float *pl = partials + ((size_t)p * T + t) * E;
        float q[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int e = lane + 32 * j;
            q[j] = (e < E) ? pl[e] : 0.0f;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j)
            v[j] = __fadd_rn(v[j], q[j]);
    }
    if (nsplit > 0 && !lazy) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int e = lane + 32 * j;
            if (e < E) {
                v[j] = router_sigmoid(v[j]);
                s[e] = v[j];
            }
        }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int e = lane + 32 * j;
        if (e < E)
            row_s[warp][e] = v[j];
    }
    __syncwarp();

    // group score: the two largest scores of the group, summed in FP32 (in
    // the lazy mode: the sigmoids of the two largest logits)
    float m1 = -INFINITY, m2 = -INFINITY;  // lane g < G: group g's two largest values
    unsigned key[8];  // order keys of v, for the warp reductions
#pragma unroll
    for (int j = 0; j < 8; ++j)
        key[j] = order_key(v[j]);
    if (gsize == 32) {
        // group j is row j: its largest value is a warp max over the keys,
        // the second the max over the other lanes (the same value again if
        // two lanes hold the largest)
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (j >= G)
                break;
            const unsigned k1 = __reduce_max_sync(full, key[j]);
            const unsigned twice = __popc(__ballot_sync(full, key[j] == k1)) > 1;
            const unsigned k2 = twice ? k1 : __reduce_max_sync(full, key[j] == k1 ? 0u : key[j]);
            if (lane == j) {
                m1 = key_value(k1);
                m2 = key_value(k2);
            }
        }
    } else if ((32 % gsize) == 0) {
        // groups are aligned runs of gsize lanes within each 32-expert row:
        // reduce (largest, second largest) pairs across the run with xor
        // shuffles, then lane g fetches group g's pair
        const int src = (lane * gsize) & 31, row = (lane * gsize) >> 5;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            float a1 = v[j], a2 = -INFINITY;
            for (int off = 1; off < gsize; off <<= 1) {
                const float o1 = __shfl_xor_sync(full, a1, off);
                const float o2 = __shfl_xor_sync(full, a2, off);
                const float lo = fminf(a1, o1);
                a1 = fmaxf(a1, o1);
                a2 = fmaxf(lo, fmaxf(a2, o2));
            }
            const float b1 = __shfl_sync(full, a1, src);
            const float b2 = __shfl_sync(full, a2, src);
            if (lane < G && row == j) {
                m1 = b1;
                m2 = b2;
            }
        }
    } else if (lane < G) {
        for (int j = 0; j < gsize; ++j) {
            const float q = row_s[warp][lane * gsize + j];
            if (q > m1) {
                m2 = m1;
                m1 = q;
            } else if (q > m2) {
                m2 = q;
            }
        }
    }
    float gs = -INFINITY;
    if (lane < G) {
        const float s1 = lazy ? router_sigmoid(m1) : m1;
        gs = (gsize == 1) ? s1 : __fadd_rn(s1, lazy ? router_sigmoid(m2) : m2);
    }
    // rank of my group under (score desc, index asc)
    int rank = 0;
    for (int g = 0; g < G; ++g) {
        const float o = __shfl_sync(full, gs, g);
        if (g != lane && (o > gs || (o == gs && g < lane)))
            ++rank;
    }
    const unsigned kept = __ballot_sync(full, lane < G && rank < TG);

    unsigned cand0 = 0;  // bit j: expert lane + 32j is in a kept group
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int e = lane + 32 * j;
        if (e < E && ((kept >> (e / gsize)) & 1u))
            cand0 |= 1u << j;
    }
    int my_e = -1;     // lane k < K: the expert of slot k
    float my_v = 0.0f;  // and its score
    bool done = false;
    if (lazy) {
        // top-K candidates by (logit desc, index asc), and the next one
        unsigned cand = cand0;
        float my_l = 0.0f;
        bool ok = true;
        for (int k = 0; k < K; ++k) {
            int be;
            const unsigned best = warp_argmax(key, cand, lane, &be);
            ok = ok && best != 0u;
            if (lane == k) {
                my_e = be;
                my_l = key_value(best);
            }
        }
        int be_next;
        const unsigned next = warp_argmax(key, cand, lane, &be_next);
        if (ok) {
            if (lane < K)
                my_v = router_sigmoid(my_l);
            const float vK = __shfl_sync(full, my_v, K - 1);
            // the K-th score is not shared with any later candidate
            if (next == 0u || router_sigmoid(key_value(next)) < vK) {
                // slot = rank under (score desc, index asc)
                int slot = 0;
                for (int j = 0; j < K; ++j) {
                    const float oj = __shfl_sync(full, my_v, j);
                    const int ej = __shfl_sync(full, my_e, j);
                    if (oj > my_v || (oj == my_v && ej < my_e))
                        ++slot;
                }
                float S = 0.0f;
                for (int k = 0; k < K; ++k) {
                    const unsigned m = __ballot_sync(full, lane < K && slot == k);
                    S = __fadd_rn(S, __shfl_sync(full, my_v, __ffs(m) - 1));
                }
                if (lane < K) {
                    ids[(size_t)t * K + slot] = my_e;
                    wts[(size_t)t * K + slot] = __fmul_rn(__fdiv_rn(my_v, S), scale);
                }
                done = true;
            }
        }
        if (!done) {  // a plateau or tie at the boundary: every candidate's score
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                v[j] = ((cand0 >> j) & 1u) ? router_sigmoid(v[j]) : -INFINITY;
                key[j] = order_key(v[j]);
            }
        }
    }
    if (!done) {
        // top-K among the kept groups' experts by repeated warp arg-max under
        // (score desc, index asc)
        unsigned cand = cand0;
        for (int k = 0; k < K; ++k) {
            int be;
            const unsigned best = warp_argmax(key, cand, lane, &be);
            if (best == 0u && lane == 0)  // no candidate left (non-finite scores)
                atomicOr(status, kStatusDevice);
            if (lane == k) {
                my_e = be;
                my_v = best != 0u ? key_value(best) : 0.0f;
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
}

}  // namespace

cudaError_t launch_router_scores(const uint16_t *x, const float *wr, int T, int H, int E,
                                 float *scores, int *status, cudaStream_t s)
{
    stage_begin(kStRouter, s);
    const dim3 grid((T + kSTM - 1) / kSTM, (E + kSTE - 1) / kSTE);
    router_scores_small<<<grid, kSThreads, 0, s>>>(x, wr, T, H, E, scores, status);
    stage_end(kStRouter, s);
    return cudaGetLastError();
}

cudaError_t launch_select(float *scores, const float *partials, int nsplit, bool write_scores,
                          int T, int E, int G, int TG, int K, float scale, int32_t *ids, float *w,
                          int *status, cudaStream_t s)
{
    stage_begin(kStSelect, s);
    select_kernel<<<(T + 7) / 8, 256, 0, s>>>(scores, partials, nsplit, write_scores ? 1 : 0, T, E,
                                             G, TG, K, scale, ids, w, status);
    stage_end(kStSelect, s);
    return cudaGetLastError();
}

}  // namespace beam
