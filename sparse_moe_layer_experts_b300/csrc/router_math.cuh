// Router score arithmetic shared by the router kernels: the FP32 sigmoid
// sigmoid(l) = 1/(1+E), E = exp(-l) rounded once to FP32 (the value
// fp32(exp((double)-l))), so every kernel turns a given FP32 logit into the
// same score bit for bit.
//
// Source of the FP32 pin: "Reflection Beam 1.0: 501B open MoE model"
// (agentlenshq.com), section "Residual stream", last paragraph (the router is
// computed in FP32); sigmoid scores: same page, section "Mixture of Experts".
#pragma once

#include "common.cuh"

#include <math.h>

namespace beam {
namespace router_math {

// Float-float (unevaluated sum h + l) helpers built from error-free
// transformations; the _rn intrinsics keep the compiler from fusing them.
struct FF {
    float h, l;
};

__device__ __forceinline__ FF ff_renorm(float s, float e)
{
    const float t = __fadd_rn(s, e);
    return {t, __fsub_rn(e, __fsub_rn(t, s))};
}

__device__ __forceinline__ FF ff_mul(FF a, FF b)
{
    const float p = __fmul_rn(a.h, b.h);
    float e = __fmaf_rn(a.h, b.h, -p);  // a.h * b.h = p + e exactly
    e = __fmaf_rn(a.h, b.l, e);
    e = __fmaf_rn(a.l, b.h, e);
    return ff_renorm(p, e);
}

__device__ __forceinline__ FF ff_add(FF a, FF b)
{
    const float s = __fadd_rn(a.h, b.h);
    const float bb = __fsub_rn(s, a.h);
    float e = __fadd_rn(__fsub_rn(a.h, __fsub_rn(s, bb)), __fsub_rn(b.h, bb));  // two-sum
    e = __fadd_rn(e, __fadd_rn(a.l, b.l));
    return ff_renorm(s, e);
}

// e^x rounded once to FP32 (nearest, ties to even).  Written from the Taylor
// series: x = k*ln2 + r (ln2 = C1 + C2 + C3; C1 has 15 significant bits, so
// k*C1 and x - k*C1 are exact), e^r = sum_{i<=11} r^i/i! with the terms up to
// r^6 summed in float-float and r^7..r^11 in float, a relative error below
// 2^-44 for |r| <= ln2/2; then scaled by 2^k.  Where that value lies within
// 2^-43 (relative) of a rounding midpoint, or |x| > 60, the double-precision
// exp decides instead, so the result always equals fp32(exp((double)x)) while
// the FP64 units (few on this part) are almost never used.
__device__ __forceinline__ float exp_rn_f32(float x)
{
    if (!(fabsf(x) <= 60.0f))
        return static_cast<float>(exp(static_cast<double>(x)));
    const float k = rintf(__fmul_rn(x, 0x1.715476p+0f));
    const float C1 = 0x1.62e4p-1f, C2 = 0x1.7f7d1cp-20f, C3 = 0x1.ef357ap-45f;
    const float r1 = __fmaf_rn(-k, C1, x);  // exact
    const float p = __fmul_rn(k, C2);
    const float pe = __fmaf_rn(k, C2, -p);  // k*C2 = p + pe exactly
    const float s = __fsub_rn(r1, p);
    const float bv = __fsub_rn(s, r1);
    float se = __fadd_rn(__fsub_rn(r1, __fsub_rn(s, bv)), __fsub_rn(-p, bv));
    se = __fsub_rn(__fsub_rn(se, pe), __fmul_rn(k, C3));
    const FF r = ff_renorm(s, se);

    // 1/i! as float-float (hi, lo); i = 0..6
    const float ch[7] = {1.0f, 1.0f, 0.5f, 0x1.555556p-3f, 0x1.555556p-5f, 0x1.111112p-7f,
                         0x1.6c16c2p-10f};
    const float cl[7] = {0.0f, 0.0f, 0.0f, -0x1.555556p-28f, -0x1.555556p-30f, -0x1.dddddep-32f,
                         -0x1.27d27ep-35f};
    float tail = 0x1.ae6456p-26f;             // 1/11!
    tail = __fmaf_rn(tail, r.h, 0x1.27e4fcp-22f);  // 1/10!
    tail = __fmaf_rn(tail, r.h, 0x1.71de3ap-19f);  // 1/9!
    tail = __fmaf_rn(tail, r.h, 0x1.a01a02p-16f);  // 1/8!
    tail = __fmaf_rn(tail, r.h, 0x1.a01a02p-13f);  // 1/7!
    FF acc = {tail, 0.0f};
#pragma unroll
    for (int i = 6; i >= 0; --i)
        acc = ff_add(ff_mul(acc, r), FF{ch[i], cl[i]});

    const float scale = __uint_as_float((uint32_t)((int)k + 127) << 23);
    const float eh = __fmul_rn(acc.h, scale), el = __fmul_rn(acc.l, scale);  // exact
    const float f = __fadd_rn(eh, el);
    const float d = __fadd_rn(__fsub_rn(eh, f), el);  // (eh + el) - f
    const uint32_t fb = __float_as_uint(f);
    const float ulp = __uint_as_float((fb & 0x7F800000u) - (23u << 23));
    const float half = (d < 0.0f && (fb & 0x7FFFFFu) == 0u) ? 0.25f * ulp : 0.5f * ulp;
    if (fabsf(half - fabsf(d)) <= f * 0x1p-43f)
        return static_cast<float>(exp(static_cast<double>(x)));
    return f;
}

__device__ __forceinline__ float router_sigmoid(float l)
{
    const float ex = exp_rn_f32(-l);
    return __fdiv_rn(1.0f, __fadd_rn(1.0f, ex));
}

}  // namespace router_math
}  // namespace beam
