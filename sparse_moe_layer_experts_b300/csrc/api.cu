// C ABI of libbeam_moe.so: argument checks, workspace layout, TMA tensor
// maps and the launch sequence of one Beam MoE layer forward.
//
//   router_scores -> select -> hist -> scan -> permute -> gate/up GEMM
//   -> down GEMM -> combine          (one stream, no host synchronisation)
#include "../../include/beam_moe.h"
#include "common.cuh"
#include "internal.h"

#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <mutex>

namespace beam {

static thread_local int64_t g_launches = 0;
static thread_local cudaEvent_t g_ev_start[kNumStages];
static thread_local cudaEvent_t g_ev_stop[kNumStages];
static thread_local int g_ev_n = 0;

void stage_begin(int stage, cudaStream_t s)
{
    if (stage < g_ev_n && g_ev_start[stage])
        cudaEventRecord(g_ev_start[stage], s);
}

void stage_end(int stage, cudaStream_t s)
{
    ++g_launches;
    if (stage < g_ev_n && g_ev_stop[stage])
        cudaEventRecord(g_ev_stop[stage], s);
}

void count_launch() { ++g_launches; }

namespace {

constexpr size_t kAlign = 1024;
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;

size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

struct Layout {
    size_t status, wr_parts, router_partials, scores, ids, wts, local_rank, cta_counts, cta_base, counts, offsets,
        chunk_start, row_of, row_src, x_perm, h, h_raw, y, row_pos, x_sf, h_sf,
        total;
};

// Prefill-size batches route on the tensor cores (router_tc.cu); smaller
// ones keep the FP32 FMA-chain router, whose logits follow the h order.
bool tc_router(int64_t T) { return T >= kTcRouterMinTokens; }

// The workspace holds the tensor-core router's partial logits for as many
// hidden-dimension splits as a GPU of up to kLayoutSms SMs would take; the
// launch never takes more.
constexpr int kLayoutSms = 256;
int tc_router_layout_splits(int64_t T, const beam_moe_cfg &c)
{
    return tc_router(T) ? router_tc_splits(T, c.n_experts, c.hidden, kLayoutSms) : 0;
}

GemmVariant pick_variant(int64_t T, const beam_moe_cfg &c)
{
    // decode: a handful of tokens per active expert
    return (T * c.top_k <= 16LL * c.n_experts) ? GemmVariant::kDecode : GemmVariant::kPrefill;
}

// Rows per token chunk (the token tile of the grouped GEMMs; both GEMMs of
// a layer use the same chunking).
int chunk_rows(int64_t T, const beam_moe_cfg &c)
{
    const GemmVariant v = pick_variant(T, c);
    return c.wtype != BEAM_MOE_W_BF16 ? fp4_chunk_rows(v) : gemm_chunk_rows(v);
}

Layout make_layout(int64_t T, const beam_moe_cfg &c)
{
    const int64_t K = c.top_k, E = c.n_experts, H = c.hidden, I = c.inter;
    const int64_t n_cta = (T + kHistTokens - 1) / kHistTokens;
    const int64_t R = T * K;
    Layout L{};
    size_t o = 0;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o = align_up(o + bytes);
        return at;
    };
    L.status = take(256);
    L.wr_parts = take(tc_router(T) ? (size_t)3 * E * H * 2 : 0);
    // partial logits of split hidden ranges (none when one range: the
    // logits then go straight into the scores buffer)
    const int splits = tc_router_layout_splits(T, c);
    L.router_partials = take(splits > 1 ? sizeof(float) * splits * T * E : 0);
    L.scores = take(sizeof(float) * T * E);
    L.ids = take(sizeof(int32_t) * R);
    L.wts = take(sizeof(float) * R);
    L.local_rank = take(sizeof(int32_t) * R);
    L.cta_counts = take(sizeof(int32_t) * n_cta * E);
    L.cta_base = take(sizeof(int32_t) * n_cta * E);
    L.counts = take(sizeof(int32_t) * E);
    L.offsets = take(sizeof(int32_t) * (E + 1));
    L.chunk_start = take(sizeof(int32_t) * (E + 1));
    L.row_of = take(sizeof(int32_t) * R);
    L.row_src = take(sizeof(int32_t) * R);
    const bool fp4 = c.wtype == BEAM_MOE_W_NVFP4, mx8 = c.wtype == BEAM_MOE_W_MXFP8;
    // activations: bf16 rows, NVFP4 codes (2 per byte) or MXFP8 codes
    L.x_perm = take(fp4 ? R * H / 2 : mx8 ? R * H : 2 * R * H);
    L.h = take(fp4 ? R * I / 2 : mx8 ? R * I : 2 * R * I);
    // FP32 h before quantisation (decode-size batches; the token-major
    // prefill kernels quantise h in their epilogue)
    L.h_raw = take((fp4 || mx8) && pick_variant(T, c) == GemmVariant::kDecode ? 4 * R * I : 0);
    L.y = take(2 * R * H);
    if (mx8) {
        // MXFP8: one chunking for both GEMMs; row_pos = chunk*256 + j; scale
        // atoms [chunk, K/128, 512] for x and h
        const int64_t cr = chunk_rows(T, c);
        const int64_t chunks = (R + cr - 1) / cr + E;
        L.row_pos = take(4 * R);
        L.x_sf = take((size_t)chunks * (H / 128) * 512);
        L.h_sf = take((size_t)chunks * (I / 128) * 512);
        L.total = o;
        return L;
    }
    // NVFP4: each row's place in the token chunking (chunk*256 + j), and the
    // activations' scales per token chunk in atoms: x [chunk, H/64, 512],
    // h [chunk, I/64, 512]
    const int64_t cr = chunk_rows(T, c);
    const int64_t chunks = fp4 ? (R + cr - 1) / cr + E : 0;
    L.row_pos = take(fp4 ? 4 * R : 0);
    L.x_sf = take((size_t)chunks * (H / 64) * 512);
    L.h_sf = take((size_t)chunks * (I / 64) * 512);
    L.total = o;
    return L;
}

template <typename T>
T *at(void *ws, size_t off)
{
    return reinterpret_cast<T *>(static_cast<char *>(ws) + off);
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_cfg(const beam_moe_cfg *c)
{
    if (!c)
        return BEAM_MOE_ERR_INVALID_ARG;
    if (c->hidden <= 0 || c->inter <= 0 || c->hidden % 128 || c->inter % 128)
        return BEAM_MOE_ERR_INVALID_ARG;
    if (c->n_experts < 1 || c->n_experts > 256 || c->n_experts % 4)
        return BEAM_MOE_ERR_INVALID_ARG;
    if (c->n_groups < 1 || c->n_groups > 32 || c->n_experts % c->n_groups)
        return BEAM_MOE_ERR_INVALID_ARG;
    const int gsize = c->n_experts / c->n_groups;
    if (gsize > 32 || c->topk_groups < 1 || c->topk_groups > c->n_groups)
        return BEAM_MOE_ERR_INVALID_ARG;
    if (c->top_k < 1 || c->top_k > 32 || c->top_k > c->topk_groups * gsize)
        return BEAM_MOE_ERR_INVALID_ARG;
    if (!(c->routed_scale == c->routed_scale))  // NaN
        return BEAM_MOE_ERR_INVALID_ARG;
    if (c->wtype != BEAM_MOE_W_BF16 && c->wtype != BEAM_MOE_W_NVFP4 &&
        c->wtype != BEAM_MOE_W_MXFP8)
        return BEAM_MOE_ERR_INVALID_ARG;
    return BEAM_MOE_OK;
}

// The block and global scales that NVFP4 / MXFP8 weights need.
int check_scale_ptrs(const beam_moe_cfg *c)
{
    if (c->wtype == BEAM_MOE_W_NVFP4) {
        const void *p[6] = {c->w_gate_sf, c->w_up_sf, c->w_down_sf,
                            c->w_gate_gs, c->w_up_gs, c->w_down_gs};
        for (const void *q : p)
            if (!q || !aligned16(q))
                return BEAM_MOE_ERR_INVALID_ARG;
    }
    if (c->wtype == BEAM_MOE_W_MXFP8) {
        const void *p[3] = {c->w_gate_sf, c->w_up_sf, c->w_down_sf};
        for (const void *q : p)
            if (!q || !aligned16(q))
                return BEAM_MOE_ERR_INVALID_ARG;
    }
    return BEAM_MOE_OK;
}

int check_T(int64_t T, const beam_moe_cfg *c)
{
    if (T < 0 || T * (int64_t)c->top_k >= (int64_t(1) << 31) || T > (int64_t(1) << 24))
        return BEAM_MOE_ERR_INVALID_ARG;
    return BEAM_MOE_OK;
}

int check_ws(int64_t T, const beam_moe_cfg *c, size_t need)
{
    if (!c->workspace || (reinterpret_cast<uintptr_t>(c->workspace) & 255u))
        return BEAM_MOE_ERR_WORKSPACE;
    if (c->workspace_bytes < need)
        return BEAM_MOE_ERR_WORKSPACE;
    (void)T;
    return BEAM_MOE_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 2-D tensor [outer, inner] (inner contiguous), box [box_outer, box_inner],
// zero fill outside.
bool make_map_2d(CUtensorMap *m, const void *base, CUtensorMapDataType dtype, int elem_bytes,
                 uint64_t inner, uint64_t outer, uint32_t box_inner, uint32_t box_outer,
                 CUtensorMapSwizzle swizzle)
{
    auto fn = encode_fn();
    if (!fn)
        return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner * (uint64_t)elem_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t es[2] = {1, 1};
    CUresult r = fn(m, dtype, 2, const_cast<void *>(base), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 16-bit operand [outer, inner], box [box_outer, 64] with the 128-byte swizzle
// the MMA descriptors name.
bool make_map(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer, uint32_t box_outer,
              CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16)
{
    return make_map_2d(m, base, dtype, 2, inner, outer, 64, box_outer, CU_TENSOR_MAP_SWIZZLE_128B);
}

// Packed E2M1 codes [outer rows, inner/2 bytes], box [box_outer rows, 128
// bytes = 256 elements] with the 128-byte swizzle; zero fill past the row end.
bool make_code_map(CUtensorMap *m, const void *base, uint64_t inner_elems, uint64_t outer,
                   uint32_t box_outer)
{
    return make_map_2d(m, base, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, inner_elems / 2, outer, 128,
                       box_outer, CU_TENSOR_MAP_SWIZZLE_128B);
}

int device_sms()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    return n;
}


#define BEAM_CUDA(call)                          \
    do {                                         \
        if ((call) != cudaSuccess)               \
            return BEAM_MOE_ERR_CUDA;            \
    } while (0)

// Steps 1-6 plus histogram/scan into the workspace.  want_scores: the
// caller reads `scores` afterwards (else the selection may skip writing them).
int run_route(const void *x, const float *router_w, int64_t T, const beam_moe_cfg &c,
              const Layout &L, float *scores, bool want_scores, int32_t *ids, float *wts,
              int rows_per_chunk, cudaStream_t s)
{
    void *ws = c.workspace;
    int *status = at<int>(ws, L.status);
    int nsplit = 0;  // 0: the FMA-chain router wrote the scores
    float *partials = scores;
    if (tc_router(T)) {
        const int sms = device_sms();
        if (sms <= 0)
            return BEAM_MOE_ERR_CUDA;
        nsplit = std::min(router_tc_splits(T, c.n_experts, c.hidden, sms),
                          tc_router_layout_splits(T, c));
        if (nsplit > 1)
            partials = at<float>(ws, L.router_partials);
        CUtensorMap mw, mx;
        // 32-deep boxes with the 64-byte swizzle the router's descriptors name
        if (!make_map_2d(&mw, at<void>(ws, L.wr_parts), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                         c.hidden, (uint64_t)3 * c.n_experts, 32, 128,
                         CU_TENSOR_MAP_SWIZZLE_64B) ||
            !make_map_2d(&mx, x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, c.hidden, (uint64_t)T, 32,
                         256, CU_TENSOR_MAP_SWIZZLE_64B))
            return BEAM_MOE_ERR_CUDA;
        const unsigned long long tmo =
            c.wait_timeout_ns > 0 ? (unsigned long long)c.wait_timeout_ns : kDefaultTimeoutNs;
        BEAM_CUDA(launch_router_tc(router_w, at<void>(ws, L.wr_parts), mw, mx, (int)T, c.hidden,
                                   c.n_experts, nsplit, partials, status, tmo, s));
    } else {
        BEAM_CUDA(launch_router_scores(static_cast<const uint16_t *>(x), router_w, (int)T,
                                       c.hidden, c.n_experts, scores, status, s));
    }
    BEAM_CUDA(launch_select(scores, partials, nsplit, want_scores, (int)T, c.n_experts,
                            c.n_groups, c.topk_groups, c.top_k, c.routed_scale, ids, wts, status,
                            s));
    BEAM_CUDA(launch_hist_scan(ids, (int)T, c.top_k, c.n_experts, rows_per_chunk,
                               at<int32_t>(ws, L.local_rank), at<int32_t>(ws, L.cta_counts),
                               at<int32_t>(ws, L.cta_base), at<int32_t>(ws, L.counts),
                               at<int32_t>(ws, L.offsets), at<int32_t>(ws, L.chunk_start), status,
                               s));
    return BEAM_MOE_OK;
}

// Fused-block epilogue: the combine also applies the post-norm and the
// residual update s_out = bf16(a * s_in + b * rmsnorm(o) * gamma).
struct BlockTail {
    const uint16_t *s_in;
    const float *gamma;
    float eps, a, b;
    uint16_t *s_out;
};

int run_forward(const void *x, const float *router_w, const void *w_gate, const void *w_up,
                const void *w_down, int64_t T, const beam_moe_cfg &c, void *out, cudaStream_t s,
                const BlockTail *tail = nullptr)
{
    const Layout L = make_layout(T, c);
    void *ws = c.workspace;
    const GemmVariant v = pick_variant(T, c);
    const bool fp4 = c.wtype == BEAM_MOE_W_NVFP4, mx8 = c.wtype == BEAM_MOE_W_MXFP8;
    int rc = run_route(x, router_w, T, c, L, at<float>(ws, L.scores), false,
                       at<int32_t>(ws, L.ids), at<float>(ws, L.wts), chunk_rows(T, c), s);
    if (rc != BEAM_MOE_OK)
        return rc;
    const int K = c.top_k, E = c.n_experts, H = c.hidden, I = c.inter;
    const int64_t R = T * K;
    if (mx8)
        BEAM_CUDA(launch_permute_mx8(
            static_cast<const uint16_t *>(x), at<int32_t>(ws, L.ids), at<int32_t>(ws, L.local_rank),
            at<int32_t>(ws, L.cta_base), at<int32_t>(ws, L.offsets), at<int32_t>(ws, L.chunk_start),
            (int)T, K, E, H, at<int32_t>(ws, L.row_of), at<int32_t>(ws, L.row_src),
            at<int32_t>(ws, L.row_pos), at<uint8_t>(ws, L.x_perm), at<uint8_t>(ws, L.x_sf), s));
    else if (fp4)
        BEAM_CUDA(launch_permute_nvfp4(
            static_cast<const uint16_t *>(x), at<int32_t>(ws, L.ids), at<int32_t>(ws, L.local_rank),
            at<int32_t>(ws, L.cta_base), at<int32_t>(ws, L.offsets), at<int32_t>(ws, L.chunk_start),
            (int)T, K, E, H, at<int32_t>(ws, L.row_of), at<int32_t>(ws, L.row_src),
            at<int32_t>(ws, L.row_pos), at<uint8_t>(ws, L.x_perm), at<uint8_t>(ws, L.x_sf), s));
    else
        BEAM_CUDA(launch_permute(static_cast<const uint16_t *>(x), at<int32_t>(ws, L.ids),
                                 at<int32_t>(ws, L.local_rank), at<int32_t>(ws, L.cta_base),
                                 at<int32_t>(ws, L.offsets), (int)T, K, E, H,
                                 at<int32_t>(ws, L.row_of), at<int32_t>(ws, L.row_src),
                                 at<void>(ws, L.x_perm), s));

    CUtensorMap m_wg, m_wu, m_wd, m_xp, m_h;
    bool maps_ok;
    if (mx8) {
        // one byte per element: the code maps' "elements" are bytes here
        const uint32_t box = (uint32_t)fp4_box_rows(v);
        maps_ok = make_code_map(&m_wg, w_gate, 2 * H, (uint64_t)E * I, 128) &&
                  make_code_map(&m_wu, w_up, 2 * H, (uint64_t)E * I, 128) &&
                  make_code_map(&m_wd, w_down, 2 * I, (uint64_t)E * H, 128) &&
                  make_code_map(&m_xp, at<void>(ws, L.x_perm), 2 * H, (uint64_t)R, box) &&
                  make_code_map(&m_h, at<void>(ws, L.h), 2 * I, (uint64_t)R, box);
    } else if (fp4) {
        const uint32_t box = (uint32_t)fp4_box_rows(v);
        maps_ok = make_code_map(&m_wg, w_gate, H, (uint64_t)E * I, 128) &&
                  make_code_map(&m_wu, w_up, H, (uint64_t)E * I, 128) &&
                  make_code_map(&m_wd, w_down, I, (uint64_t)E * H, 128) &&
                  make_code_map(&m_xp, at<void>(ws, L.x_perm), H, (uint64_t)R, box) &&
                  make_code_map(&m_h, at<void>(ws, L.h), I, (uint64_t)R, box);
    } else {
        const uint32_t box = (uint32_t)gemm_box_rows(v);
        maps_ok = make_map(&m_wg, w_gate, H, (uint64_t)E * I, 128) &&
                  make_map(&m_wu, w_up, H, (uint64_t)E * I, 128) &&
                  make_map(&m_wd, w_down, I, (uint64_t)E * H, 128) &&
                  make_map(&m_xp, at<void>(ws, L.x_perm), H, (uint64_t)R, box) &&
                  make_map(&m_h, at<void>(ws, L.h), I, (uint64_t)R, box);
    }
    if (!maps_ok)
        return BEAM_MOE_ERR_CUDA;

    const int sms = device_sms();
    if (sms <= 0)
        return BEAM_MOE_ERR_CUDA;
    GemmArgs a{};
    a.offsets = at<int32_t>(ws, L.offsets);
    a.chunk_start = at<int32_t>(ws, L.chunk_start);
    a.E = E;
    a.status = at<int>(ws, L.status);
    a.timeout_ns = c.wait_timeout_ns > 0 ? (unsigned long long)c.wait_timeout_ns : kDefaultTimeoutNs;
    a.debug_flags = c.debug_flags;

    a.m_tiles = I / 128;
    a.ksteps = H / 64;
    a.out = at<void>(ws, L.h);
    a.out_ld = I;
    const bool tm = v == GemmVariant::kPrefill;
    if ((mx8 || fp4) && tm) {
        // token-major gate/up with h quantised in the epilogue
        Fp4Weights f{static_cast<const uint8_t *>(c.w_gate_sf),
                     static_cast<const uint8_t *>(c.w_up_sf), mx8 ? nullptr : c.w_gate_gs,
                     mx8 ? nullptr : c.w_up_gs, at<uint8_t>(ws, L.x_sf)};
        a.out = at<void>(ws, L.h);
        BEAM_CUDA(launch_gateup_tm(mx8, m_wg, m_wu, m_xp, a, f, mx8 ? H / 128 : H / 64,
                                   at<uint8_t>(ws, L.h_sf), at<int32_t>(ws, L.row_pos), sms, s));
    } else if (mx8) {
        Fp4Weights f{static_cast<const uint8_t *>(c.w_gate_sf),
                     static_cast<const uint8_t *>(c.w_up_sf), nullptr, nullptr,
                     at<uint8_t>(ws, L.x_sf)};
        a.out = at<void>(ws, L.h_raw);
        BEAM_CUDA(launch_gateup_mx8(v, m_wg, m_wu, m_xp, a, f, H / 128, sms, s));
        BEAM_CUDA(launch_quantize_rows_mx8(at<float>(ws, L.h_raw), R, I, at<int32_t>(ws, L.row_pos),
                                           at<uint8_t>(ws, L.h), at<uint8_t>(ws, L.h_sf), s));
    } else if (fp4) {
        Fp4Weights f{static_cast<const uint8_t *>(c.w_gate_sf),
                     static_cast<const uint8_t *>(c.w_up_sf), c.w_gate_gs, c.w_up_gs,
                     at<uint8_t>(ws, L.x_sf)};
        a.out = at<void>(ws, L.h_raw);
        BEAM_CUDA(launch_gateup_fp4(v, m_wg, m_wu, m_xp, a, f, H / 64, sms, s));
        BEAM_CUDA(launch_quantize_rows(at<float>(ws, L.h_raw), R, I, at<int32_t>(ws, L.row_pos),
                                       at<uint8_t>(ws, L.h), at<uint8_t>(ws, L.h_sf), s));
    } else {
        BEAM_CUDA(launch_gateup(v, m_wg, m_wu, m_xp, a, sms, s));
    }

    a.m_tiles = H / 128;
    a.ksteps = I / 64;
    a.out = at<void>(ws, L.y);
    a.out_ld = H;
    a.debug_flags = 0;
    if (mx8) {
        Fp4Weights f{static_cast<const uint8_t *>(c.w_down_sf), nullptr, nullptr, nullptr,
                     at<uint8_t>(ws, L.h_sf)};
        if (tm && (H / 128) % 2 == 0)
            BEAM_CUDA(launch_down_tm(true, m_wd, m_h, a, f, I / 128, sms, s));
        else
            BEAM_CUDA(launch_down_mx8(v, m_wd, m_h, a, f, I / 128, sms, s));
    } else if (fp4) {
        Fp4Weights f{static_cast<const uint8_t *>(c.w_down_sf), nullptr, c.w_down_gs, nullptr,
                     at<uint8_t>(ws, L.h_sf)};
        if (tm && (H / 128) % 2 == 0)
            BEAM_CUDA(launch_down_tm(false, m_wd, m_h, a, f, I / 64, sms, s));
        else
            BEAM_CUDA(launch_down_fp4(v, m_wd, m_h, a, f, I / 64, sms, s));
    } else {
        BEAM_CUDA(launch_down(v, m_wd, m_h, a, sms, s));
    }

    if (tail)
        BEAM_CUDA(launch_combine_block(at<uint16_t>(ws, L.y), at<float>(ws, L.wts),
                                       at<int32_t>(ws, L.row_of), (int)T, K, H, tail->s_in,
                                       tail->gamma, tail->eps, tail->a, tail->b, tail->s_out, s));
    else
        BEAM_CUDA(launch_combine(at<uint16_t>(ws, L.y), at<float>(ws, L.wts),
                                 at<int32_t>(ws, L.row_of), (int)T, K, H,
                                 static_cast<uint16_t *>(out), s));
    return BEAM_MOE_OK;
}

// ---- dense SwiGLU layers (the first three decoder layers): the same
// grouped GEMMs with one segment of all T rows, x read in place and the
// down GEMM writing the output rows.
struct DenseLayout {
    size_t status, offsets, chunk_start, h, total;
};

DenseLayout make_dense_layout(int64_t T, const beam_moe_cfg &c)
{
    DenseLayout L{};
    size_t o = 0;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o = align_up(o + bytes);
        return at;
    };
    L.status = take(256);
    L.offsets = take(sizeof(int32_t) * 2);
    L.chunk_start = take(sizeof(int32_t) * 2);
    L.h = take((size_t)2 * T * c.inter);
    L.total = o;
    return L;
}

int check_dense_cfg(const beam_moe_cfg *c)
{
    if (!c)
        return BEAM_MOE_ERR_INVALID_ARG;
    if (c->hidden <= 0 || c->inter <= 0 || c->hidden % 128 || c->inter % 128)
        return BEAM_MOE_ERR_INVALID_ARG;
    if (c->wtype != BEAM_MOE_W_BF16)
        return c->wtype == BEAM_MOE_W_NVFP4 ? BEAM_MOE_ERR_UNSUPPORTED : BEAM_MOE_ERR_INVALID_ARG;
    return BEAM_MOE_OK;
}

int run_dense(const void *x, const void *w_gate, const void *w_up, const void *w_down, int64_t T,
              const beam_moe_cfg &c, void *out, cudaStream_t s)
{
    const DenseLayout L = make_dense_layout(T, c);
    void *ws = c.workspace;
    const int H = c.hidden, I = c.inter;
    const GemmVariant v = T <= 16 ? GemmVariant::kDecode : GemmVariant::kPrefill;
    BEAM_CUDA(launch_dense_setup((int)T, gemm_chunk_rows(v), at<int32_t>(ws, L.offsets),
                                 at<int32_t>(ws, L.chunk_start), at<int>(ws, L.status), s));
    const uint32_t box = (uint32_t)gemm_box_rows(v);
    CUtensorMap m_wg, m_wu, m_wd, m_x, m_h;
    if (!make_map(&m_wg, w_gate, H, (uint64_t)I, 128) ||
        !make_map(&m_wu, w_up, H, (uint64_t)I, 128) ||
        !make_map(&m_wd, w_down, I, (uint64_t)H, 128) ||
        !make_map(&m_x, x, H, (uint64_t)T, box) ||
        !make_map(&m_h, at<void>(ws, L.h), I, (uint64_t)T, box))
        return BEAM_MOE_ERR_CUDA;
    const int sms = device_sms();
    if (sms <= 0)
        return BEAM_MOE_ERR_CUDA;
    GemmArgs a{};
    a.offsets = at<int32_t>(ws, L.offsets);
    a.chunk_start = at<int32_t>(ws, L.chunk_start);
    a.E = 1;
    a.status = at<int>(ws, L.status);
    a.timeout_ns = c.wait_timeout_ns > 0 ? (unsigned long long)c.wait_timeout_ns : kDefaultTimeoutNs;
    a.m_tiles = I / 128;
    a.ksteps = H / 64;
    a.out = at<void>(ws, L.h);
    a.out_ld = I;
    BEAM_CUDA(launch_gateup(v, m_wg, m_wu, m_x, a, sms, s));
    a.m_tiles = H / 128;
    a.ksteps = I / 64;
    a.out = out;
    a.out_ld = H;
    BEAM_CUDA(launch_down(v, m_wd, m_h, a, sms, s));
    return BEAM_MOE_OK;
}

}  // namespace
}  // namespace beam

using namespace beam;

extern "C" {

void beam_moe_cfg_init_beam(beam_moe_cfg *cfg)
{
    if (!cfg)
        return;
    *cfg = beam_moe_cfg{};
    cfg->hidden = 5120;
    cfg->inter = 2560;
    cfg->n_experts = 256;
    cfg->n_groups = 8;
    cfg->topk_groups = 4;
    cfg->top_k = 8;
    cfg->routed_scale = 2.5f;
    cfg->wtype = BEAM_MOE_W_BF16;
}

size_t beam_moe_workspace_size(int64_t T, const beam_moe_cfg *cfg)
{
    if (check_cfg(cfg) != BEAM_MOE_OK || T < 0)
        return 0;
    return make_layout(T, *cfg).total;
}

int beam_moe_router_arith(int64_t T, const beam_moe_cfg *cfg)
{
    if (check_cfg(cfg) != BEAM_MOE_OK || T < 0)
        return BEAM_MOE_ERR_INVALID_ARG;
    return tc_router(T) ? BEAM_MOE_ROUTER_TENSOR : BEAM_MOE_ROUTER_FMA_CHAIN;
}

size_t beam_moe_hostio_extra_bytes(int64_t T, const beam_moe_cfg *cfg)
{
    if (check_cfg(cfg) != BEAM_MOE_OK || T < 0)
        return 0;
    return 2 * align_up((size_t)T * cfg->hidden * 2);
}

int beam_moe_route(const void *x, const float *router_w, int64_t T, const beam_moe_cfg *cfg,
                   int32_t *topk_ids, float *topk_w, float *scores, int32_t *counts,
                   int32_t *offsets, int32_t *row_of, void *stream)
{
    int rc = check_cfg(cfg);
    if (rc != BEAM_MOE_OK)
        return rc;
    if ((rc = check_T(T, cfg)) != BEAM_MOE_OK)
        return rc;
    if (T == 0)
        return BEAM_MOE_OK;
    if (!x || !router_w || !topk_ids || !topk_w || !aligned16(x) || !aligned16(router_w))
        return BEAM_MOE_ERR_INVALID_ARG;
    const beam_moe_cfg &c = *cfg;
    const Layout L = make_layout(T, c);
    if ((rc = check_ws(T, cfg, L.total)) != BEAM_MOE_OK)
        return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    void *ws = c.workspace;
    float *sc = scores ? scores : at<float>(ws, L.scores);
    rc = run_route(x, router_w, T, c, L, sc, scores != nullptr, topk_ids, topk_w,
                   chunk_rows(T, c), s);
    if (rc != BEAM_MOE_OK)
        return rc;
    const int E = c.n_experts;
    if (counts)
        BEAM_CUDA(cudaMemcpyAsync(counts, at<int32_t>(ws, L.counts), sizeof(int32_t) * E,
                                  cudaMemcpyDeviceToDevice, s));
    if (offsets)
        BEAM_CUDA(cudaMemcpyAsync(offsets, at<int32_t>(ws, L.offsets), sizeof(int32_t) * (E + 1),
                                  cudaMemcpyDeviceToDevice, s));
    if (row_of)
        BEAM_CUDA(launch_rows(topk_ids, at<int32_t>(ws, L.local_rank), at<int32_t>(ws, L.cta_base),
                              at<int32_t>(ws, L.offsets), (int)T, c.top_k, E, row_of, s));
    return BEAM_MOE_OK;
}

int beam_moe_forward(const void *x, const float *router_w, const void *w_gate, const void *w_up,
                     const void *w_down, int64_t T, const beam_moe_cfg *cfg, void *out,
                     void *stream)
{
    int rc = check_cfg(cfg);
    if (rc != BEAM_MOE_OK)
        return rc;
    if ((rc = check_T(T, cfg)) != BEAM_MOE_OK)
        return rc;
    if (T == 0)
        return BEAM_MOE_OK;
    if (!x || !router_w || !w_gate || !w_up || !w_down || !out)
        return BEAM_MOE_ERR_INVALID_ARG;
    if ((rc = check_scale_ptrs(cfg)) != BEAM_MOE_OK)
        return rc;
    if (!aligned16(x) || !aligned16(router_w) || !aligned16(w_gate) || !aligned16(w_up) ||
        !aligned16(w_down) || !aligned16(out))
        return BEAM_MOE_ERR_INVALID_ARG;
    if ((rc = check_ws(T, cfg, make_layout(T, *cfg).total)) != BEAM_MOE_OK)
        return rc;
    return run_forward(x, router_w, w_gate, w_up, w_down, T, *cfg, out,
                       static_cast<cudaStream_t>(stream));
}

int beam_moe_forward_hostio(const void *x_host, const float *router_w, const void *w_gate,
                            const void *w_up, const void *w_down, int64_t T,
                            const beam_moe_cfg *cfg, void *out_host, void *stream)
{
    int rc = check_cfg(cfg);
    if (rc != BEAM_MOE_OK)
        return rc;
    if ((rc = check_T(T, cfg)) != BEAM_MOE_OK)
        return rc;
    if (T == 0)
        return BEAM_MOE_OK;
    if (!x_host || !out_host)
        return BEAM_MOE_ERR_INVALID_ARG;
    const size_t base = make_layout(T, *cfg).total;
    const size_t act = align_up((size_t)T * cfg->hidden * 2);
    if ((rc = check_ws(T, cfg, base + 2 * act)) != BEAM_MOE_OK)
        return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    void *x_dev = at<void>(cfg->workspace, base);
    void *o_dev = at<void>(cfg->workspace, base + act);
    const size_t bytes = (size_t)T * cfg->hidden * 2;
    BEAM_CUDA(cudaMemcpyAsync(x_dev, x_host, bytes, cudaMemcpyHostToDevice, s));
    rc = beam_moe_forward(x_dev, router_w, w_gate, w_up, w_down, T, cfg, o_dev, stream);
    if (rc != BEAM_MOE_OK)
        return rc;
    BEAM_CUDA(cudaMemcpyAsync(out_host, o_dev, bytes, cudaMemcpyDeviceToHost, s));
    BEAM_CUDA(cudaStreamSynchronize(s));
    return BEAM_MOE_OK;
}

int beam_moe_quantize_nvfp4(const void *w, int64_t n_mat, int64_t rows, int64_t cols,
                            void *packed, void *block_sf, float *global_sf, void *stream)
{
    if (n_mat == 0 || rows == 0)
        return BEAM_MOE_OK;
    if (n_mat < 0 || rows < 0 || cols <= 0 || rows % 128 || cols % 64 || rows > (1 << 24) ||
        cols > (1 << 24) || n_mat > (1 << 20))
        return BEAM_MOE_ERR_INVALID_ARG;
    if (!w || !packed || !block_sf || !global_sf || !aligned16(w) || !aligned16(packed) ||
        !aligned16(block_sf) || !aligned16(global_sf))
        return BEAM_MOE_ERR_INVALID_ARG;
    BEAM_CUDA(launch_quantize_nvfp4(static_cast<const uint16_t *>(w), n_mat, (int)rows, (int)cols,
                                    static_cast<uint8_t *>(packed),
                                    static_cast<uint8_t *>(block_sf), global_sf,
                                    static_cast<cudaStream_t>(stream)));
    return BEAM_MOE_OK;
}

int beam_moe_quantize_mxfp8(const void *w, int64_t n_mat, int64_t rows, int64_t cols,
                            void *codes, void *block_sf, void *stream)
{
    if (n_mat == 0 || rows == 0)
        return BEAM_MOE_OK;
    if (n_mat < 0 || rows < 0 || cols <= 0 || rows % 128 || cols % 128 || rows > (1 << 24) ||
        cols > (1 << 24) || n_mat > (1 << 20))
        return BEAM_MOE_ERR_INVALID_ARG;
    if (!w || !codes || !block_sf || !aligned16(w) || !aligned16(codes) || !aligned16(block_sf))
        return BEAM_MOE_ERR_INVALID_ARG;
    BEAM_CUDA(launch_quantize_mxfp8(static_cast<const uint16_t *>(w), n_mat, (int)rows, (int)cols,
                                    static_cast<uint8_t *>(codes), static_cast<uint8_t *>(block_sf),
                                    static_cast<cudaStream_t>(stream)));
    return BEAM_MOE_OK;
}

int beam_moe_quantize_act(int wtype, const float *x, int64_t rows, int64_t cols, void *codes,
                          void *sf, void *stream)
{
    if (wtype != BEAM_MOE_W_NVFP4 && wtype != BEAM_MOE_W_MXFP8)
        return BEAM_MOE_ERR_INVALID_ARG;
    const bool mx8 = wtype == BEAM_MOE_W_MXFP8;
    if (rows < 0 || cols <= 0 || cols % (mx8 ? 32 : 16) || cols > (1 << 24) ||
        rows > (int64_t(1) << 31))
        return BEAM_MOE_ERR_INVALID_ARG;
    if (rows == 0)
        return BEAM_MOE_OK;
    if (!x || !codes || !sf || !aligned16(x) || !aligned16(codes))
        return BEAM_MOE_ERR_INVALID_ARG;
    BEAM_CUDA(launch_quantize_act(mx8, x, rows, (int)cols, static_cast<uint8_t *>(codes),
                                  static_cast<uint8_t *>(sf), static_cast<cudaStream_t>(stream)));
    return BEAM_MOE_OK;
}

int beam_moe_read_status(const beam_moe_cfg *cfg, void *stream)
{
    if (!cfg || !cfg->workspace || cfg->workspace_bytes < 256)
        return BEAM_MOE_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int word = 0;
    if (cudaMemcpyAsync(&word, cfg->workspace, sizeof(int), cudaMemcpyDeviceToHost, s) !=
            cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return BEAM_MOE_ERR_CUDA;
    if (cudaMemsetAsync(cfg->workspace, 0, sizeof(int), s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return BEAM_MOE_ERR_CUDA;
    if (word & kStatusTimeout)
        return BEAM_MOE_ERR_TIMEOUT;
    if (word & kStatusDevice)
        return BEAM_MOE_ERR_DEVICE;
    return BEAM_MOE_OK;
}

const char *beam_moe_status_string(int code)
{
    switch (code) {
    case BEAM_MOE_OK: return "ok";
    case BEAM_MOE_ERR_INVALID_ARG: return "invalid argument";
    case BEAM_MOE_ERR_UNSUPPORTED: return "unsupported configuration";
    case BEAM_MOE_ERR_CUDA: return "CUDA call failed";
    case BEAM_MOE_ERR_WORKSPACE: return "workspace missing or too small";
    case BEAM_MOE_ERR_TIMEOUT: return "device wait timed out";
    case BEAM_MOE_ERR_DEVICE: return "device-side check failed";
    default: return "unknown status";
    }
}

int64_t beam_moe_launch_count(void) { return g_launches; }

int beam_moe_set_kernel_events(void *const *start, void *const *stop, int n)
{
    if (n < 0 || n > kNumStages || (n > 0 && (!start || !stop)))
        return BEAM_MOE_ERR_INVALID_ARG;
    for (int i = 0; i < kNumStages; ++i) {
        g_ev_start[i] = i < n ? static_cast<cudaEvent_t>(start[i]) : nullptr;
        g_ev_stop[i] = i < n ? static_cast<cudaEvent_t>(stop[i]) : nullptr;
    }
    g_ev_n = n;
    return BEAM_MOE_OK;
}

int beam_moe_device_sms(void) { return device_sms(); }

size_t beam_moe_dense_workspace_size(int64_t T, const beam_moe_cfg *cfg)
{
    if (check_dense_cfg(cfg) != BEAM_MOE_OK || T < 0)
        return 0;
    return make_dense_layout(T, *cfg).total;
}

int beam_moe_dense_forward(const void *x, const void *w_gate, const void *w_up, const void *w_down,
                           int64_t T, const beam_moe_cfg *cfg, void *out, void *stream)
{
    int rc = check_dense_cfg(cfg);
    if (rc != BEAM_MOE_OK)
        return rc;
    if (T < 0 || T > (int64_t(1) << 24))
        return BEAM_MOE_ERR_INVALID_ARG;
    if (T == 0)
        return BEAM_MOE_OK;
    if (!x || !w_gate || !w_up || !w_down || !out)
        return BEAM_MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w_gate) || !aligned16(w_up) || !aligned16(w_down) ||
        !aligned16(out))
        return BEAM_MOE_ERR_INVALID_ARG;
    if ((rc = check_ws(T, cfg, make_dense_layout(T, *cfg).total)) != BEAM_MOE_OK)
        return rc;
    return run_dense(x, w_gate, w_up, w_down, T, *cfg, out, static_cast<cudaStream_t>(stream));
}

size_t beam_moe_block_workspace_size(int64_t T, const beam_moe_cfg *cfg)
{
    if (check_cfg(cfg) != BEAM_MOE_OK || T < 0)
        return 0;
    return make_layout(T, *cfg).total + align_up((size_t)2 * T * cfg->hidden);
}

int beam_moe_block_forward(const void *stream_in, int step, const float *norm_pre,
                           const float *norm_post, float eps, const float *router_w,
                           const void *w_gate, const void *w_up, const void *w_down, int64_t T,
                           const beam_moe_cfg *cfg, void *stream_out, void *stream)
{
    int rc = check_cfg(cfg);
    if (rc != BEAM_MOE_OK)
        return rc;
    if (cfg->hidden > 8192)
        return BEAM_MOE_ERR_UNSUPPORTED;
    if ((rc = check_T(T, cfg)) != BEAM_MOE_OK)
        return rc;
    if (step < 1 || !(eps >= 0.0f) || eps > 1.0f)
        return BEAM_MOE_ERR_INVALID_ARG;
    if (T == 0)
        return BEAM_MOE_OK;
    if (!stream_in || !norm_pre || !norm_post || !router_w || !w_gate || !w_up || !w_down ||
        !stream_out)
        return BEAM_MOE_ERR_INVALID_ARG;
    if ((rc = check_scale_ptrs(cfg)) != BEAM_MOE_OK)
        return rc;
    if (!aligned16(stream_in) || !aligned16(norm_pre) || !aligned16(norm_post) ||
        !aligned16(router_w) || !aligned16(w_gate) || !aligned16(w_up) || !aligned16(w_down) ||
        !aligned16(stream_out))
        return BEAM_MOE_ERR_INVALID_ARG;
    const size_t base = make_layout(T, *cfg).total;
    if ((rc = check_ws(T, cfg, base + align_up((size_t)2 * T * cfg->hidden))) != BEAM_MOE_OK)
        return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint16_t *x = at<uint16_t>(cfg->workspace, base);
    BEAM_CUDA(launch_rmsnorm_bf16(static_cast<const uint16_t *>(stream_in), norm_pre, eps, (int)T,
                                  cfg->hidden, x, s));
    BlockTail tail;
    tail.s_in = static_cast<const uint16_t *>(stream_in);
    tail.gamma = norm_post;
    tail.eps = eps;
    tail.a = (float)std::sqrt((double)(step - 1) / (double)step);
    tail.b = (float)(1.0 / std::sqrt((double)step));
    tail.s_out = static_cast<uint16_t *>(stream_out);
    return run_forward(x, router_w, w_gate, w_up, w_down, T, *cfg, nullptr, s, &tail);
}

}  // extern "C"
