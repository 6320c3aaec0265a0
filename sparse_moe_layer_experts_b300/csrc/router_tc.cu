// Router logits on the sm_103a tensor cores for prefill-size batches.
//
// The router is computed in FP32 ("Reflection Beam 1.0: 501B open MoE model"
// (agentlenshq.com), section "Residual stream", last paragraph), over the
// sigmoid scores of all experts (same page, section "Mixture of Experts").
//
// x is bf16, so every product x[t,h] * Wr[h,e] needs only Wr's 24-bit
// significand to be exact.  Wr is split once per call into three bf16 parts,
// Wr = hi + mid + lo exactly (hi = bf16(Wr), mid = bf16(Wr - hi),
// lo = Wr - hi - mid, which has at most 8 significant bits), and the logit is
//     l[t,e] = sum_h x[t,h]*hi[e,h] + x[t,h]*mid[e,h] + x[t,h]*lo[e,h]
// on kind::f16 MMAs with FP32 accumulation.  Each product of two bf16 values
// is exact in FP32, so the only difference from a sequential FP32 dot
// product is the order (and grouping) in which the tensor cores add the
// exact products.  The split is exact for |Wr| >= 2^-110; below that lo is
// rounded to bf16's subnormal grid (an error under 2^-133 per weight).
//
// Tile: 128 experts (MMA M, one expert per TMEM lane) x 256 tokens (MMA N,
// the widest MMA, which costs about as much per instruction as narrower
// ones), K = H in 32-deep stages (one 64-byte swizzled row per operand row,
// so that five 40 KB stages fit and four are in flight while the MMAs run).
// Per stage: the three 128 x 32 weight parts and the 256 x 32 x tile by TMA;
// per 16-deep k step three MMAs (hi, mid, lo) into one FP32 accumulator.
// Small batches leave SMs idle with one CTA per (expert tile, token tile),
// so the hidden dimension is split into S ranges (S a power of two chosen
// on the host): CTA (tile, s) sums its range and stores FP32 partial
// logits [S][T][E]; the selection kernel adds the S partials in order
// s = 0..S-1 and applies the sigmoid where the selection needs it (to every
// logit when the caller asks for the scores).  With S = 1 the partials are
// the logits themselves, stored straight into the scores buffer.
// Warp 0 produces, warp 1 owns tensor memory and issues the MMAs, warps 2-5
// read the accumulator and store it.
#include "common.cuh"
#include "gemm_common.cuh"
#include "internal.h"
#include "router_math.cuh"

#include <mutex>

namespace beam {

namespace {

constexpr int kRE = 128;    // experts per tile (MMA M)
constexpr int kRN = 256;    // tokens per tile (MMA N)
constexpr int kRK = 32;     // bf16 per swizzled row (64 bytes)
constexpr int kParts = 3;   // hi, mid, lo
constexpr int kRThreads = 192;
constexpr int kRStages = 5;

struct RCfg {
    static constexpr int PART_BYTES = kRE * kRK * 2;
    static constexpr int A_BYTES = kParts * PART_BYTES;  // weight parts
    static constexpr int B_BYTES = kRN * kRK * 2;        // x tile
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int STAGES = kRStages;
    static constexpr int TMEM_COLS = kRN;
    static constexpr int N_BARS = 2 * STAGES + 2;  // full, empty, accumulator full, drain
    static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + N_BARS * 8 + 16;
    static_assert(STAGE_BYTES % 1024 == 0 && PART_BYTES % 1024 == 0, "swizzle atoms");
    static_assert(kRK * 2 == 64, "the tensor maps and descriptors use the 64-byte swizzle");
    static_assert(SMEM_BYTES <= 232448, "shared memory");
};

// Shared-memory matrix descriptor of a K-major bf16 tile written by TMA with
// the 64-byte swizzle: rows of 32 bf16 (64 B), 8-row atoms of 512 B.
//   bits  0-13 start address >> 4     bits 16-29 leading byte offset >> 4
//   bits 32-45 stride byte offset >> 4 (512 B between 8-row atoms)
//   bits 46-47 descriptor version (1)  bits 61-63 layout (4 = 64B swizzle)
__device__ __forceinline__ uint64_t smem_desc_k64sw(uint32_t saddr)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(16u >> 4) << 16;
    d |= static_cast<uint64_t>(512u >> 4) << 32;
    d |= static_cast<uint64_t>(1u) << 46;
    d |= static_cast<uint64_t>(4u) << 61;
    return d;
}

// Wr [H,E] fp32 (hidden-major) -> parts [3][E][H] bf16 (K-major rows of the
// MMA's B operand).  32 x 32 tiles through shared memory so both the reads
// (E contiguous) and the writes (H contiguous) are coalesced.  Also clears
// the call's status word (this is the call's first kernel).
__global__ void __launch_bounds__(256)
router_split_kernel(const float *__restrict__ wr, int H, int E, __nv_bfloat16 *__restrict__ parts,
                    int *status)
{
    if (status && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0)
        *status = 0;
    __shared__ float tile[32][33];
    const int h0 = blockIdx.x * 32, e0 = blockIdx.y * 32;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 8 rows per pass
    for (int r = ty; r < 32; r += 8) {
        const int h = h0 + r, e = e0 + tx;
        tile[r][tx] = (h < H && e < E) ? wr[(size_t)h * E + e] : 0.0f;
    }
    __syncthreads();
    for (int r = ty; r < 32; r += 8) {
        const int e = e0 + r, h = h0 + tx;
        if (e >= E || h >= H)
            continue;
        const float w = tile[tx][r];
        const __nv_bfloat16 hi = __float2bfloat16_rn(w);
        const float r1 = __fsub_rn(w, __bfloat162float(hi));  // exact
        const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
        const float r2 = __fsub_rn(r1, __bfloat162float(mid));  // exact
        const __nv_bfloat16 lo = __float2bfloat16_rn(r2);      // exact for |w| >= 2^-110
        const size_t o = (size_t)e * H + h, plane = (size_t)E * H;
        parts[o] = hi;
        parts[plane + o] = mid;
        parts[2 * plane + o] = lo;
    }
}

__global__ void __launch_bounds__(kRThreads, 1)
router_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                 int T, int E, int ksteps, int nsplit, float *__restrict__ partials, int *status,
                 unsigned long long timeout_ns)
{
    using C = RCfg;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t base_u32 = (raw_u32 + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (base_u32 - raw_u32);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::STAGES * C::STAGE_BYTES);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + C::N_BARS);
    volatile int *s_abort = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const uint32_t bar_u32 = smem_u32(bars);
    auto full_bar = [&](int s) { return bar_u32 + 8u * s; };
    auto empty_bar = [&](int s) { return bar_u32 + 8u * (C::STAGES + s); };
    const uint32_t tfull_bar = bar_u32 + 8u * (2 * C::STAGES);
    const uint32_t drain_bar = tfull_bar + 8u;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // CTA index = ((token tile * nsplit) + split) * expert tiles + expert tile:
    // the expert tiles (which share the x tile) are adjacent, then the splits
    const int n_etiles = (E + kRE - 1) / kRE;
    const int et = (int)(blockIdx.x % n_etiles);
    const int rest = (int)(blockIdx.x / n_etiles);
    const int split = rest % nsplit, tt = rest / nsplit;
    const int e0 = et * kRE, t0 = tt * kRN;
    const int k_begin = (int)((long long)ksteps * split / nsplit);
    const int k_end = (int)((long long)ksteps * (split + 1) / nsplit);

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        mbar_init(tfull_bar, 1);
        mbar_init(drain_bar, 1);
        *s_abort = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmW);
        tma_prefetch_desc(&tmX);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const uint64_t tmo = timeout_ns;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------------------------------------------- TMA producer
            int stage = 0;
            uint32_t phase = 0, armed = 0, armed_par = 0;
            bool ok = true;
            for (int k = k_begin; k < k_end; ++k) {
                if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, tmo, s_abort, status)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(full_bar(stage), C::STAGE_BYTES);
                armed |= 1u << stage;
                armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
                const uint32_t sa = base_u32 + stage * C::STAGE_BYTES;
#pragma unroll
                for (int p = 0; p < kParts; ++p)
                    tma_load_2d(sa + p * C::PART_BYTES, &tmW, k * kRK, p * E + e0,
                                full_bar(stage));
                tma_load_2d(sa + C::A_BYTES, &tmX, k * kRK, t0, full_bar(stage));
                if (++stage == C::STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) {
                for (int s = 0; s < C::STAGES; ++s)
                    if ((armed >> s) & 1u)
                        mbar_wait_drain(full_bar(s), (armed_par >> s) & 1u, tmo);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------------ MMA issuer
            const uint32_t idesc = idesc_bf16_f32(kRE, kRN);
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int k = k_begin; k < k_end; ++k) {
                if (!mbar_wait_bounded(full_bar(stage), phase, tmo, s_abort, status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t sa = base_u32 + stage * C::STAGE_BYTES;
                const uint32_t sb = sa + C::A_BYTES;
#pragma unroll
                for (int kk = 0; kk < kRK / 16; ++kk) {
                    const uint64_t bd = smem_desc_k64sw(sb + kk * 32);
#pragma unroll
                    for (int p = 0; p < kParts; ++p)
                        mma_bf16_ss(tmem_base, smem_desc_k64sw(sa + p * C::PART_BYTES + kk * 32), bd,
                                    idesc, (k != k_begin || kk != 0 || p != 0) ? 1u : 0u);
                }
                mma_commit(empty_bar(stage));
                if (++stage == C::STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (ok) {
                mma_commit(tfull_bar);
            } else {
                mma_commit(drain_bar);
                mbar_wait_drain(drain_bar, 0, tmo);
            }
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------- epilogue
        // lane quarter q holds experts e0 + 32q .. +31; a 16-column load gives
        // one expert 16 tokens, and each store of a warp covers 32
        // consecutive experts of one token (128 bytes)
        const int q = warp & 3;
        const int e = e0 + q * 32 + lane;
        if (mbar_wait_bounded(tfull_bar, 0, tmo, s_abort, status)) {
            tc_fence_after();
            const uint32_t ta = tmem_base + ((uint32_t)(q * 32) << 16);
            float *dst = partials + (size_t)split * T * E;
#pragma unroll 1
            for (int c0 = 0; c0 < kRN && t0 + c0 < T; c0 += 16) {
                uint32_t r[16];
                tmem_ld16(ta + c0, r);
                tmem_ld_wait();
                if (e < E) {
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        if (t0 + c0 + j < T)
                            dst[(size_t)(t0 + c0 + j) * E + e] = __uint_as_float(r[j]);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

}  // namespace

int router_tc_splits(int64_t T, int E, int H, int sms)
{
    // the largest power of two that keeps the CTA count within the SMs and
    // gives every split at least one 32-deep k step
    const int64_t tiles = ((T + kRN - 1) / kRN) * ((E + kRE - 1) / kRE);
    int s = 1;
    while (s < kRouterMaxSplits && tiles * 2 * s <= sms && 2 * s <= H / kRK)
        s *= 2;
    return s;
}

cudaError_t launch_router_tc(const float *wr, void *parts, const CUtensorMap &w_map,
                             const CUtensorMap &x_map, int T, int H, int E, int nsplit,
                             float *partials, int *status, unsigned long long timeout_ns,
                             cudaStream_t s)
{
    using C = RCfg;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(router_tc_kernel,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    });
    if (attr_err != cudaSuccess)
        return attr_err;
    if (nsplit < 1 || nsplit > kRouterMaxSplits || nsplit > H / kRK)
        return cudaErrorInvalidValue;
    cudaError_t err;
    // the router stage's events bracket both kernels: the split and the GEMM
    stage_begin(kStRouter, s);
    const dim3 sgrid((H + 31) / 32, (E + 31) / 32);
    router_split_kernel<<<sgrid, 256, 0, s>>>(wr, H, E, static_cast<__nv_bfloat16 *>(parts),
                                              status);
    count_launch();
    if ((err = cudaGetLastError()) != cudaSuccess)
        return err;
    const unsigned grid = (unsigned)((E + kRE - 1) / kRE) * (unsigned)nsplit *
                          (unsigned)((T + kRN - 1) / kRN);
    router_tc_kernel<<<grid, kRThreads, C::SMEM_BYTES, s>>>(w_map, x_map, T, E, H / kRK, nsplit,
                                                          partials, status, timeout_ns);
    stage_end(kStRouter, s);
    return cudaGetLastError();
}

}  // namespace beam
