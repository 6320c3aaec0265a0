// Grouped expert GEMMs of the Beam MoE layer on the sm_103a tensor cores
// (tcgen05.mma, accumulators in tensor memory, operands staged by TMA).
//
// Each expert is a SwiGLU MLP ("Reflection Beam 1.0" (agentlenshq.com),
// section "Mixture of Experts": SwiGLU experts of intermediate size 2560)
// with the SiLU(gate) * up product in FP32 (same page, section "Residual
// stream", last paragraph).
//
// Layout: the weights are the MMA's M operand (128 weight rows per tile) and
// the expert's token rows the N operand ("swap AB"), so one tile covers
// between 16 and BN tokens of one expert in steps of 16 and a lightly loaded
// expert wastes little work.  Both operands are K-major; TMA writes them with
// the 128-byte swizzle that the MMA descriptors name.
//
//   gate/up: D_g[i, n] = sum_h Wg[e, m0+i, h] * Xp[row0+n, h]  (TMEM cols 0..BN)
//            D_u[i, n] = sum_h Wu[e, m0+i, h] * Xp[row0+n, h]  (cols BN..2BN)
//            h[row0+n, m0+i] = bf16( silu(D_g) * D_u )   in FP32
//   down:    D[i, n]   = sum_j Wd[e, m0+i, j] * Hp[row0+n, j]
//            y[row0+n, m0+i] = bf16(D)   (the combine sums the K rows in FP32)
//
// Persistent kernel, one CTA per SM, warp-specialised:
//   warp 0      TMA producer (one thread)
//   warp 1      TMEM allocator and MMA issuer (one thread)
//   warps 2..   epilogue warpgroup(s): tcgen05.ld from TMEM, SwiGLU, global
//               stores; with two warpgroups each takes every other 16-column
//               chunk of the tile
// Tiles are enumerated expert by expert, weight tile by weight tile, token
// chunk fastest, so CTAs that run at the same time share weight tiles in L2.
#include "common.cuh"
#include "gemm_common.cuh"
#include "internal.h"

#include <mutex>

namespace beam {

namespace {

constexpr int kNonEpiThreads = 64;  // producer warp + MMA warp
constexpr int kBlockM = 128;
constexpr int kBlockK = 64;  // 64 bf16 = one 128-byte swizzle row
constexpr int kABytes = kBlockM * kBlockK * 2;
constexpr int kMaxExperts = 256;

// BOX: token rows per TMA box of the B operand (bigger boxes, fewer TMA
// operations); EPI_WG: epilogue warpgroups, which split a tile's columns.
template <bool GATEUP, int BN, int STAGES, int ACC_BUFS, int BOX, int EPI_WG>
struct Cfg {
    static constexpr int NA = GATEUP ? 2 : 1;
    static constexpr int THREADS = kNonEpiThreads + 128 * EPI_WG;
    static constexpr int BOX_BYTES = BOX * kBlockK * 2;
    static constexpr int B_BYTES = BN * kBlockK * 2;
    static constexpr int STAGE_BYTES = NA * kABytes + B_BYTES;
    static constexpr int ACC_COLS = NA * BN;
    static constexpr int COLS_RAW = ACC_BUFS * ACC_COLS;
    static constexpr int TMEM_COLS = COLS_RAW <= 32    ? 32
                                     : COLS_RAW <= 64  ? 64
                                     : COLS_RAW <= 128 ? 128
                                     : COLS_RAW <= 256 ? 256
                                                       : 512;
    static constexpr int N_BARS = 2 * STAGES + 2 * ACC_BUFS + 1;
    // barriers, tmem slot, abort flag, offsets[E+1], chunk_start[E+1]
    static constexpr int AUX_BYTES = N_BARS * 8 + 16 + 2 * (kMaxExperts + 1) * 4;
    static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + ((AUX_BYTES + 127) / 128) * 128;
    static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "MMA N");
    static_assert(BN % BOX == 0 && BOX % 16 == 0, "token boxes tile the B operand");
    static_assert(COLS_RAW <= 512, "TMEM columns");
    static_assert(SMEM_BYTES <= 232448, "shared memory");
};

__device__ __forceinline__ float silu_mul(float g, float u)
{
    return __fdividef(g, 1.0f + __expf(-g)) * u;
}

template <bool GATEUP, int BN, int STAGES, int ACC_BUFS, int BOX, int EPI_WG>
__global__ void __launch_bounds__(kNonEpiThreads + 128 * EPI_WG, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA0,
                    const __grid_constant__ CUtensorMap tmA1,
                    const __grid_constant__ CUtensorMap tmB, const GemmArgs p)
{
    using C = Cfg<GATEUP, BN, STAGES, ACC_BUFS, BOX, EPI_WG>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t base_u32 = (raw_u32 + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (base_u32 - raw_u32);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + STAGES * C::STAGE_BYTES);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + C::N_BARS);
    volatile int *s_abort = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int *s_off = reinterpret_cast<int *>(tmem_slot + 4);
    int *s_cs = s_off + (kMaxExperts + 1);

    const uint32_t tiles_u32 = base_u32;
    const uint32_t bar_u32 = smem_u32(bars);
    auto full_bar = [&](int s) { return bar_u32 + 8u * s; };
    auto empty_bar = [&](int s) { return bar_u32 + 8u * (STAGES + s); };
    auto tfull_bar = [&](int a) { return bar_u32 + 8u * (2 * STAGES + a); };
    auto tempty_bar = [&](int a) { return bar_u32 + 8u * (2 * STAGES + ACC_BUFS + a); };
    const uint32_t drain_bar = bar_u32 + 8u * (2 * STAGES + 2 * ACC_BUFS);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int E = p.E;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < ACC_BUFS; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), 128 * EPI_WG);
        }
        mbar_init(drain_bar, 1);
        *s_abort = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA0);
        if (GATEUP)
            tma_prefetch_desc(&tmA1);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    for (int i = threadIdx.x; i <= E; i += C::THREADS) {
        s_off[i] = p.offsets[i];
        s_cs[i] = p.chunk_start[i];
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int n_tiles = p.m_tiles * s_cs[E];
    const uint64_t tmo = p.timeout_ns;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            int stage = 0;
            uint32_t phase = 0;
            uint32_t armed = 0, armed_par = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
                const Tile tl = decode_tile(t, s_off, s_cs, E, p.m_tiles);
                const int arow = tl.e * p.m_tiles * kBlockM + tl.m * kBlockM;
                const int nb = (tl.nrows + BOX - 1) / BOX;
                const uint32_t bytes = C::NA * kABytes + nb * C::BOX_BYTES;
                for (int k = 0; k < p.ksteps; ++k) {
                    if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, tmo, s_abort, p.status)) {
                        ok = false;
                        break;
                    }
                    const bool drop = (p.debug_flags & 1u) && blockIdx.x == 0 &&
                                      t == (int)blockIdx.x && k == 1;
                    if (!drop) {
                        mbar_arrive_expect_tx(full_bar(stage), bytes);
                        armed |= 1u << stage;
                        armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
                        const uint32_t sa = tiles_u32 + stage * C::STAGE_BYTES;
                        tma_load_2d(sa, &tmA0, k * kBlockK, arow, full_bar(stage));
                        if (GATEUP)
                            tma_load_2d(sa + kABytes, &tmA1, k * kBlockK, arow, full_bar(stage));
                        const uint32_t sb = sa + C::NA * kABytes;
                        for (int b = 0; b < nb; ++b)
                            tma_load_2d(sb + b * C::BOX_BYTES, &tmB, k * kBlockK,
                                        tl.row0 + b * BOX, full_bar(stage));
                    }
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                for (int s = 0; s < STAGES; ++s)
                    if ((armed >> s) & 1u)
                        mbar_wait_drain(full_bar(s), (armed_par >> s) & 1u, tmo);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------ MMA issuer
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
                const Tile tl = decode_tile(t, s_off, s_cs, E, p.m_tiles);
                const uint32_t n = (uint32_t)((tl.nrows + 15) & ~15);
                const uint32_t idesc = idesc_bf16_f32(kBlockM, n);
                if (!mbar_wait_bounded(tempty_bar(acc), acc_phase ^ 1u, tmo, s_abort, p.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem_base + acc * C::ACC_COLS;
                for (int k = 0; k < p.ksteps; ++k) {
                    if (!mbar_wait_bounded(full_bar(stage), phase, tmo, s_abort, p.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = tiles_u32 + stage * C::STAGE_BYTES;
                    const uint32_t sb = sa + C::NA * kABytes;
#pragma unroll
                    for (int kk = 0; kk < kBlockK / 16; ++kk) {
                        const uint64_t bd = smem_desc_k128(sb + kk * 32);
                        const uint32_t accum = (k | kk) != 0;
                        mma_bf16_ss(d, smem_desc_k128(sa + kk * 32), bd, idesc, accum);
                        if (GATEUP)
                            mma_bf16_ss(d + BN, smem_desc_k128(sa + kABytes + kk * 32), bd, idesc,
                                        accum);
                    }
                    mma_commit(empty_bar(stage));
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok)
                    break;
                mma_commit(tfull_bar(acc));
                if (++acc == ACC_BUFS) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            if (!ok) {
                mma_commit(drain_bar);
                mbar_wait_drain(drain_bar, 0, tmo);
            }
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------- epilogue
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const int i = q * 32 + lane;
        const int wg = (warp - 2) >> 2;  // this warpgroup takes column chunks wg, wg+EPI_WG, ...
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int t = blockIdx.x; t < n_tiles; t += gridDim.x) {
            const Tile tl = decode_tile(t, s_off, s_cs, E, p.m_tiles);
            if (!mbar_wait_bounded(tfull_bar(acc), acc_phase, tmo, s_abort, p.status))
                break;
            tc_fence_after();
            const uint32_t ta = tmem_base + ((uint32_t)(q * 32) << 16) + acc * C::ACC_COLS;
            const int col = tl.m * kBlockM + i;
            for (int c0 = wg * 16; c0 < tl.nrows; c0 += 16 * EPI_WG) {
                uint32_t g[16];
                tmem_ld16(ta + c0, g);
                if (GATEUP) {
                    uint32_t u[16];
                    tmem_ld16(ta + BN + c0, u);
                    tmem_ld_wait();
                    __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(p.out);
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        if (c0 + j < tl.nrows)
                            out[(size_t)(tl.row0 + c0 + j) * p.out_ld + col] = __float2bfloat16_rn(
                                silu_mul(__uint_as_float(g[j]), __uint_as_float(u[j])));
                } else {
                    tmem_ld_wait();
                    __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(p.out);
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        if (c0 + j < tl.nrows)
                            out[(size_t)(tl.row0 + c0 + j) * p.out_ld + col] =
                                __float2bfloat16_rn(__uint_as_float(g[j]));
                }
            }
            tc_fence_before();
            mbar_arrive(tempty_bar(acc));
            if (++acc == ACC_BUFS) {
                acc = 0;
                acc_phase ^= 1u;
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

template <bool GATEUP, int BN, int STAGES, int ACC_BUFS, int BOX, int EPI_WG>
cudaError_t launch_variant(const CUtensorMap &a0, const CUtensorMap &a1, const CUtensorMap &b,
                           const GemmArgs &args, int grid, int stage, cudaStream_t s)
{
    using C = Cfg<GATEUP, BN, STAGES, ACC_BUFS, BOX, EPI_WG>;
    auto kern = grouped_gemm_kernel<GATEUP, BN, STAGES, ACC_BUFS, BOX, EPI_WG>;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        C::SMEM_BYTES);
    });
    if (attr_err != cudaSuccess)
        return attr_err;
    stage_begin(stage, s);
    kern<<<grid, C::THREADS, C::SMEM_BYTES, s>>>(a0, a1, b, args);
    stage_end(stage, s);
    return cudaGetLastError();
}

}  // namespace

int gemm_chunk_rows(GemmVariant v)
{
    return v == GemmVariant::kDecode ? 32 : 256;
}

int gemm_box_rows(GemmVariant v)
{
    return v == GemmVariant::kDecode ? 16 : 128;
}

cudaError_t launch_gateup(GemmVariant v, const CUtensorMap &wg, const CUtensorMap &wu,
                          const CUtensorMap &xp, const GemmArgs &a, int grid, cudaStream_t s)
{
    if (v == GemmVariant::kDecode)
        return launch_variant<true, 32, 6, 2, 16, 1>(wg, wu, xp, a, grid, kStGateUp, s);
    return launch_variant<true, 256, 3, 1, 128, 2>(wg, wu, xp, a, grid, kStGateUp, s);
}

cudaError_t launch_down(GemmVariant v, const CUtensorMap &wd, const CUtensorMap &hp,
                        const GemmArgs &a, int grid, cudaStream_t s)
{
    if (v == GemmVariant::kDecode)
        return launch_variant<false, 32, 10, 2, 16, 1>(wd, wd, hp, a, grid, kStDown, s);
    if (a.m_tiles % 2 == 0)
        return launch_down_pair(wd, hp, a, grid, s);
    return launch_variant<false, 256, 4, 2, 128, 2>(wd, wd, hp, a, grid, kStDown, s);
}

}  // namespace beam
