// Grouped expert GEMMs with NVFP4 expert weights (E2M1 codes, one E4M3
// scale per 16 elements, an FP32 scale per expert and projection).
//
// The pages name NVFP4 as the checkpoint for Blackwell ("Reflection Beam
// 1.0", section on hardware requirements: most parameters in 4 bits); the
// recipe is a reading (see nvfp4.cuh).  Each expert is still the SwiGLU MLP of
// the "Mixture of Experts" section with the product in FP32.
//
// The weights stream from HBM as 4-bit codes plus scales (0.5625 B per
// weight).  Converter warps expand each 128x64 tile in shared memory into the
// FP16 values q*sf, which are exact because they need at most 6 significant
// bits.  The tensor cores then run the same kind::f16 MMA as the bf16 path:
// activations are FP16 too, holding the exact NVFP4 values of x (quantised in
// the permute kernel) and of h (the gate/up epilogue writes h in FP32 and a
// streaming pass quantises it).  The global scale multiplies the FP32
// accumulator in the epilogue.
//
// Warp roles:
//   warp 0      producer: TMA of the code tile + bulk copy of its 512 scale
//               bytes into a deep "raw" ring, and TMA of the token tile into
//               the B ring
//   warp 1      TMEM allocator and MMA issuer
//   next 4*EPI_WG warps: epilogue warpgroup(s), splitting a tile's columns
//   last 4 warps converters, one weight row per thread: raw ring -> FP16 A
//               tiles (128-byte swizzled, K-major) of the A ring
#include "common.cuh"
#include "gemm_common.cuh"
#include "internal.h"
#include "nvfp4.cuh"

#include <mutex>

namespace beam {

namespace {

constexpr int kBlockM = 128;
constexpr int kBlockK = 64;
constexpr int kCodeBytes = kBlockM * kBlockK / 2;  // 4096
constexpr int kSfBytes = kBlockM * kBlockK / 16;   // 512
constexpr int kAF16Bytes = kBlockM * kBlockK * 2;  // 16384
constexpr int kMaxExperts = 256;

template <bool GATEUP, int BN, int RS, int AS, int BS, int ACC_BUFS, int BOX, int EPI_WG>
struct CfgF {
    static constexpr int NA = GATEUP ? 2 : 1;
    static constexpr int THREADS = 64 + 128 * EPI_WG + 128;
    static constexpr int CONV_WARP0 = 2 + 4 * EPI_WG;
    static constexpr int BOX_BYTES = BOX * kBlockK * 2;
    static constexpr int RAW_BYTES = NA * (kCodeBytes + kSfBytes);
    static constexpr int A_BYTES = NA * kAF16Bytes;     // converted weight tiles
    static constexpr int B_BYTES = BN * kBlockK * 2;    // token tile
    static constexpr int ACC_COLS = NA * BN;
    static constexpr int COLS_RAW = ACC_BUFS * ACC_COLS;
    static constexpr int TMEM_COLS = COLS_RAW <= 32    ? 32
                                     : COLS_RAW <= 64  ? 64
                                     : COLS_RAW <= 128 ? 128
                                     : COLS_RAW <= 256 ? 256
                                                       : 512;
    static constexpr int N_BARS = 2 * RS + 2 * AS + 2 * BS + 2 * ACC_BUFS + 1;
    static constexpr int AUX_BYTES = N_BARS * 8 + 16 + 2 * (kMaxExperts + 1) * 4;
    static constexpr int SMEM_BYTES = 1024 + AS * A_BYTES + BS * B_BYTES + RS * RAW_BYTES +
                                      ((AUX_BYTES + 127) / 128) * 128;
    static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "MMA N");
    static_assert(BN % BOX == 0 && BOX % 16 == 0, "token boxes tile the B operand");
    static_assert(COLS_RAW <= 512, "TMEM columns");
    static_assert(A_BYTES % 1024 == 0 && B_BYTES % 1024 == 0 && RAW_BYTES % 128 == 0,
                  "alignment");
    static_assert(SMEM_BYTES <= 232448, "shared memory");
};

struct Fp4Params {
    GemmArgs a;
    Fp4Weights f;
    int ksteps_total;  // k-steps per weight matrix row block (for scale tiles)
};

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                         uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// two E2M1 codes (low nibble first) -> f16x2 {low, high}
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte)
{
    uint32_t r;
    const uint16_t b = (uint16_t)byte;
    asm("{\n\t.reg .b8 t;\n\tcvt.u8.u16 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}"
        : "=r"(r)
        : "h"(b));
    return r;
}

// two E4M3 codes (low byte first) -> f16x2 {low, high}
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two)
{
    uint32_t r;
    const uint16_t b = (uint16_t)two;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(b));
    return r;
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b)
{
    const __half2 r = __hmul2(*reinterpret_cast<const __half2 *>(&a),
                              *reinterpret_cast<const __half2 *>(&b));
    return *reinterpret_cast<const uint32_t *>(&r);
}

__device__ __forceinline__ float silu_mul_f(float g, float u)
{
    return __fdividef(g, 1.0f + __expf(-g)) * u;
}

template <bool GATEUP, int BN, int RS, int AS, int BS, int ACC_BUFS, int BOX, int EPI_WG>
__global__ void __launch_bounds__(64 + 128 * EPI_WG + 128, 1)
grouped_gemm_fp4_kernel(const __grid_constant__ CUtensorMap tmA0,
                        const __grid_constant__ CUtensorMap tmA1,
                        const __grid_constant__ CUtensorMap tmB, const Fp4Params P)
{
    using C = CfgF<GATEUP, BN, RS, AS, BS, ACC_BUFS, BOX, EPI_WG>;
    const GemmArgs &p = P.a;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t base_u32 = (raw_u32 + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (base_u32 - raw_u32);
    // [A ring (converted weights) | B ring (tokens) | raw ring | barriers | aux]
    const uint32_t a_u32 = base_u32;
    const uint32_t b_u32 = base_u32 + AS * C::A_BYTES;
    uint8_t *raw_ring = smem + AS * C::A_BYTES + BS * C::B_BYTES;
    const uint32_t rawring_u32 = b_u32 + BS * C::B_BYTES;
    uint64_t *bars = reinterpret_cast<uint64_t *>(raw_ring + RS * C::RAW_BYTES);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + C::N_BARS);
    volatile int *s_abort = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int *s_off = reinterpret_cast<int *>(tmem_slot + 4);
    int *s_cs = s_off + (kMaxExperts + 1);

    const uint32_t bar_u32 = smem_u32(bars);
    auto raw_full = [&](int s) { return bar_u32 + 8u * s; };
    auto raw_empty = [&](int s) { return bar_u32 + 8u * (RS + s); };
    auto a_full = [&](int s) { return bar_u32 + 8u * (2 * RS + s); };
    auto a_empty = [&](int s) { return bar_u32 + 8u * (2 * RS + AS + s); };
    auto b_full = [&](int s) { return bar_u32 + 8u * (2 * RS + 2 * AS + s); };
    auto b_empty = [&](int s) { return bar_u32 + 8u * (2 * RS + 2 * AS + BS + s); };
    constexpr int TB = 2 * RS + 2 * AS + 2 * BS;
    auto tfull_bar = [&](int a) { return bar_u32 + 8u * (TB + a); };
    auto tempty_bar = [&](int a) { return bar_u32 + 8u * (TB + ACC_BUFS + a); };
    const uint32_t drain_bar = bar_u32 + 8u * (TB + 2 * ACC_BUFS);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int E = p.E;

    if (threadIdx.x == 0) {
        for (int s = 0; s < RS; ++s) {
            mbar_init(raw_full(s), 1);
            mbar_init(raw_empty(s), 128);
        }
        for (int s = 0; s < AS; ++s) {
            mbar_init(a_full(s), 128);
            mbar_init(a_empty(s), 1);
        }
        for (int s = 0; s < BS; ++s) {
            mbar_init(b_full(s), 1);
            mbar_init(b_empty(s), 1);
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
            // ------------------- producer: weight codes + scales, token tiles
            int rs = 0, bs = 0;
            uint32_t rph = 0, bph = 0, armed = 0, armed_par = 0, barmed = 0, barmed_par = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
                const Tile tl = decode_tile(t, s_off, s_cs, E, p.m_tiles);
                const int arow = tl.e * p.m_tiles * kBlockM + tl.m * kBlockM;
                const size_t sf_tile = ((size_t)tl.e * p.m_tiles + tl.m) * P.ksteps_total;
                const int nb = (tl.nrows + BOX - 1) / BOX;
                for (int k = 0; k < p.ksteps; ++k) {
                    if (!mbar_wait_bounded(raw_empty(rs), rph ^ 1u, tmo, s_abort, p.status)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(raw_full(rs), C::RAW_BYTES);
                    armed |= 1u << rs;
                    armed_par = (armed_par & ~(1u << rs)) | (rph << rs);
                    const uint32_t dst = rawring_u32 + rs * C::RAW_BYTES;
                    tma_load_2d(dst, &tmA0, k * (kBlockK / 2), arow, raw_full(rs));
                    bulk_g2s(dst + C::NA * kCodeBytes, P.f.sf0 + (sf_tile + k) * kSfBytes, kSfBytes,
                             raw_full(rs));
                    if (GATEUP) {
                        tma_load_2d(dst + kCodeBytes, &tmA1, k * (kBlockK / 2), arow,
                                    raw_full(rs));
                        bulk_g2s(dst + C::NA * kCodeBytes + kSfBytes,
                                 P.f.sf1 + (sf_tile + k) * kSfBytes, kSfBytes, raw_full(rs));
                    }
                    if (++rs == RS) {
                        rs = 0;
                        rph ^= 1u;
                    }
                    if (!mbar_wait_bounded(b_empty(bs), bph ^ 1u, tmo, s_abort, p.status)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(b_full(bs), nb * C::BOX_BYTES);
                    barmed |= 1u << bs;
                    barmed_par = (barmed_par & ~(1u << bs)) | (bph << bs);
                    const uint32_t sb = b_u32 + bs * C::B_BYTES;
                    for (int bb = 0; bb < nb; ++bb)
                        tma_load_2d(sb + bb * C::BOX_BYTES, &tmB, k * kBlockK, tl.row0 + bb * BOX,
                                    b_full(bs));
                    if (++bs == BS) {
                        bs = 0;
                        bph ^= 1u;
                    }
                }
            }
            if (!ok) {
                for (int s = 0; s < RS; ++s)
                    if ((armed >> s) & 1u)
                        mbar_wait_drain(raw_full(s), (armed_par >> s) & 1u, tmo);
                for (int s = 0; s < BS; ++s)
                    if ((barmed >> s) & 1u)
                        mbar_wait_drain(b_full(s), (barmed_par >> s) & 1u, tmo);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            // --------------------------------------------- MMA issuer
            int as = 0, bs = 0, acc = 0;
            uint32_t aph = 0, bph = 0, acc_phase = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
                const Tile tl = decode_tile(t, s_off, s_cs, E, p.m_tiles);
                const uint32_t n = (uint32_t)((tl.nrows + 15) & ~15);
                // f16 x f16 -> f32: the bf16 descriptor with both formats = 0
                const uint32_t idesc = idesc_bf16_f32(kBlockM, n) & ~((7u << 7) | (7u << 10));
                if (!mbar_wait_bounded(tempty_bar(acc), acc_phase ^ 1u, tmo, s_abort, p.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem_base + acc * C::ACC_COLS;
                for (int k = 0; k < p.ksteps; ++k) {
                    if (!mbar_wait_bounded(b_full(bs), bph, tmo, s_abort, p.status) ||
                        !mbar_wait_bounded(a_full(as), aph, tmo, s_abort, p.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = a_u32 + as * C::A_BYTES;
                    const uint32_t sb = b_u32 + bs * C::B_BYTES;
#pragma unroll
                    for (int kk = 0; kk < kBlockK / 16; ++kk) {
                        const uint64_t bd = smem_desc_k128(sb + kk * 32);
                        const uint32_t accum = (k | kk) != 0;
                        mma_bf16_ss(d, smem_desc_k128(sa + kk * 32), bd, idesc, accum);
                        if (GATEUP)
                            mma_bf16_ss(d + BN, smem_desc_k128(sa + kAF16Bytes + kk * 32), bd,
                                        idesc, accum);
                    }
                    mma_commit(a_empty(as));
                    mma_commit(b_empty(bs));
                    if (++as == AS) {
                        as = 0;
                        aph ^= 1u;
                    }
                    if (++bs == BS) {
                        bs = 0;
                        bph ^= 1u;
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
    } else if (warp < C::CONV_WARP0) {
        // ------------------------------------------------- epilogue
        const int q = warp & 3;
        const int i = q * 32 + lane;
        const int wg = (warp - 2) >> 2;  // column chunks wg, wg+EPI_WG, ...
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int t = blockIdx.x; t < n_tiles; t += gridDim.x) {
            const Tile tl = decode_tile(t, s_off, s_cs, E, p.m_tiles);
            const float g0 = P.f.gs0[tl.e];
            const float g1 = GATEUP ? P.f.gs1[tl.e] : 0.0f;
            if (!mbar_wait_bounded(tfull_bar(acc), acc_phase, tmo, s_abort, p.status))
                break;
            tc_fence_after();
            const uint32_t ta = tmem_base + ((uint32_t)(q * 32) << 16) + acc * C::ACC_COLS;
            const int col = tl.m * kBlockM + i;
            for (int c0 = wg * 16; c0 < tl.nrows; c0 += 16 * EPI_WG) {
                uint32_t g[16];
                tmem_ld16(ta + c0, g);
                if constexpr (GATEUP) {
                    uint32_t u[16];
                    tmem_ld16(ta + BN + c0, u);
                    tmem_ld_wait();
                    // h = silu(g) * u, kept in FP32 for a separate pass that
                    // quantises it to NVFP4 before the down GEMM
                    float *out = static_cast<float *>(p.out);
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        if (c0 + j < tl.nrows)
                            out[(size_t)(tl.row0 + c0 + j) * p.out_ld + col] =
                                silu_mul_f(__fmul_rn(__uint_as_float(g[j]), g0),
                                           __fmul_rn(__uint_as_float(u[j]), g1));
                } else {
                    tmem_ld_wait();
                    __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(p.out);
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        if (c0 + j < tl.nrows)
                            out[(size_t)(tl.row0 + c0 + j) * p.out_ld + col] =
                                __float2bfloat16_rn(__fmul_rn(__uint_as_float(g[j]), g0));
                }
            }
            tc_fence_before();
            mbar_arrive(tempty_bar(acc));
            if (++acc == ACC_BUFS) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
    } else {
        // ------------------------------------------------ converters
        const int r = (warp - C::CONV_WARP0) * 32 + lane;  // weight row of the tile
        int rs = 0, as = 0;
        uint32_t rph = 0, aph = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
            for (int k = 0; k < p.ksteps; ++k) {
                if (!mbar_wait_bounded(raw_full(rs), rph, tmo, s_abort, p.status) ||
                    !mbar_wait_bounded(a_empty(as), aph ^ 1u, tmo, s_abort, p.status)) {
                    ok = false;
                    break;
                }
                const uint32_t sa = a_u32 + as * C::A_BYTES;
                const uint8_t *raw = raw_ring + rs * C::RAW_BYTES;
#pragma unroll
                for (int mat = 0; mat < C::NA; ++mat) {
                    const uint4 c0 = *reinterpret_cast<const uint4 *>(raw + mat * kCodeBytes + r * 32);
                    const uint4 c1 =
                        *reinterpret_cast<const uint4 *>(raw + mat * kCodeBytes + r * 32 + 16);
                    const uint32_t sfw = *reinterpret_cast<const uint32_t *>(
                        raw + C::NA * kCodeBytes + mat * kSfBytes + r * 4);
                    const uint32_t s01 = e4m3x2_to_f16x2(sfw & 0xFFFFu);
                    const uint32_t s23 = e4m3x2_to_f16x2(sfw >> 16);
                    const uint32_t sfb[4] = {__byte_perm(s01, 0, 0x1010), __byte_perm(s01, 0, 0x3232),
                                             __byte_perm(s23, 0, 0x1010), __byte_perm(s23, 0, 0x3232)};
                    const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
                    const uint32_t row_base = sa + mat * kAF16Bytes + r * 128;
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const uint32_t sc = sfb[c >> 1];
                        const uint32_t o0 = hmul2_u32(e2m1x2_to_f16x2(w[c] & 0xFFu), sc);
                        const uint32_t o1 = hmul2_u32(e2m1x2_to_f16x2((w[c] >> 8) & 0xFFu), sc);
                        const uint32_t o2 = hmul2_u32(e2m1x2_to_f16x2((w[c] >> 16) & 0xFFu), sc);
                        const uint32_t o3 = hmul2_u32(e2m1x2_to_f16x2(w[c] >> 24), sc);
                        const uint32_t dst = row_base + ((uint32_t)(c ^ (r & 7)) << 4);
                        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(o0),
                                     "r"(o1), "r"(o2), "r"(o3)
                                     : "memory");
                    }
                }
                fence_proxy_async_smem();
                mbar_arrive(raw_empty(rs));
                mbar_arrive(a_full(as));
                if (++rs == RS) {
                    rs = 0;
                    rph ^= 1u;
                }
                if (++as == AS) {
                    as = 0;
                    aph ^= 1u;
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

template <bool GATEUP, int BN, int RS, int AS, int BS, int ACC_BUFS, int BOX, int EPI_WG>
cudaError_t launch_fp4_variant(const CUtensorMap &a0, const CUtensorMap &a1, const CUtensorMap &b,
                               const GemmArgs &args, const Fp4Weights &f, int grid, int stage,
                               cudaStream_t s)
{
    using C = CfgF<GATEUP, BN, RS, AS, BS, ACC_BUFS, BOX, EPI_WG>;
    auto kern = grouped_gemm_fp4_kernel<GATEUP, BN, RS, AS, BS, ACC_BUFS, BOX, EPI_WG>;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        C::SMEM_BYTES);
    });
    if (attr_err != cudaSuccess)
        return attr_err;
    Fp4Params P;
    P.a = args;
    P.f = f;
    P.ksteps_total = args.ksteps;
    stage_begin(stage, s);
    kern<<<grid, C::THREADS, C::SMEM_BYTES, s>>>(a0, a1, b, P);
    stage_end(stage, s);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gateup_fp4(GemmVariant v, const CUtensorMap &wg, const CUtensorMap &wu,
                              const CUtensorMap &xp, const GemmArgs &a, const Fp4Weights &f,
                              int grid, cudaStream_t s)
{
    if (v == GemmVariant::kDecode)
        return launch_fp4_variant<true, 32, 12, 3, 4, 2, 16, 1>(wg, wu, xp, a, f, grid, kStGateUp, s);
    return launch_fp4_variant<true, 256, 6, 2, 3, 1, 128, 2>(wg, wu, xp, a, f, grid, kStGateUp, s);
}

cudaError_t launch_down_fp4(GemmVariant v, const CUtensorMap &wd, const CUtensorMap &hp,
                            const GemmArgs &a, const Fp4Weights &f, int grid, cudaStream_t s)
{
    if (v == GemmVariant::kDecode)
        return launch_fp4_variant<false, 32, 16, 4, 6, 2, 16, 1>(wd, wd, hp, a, f, grid, kStDown, s);
    return launch_fp4_variant<false, 256, 10, 2, 4, 2, 128, 2>(wd, wd, hp, a, f, grid, kStDown, s);
}

}  // namespace beam
