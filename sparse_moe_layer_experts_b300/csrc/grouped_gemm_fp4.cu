// Grouped expert GEMMs in NVFP4 on the FP4 tensor cores: E2M1 weights and
// activations, one E4M3 scale per 16 elements, an FP32 scale per expert and
// projection.
//
// The pages name NVFP4 as the checkpoint for Blackwell ("Reflection Beam
// 1.0", section on hardware requirements: most parameters in 4 bits); the
// recipe is a reading (see nvfp4.cuh).  Each expert is still the SwiGLU MLP of
// the "Mixture of Experts" section with the product in FP32.
//
// Both operands stay 4-bit from HBM to the tensor core.  Weights are the
// M = 128 operand (swap-AB, as in the bf16 kernels), an expert's token rows
// the N operand (16..128).  One k-step covers 256 elements: a 128-byte
// swizzled row of codes per operand row, and four 512-byte scale atoms per
// operand (the scales of 128 rows x 64 elements, row r = m0 + 32*m1 at byte
// 16*m0 + 4*m1).  The MMA issuer copies the atoms from shared memory into
// tensor memory (tcgen05.cp, 32x128b, replicated to the four lane quarters)
// and runs tcgen05.mma kind::mxf4nvf4 with block16 scales, which
// accumulates sum(q_a*sf_a * q_b*sf_b) in FP32.  The FP32 global scale of
// the weights multiplies the accumulator in the epilogue (activations have
// global scale 1).
//
// Activation scales are laid out per token chunk (the N tile of one work
// unit), written by the kernels that quantise x and h: atoms
// [chunk, K/64, 512] for chunks of <= 128 rows.  K must be a multiple of
// 64: a last k-step with fewer than four 64-blocks issues fewer MMAs, and its
// code tiles are zero-filled by TMA past the row end.  (Prefill-size batches
// mostly run the token-major kernels of grouped_gemm_tm.cu.)
//
// MX8 variants run the MXFP8 experts (E4M3 values, one power-of-two UE8M0
// scale per 32 elements, no global scale) through the same pipeline: a
// k-step is 128 FP8 elements (the same 128-byte row), its scales one atom
// per operand (4 bytes per row, one per 32-block), copied once, and the four
// MMAs of kind::mxf8f6f4 (K = 32, scale_vec::1X) pick byte kk of it with the
// scale-factor ids of the instruction descriptor.
//
// Warp roles: warp 0 TMA/bulk-copy producer, warp 1 TMEM allocator and MMA
// issuer, then EPI_WG epilogue warpgroups splitting a tile's columns, and
// with SFST a scale warpgroup: it writes each stage's scale atoms into tensor
// memory with tcgen05.st (each warp its lane quarter, the layout of a
// 32x128b.warpx4 copy) and signals the MMA thread, so the tensor pipe issues
// only MMAs.  A stage's scale columns are its atoms in shared-memory order
// (weights A0, A1, then tokens), column c = word c % 4 of atom c / 4.
#include "common.cuh"
#include "gemm_common.cuh"
#include "internal.h"
#include "blockscaled.cuh"
#include "nvfp4.cuh"

#include <mutex>

namespace beam {

namespace {

constexpr int kBlockM = 128;
constexpr int kKStep = 256;                       // FP4 elements per k-step
constexpr int kRowBytes = kKStep / 2;             // 128: one swizzle row
constexpr int kACodeBytes = kBlockM * kRowBytes;  // 16384
constexpr int kAtom = 512;                        // scales of 128 rows x 64 elements
constexpr int kSfStep = 4 * kAtom;                // scales of one k-step
constexpr int kMaxExperts = 256;

template <bool GATEUP, int BN, int STAGES, int ACC_BUFS, int BOX, int EPI_WG, bool MX8 = false,
          bool SFST = false>
struct CfgN {
    static constexpr int NA = GATEUP ? 2 : 1;
    static constexpr int THREADS = 64 + 128 * EPI_WG + (SFST ? 128 : 0);
    static constexpr int SF_W0 = 2 + 4 * EPI_WG;  // first scale warp (SFST)
    static constexpr int A_BYTES = NA * kACodeBytes;
    static constexpr int B_BYTES = BN * kRowBytes;
    static constexpr int SFA_MAT = MX8 ? kAtom : kSfStep;  // one weight matrix's scales per stage
    static constexpr int SFA_BYTES = NA * SFA_MAT;
    static constexpr int SFB_KB_BYTES = kAtom;  // token scales of one 64-block
    static constexpr int SFB_BYTES = MX8 ? kAtom : 4 * SFB_KB_BYTES;
    static constexpr int SF_BYTES = ((SFA_BYTES + SFB_BYTES + 1023) / 1024) * 1024;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SF_BYTES;
    static constexpr int BOX_BYTES = BOX * kRowBytes;
    static constexpr int ACC_COLS = NA * BN;
    static constexpr int SFA_COLS = MX8 ? 4 : 16;  // per weight matrix and stage
    static constexpr int SFB_COLS = MX8 ? 4 : 16;
    static constexpr int SF_COLS = NA * SFA_COLS + SFB_COLS;
    static constexpr int SF_COL0 = ACC_BUFS * ACC_COLS;
    static constexpr int COLS_NEED = SF_COL0 + STAGES * SF_COLS;
    static constexpr int TMEM_COLS = COLS_NEED <= 32    ? 32
                                     : COLS_NEED <= 64  ? 64
                                     : COLS_NEED <= 128 ? 128
                                     : COLS_NEED <= 256 ? 256
                                                        : 512;
    static constexpr int N_BARS = 3 * STAGES + 2 * ACC_BUFS + 1;
    static constexpr int AUX_BYTES = N_BARS * 8 + 16 + 2 * (kMaxExperts + 1) * 4;
    static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + ((AUX_BYTES + 127) / 128) * 128;
    static_assert(BN % 16 == 0 && BN >= 16 && BN <= 128, "MMA N; token scale atoms per chunk");
    static_assert(BN % BOX == 0 && BOX % 8 == 0, "token boxes tile the B operand");
    static_assert(COLS_NEED <= 512, "TMEM columns");
    static_assert(STAGE_BYTES % 1024 == 0 && B_BYTES % 1024 == 0, "swizzle-atom alignment");
    static_assert(SMEM_BYTES <= 232448, "shared memory");
    static_assert(!SFST || (!MX8 && SF_COLS % 16 == 0 && SF_COL0 % 16 == 0),
                  "scale staging: NVFP4, whole 16-column stores");
};

struct Fp4Params {
    GemmArgs a;
    Fp4Weights f;
    int kblocks;  // 512-byte scale atoms per operand row tile: K / 64 (NVFP4), K / 128 (MXFP8)
};

template <bool GATEUP, int BN, int STAGES, int ACC_BUFS, int BOX, int EPI_WG, bool MX8, bool SFST>
__global__ void __launch_bounds__(CfgN<GATEUP, BN, STAGES, ACC_BUFS, BOX, EPI_WG, MX8, SFST>::THREADS, 1)
grouped_gemm_nvf4_kernel(const __grid_constant__ CUtensorMap tmA0,
                         const __grid_constant__ CUtensorMap tmA1,
                         const __grid_constant__ CUtensorMap tmB, const Fp4Params P)
{
    using C = CfgN<GATEUP, BN, STAGES, ACC_BUFS, BOX, EPI_WG, MX8, SFST>;
    const GemmArgs &p = P.a;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t base_u32 = (raw_u32 + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (base_u32 - raw_u32);
    // stage s: [A codes | B codes | A scale atoms | B scale atoms]
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + STAGES * C::STAGE_BYTES);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + C::N_BARS);
    volatile int *s_abort = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int *s_off = reinterpret_cast<int *>(tmem_slot + 4);
    int *s_cs = s_off + (kMaxExperts + 1);

    const uint32_t bar_u32 = smem_u32(bars);
    auto full_bar = [&](int s) { return bar_u32 + 8u * s; };
    auto empty_bar = [&](int s) { return bar_u32 + 8u * (STAGES + s); };
    auto tfull_bar = [&](int a) { return bar_u32 + 8u * (2 * STAGES + a); };
    auto tempty_bar = [&](int a) { return bar_u32 + 8u * (2 * STAGES + ACC_BUFS + a); };
    const uint32_t drain_bar = bar_u32 + 8u * (2 * STAGES + 2 * ACC_BUFS);
    auto sfready_bar = [&](int s) { return bar_u32 + 8u * (2 * STAGES + 2 * ACC_BUFS + 1 + s); };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int E = p.E;
    const int KB = P.kblocks;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < ACC_BUFS; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), 128 * EPI_WG);
        }
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(sfready_bar(s), 4);  // one arrive per scale warp (SFST)
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
            // ------------------------- producer: codes by TMA, scales by bulk copy
            int stage = 0;
            uint32_t phase = 0, armed = 0, armed_par = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
                const Tile tl = decode_tile(t, s_off, s_cs, E, p.m_tiles);
                const size_t wtile = (size_t)tl.e * p.m_tiles + tl.m;
                const int arow = (int)wtile * kBlockM;
                const uint8_t *sfa0 = P.f.sf0 + wtile * KB * kAtom;
                const uint8_t *sfa1 = GATEUP ? P.f.sf1 + wtile * KB * kAtom : nullptr;
                // the tile's token chunk (its first row sits at position 0)
                int j0;
                const int chunk =
                    s_cs[tl.e] + nvfp4_chunk_of_row(tl.row0 - s_off[tl.e], s_off[tl.e + 1] - s_off[tl.e],
                                                    s_cs[tl.e + 1] - s_cs[tl.e], &j0);
                const uint8_t *sfb = P.f.act_sf + (size_t)chunk * KB * C::SFB_KB_BYTES;
                const int nb = (tl.nrows + BOX - 1) / BOX;
                for (int k = 0; k < p.ksteps; ++k) {
                    // scale atoms of this k-step: MXFP8 one per operand, NVFP4
                    // one per 64-block (a short last k-step has fewer)
                    const int nkb = MX8 ? 1 : min(4, KB - 4 * k);
                    const int atom0 = MX8 ? k : 4 * k;
                    if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, tmo, s_abort, p.status)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(full_bar(stage),
                                          (uint32_t)(C::A_BYTES + nb * C::BOX_BYTES +
                                                     nkb * (kAtom * C::NA + C::SFB_KB_BYTES)));
                    armed |= 1u << stage;
                    armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
                    const uint32_t st = base_u32 + stage * C::STAGE_BYTES;
                    const uint32_t sf = st + C::A_BYTES + C::B_BYTES;
                    tma_load_2d(st, &tmA0, k * kRowBytes, arow, full_bar(stage));
                    if (GATEUP)
                        tma_load_2d(st + kACodeBytes, &tmA1, k * kRowBytes, arow, full_bar(stage));
                    for (int bb = 0; bb < nb; ++bb)
                        tma_load_2d(st + C::A_BYTES + bb * C::BOX_BYTES, &tmB, k * kRowBytes,
                                    tl.row0 + bb * BOX, full_bar(stage));
                    bulk_g2s(sf, sfa0 + (size_t)atom0 * kAtom, nkb * kAtom, full_bar(stage));
                    if (GATEUP)
                        bulk_g2s(sf + C::SFA_MAT, sfa1 + (size_t)atom0 * kAtom, nkb * kAtom,
                                 full_bar(stage));
                    bulk_g2s(sf + C::SFA_BYTES, sfb + (size_t)atom0 * C::SFB_KB_BYTES,
                             nkb * C::SFB_KB_BYTES, full_bar(stage));
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok)
                for (int s = 0; s < STAGES; ++s)
                    if ((armed >> s) & 1u)
                        mbar_wait_drain(full_bar(s), (armed_par >> s) & 1u, tmo);
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            // --------------------------------------------- MMA issuer
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
                const Tile tl = decode_tile(t, s_off, s_cs, E, p.m_tiles);
                const uint32_t n_mma = (uint32_t)((tl.nrows + 15) & ~15);
                const uint32_t idesc = MX8 ? idesc_mx8(kBlockM, n_mma) : idesc_nvf4(kBlockM, n_mma);
                if (!mbar_wait_bounded(tempty_bar(acc), acc_phase ^ 1u, tmo, s_abort, p.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem_base + acc * C::ACC_COLS;
                for (int k = 0; k < p.ksteps; ++k) {
                    const int nkb = MX8 ? 4 : min(4, KB - 4 * k);  // MMAs of this k-step
                    if (!mbar_wait_bounded(full_bar(stage), phase, tmo, s_abort, p.status) ||
                        (SFST &&
                         !mbar_wait_bounded(sfready_bar(stage), phase, tmo, s_abort, p.status))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t st = base_u32 + stage * C::STAGE_BYTES;
                    const uint32_t sf = st + C::A_BYTES + C::B_BYTES;
                    // this stage's scale columns: A0 | A1 (16 each) | B (16; MXFP8
                    // 4 each); every MMA scale address is a multiple of 4 columns
                    const uint32_t ts = tmem_base + C::SF_COL0 + stage * C::SF_COLS;
                    const uint32_t tsb = ts + C::SFA_COLS * C::NA;
                    if constexpr (MX8) {
                        // one atom per operand; MMA kb reads byte kb of it
                        tmem_cp_atom(ts, sf);
                        if (GATEUP)
                            tmem_cp_atom(ts + 4, sf + C::SFA_MAT);
                        tmem_cp_atom(tsb, sf + C::SFA_BYTES);
                        for (int kb = 0; kb < 4; ++kb) {
                            const uint64_t bd = smem_desc_k128(st + C::A_BYTES + kb * 32);
                            const uint32_t accum = (k | kb) != 0;
                            const uint32_t id = idesc | ((uint32_t)kb << 29) | ((uint32_t)kb << 4);
                            mma_mx8(d, smem_desc_k128(st + kb * 32), bd, id, ts, tsb, accum);
                            if (GATEUP)
                                mma_mx8(d + BN, smem_desc_k128(st + kACodeBytes + kb * 32), bd, id,
                                        ts + 4, tsb, accum);
                        }
                    } else {
                        if constexpr (!SFST) {
                            for (int kb = 0; kb < nkb; ++kb) {
                                tmem_cp_atom(ts + 4 * kb, sf + kb * kAtom);
                                if (GATEUP)
                                    tmem_cp_atom(ts + 16 + 4 * kb, sf + kSfStep + kb * kAtom);
                                tmem_cp_atom(tsb + 4 * kb, sf + C::SFA_BYTES + kb * kAtom);
                            }
                        }
                        for (int kb = 0; kb < nkb; ++kb) {
                            const uint64_t bd = smem_desc_k128(st + C::A_BYTES + kb * 32);
                            const uint32_t accum = (k | kb) != 0;
                            mma_nvf4(d, smem_desc_k128(st + kb * 32), bd, idesc, ts + 4 * kb,
                                     tsb + 4 * kb, accum);
                            if (GATEUP)
                                mma_nvf4(d + BN, smem_desc_k128(st + kACodeBytes + kb * 32), bd,
                                         idesc, ts + 16 + 4 * kb, tsb + 4 * kb, accum);
                        }
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
    } else if (warp < C::SF_W0) {
        // ------------------------------------------------- epilogue
        const int q = warp & 3;
        const int i = q * 32 + lane;
        const int wg = (warp - 2) >> 2;  // column chunks wg, wg+EPI_WG, ...
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int t = blockIdx.x; t < n_tiles; t += gridDim.x) {
            const Tile tl = decode_tile(t, s_off, s_cs, E, p.m_tiles);
            const float g0 = MX8 ? 1.0f : P.f.gs0[tl.e];
            const float g1 = GATEUP ? (MX8 ? 1.0f : P.f.gs1[tl.e]) : 0.0f;
            if (!mbar_wait_bounded(tfull_bar(acc), acc_phase, tmo, s_abort, p.status))
                break;
            tc_fence_after();
            const uint32_t ta = tmem_base + ((uint32_t)(q * 32) << 16) + acc * C::ACC_COLS;
            const int col = tl.m * kBlockM + i;
            // Drain this thread's columns into registers first and release
            // the accumulator, so the next tile's MMAs overlap the stores.
            // Column chunks of this warpgroup: (ch * EPI_WG + wg) * 16.
            constexpr int NCH = BN / 16 / EPI_WG;
            if constexpr (GATEUP) {
                // h = silu(g) * u in FP32, for the pass that quantises it
                float hv[NCH][16];
#pragma unroll
                for (int ch = 0; ch < NCH; ++ch) {
                    const int c0 = (ch * EPI_WG + wg) * 16;
                    if (c0 < tl.nrows) {
                        uint32_t g[16], u[16];
                        tmem_ld16(ta + c0, g);
                        tmem_ld16(ta + BN + c0, u);
                        tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            hv[ch][j] = silu_mul_f(__fmul_rn(__uint_as_float(g[j]), g0),
                                                   __fmul_rn(__uint_as_float(u[j]), g1));
                    }
                }
                tc_fence_before();
                mbar_arrive(tempty_bar(acc));
                float *out = static_cast<float *>(p.out);
#pragma unroll
                for (int ch = 0; ch < NCH; ++ch) {
                    const int c0 = (ch * EPI_WG + wg) * 16;
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        if (c0 + j < tl.nrows)
                            out[(size_t)(tl.row0 + c0 + j) * p.out_ld + col] = hv[ch][j];
                }
            } else {
                __nv_bfloat16 yv[NCH][16];
#pragma unroll
                for (int ch = 0; ch < NCH; ++ch) {
                    const int c0 = (ch * EPI_WG + wg) * 16;
                    if (c0 < tl.nrows) {
                        uint32_t g[16];
                        tmem_ld16(ta + c0, g);
                        tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            yv[ch][j] = __float2bfloat16_rn(__fmul_rn(__uint_as_float(g[j]), g0));
                    }
                }
                tc_fence_before();
                mbar_arrive(tempty_bar(acc));
                __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(p.out);
#pragma unroll
                for (int ch = 0; ch < NCH; ++ch) {
                    const int c0 = (ch * EPI_WG + wg) * 16;
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        if (c0 + j < tl.nrows)
                            out[(size_t)(tl.row0 + c0 + j) * p.out_ld + col] = yv[ch][j];
                }
            }
            if (++acc == ACC_BUFS) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
    } else if constexpr (SFST) {
        // --------------------------------------- scale staging (SFST)
        // lane i of warp quarter q: column c of the stage = word c % 4 of
        // row i of atom c / 4 (atoms contiguous in the stage's scale region)
        const int q = warp & 3;
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
            for (int k = 0; k < p.ksteps; ++k) {
                if (!mbar_wait_bounded(full_bar(stage), phase, tmo, s_abort, p.status)) {
                    ok = false;
                    break;
                }
                const uint8_t *sf = smem + stage * C::STAGE_BYTES + C::A_BYTES + C::B_BYTES;
                const uint32_t ta =
                    tmem_base + ((uint32_t)(q * 32) << 16) + C::SF_COL0 + stage * C::SF_COLS;
#pragma unroll
                for (int g = 0; g < C::SF_COLS / 16; ++g) {
                    uint32_t r[16];
#pragma unroll
                    for (int a = 0; a < 4; ++a) {
                        const uint4 v =
                            *reinterpret_cast<const uint4 *>(sf + (4 * g + a) * kAtom + 16 * lane);
                        r[4 * a] = v.x;
                        r[4 * a + 1] = v.y;
                        r[4 * a + 2] = v.z;
                        r[4 * a + 3] = v.w;
                    }
                    tmem_st16(ta + 16 * g, r);
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(sfready_bar(stage));
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
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

template <bool GATEUP, int BN, int STAGES, int ACC_BUFS, int BOX, int EPI_WG, bool MX8 = false,
          bool SFST = false>
cudaError_t launch_nvf4_variant(const CUtensorMap &a0, const CUtensorMap &a1, const CUtensorMap &b,
                                const GemmArgs &args, const Fp4Weights &f, int kblocks, int grid,
                                int stage, cudaStream_t s)
{
    using C = CfgN<GATEUP, BN, STAGES, ACC_BUFS, BOX, EPI_WG, MX8, SFST>;
    auto kern = grouped_gemm_nvf4_kernel<GATEUP, BN, STAGES, ACC_BUFS, BOX, EPI_WG, MX8, SFST>;
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
    P.a.ksteps = MX8 ? kblocks : (kblocks + 3) / 4;
    P.f = f;
    P.kblocks = kblocks;
    stage_begin(stage, s);
    kern<<<grid, C::THREADS, C::SMEM_BYTES, s>>>(a0, a1, b, P);
    stage_end(stage, s);
    return cudaGetLastError();
}

}  // namespace

int fp4_chunk_rows(GemmVariant v)
{
    return v == GemmVariant::kDecode ? 32 : 128;
}

int fp4_box_rows(GemmVariant v)
{
    return v == GemmVariant::kDecode ? 16 : 128;
}

cudaError_t launch_gateup_fp4(GemmVariant v, const CUtensorMap &wg, const CUtensorMap &wu,
                              const CUtensorMap &xq, const GemmArgs &a, const Fp4Weights &f,
                              int kblocks, int grid, cudaStream_t s)
{
    // prefill-size batches run the token-major kernel (grouped_gemm_tm.cu)
    if (v != GemmVariant::kDecode)
        return cudaErrorInvalidValue;
    return launch_nvf4_variant<true, 32, 5, 2, 16, 1, false, true>(wg, wu, xq, a, f, kblocks, grid,
                                                                   kStGateUp, s);
}

cudaError_t launch_down_fp4(GemmVariant v, const CUtensorMap &wd, const CUtensorMap &hq,
                            const GemmArgs &a, const Fp4Weights &f, int kblocks, int grid,
                            cudaStream_t s)
{
    if (v == GemmVariant::kDecode)
        return launch_nvf4_variant<false, 32, 9, 2, 16, 1, false, true>(wd, wd, hq, a, f, kblocks,
                                                                        grid, kStDown, s);
    // prefill size with an odd H/128 (even H/128 runs token-major)
    return launch_nvf4_variant<false, 128, 6, 2, 128, 2>(wd, wd, hq, a, f, kblocks, grid, kStDown,
                                                         s);
}

cudaError_t launch_gateup_mx8(GemmVariant v, const CUtensorMap &wg, const CUtensorMap &wu,
                              const CUtensorMap &xq, const GemmArgs &a, const Fp4Weights &f,
                              int kblocks, int grid, cudaStream_t s)
{
    // prefill-size batches run the token-major kernel (grouped_gemm_tm.cu)
    if (v != GemmVariant::kDecode)
        return cudaErrorInvalidValue;
    return launch_nvf4_variant<true, 32, 5, 2, 16, 1, true>(wg, wu, xq, a, f, kblocks, grid,
                                                                   kStGateUp, s);
}

cudaError_t launch_down_mx8(GemmVariant v, const CUtensorMap &wd, const CUtensorMap &hq,
                            const GemmArgs &a, const Fp4Weights &f, int kblocks, int grid,
                            cudaStream_t s)
{
    if (v == GemmVariant::kDecode)
        return launch_nvf4_variant<false, 32, 10, 2, 16, 1, true>(wd, wd, hq, a, f, kblocks,
                                                                         grid, kStDown, s);
    return launch_nvf4_variant<false, 128, 6, 2, 128, 2, true>(wd, wd, hq, a, f, kblocks,
                                                                      grid, kStDown, s);
}

}  // namespace beam
