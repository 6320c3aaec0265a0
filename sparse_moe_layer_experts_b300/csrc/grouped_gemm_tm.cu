// Token-major NVFP4 / MXFP8 grouped expert GEMMs for token-heavy (prefill-size)
// batches: the expert's token rows are the M = 128 operand and 256 weight
// rows the N operand, so each block-scaled MMA is 128 x 256.
//
// Same computation as the weight-major GEMMs of grouped_gemm_fp4.cu, which
// serve decode-size batches (the SwiGLU experts of "Reflection Beam 1.0",
// section "Mixture of Experts", with NVFP4 or MXFP8 operands), laid out for
// the tensor pipe's cost model: every tcgen05 instruction costs a roughly
// fixed number of cycles (about 142 for an N <= 128 MMA, 161 for N = 256,
// plus the scale copies), so one 128 x 256 MMA per 64-block does the work of
// the two 128 x 128 MMAs a weight-major gate/up tile issues.
//
// Gate/up: the N operand is gate tile m (rows 0-127) stacked on up tile m
// (rows 128-255), so one accumulator holds g and u side by side for 128
// tokens x 128 features.  Each epilogue thread owns one token row and 64
// consecutive features, i.e. whole quantisation blocks of h: it computes
// h = silu(g) * u in FP32 and quantises h itself (NVFP4: 16-blocks with E4M3
// scales; MXFP8: 32-blocks with power-of-two scales), writing the codes and
// the token-chunk scale atoms the down GEMM reads.  No FP32 h goes to
// memory.  Down: the N operand is weight tiles 2m and 2m+1 (256 output
// features); the epilogue writes bf16 y rows.
//
// Scales: the token chunk's atom per 64-block (NVFP4) or per 128-deep k-step
// (MXFP8) goes to tensor memory as the A scales; the two weight tiles'
// atoms as the B scales, the second one 4 columns after the first (rows
// 128-255 of an N = 256 operand).  Every B scale address is a multiple of 8
// columns, every A scale address a multiple of 4.
//
// Scale staging: with SFST, a fourth warpgroup reads each stage's atoms from
// shared memory and writes them into tensor memory with tcgen05.st (each
// warp its lane quarter: lane 32q + i, columns c..c+3 = words 0-3 of atom
// row i, the layout a 32x128b.warpx4 copy produces), then signals the MMA
// thread; the tensor pipe then runs only MMAs.  The producer issues a
// stage's scale atoms before its operand tiles and counts them on a barrier
// of their own, so the staging overlaps the operand copies instead of
// following them.  Without SFST the MMA thread
// copies the atoms with tcgen05.cp.  NVFP4 (12 atoms per k-step) uses SFST;
// MXFP8 (3 atoms per four MMAs) copies, which measured faster there.
//
// Warp roles: warp 0 TMA / bulk-copy producer, warp 1 TMEM allocator and MMA
// issuer, two epilogue warpgroups (features split in halves), and with SFST
// the scale warpgroup (warps 12-15; warps 2-3 idle).  One accumulator: the
// epilogue drains it into registers in two halves, computing between the
// loads, and releases it before quantising and storing.  Waits are bounded.
#include "blockscaled.cuh"
#include "common.cuh"
#include "gemm_common.cuh"
#include "internal.h"
#include "nvfp4.cuh"

#include <mutex>

namespace beam {

namespace {

constexpr int kBlockM = 128;   // token rows per tile
constexpr int kRowBytes = 128;  // one 128-byte swizzle row of codes per k-step
constexpr int kAtom = 512;
constexpr int kMaxExperts = 256;
constexpr int kEpiWG = 2;

template <bool GATEUP, bool MX8, int STAGES, bool SFST>
struct TmCfg {
    static constexpr int THREADS = SFST ? 512 : 64 + 128 * kEpiWG;
    static constexpr int EPI_W0 = SFST ? 4 : 2;  // first epilogue warp
    static constexpr int SF_W0 = 12;             // first scale warp (SFST)
    static constexpr int A_BYTES = kBlockM * kRowBytes;  // token codes
    static constexpr int B_BYTES = 256 * kRowBytes;      // two weight tiles
    static constexpr int ATOMS = MX8 ? 1 : 4;            // scale atoms per operand and k-step
    static constexpr int SF_OP = ATOMS * kAtom;          // one operand's scales per stage
    static constexpr int SF_BYTES = ((3 * SF_OP + 1023) / 1024) * 1024;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SF_BYTES;
    static constexpr int ACC_COLS = 256;
    // per stage: A scales (4 per atom), then B scales (8 per atom: tile 0 at
    // +0, tile 1 at +4), B starting on a multiple of 8
    static constexpr int SFA_COLS = MX8 ? 8 : 16;
    static constexpr int SF_COLS = SFA_COLS + 8 * ATOMS;
    static constexpr int SF_COL0 = ACC_COLS;
    static constexpr int COLS_NEED = SF_COL0 + STAGES * SF_COLS;
    static constexpr int TMEM_COLS = COLS_NEED <= 256 ? 256 : 512;
    // full, empty, sfready per stage; tfull, tempty, drain; sffull per stage
    static constexpr int N_BARS = 4 * STAGES + 3;
    static constexpr int AUX_BYTES = N_BARS * 8 + 16 + 2 * (kMaxExperts + 1) * 4;
    static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + ((AUX_BYTES + 127) / 128) * 128;
    static_assert(SF_COL0 % 8 == 0 && SF_COLS % 8 == 0 && SFA_COLS % 8 == 0,
                  "B scale columns on multiples of 8");
    static_assert(COLS_NEED <= 512, "TMEM columns");
    static_assert(STAGE_BYTES % 1024 == 0, "swizzle-atom alignment");
    static_assert(SMEM_BYTES <= 232448, "shared memory");
};

struct TmParams {
    GemmArgs a;      // m_tiles = N tiles (256 weight rows) per expert; out = h codes / y
    Fp4Weights f;    // sf0 / sf1 weight atoms, gs0 / gs1 (NVFP4), act_sf token atoms
    int kblocks;     // scale atoms per operand row tile: K/64 (NVFP4), K/128 (MXFP8)
    int n_tiles_w;   // 128-row weight tiles per expert in sf0 / the B maps
    uint8_t *h_sf;   // gate/up: scale atoms of h [chunk, I/64 (NVFP4) or I/128 (MXFP8), 512]
    const int32_t *row_pos;  // gate/up: row -> chunk * 256 + position (down GEMM's chunking)
};

template <bool GATEUP, bool MX8, int STAGES, bool SFST>
__global__ void __launch_bounds__(TmCfg<GATEUP, MX8, STAGES, SFST>::THREADS, 1)
grouped_gemm_tm_kernel(const __grid_constant__ CUtensorMap tmA,
                       const __grid_constant__ CUtensorMap tmB0,
                       const __grid_constant__ CUtensorMap tmB1, const TmParams P)
{
    using C = TmCfg<GATEUP, MX8, STAGES, SFST>;
    const GemmArgs &p = P.a;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t base_u32 = (raw_u32 + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (base_u32 - raw_u32);
    // stage s: [token codes | weight codes (2 tiles) | token atoms | tile-0 atoms | tile-1 atoms]
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + STAGES * C::STAGE_BYTES);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + C::N_BARS);
    volatile int *s_abort = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int *s_off = reinterpret_cast<int *>(tmem_slot + 4);
    int *s_cs = s_off + (kMaxExperts + 1);

    const uint32_t bar_u32 = smem_u32(bars);
    auto full_bar = [&](int s) { return bar_u32 + 8u * s; };
    auto empty_bar = [&](int s) { return bar_u32 + 8u * (STAGES + s); };
    auto sfready_bar = [&](int s) { return bar_u32 + 8u * (2 * STAGES + s); };
    const uint32_t tfull_bar = bar_u32 + 8u * (3 * STAGES);
    const uint32_t tempty_bar = bar_u32 + 8u * (3 * STAGES + 1);
    const uint32_t drain_bar = bar_u32 + 8u * (3 * STAGES + 2);
    // SFST: the stage's scale atoms complete on their own barrier, so the
    // scale warpgroup stages them while the operand tiles are still landing
    auto sffull_bar = [&](int s) { return bar_u32 + 8u * (3 * STAGES + 3 + s); };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int E = p.E;
    const int KB = P.kblocks;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
            mbar_init(sfready_bar(s), 4);  // one arrive per scale warp
            mbar_init(sffull_bar(s), 1);
        }
        mbar_init(tfull_bar, 1);
        mbar_init(tempty_bar, 128 * kEpiWG);
        mbar_init(drain_bar, 1);
        *s_abort = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB0);
        if (GATEUP)
            tma_prefetch_desc(&tmB1);
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

    // weight tiles (128 rows) of work unit m: gate/up m in both maps, down 2m, 2m+1
    auto wtile0 = [&](const Tile &tl) { return tl.e * P.n_tiles_w + (GATEUP ? tl.m : 2 * tl.m); };

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------- producer: codes by TMA, scales by bulk copy
            int stage = 0;
            uint32_t phase = 0, armed = 0, armed_par = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
                const Tile tl = decode_tile(t, s_off, s_cs, E, p.m_tiles);
                const int w0 = wtile0(tl);
                const int w1 = GATEUP ? w0 : w0 + 1;
                const uint8_t *sfb0 = P.f.sf0 + (size_t)w0 * KB * kAtom;
                const uint8_t *sfb1 = (GATEUP ? P.f.sf1 : P.f.sf0) + (size_t)w1 * KB * kAtom;
                int j0;
                const int chunk =
                    s_cs[tl.e] + nvfp4_chunk_of_row(tl.row0 - s_off[tl.e], s_off[tl.e + 1] - s_off[tl.e],
                                                    s_cs[tl.e + 1] - s_cs[tl.e], &j0);
                const uint8_t *sfa = P.f.act_sf + (size_t)chunk * KB * kAtom;
                for (int k = 0; k < p.ksteps; ++k) {
                    const int nkb = MX8 ? 1 : min(4, KB - 4 * k);
                    const int atom0 = MX8 ? k : 4 * k;
                    if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, tmo, s_abort, p.status)) {
                        ok = false;
                        break;
                    }
                    armed |= 1u << stage;
                    armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
                    const uint32_t st = base_u32 + stage * C::STAGE_BYTES;
                    const uint32_t sb = st + C::A_BYTES;
                    const uint32_t sf = sb + C::B_BYTES;
                    // scales first (on their own barrier with SFST), then the
                    // operand tiles
                    const uint32_t sbar = SFST ? sffull_bar(stage) : full_bar(stage);
                    if (SFST) {
                        mbar_arrive_expect_tx(sbar, (uint32_t)(3 * nkb * kAtom));
                        mbar_arrive_expect_tx(full_bar(stage), (uint32_t)(C::A_BYTES + C::B_BYTES));
                    } else {
                        mbar_arrive_expect_tx(full_bar(stage), (uint32_t)(C::A_BYTES + C::B_BYTES +
                                                                          3 * nkb * kAtom));
                    }
                    bulk_g2s(sf, sfa + (size_t)atom0 * kAtom, nkb * kAtom, sbar);
                    bulk_g2s(sf + C::SF_OP, sfb0 + (size_t)atom0 * kAtom, nkb * kAtom, sbar);
                    bulk_g2s(sf + 2 * C::SF_OP, sfb1 + (size_t)atom0 * kAtom, nkb * kAtom, sbar);
                    tma_load_2d(st, &tmA, k * kRowBytes, tl.row0, full_bar(stage));
                    tma_load_2d(sb, &tmB0, k * kRowBytes, w0 * kBlockM, full_bar(stage));
                    tma_load_2d(sb + 128 * kRowBytes, GATEUP ? &tmB1 : &tmB0, k * kRowBytes,
                                w1 * kBlockM, full_bar(stage));
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok)
                for (int s = 0; s < STAGES; ++s)
                    if ((armed >> s) & 1u) {
                        mbar_wait_drain(full_bar(s), (armed_par >> s) & 1u, tmo);
                        if (SFST)
                            mbar_wait_drain(sffull_bar(s), (armed_par >> s) & 1u, tmo);
                    }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            // --------------------------------------------- MMA issuer
            const uint32_t idesc = MX8 ? idesc_mx8(kBlockM, 256) : idesc_nvf4(kBlockM, 256);
            int stage = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
                if (!mbar_wait_bounded(tempty_bar, acc_phase ^ 1u, tmo, s_abort, p.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem_base;
                for (int k = 0; k < p.ksteps; ++k) {
                    const int nkb = MX8 ? 1 : min(4, KB - 4 * k);
                    // operands in shared memory, and (SFST) the scales in tensor memory
                    if (!mbar_wait_bounded(full_bar(stage), phase, tmo, s_abort, p.status) ||
                        (SFST &&
                         !mbar_wait_bounded(sfready_bar(stage), phase, tmo, s_abort, p.status))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t st = base_u32 + stage * C::STAGE_BYTES;
                    const uint32_t sb = st + C::A_BYTES;
                    const uint32_t sf = sb + C::B_BYTES;
                    const uint32_t ta = tmem_base + C::SF_COL0 + stage * C::SF_COLS;
                    const uint32_t tb = ta + C::SFA_COLS;
                    if constexpr (!SFST) {
                        for (int kb = 0; kb < nkb; ++kb) {
                            tmem_cp_atom(ta + 4 * kb, sf + kb * kAtom);
                            tmem_cp_atom(tb + 8 * kb, sf + C::SF_OP + kb * kAtom);
                            tmem_cp_atom(tb + 8 * kb + 4, sf + 2 * C::SF_OP + kb * kAtom);
                        }
                    }
                    if constexpr (MX8) {
                        // four K = 32 MMAs pick byte kk of the one atom per operand
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint32_t id = idesc | ((uint32_t)kk << 29) | ((uint32_t)kk << 4);
                            mma_mx8(d, smem_desc_k128(st + kk * 32), smem_desc_k128(sb + kk * 32),
                                    id, ta, tb, (k | kk) != 0);
                        }
                    } else {
                        for (int kb = 0; kb < nkb; ++kb)
                            mma_nvf4(d, smem_desc_k128(st + kb * 32), smem_desc_k128(sb + kb * 32),
                                     idesc, ta + 4 * kb, tb + 8 * kb, (k | kb) != 0);
                    }
                    mma_commit(empty_bar(stage));
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok)
                    break;
                mma_commit(tfull_bar);
                acc_phase ^= 1u;
            }
            if (!ok) {
                mma_commit(drain_bar);
                mbar_wait_drain(drain_bar, 0, tmo);
            }
        }
        __syncwarp();
    } else if (warp >= C::EPI_W0 && warp < C::EPI_W0 + 4 * kEpiWG) {
        // ------------------------------------------------- epilogue
        const int q = warp & 3;                   // TMEM lane quarter of this warp
        const int j = q * 32 + lane;              // token row in the tile
        const int wg = (warp - C::EPI_W0) >> 2;  // feature half
        uint32_t acc_phase = 0;
        for (int t = blockIdx.x; t < n_tiles; t += gridDim.x) {
            const Tile tl = decode_tile(t, s_off, s_cs, E, p.m_tiles);
            const float g0 = MX8 ? 1.0f : P.f.gs0[tl.e];
            const float g1 = (MX8 || !GATEUP) ? 1.0f : P.f.gs1[tl.e];
            if (!mbar_wait_bounded(tfull_bar, acc_phase, tmo, s_abort, p.status))
                break;
            tc_fence_after();
            const uint32_t ta = tmem_base + ((uint32_t)(q * 32) << 16);
            const int row = tl.row0 + j;
            const bool live = j < tl.nrows;
            if constexpr (GATEUP) {
                // features 64wg + 32c + i: g in column 64wg + 32c + i, u 128 further.
                // Two halves: h of the first is computed before the second is
                // loaded; the accumulator is released after the second load.
                float h[2][32];
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    uint32_t g[2][16], u[2][16];
                    tmem_ld16(ta + 64 * wg + 32 * c, g[0]);
                    tmem_ld16(ta + 64 * wg + 32 * c + 16, g[1]);
                    tmem_ld16(ta + 128 + 64 * wg + 32 * c, u[0]);
                    tmem_ld16(ta + 128 + 64 * wg + 32 * c + 16, u[1]);
                    tmem_ld_wait();
                    if (c == 1) {
                        tc_fence_before();
                        mbar_arrive(tempty_bar);
                    }
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        h[c][i] = silu_mul_f(__fmul_rn(__uint_as_float(g[i / 16][i % 16]), g0),
                                             __fmul_rn(__uint_as_float(u[i / 16][i % 16]), g1));
                }
                if (live) {
                    const int I = p.out_ld;  // h elements per row
                    const int ps = P.row_pos[row];
                    const int jc = ps & 255;
                    uint8_t *hq = static_cast<uint8_t *>(p.out);
                    if constexpr (MX8) {
                        // half c is the 32-block 2wg + c of the 128-block m
                        uint32_t sc = 0;
#pragma unroll
                        for (int c = 0; c < 2; ++c) {
                            float amax = 0.0f;
#pragma unroll
                            for (int i = 0; i < 32; ++i)
                                amax = fmaxf(amax, fabsf(h[c][i]));
                            const int e = mx_shared_exp(amax);
                            const float inv = mx_inv_scale(e);
                            uint32_t w[8];
#pragma unroll
                            for (int v = 0; v < 8; ++v)
                                w[v] = mx_code4(&h[c][4 * v], inv);
                            uint4 *dst = reinterpret_cast<uint4 *>(
                                hq + (size_t)row * I + tl.m * 128 + 64 * wg + 32 * c);
                            dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
                            dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
                            sc |= (uint32_t)(e + 127) << (8 * c);
                        }
                        // atom of (chunk, 128-block m): bytes 2wg, 2wg+1 of the row's word
                        *reinterpret_cast<uint16_t *>(
                            P.h_sf + ((size_t)(ps >> 8) * (I / 128) + tl.m) * kAtom +
                            nvfp4_atom_offset(jc) + 2 * wg) = (uint16_t)sc;
                    } else {
                        // four 16-blocks = the 64-block 2m + wg
                        uint32_t lo[4], hi[4], word = 0;
#pragma unroll
                        for (int b = 0; b < 4; ++b) {
                            float v[16];
#pragma unroll
                            for (int i = 0; i < 16; ++i)
                                v[i] = h[b / 2][16 * (b % 2) + i];
                            word |= nvfp4_quant16(v, &lo[b], &hi[b]) << (8 * b);
                        }
                        uint4 *dst = reinterpret_cast<uint4 *>(hq + (size_t)row * (I / 2) +
                                                               tl.m * 64 + 32 * wg);
                        dst[0] = make_uint4(lo[0], hi[0], lo[1], hi[1]);
                        dst[1] = make_uint4(lo[2], hi[2], lo[3], hi[3]);
                        // atom of (chunk, 64-block 2m + wg): the row's word
                        *reinterpret_cast<uint32_t *>(
                            P.h_sf + ((size_t)(ps >> 8) * (I / 64) + 2 * tl.m + wg) * kAtom +
                            nvfp4_atom_offset(jc)) = word;
                    }
                }
            } else {
                // y columns 128wg .. 128wg + 127 of the 256-feature tile, in
                // four loads of 32 packed to bf16 pairs; release after the last
                uint32_t w[4][16];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t v[2][16];
                    tmem_ld16(ta + 128 * wg + 32 * c, v[0]);
                    tmem_ld16(ta + 128 * wg + 32 * c + 16, v[1]);
                    tmem_ld_wait();
                    if (c == 3) {
                        tc_fence_before();
                        mbar_arrive(tempty_bar);
                    }
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        w[c][i] = pack_bf16x2(
                            __fmul_rn(__uint_as_float(v[(2 * i) / 16][(2 * i) % 16]), g0),
                            __fmul_rn(__uint_as_float(v[(2 * i + 1) / 16][(2 * i + 1) % 16]), g0));
                }
                if (live) {
                    // 256 contiguous bytes of the row in eight 256-bit stores
                    // (the row's 32 lanes each write another row, so fewer,
                    // wider stores keep the load/store pipe free for the
                    // scale staging); 32-byte aligned: H * 2, the tile offset
                    // (multiples of 256 bytes) and the 1 KB-aligned y region
                    uint8_t *dst = reinterpret_cast<uint8_t *>(static_cast<__nv_bfloat16 *>(p.out) +
                                                               (size_t)row * p.out_ld +
                                                               tl.m * 256 + 128 * wg);
#pragma unroll
                    for (int c = 0; c < 4; ++c)
#pragma unroll
                        for (int v = 0; v < 2; ++v)
                            st_global_v8(dst + 64 * c + 32 * v, w[c][8 * v], w[c][8 * v + 1],
                                         w[c][8 * v + 2], w[c][8 * v + 3], w[c][8 * v + 4],
                                         w[c][8 * v + 5], w[c][8 * v + 6], w[c][8 * v + 7]);
                }
            }
            acc_phase ^= 1u;
        }
    } else if (SFST && warp >= C::SF_W0) {
        // --------------------------------------- scale staging (SFST)
        // Each warp writes its lane quarter: lane 32q + i, column c + w =
        // word w of row i of the atom placed at column c.
        const int q = warp & 3;
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
            for (int k = 0; k < p.ksteps; ++k) {
                if (!mbar_wait_bounded(sffull_bar(stage), phase, tmo, s_abort, p.status)) {
                    ok = false;
                    break;
                }
                const uint8_t *sf = smem + stage * C::STAGE_BYTES + C::A_BYTES + C::B_BYTES;
                const uint32_t ta =
                    tmem_base + ((uint32_t)(q * 32) << 16) + C::SF_COL0 + stage * C::SF_COLS;
                if constexpr (MX8) {
                    // columns: token atom 0-3, (unused) 4-7, tile 0 8-11, tile 1 12-15
                    const uint4 a = *reinterpret_cast<const uint4 *>(sf + 16 * lane);
                    const uint4 b0 = *reinterpret_cast<const uint4 *>(sf + C::SF_OP + 16 * lane);
                    const uint4 b1 =
                        *reinterpret_cast<const uint4 *>(sf + 2 * C::SF_OP + 16 * lane);
                    const uint32_t r[16] = {a.x,  a.y,  a.z,  a.w,  0u,   0u,   0u,   0u,
                                            b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
                    tmem_st16(ta, r);
                } else {
                    // columns: token atoms 4kb..4kb+3; weight atoms 16 + 8kb (tile 0)
                    // and 20 + 8kb (tile 1)
                    uint32_t r[3][16];
#pragma unroll
                    for (int kb = 0; kb < 4; ++kb) {
                        const uint4 a = *reinterpret_cast<const uint4 *>(sf + kb * kAtom + 16 * lane);
                        const uint4 b0 = *reinterpret_cast<const uint4 *>(sf + C::SF_OP +
                                                                          kb * kAtom + 16 * lane);
                        const uint4 b1 = *reinterpret_cast<const uint4 *>(sf + 2 * C::SF_OP +
                                                                          kb * kAtom + 16 * lane);
                        r[0][4 * kb] = a.x;
                        r[0][4 * kb + 1] = a.y;
                        r[0][4 * kb + 2] = a.z;
                        r[0][4 * kb + 3] = a.w;
                        const int x = 8 * kb;  // column 16 + x of the stage = r[1 + x/16][x%16]
                        r[1 + x / 16][x % 16] = b0.x;
                        r[1 + x / 16][x % 16 + 1] = b0.y;
                        r[1 + x / 16][x % 16 + 2] = b0.z;
                        r[1 + x / 16][x % 16 + 3] = b0.w;
                        r[1 + x / 16][x % 16 + 4] = b1.x;
                        r[1 + x / 16][x % 16 + 5] = b1.y;
                        r[1 + x / 16][x % 16 + 6] = b1.z;
                        r[1 + x / 16][x % 16 + 7] = b1.w;
                    }
                    tmem_st16(ta, r[0]);
                    tmem_st16(ta + 16, r[1]);
                    tmem_st16(ta + 32, r[2]);
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

template <bool GATEUP, bool MX8, int STAGES, bool SFST>
cudaError_t launch_tm(const CUtensorMap &a, const CUtensorMap &b0, const CUtensorMap &b1,
                      const TmParams &P, int grid, int stage, cudaStream_t s)
{
    using C = TmCfg<GATEUP, MX8, STAGES, SFST>;
    auto kern = grouped_gemm_tm_kernel<GATEUP, MX8, STAGES, SFST>;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        C::SMEM_BYTES);
    });
    if (attr_err != cudaSuccess)
        return attr_err;
    stage_begin(stage, s);
    kern<<<grid, C::THREADS, C::SMEM_BYTES, s>>>(a, b0, b1, P);
    stage_end(stage, s);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gateup_tm(bool mx8, const CUtensorMap &wg, const CUtensorMap &wu,
                             const CUtensorMap &xq, const GemmArgs &a, const Fp4Weights &f,
                             int kblocks, uint8_t *h_sf, const int32_t *row_pos, int grid,
                             cudaStream_t s)
{
    TmParams P;
    P.a = a;
    P.a.ksteps = mx8 ? kblocks : (kblocks + 3) / 4;
    P.f = f;
    P.kblocks = kblocks;
    P.n_tiles_w = a.m_tiles;
    P.h_sf = h_sf;
    P.row_pos = row_pos;
    // NVFP4 (12 scale atoms per k-step) stages its scales with tcgen05.st;
    // MXFP8 (3 per k-step) copies them in the tensor pipe, which measured faster
    if (mx8)
        return launch_tm<true, true, 4, false>(xq, wg, wu, P, grid, kStGateUp, s);
    return launch_tm<true, false, 4, true>(xq, wg, wu, P, grid, kStGateUp, s);
}

cudaError_t launch_down_tm(bool mx8, const CUtensorMap &wd, const CUtensorMap &hq,
                           const GemmArgs &a, const Fp4Weights &f, int kblocks, int grid,
                           cudaStream_t s)
{
    if (a.m_tiles % 2)
        return cudaErrorInvalidValue;
    TmParams P;
    P.a = a;
    P.a.m_tiles = a.m_tiles / 2;  // 256-feature tiles
    P.a.ksteps = mx8 ? kblocks : (kblocks + 3) / 4;
    P.f = f;
    P.kblocks = kblocks;
    P.n_tiles_w = a.m_tiles;
    P.h_sf = nullptr;
    P.row_pos = nullptr;
    if (mx8)
        return launch_tm<false, true, 4, false>(hq, wd, wd, P, grid, kStDown, s);
    return launch_tm<false, false, 4, true>(hq, wd, wd, P, grid, kStDown, s);
}

}  // namespace beam
