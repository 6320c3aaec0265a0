// Internal launchers shared by the translation units of libbeam_moe.so.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace beam {

// Kernel stages, in launch order; the index of the optional timing events.
enum Stage {
    kStRouter = 0,
    kStSelect,
    kStHist,
    kStScan,
    kStPermute,
    kStGateUp,
    kStDown,
    kStCombine,
    kStQuantH,  // NVFP4 layers only: quantise h before the down GEMM
    kStNorm,    // fused block only: the pre-norm of the residual stream
    kNumStages
};
// Bracket one kernel launch: records the calling thread's timing events for
// the stage (if any are set) and counts the launch.
void stage_begin(int stage, cudaStream_t s);
void stage_end(int stage, cudaStream_t s);
// Count a launch that shares its stage's events with the stage's last kernel.
void count_launch();

// ---- router.cu
// scores[t,e] = sigmoid(sum_h x[t,h] * wr[h,e]) with an FP32 FMA chain in
// ascending h per output.
// Also resets *status (the call's device status word) to 0.
cudaError_t launch_router_scores(const uint16_t *x, const float *wr, int T, int H, int E,
                                 float *scores, int *status, cudaStream_t s);
// ---- router_tc.cu
// Batches of at least kTcRouterMinTokens tokens take the tensor-core router:
// wr is split into three exact bf16 parts [3][E][H] (`parts`, 3*E*H*2 bytes
// of workspace), then the FP32 tensor-core sums of the exact products
// x[t,h]*part[e,h] over nsplit ranges of h go to partials [nsplit][T][E]
// (nsplit a power of two <= kRouterMaxSplits; router_tc_splits picks it from
// the tile count and the SM count).  w_map: parts as [3E, H] bf16, box 64 x
// 128 rows; x_map: x [T,H] bf16, box 64 x 256 rows (both 128-byte
// swizzled).  Two launches; the first resets *status.  launch_select then
// turns the partials into scores.
constexpr int kTcRouterMinTokens = 256;
constexpr int kRouterMaxSplits = 8;
int router_tc_splits(int64_t T, int E, int H, int sms);
cudaError_t launch_router_tc(const float *wr, void *parts, const CUtensorMap &w_map,
                             const CUtensorMap &x_map, int T, int H, int E, int nsplit,
                             float *partials, int *status, unsigned long long timeout_ns,
                             cudaStream_t s);
// Group-limited top-k over scores -> ids [T,K], w [T,K].  With nsplit > 0
// the logits are first summed from the router's partials [nsplit][T][E] (in
// order); with write_scores every score is then computed and written to
// scores (partials may equal scores when nsplit == 1), without it only the
// scores the selection needs are evaluated and scores is not written.  The
// selection is the same either way.
cudaError_t launch_select(float *scores, const float *partials, int nsplit, bool write_scores,
                          int T, int E, int G, int TG, int K, float scale, int32_t *ids, float *w,
                          int *status, cudaStream_t s);

// ---- dispatch.cu
constexpr int kHistTokens = 256;  // tokens per histogram CTA
// Per-CTA histograms (local_rank, cta_counts), then the scan over experts:
// cta_base, counts, offsets and the token chunks of chunk_rows rows per
// expert (chunk_start).  With one histogram CTA (T <= 256) that CTA does the
// scan too and the scan kernel is not launched.
cudaError_t launch_hist_scan(const int32_t *ids, int T, int K, int E, int chunk_rows,
                             int32_t *local_rank, int32_t *cta_counts, int32_t *cta_base,
                             int32_t *counts, int32_t *offsets, int32_t *chunk_start, int *status,
                             cudaStream_t s);
cudaError_t launch_permute(const uint16_t *x, const int32_t *ids, const int32_t *local_rank,
                           const int32_t *cta_base, const int32_t *offsets, int T, int K, int E,
                           int H, int32_t *row_of, int32_t *row_src, void *x_perm,
                           cudaStream_t s);
// MXFP8 layers: x rows into E4M3 codes [R, H] and scale atoms
// [chunk, H/128, 512] of the chunking (chunk_start); row_pos[row] = chunk*256 + j
cudaError_t launch_permute_mx8(const uint16_t *x, const int32_t *ids, const int32_t *local_rank,
                               const int32_t *cta_base, const int32_t *offsets,
                               const int32_t *chunk_start, int T, int K, int E, int H,
                               int32_t *row_of, int32_t *row_src, int32_t *row_pos,
                               uint8_t *x_codes, uint8_t *x_sf, cudaStream_t s);
// MXFP8 h: FP32 [rows, cols] -> E4M3 codes [rows, cols] and scale atoms
// [chunk, cols/128, 512] at row_pos
cudaError_t launch_quantize_rows_mx8(const float *in, int64_t rows, int cols, const int32_t *row_pos,
                                     uint8_t *codes, uint8_t *sf, cudaStream_t s);
// NVFP4 layers: x rows quantised (global scale 1) into codes [R, H/2] and
// scale atoms [chunk, H/64, 512] of the token chunking (chunk_start);
// row_pos[row] = chunk*256 + j, the row's place in that chunking
cudaError_t launch_permute_nvfp4(const uint16_t *x, const int32_t *ids, const int32_t *local_rank,
                                 const int32_t *cta_base, const int32_t *offsets,
                                 const int32_t *chunk_start, int T, int K, int E, int H,
                                 int32_t *row_of, int32_t *row_src, int32_t *row_pos,
                                 uint8_t *x_codes, uint8_t *x_sf, cudaStream_t s);
// route-only variant: row_of without moving activations
cudaError_t launch_rows(const int32_t *ids, const int32_t *local_rank, const int32_t *cta_base,
                        const int32_t *offsets, int T, int K, int E, int32_t *row_of,
                        cudaStream_t s);
// NVFP4 activations: FP32 [rows, cols] -> codes [rows, cols/2] and scales at
// the token-chunk positions row_pos names (global scale 1): atoms
// [chunk, cols/64, 512]
cudaError_t launch_quantize_rows(const float *in, int64_t rows, int cols, const int32_t *row_pos,
                                 uint8_t *codes, uint8_t *sf, cudaStream_t s);
cudaError_t launch_combine(const uint16_t *y, const float *w, const int32_t *row_of, int T, int K,
                           int H, uint16_t *out, cudaStream_t s);
// fused MoE block: x = bf16(rmsnorm(s_in) * gamma) (FP64 sum of squares,
// FP32 r = 1/sqrt(mean + eps)), and the combine with post-norm and the
// residual s_out = bf16(a * s_in + b * rmsnorm(o) * gamma) (H <= 8192;
// s_out may be s_in)
cudaError_t launch_rmsnorm_bf16(const uint16_t *s_in, const float *gamma, float eps, int T, int H,
                               uint16_t *x, cudaStream_t st);
cudaError_t launch_combine_block(const uint16_t *y, const float *w, const int32_t *row_of, int T,
                                 int K, int H, const uint16_t *s_in, const float *gamma, float eps,
                                 float a, float b, uint16_t *s_out, cudaStream_t st);
// dense layers: offsets {0, T}, chunk_start {0, ceil(T/chunk_rows)}, status 0
cudaError_t launch_dense_setup(int T, int chunk_rows, int32_t *offsets, int32_t *chunk_start,
                               int *status, cudaStream_t s);

// ---- grouped_gemm.cu
struct GemmArgs {
    const int32_t *offsets;      // [E+1] rows of each expert in the permuted order
    const int32_t *chunk_start;  // [E+1] prefix of per-expert row chunks
    int E;
    int m_tiles;    // weight rows per expert / 128
    int ksteps;     // reduction length / 64
    void *out;      // gate/up: h bf16 [R, ld] (NVFP4 / MXFP8: FP32, or codes from the
                    // token-major kernel); down: y bf16 [R, ld]
    int out_ld;
    int *status;
    unsigned long long timeout_ns;
    unsigned debug_flags;
};

enum class GemmVariant { kDecode, kPrefill };

// NVFP4 operands: E2M1 codes (via TMA maps), tiled E4M3 block scales of the
// weights, FP32 global scales of the weights, and the activations' scales
// in token-chunk atoms.
struct Fp4Weights {
    const uint8_t *sf0, *sf1;  // block scales of A0 / A1 (A1: up projection)
    const float *gs0, *gs1;    // global scales [E]
    const uint8_t *act_sf;     // [chunk, K/64, 512] scales of the B operand
};

// ---- nvfp4.cu
// FP32 activation rows -> codes and row-major scales (global scale 1)
cudaError_t launch_quantize_act(bool mx8, const float *x, int64_t rows, int cols, uint8_t *codes,
                                uint8_t *sf, cudaStream_t s);
cudaError_t launch_quantize_nvfp4(const uint16_t *w, int64_t n_mat, int rows, int cols,
                                  uint8_t *packed, uint8_t *block_sf, float *global_sf,
                                  cudaStream_t s);
// MXFP8: codes [n_mat, rows, cols] E4M3, block_sf [n_mat, rows/128, cols/128, 512]
cudaError_t launch_quantize_mxfp8(const uint16_t *w, int64_t n_mat, int rows, int cols,
                                  uint8_t *codes, uint8_t *block_sf, cudaStream_t s);

// chunk height (rows of one expert handled by one tile) of a variant
int gemm_chunk_rows(GemmVariant v);
// token rows per TMA box of the B operand (the B tensor maps' box height)
int gemm_box_rows(GemmVariant v);

// h = silu(x_perm . Wg^T) * (x_perm . Wu^T) per expert segment (bf16 out)
cudaError_t launch_gateup(GemmVariant v, const CUtensorMap &wg, const CUtensorMap &wu,
                          const CUtensorMap &xp, const GemmArgs &a, int grid, cudaStream_t s);
// y = h . Wd^T per expert segment (bf16 out)
cudaError_t launch_down(GemmVariant v, const CUtensorMap &wd, const CUtensorMap &hp,
                        const GemmArgs &a, int grid, cudaStream_t s);

// ---- grouped_gemm_pair.cu: the prefill-size down GEMM on CTA pairs with the
// 2-SM MMA (weight tiles of 256 rows; needs an even a.m_tiles and 128-row
// token boxes in the B map)
cudaError_t launch_down_pair(const CUtensorMap &wd, const CUtensorMap &hp, const GemmArgs &a,
                             int grid, cudaStream_t s);

// ---- grouped_gemm_fp4.cu: the same GEMMs in NVFP4 on the FP4 tensor cores
// (E2M1 codes of weights and activations via 128-byte TMA rows, block
// scales via bulk copies).  Gate/up here is the decode-size kernel only
// (prefill-size batches: launch_gateup_tm); it writes h in FP32 for
// launch_quantize_rows.  Down here: decode size, and prefill size with an
// odd H/128 (else launch_down_tm).  kblocks = K/64.  Token chunks are
// fp4_chunk_rows(v) rows at most; the activation maps use fp4_box_rows(v)-row
// boxes; activation scales are atoms [chunk, K/64, 512].
int fp4_chunk_rows(GemmVariant v);
int fp4_box_rows(GemmVariant v);
// MXFP8 experts on the same kernels (kind::mxf8f6f4): E4M3 codes, one
// UE8M0 scale per 32 elements, scale atoms [.., K/128, 512]; kblocks = K/128;
// chunks of fp4_chunk_rows(v) rows for both GEMMs, activation scales in
// atoms.  Gate/up: decode size only, writing h in FP32 for
// launch_quantize_rows_mx8; down: any size (prefill-size batches with an
// even H/128 use launch_down_tm_mx8).
cudaError_t launch_gateup_mx8(GemmVariant v, const CUtensorMap &wg, const CUtensorMap &wu,
                              const CUtensorMap &xq, const GemmArgs &a, const Fp4Weights &f,
                              int kblocks, int grid, cudaStream_t s);
cudaError_t launch_down_mx8(GemmVariant v, const CUtensorMap &wd, const CUtensorMap &hq,
                            const GemmArgs &a, const Fp4Weights &f, int kblocks, int grid,
                            cudaStream_t s);
// ---- grouped_gemm_tm.cu: token-major prefill-size GEMMs (tokens the
// M = 128 operand, 256 weight rows the N operand).  Gate/up (NVFP4 or MXFP8,
// chunks of fp4_chunk_rows(kPrefill) rows, 128-row token boxes) writes h
// already quantised: codes [R, I] (NVFP4 two per byte) and scale atoms at
// row_pos.  a.out = h codes, a.out_ld = I, a.m_tiles = I/128.  Down
// (a.m_tiles = H/128 even; kblocks = I/64 NVFP4, I/128 MXFP8) writes y
// bf16 [R, H].
cudaError_t launch_gateup_tm(bool mx8, const CUtensorMap &wg, const CUtensorMap &wu,
                             const CUtensorMap &xq, const GemmArgs &a, const Fp4Weights &f,
                             int kblocks, uint8_t *h_sf, const int32_t *row_pos, int grid,
                             cudaStream_t s);
cudaError_t launch_down_tm(bool mx8, const CUtensorMap &wd, const CUtensorMap &hq,
                           const GemmArgs &a, const Fp4Weights &f, int kblocks, int grid,
                           cudaStream_t s);
cudaError_t launch_gateup_fp4(GemmVariant v, const CUtensorMap &wg, const CUtensorMap &wu,
                              const CUtensorMap &xq, const GemmArgs &a, const Fp4Weights &f,
                              int kblocks, int grid, cudaStream_t s);
cudaError_t launch_down_fp4(GemmVariant v, const CUtensorMap &wd, const CUtensorMap &hq,
                            const GemmArgs &a, const Fp4Weights &f, int kblocks, int grid,
                            cudaStream_t s);

}  // namespace beam
