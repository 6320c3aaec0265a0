// The down-projection grouped GEMM on CTA pairs with the 2-SM tensor-core MMA
// (tcgen05 cta_group::2), for token-heavy (prefill-size) batches.
//
// Same computation as the down GEMM of grouped_gemm.cu (expert output
// h W_down^T of the SwiGLU experts of "Reflection Beam 1.0", section
// "Mixture of Experts"), but two CTAs on two SMs share each MMA of
// M = 256 weight rows: CTA r holds
// weight rows [128r, 128r+128) of the pair's 256-row tile and token rows
// [r*N/2, (r+1)*N/2) of the N-token chunk, and receives its 128 rows of the
// result in its own tensor memory.  Per SM this halves the token tile that
// TMA writes into shared memory and that the MMA reads back.  (The gate/up
// GEMM stays on the 1-SM kernel: at large batch it runs at the power-capped
// tensor rate, and the pair form measured no faster there.)
//
// Roles (both CTAs): warp 0 issues the TMA loads of its CTA's operands, with
// completion counted on the leader CTA's barriers; warp 1 of the leader
// (rank 0) issues the MMAs and commits them to both CTAs; the epilogue
// warpgroups of each CTA drain its own accumulators, and warp 1 of the
// follower relays "drained" to the leader once per tile.  Waits are bounded
// as in the 1-SM kernel.
#include "common.cuh"
#include "gemm_common.cuh"
#include "internal.h"

#include <mutex>

namespace beam {

namespace {

constexpr int kBlockM = 128;   // weight rows per CTA (256 per pair)
constexpr int kBlockK = 64;    // one 128-byte swizzle row of bf16
constexpr int kABytes = kBlockM * kBlockK * 2;
constexpr int kHalfRows = 128;  // token rows one CTA stages (half of N <= 256)
constexpr int kBBytes = kHalfRows * kBlockK * 2;
constexpr int kMaxExperts = 256;
constexpr int kEpiWG = 2;
constexpr int kThreads = 64 + 128 * kEpiWG;

template <int STAGES, int ACC_BUFS>
struct PairCfg {
    static constexpr int STAGE_BYTES = kABytes + kBBytes;
    static constexpr int ACC_COLS = 256;
    static constexpr int TMEM_COLS = ACC_BUFS * ACC_COLS;
    static constexpr uint32_t PAIR_TX = 2 * STAGE_BYTES;  // both CTAs' loads of a stage
    static constexpr int N_BARS = 2 * STAGES + 2 * ACC_BUFS + 1;
    static constexpr int AUX_BYTES = N_BARS * 8 + 16 + 2 * (kMaxExperts + 1) * 4;
    static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + ((AUX_BYTES + 127) / 128) * 128;
    static_assert(TMEM_COLS == 256 || TMEM_COLS == 512, "TMEM allocation");
    static_assert(SMEM_BYTES <= 232448, "shared memory");
};

template <int STAGES, int ACC_BUFS>
__global__ void __launch_bounds__(kThreads, 1)
grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                         const __grid_constant__ CUtensorMap tmB, const GemmArgs p)
{
    using C = PairCfg<STAGES, ACC_BUFS>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t base_u32 = (raw_u32 + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (base_u32 - raw_u32);
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

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int E = p.E;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);   // leader: its arrive + both CTAs' bytes
            mbar_init(empty_bar(s), 1);  // the leader's commit, in both CTAs
        }
        for (int a = 0; a < ACC_BUFS; ++a) {
            mbar_init(tfull_bar(a), 1);
            // leader: its epilogue threads + one relayed arrive from the
            // follower; follower: its own epilogue threads
            mbar_init(tempty_bar(a), 128 * kEpiWG + (rank == 0 ? 1 : 0));
        }
        mbar_init(drain_bar, 1);
        *s_abort = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        tmem_alloc2(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish2();
    }
    for (int i = threadIdx.x; i <= E; i += kThreads) {
        s_off[i] = p.offsets[i];
        s_cs[i] = p.chunk_start[i];
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // both CTAs' barriers exist before any cross-CTA signal
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    // work unit = (expert, weight-tile pair, token chunk); this CTA's weight
    // tile is m = 2*pair + rank
    const int unit_mtiles = p.m_tiles / 2;
    const int n_units = unit_mtiles * s_cs[E];
    const int first = (int)(blockIdx.x >> 1), stride = (int)(gridDim.x >> 1);
    auto tile_of = [&](int u) {
        Tile tl = decode_tile(u, s_off, s_cs, E, unit_mtiles);
        tl.m = 2 * tl.m + (int)rank;
        return tl;
    };
    const uint64_t tmo = p.timeout_ns;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            int stage = 0;
            uint32_t phase = 0, armed = 0, armed_par = 0;
            bool ok = true;
            for (int u = first; u < n_units && ok; u += stride) {
                const Tile tl = tile_of(u);
                const int arow = tl.e * p.m_tiles * kBlockM + tl.m * kBlockM;
                const int half = ((tl.nrows + 31) & ~31) / 2;
                const int brow = tl.row0 + (int)rank * half;
                for (int k = 0; k < p.ksteps; ++k) {
                    if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, tmo, s_abort, p.status)) {
                        ok = false;
                        break;
                    }
                    if (leader) {
                        mbar_arrive_expect_tx(full_bar(stage), C::PAIR_TX);
                        armed |= 1u << stage;
                        armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
                    }
                    const uint32_t fb = mapa_shared(full_bar(stage), 0);
                    const uint32_t sa = base_u32 + stage * C::STAGE_BYTES;
                    tma_load_2d_pair(sa, &tmA, k * kBlockK, arow, fb);
                    tma_load_2d_pair(sa + kABytes, &tmB, k * kBlockK, brow, fb);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok && leader)
                for (int s = 0; s < STAGES; ++s)
                    if ((armed >> s) & 1u)
                        mbar_wait_drain(full_bar(s), (armed_par >> s) & 1u, tmo);
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0 && !leader) {
            // follower: relay "accumulator drained" to the leader, once per tile
            int acc = 0;
            uint32_t acc_phase = 0;
            for (int u = first; u < n_units; u += stride) {
                if (!mbar_wait_bounded(tempty_bar(acc), acc_phase, tmo, s_abort, p.status))
                    break;
                mbar_arrive_cluster(mapa_shared(tempty_bar(acc), 0));
                if (++acc == ACC_BUFS) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
        }
        if (lane == 0 && leader) {
            // ------------------------------------------------ MMA issuer
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            for (int u = first; u < n_units && ok; u += stride) {
                const Tile tl = tile_of(u);
                const uint32_t n = (uint32_t)((tl.nrows + 31) & ~31);
                const uint32_t idesc = idesc_bf16_f32(2 * kBlockM, n);
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
                    const uint32_t sa = base_u32 + stage * C::STAGE_BYTES;
                    const uint32_t sb = sa + kABytes;
#pragma unroll
                    for (int kk = 0; kk < kBlockK / 16; ++kk)
                        mma_bf16_ss_pair(d, smem_desc_k128(sa + kk * 32),
                                         smem_desc_k128(sb + kk * 32), idesc, (k | kk) != 0);
                    mma_commit_pair(empty_bar(stage), 0x3);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok)
                    break;
                mma_commit_pair(tfull_bar(acc), 0x3);
                if (++acc == ACC_BUFS) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            if (!ok) {
                mma_commit_pair(drain_bar, 0x1);
                mbar_wait_drain(drain_bar, 0, tmo);
            }
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------- epilogue
        const int q = warp & 3;
        const int i = q * 32 + lane;
        const int wg = (warp - 2) >> 2;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int u = first; u < n_units; u += stride) {
            const Tile tl = tile_of(u);
            if (!mbar_wait_bounded(tfull_bar(acc), acc_phase, tmo, s_abort, p.status))
                break;
            tc_fence_after();
            const uint32_t ta = tmem_base + ((uint32_t)(q * 32) << 16) + acc * C::ACC_COLS;
            const int col = tl.m * kBlockM + i;
            for (int c0 = wg * 16; c0 < tl.nrows; c0 += 16 * kEpiWG) {
                uint32_t v[16];
                tmem_ld16(ta + c0, v);
                tmem_ld_wait();
                __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(p.out);
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    if (c0 + j < tl.nrows)
                        out[(size_t)(tl.row0 + c0 + j) * p.out_ld + col] =
                            __float2bfloat16_rn(__uint_as_float(v[j]));
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
    cluster_sync();  // the leader's MMAs into this CTA's memory are done
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc2(tmem_base, C::TMEM_COLS);
    }
}

template <int STAGES, int ACC_BUFS>
cudaError_t launch_pair(const CUtensorMap &a, const CUtensorMap &b, const GemmArgs &args,
                        int grid, int stage, cudaStream_t s)
{
    using C = PairCfg<STAGES, ACC_BUFS>;
    auto kern = grouped_gemm_pair_kernel<STAGES, ACC_BUFS>;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    static int max_pairs = 0;
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        C::SMEM_BYTES);
        if (attr_err != cudaSuccess)
            return;
        // pairs that fit at once (the two SMs of a pair sit in one GPC)
        cudaLaunchConfig_t q = {};
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = 2;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        q.gridDim = dim3(2, 1, 1);
        q.blockDim = dim3(kThreads, 1, 1);
        q.dynamicSmemBytes = C::SMEM_BYTES;
        q.attrs = at;
        q.numAttrs = 1;
        attr_err = cudaOccupancyMaxActiveClusters(&max_pairs, kern, &q);
    });
    if (attr_err != cudaSuccess)
        return attr_err;
    const int pairs = grid / 2 < max_pairs ? grid / 2 : max_pairs;
    if (pairs < 1)
        return cudaErrorInvalidConfiguration;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2 * pairs, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = s;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    stage_begin(stage, s);
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, a, b, args);
    stage_end(stage, s);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

cudaError_t launch_down_pair(const CUtensorMap &wd, const CUtensorMap &hp, const GemmArgs &a,
                             int grid, cudaStream_t s)
{
    return launch_pair<6, 2>(wd, hp, a, grid, kStDown, s);
}

}  // namespace beam
