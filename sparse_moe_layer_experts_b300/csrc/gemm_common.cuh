// Pieces shared by the grouped GEMM kernels (bf16 and NVFP4 weights).
#pragma once

#include "common.cuh"

namespace beam {

struct Tile {
    int e, m, row0, nrows;
};

// Tile t -> (expert, weight tile, token rows).  Tiles of expert e occupy
// [m_tiles*cs[e], m_tiles*cs[e+1]); inside, weight tile major, chunk minor.
// The expert's n rows are split into nc = cs[e+1]-cs[e] near-equal chunks.
__device__ __forceinline__ Tile decode_tile(int t, const int *off, const int *cs, int E,
                                            int m_tiles)
{
    int lo = 0, hi = E - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (m_tiles * cs[mid] <= t)
            lo = mid;
        else
            hi = mid - 1;
    }
    Tile r;
    r.e = lo;
    const int nc = cs[lo + 1] - cs[lo];
    const int local = t - m_tiles * cs[lo];
    r.m = local / nc;
    const int c = local - r.m * nc;
    const int n = off[lo + 1] - off[lo];
    const int r0 = (int)(((long long)c * n) / nc);
    const int r1 = (int)(((long long)(c + 1) * n) / nc);
    r.row0 = off[lo] + r0;
    r.nrows = r1 - r0;
    return r;
}

// Drain-only wait (ignores the abort flag): used on the error path to let
// copies and MMAs that were already issued finish before the CTA exits.
__device__ __forceinline__ void mbar_wait_drain(uint32_t bar, uint32_t parity, uint64_t timeout_ns)
{
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_timer_ns() - t0 > timeout_ns)
            return;
}

}  // namespace beam
