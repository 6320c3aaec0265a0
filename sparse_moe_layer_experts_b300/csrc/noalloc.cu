// beam_moe_forward_noalloc: the layer forward for callers that cannot
// allocate device memory.
//
// beam_moe_forward needs a caller-provided workspace.  Some callers have no
// way to get one: code running where the allocator is owned by someone else
// (a host application that forbids allocations after start-up, a
// pre-allocated inference arena, a plug-in with no handle on the process's
// allocator), or a call made from a context where cudaMalloc is not allowed.
// This entry point keeps its scratch in a fixed array compiled into the
// library, so it allocates nothing at call time.
//
// Cost and limits: the array (kNoAllocScratchBytes) lives in this file's own
// CUDA module.  Under lazy module loading (the CUDA default) a device holds
// it from the first call of this entry point on that device until the
// process exits; under eager loading (CUDA_MODULE_LOADING=EAGER) every
// device on which the process creates a context holds it, whether or not the
// entry point is called.  A call is rejected when the layer's workspace for
// T tokens exceeds the array.  All calls share the one array, so calls that
// overlap on the GPU (different streams, different host threads) race;
// serialise them.
#include "../../include/beam_moe.h"

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(24) << 20;  // 24 MiB
constexpr int kCacheSlots = 64;

// The shared scratch.  In host code this name is only a host-side stand-in:
// its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device addresses of the array, one per CUDA context that has called this
// entry point.  The key is the driver's context id, which is unique for the
// life of the process: a context created after cudaDeviceReset, or a
// non-primary context made current by the caller, gets an id of its own and
// so a fresh lookup, never a stale address.
struct Slot {
    unsigned long long ctx_id;
    void *addr;
};

std::mutex g_mu;
Slot g_slots[kCacheSlots];
int g_next_slot = 0;

PFN_cuCtxGetCurrent_v4000 g_get_current = nullptr;
PFN_cuCtxGetId_v12000 g_get_id = nullptr;

bool driver_entry_points()
{
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    });
    return g_get_current && g_get_id;
}

// Device address of the scratch in the current context.  The first call in
// a context looks it up (cudaGetSymbolAddress, with that context current);
// later calls in the same context reuse it.
int scratch_address(void **out)
{
    if (!driver_entry_points())
        return BEAM_MOE_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    CUcontext ctx = nullptr;
    void *p = nullptr;
    if (g_get_current(&ctx) != CUDA_SUCCESS)
        return BEAM_MOE_ERR_CUDA;
    if (!ctx) {
        // No context is current on this thread yet: the runtime binds the
        // current device's primary context on its first call, this lookup.
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p)
            return BEAM_MOE_ERR_CUDA;
        if (g_get_current(&ctx) != CUDA_SUCCESS || !ctx)
            return BEAM_MOE_ERR_CUDA;
    }
    unsigned long long id = 0;
    if (g_get_id(ctx, &id) != CUDA_SUCCESS)
        return BEAM_MOE_ERR_CUDA;
    for (const Slot &s : g_slots)
        if (s.addr && s.ctx_id == id) {
            *out = s.addr;
            return BEAM_MOE_OK;
        }
    if (!p && (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p))
        return BEAM_MOE_ERR_CUDA;
    g_slots[g_next_slot] = Slot{id, p};
    g_next_slot = (g_next_slot + 1) % kCacheSlots;
    *out = p;
    return BEAM_MOE_OK;
}

}  // namespace

extern "C" int beam_moe_forward_noalloc(const void *x, const float *router_w,
                                        const void *w_gate, const void *w_up,
                                        const void *w_down, int64_t T,
                                        const beam_moe_cfg *cfg, void *out, void *stream)
{
    const size_t need = beam_moe_workspace_size(T, cfg);
    if (need == 0)
        return BEAM_MOE_ERR_INVALID_ARG;  // invalid configuration or T < 0
    if (need > kNoAllocScratchBytes)
        return BEAM_MOE_ERR_WORKSPACE;  // more tokens than the fixed scratch holds
    if (T == 0)
        return BEAM_MOE_OK;
    void *scratch = nullptr;
    const int rc = scratch_address(&scratch);
    if (rc != BEAM_MOE_OK)
        return rc;
    // Same kernels as beam_moe_forward; only the workspace differs.  The
    // first kernel resets the status word, the only scratch value read before
    // it is written, so the previous call's contents do no harm.
    beam_moe_cfg c = *cfg;
    c.workspace = scratch;
    c.workspace_bytes = kNoAllocScratchBytes;
    return beam_moe_forward(x, router_w, w_gate, w_up, w_down, T, &c, out, stream);
}
