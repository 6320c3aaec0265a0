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
// Cost and limits: every GPU on which this entry point runs holds the array
// (kNoAllocScratchBytes) until the process exits.  A call is rejected when
// the layer's workspace for T tokens exceeds the array.  All calls share the
// one array, so calls that overlap on the GPU (different streams, different
// host threads) race; serialise them.
#include "../../include/beam_moe.h"

#include <cuda_runtime.h>

#include <mutex>

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(24) << 20;  // 24 MiB
constexpr int kMaxDevices = 64;

// The shared scratch.  In host code this name is only a host-side stand-in:
// its device address comes from cudaGetSymbolAddress, once per device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void *g_scratch_addr[kMaxDevices];

// Device address of the scratch on the current device (looked up on the
// first call per device, with that device current).
int scratch_address(void **out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return BEAM_MOE_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p)
            return BEAM_MOE_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
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
