/*
 * beam_moe.h -- C ABI of the B300 (sm_103a) Beam-style sparse MoE layer.
 *
 * The layer (one forward pass, no shared expert):
 *   1. router logits  l[t,e] = sum_h x[t,h] * Wr[h,e]          (FP32)
 *   2. scores         s[t,e] = sigmoid(l[t,e])                 (FP32)
 *   3. group score    gs[t,g] = sum of the two largest s in group g
 *   4. keep the topk_groups groups with the largest gs
 *   5. pick the top_k experts by s inside the kept groups
 *   6. weights        w[t,k] = s_k / sum_j s_j * routed_scale
 *   7. out[t] = sum_k w[t,k] * SwiGLU_{e_k}(x[t]),
 *      SwiGLU_e(x) = W_down[e] (silu(W_gate[e] x) * (W_up[e] x))
 * Source: "Reflection Beam 1.0: 501B open MoE model, 1M context, Apache 2.0"
 * (agentlenshq.com), section "Mixture of Experts: 256 experts, 8 routed per
 * token" (256 experts, sigmoid scores, 8 groups of 32, rank groups by the sum
 * of their top-2 scores, keep 4 groups, top-8 experts, no shared expert,
 * normalised weights scaled by 2.5, SwiGLU experts of intermediate 2560), and
 * the same page's section "Residual stream", last paragraph (router and the
 * SwiGLU product in FP32).  Restated by "Beam 501B open model" (aixai.ru),
 * section "256 experts per layer", and by the dothoosh.com news article,
 * section "Architecture and memory efficiency".
 *
 * Readings taken where the pages are silent: ties go to the lower group or
 * expert index; the selected slots are ordered by score descending, index
 * ascending; the router logits are FP32 sums of exact products (a sequential
 * FMA chain for small batches, tensor cores for large ones: see
 * beam_moe_router_arith); sigmoid(l) = 1/(1 + fp32(exp(-l))).
 *
 * Conventions shared by every call:
 *  - Pointers named as device pointers are CUDA device memory owned by the
 *    caller.  The library never allocates, frees or synchronises device
 *    memory, except where a function says so.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Work is enqueued asynchronously on it; host-detectable errors
 *    return before anything is enqueued.
 *  - Device-detected errors (a bounded wait that ran out, a failed debug
 *    check) are written to a status word inside the workspace; read it with
 *    beam_moe_read_status() before the next call on that workspace, whose
 *    first kernel clears it.
 *  - bf16 tensors are IEEE bfloat16, row-major, densely packed.
 *  - All device pointers must be 16-byte aligned.
 *  - Calls that share a workspace must not overlap on the GPU; calls with
 *    distinct workspaces may run concurrently from any threads.
 */
#ifndef BEAM_MOE_H
#define BEAM_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes.  Negative = error. */
typedef enum {
    BEAM_MOE_OK = 0,
    BEAM_MOE_ERR_INVALID_ARG = -1,  /* bad pointer, size or configuration  */
    BEAM_MOE_ERR_UNSUPPORTED = -2,  /* valid but not implemented           */
    BEAM_MOE_ERR_CUDA = -3,         /* a CUDA runtime/driver call failed   */
    BEAM_MOE_ERR_WORKSPACE = -4,    /* workspace missing or too small      */
    BEAM_MOE_ERR_TIMEOUT = -5,      /* device: a bounded wait ran out      */
    BEAM_MOE_ERR_DEVICE = -6        /* device: an internal check failed    */
} beam_moe_status;

/* Expert weight formats. */
typedef enum {
    BEAM_MOE_W_BF16 = 0,
    BEAM_MOE_W_NVFP4 = 1,
    BEAM_MOE_W_MXFP8 = 2
} beam_moe_wtype;

/* debug_flags bits (tests only). */
#define BEAM_MOE_DEBUG_DROP_ONE_LOAD 0x1u /* CTA 0 of the gate/up GEMM never
                                             arms one pipeline stage, so its
                                             consumer's bounded wait runs out
                                             and the call reports
                                             BEAM_MOE_ERR_TIMEOUT            */

/*
 * Layer configuration.  Beam: hidden 5120, inter 2560, n_experts 256,
 * n_groups 8, topk_groups 4, top_k 8, routed_scale 2.5.
 * Requirements: hidden, inter multiples of 128; 4 <= n_experts <= 256 with
 * n_experts % 4 == 0; 1 <= n_groups <= 32; n_experts % n_groups == 0;
 * n_experts / n_groups <= 32; 1 <= topk_groups <= n_groups;
 * 1 <= top_k <= min(32, topk_groups * n_experts / n_groups).
 * Anything else returns BEAM_MOE_ERR_INVALID_ARG with nothing enqueued.
 */
typedef struct {
    int hidden;          /* H */
    int inter;           /* I */
    int n_experts;       /* E */
    int n_groups;        /* G */
    int topk_groups;     /* groups kept per token */
    int top_k;           /* experts per token (K) */
    float routed_scale;  /* 2.5 for Beam */
    int wtype;           /* beam_moe_wtype */
    /* NVFP4 weights only (else NULL): per-16-element E4M3 block scales and
       FP32 per-(expert, projection) global scales, see beam_moe_quantize_nvfp4 */
    const void *w_gate_sf, *w_up_sf, *w_down_sf;
    const float *w_gate_gs, *w_up_gs, *w_down_gs;
    /* caller-owned device scratch, >= beam_moe_workspace_size() bytes,
       256-byte aligned */
    void *workspace;
    size_t workspace_bytes;
    /* bounded device waits give up after this many nanoseconds (0 = 2 s) */
    int64_t wait_timeout_ns;
    unsigned debug_flags; /* 0 in production */
} beam_moe_cfg;

/* Fill *cfg with the Beam layer sizes and no workspace. */
void beam_moe_cfg_init_beam(beam_moe_cfg *cfg);

/*
 * Bytes of device workspace a call with T tokens needs (0 on an invalid
 * configuration).  The size grows linearly with T.
 */
size_t beam_moe_workspace_size(int64_t T, const beam_moe_cfg *cfg);

/*
 * Routing only (steps 1-6) plus the expert histogram.
 *   x        [T,H] bf16, device
 *   router_w [H,E] fp32, device (hidden-major)
 *   topk_ids [T,K] int32, device, out: expert ids in slot order
 *   topk_w   [T,K] fp32, device, out: combine weights (sum = routed_scale)
 *   scores   [T,E] fp32, device, out, or NULL: the sigmoid scores
 *   counts   [E]   int32, device, out, or NULL: tokens routed to each expert
 *   offsets  [E+1] int32, device, out, or NULL: exclusive prefix of counts
 *   row_of   [T,K] int32, device, out, or NULL: row of pair (t,k) in the
 *            expert-grouped order (experts ascending, tokens ascending)
 * T = 0 is a successful no-op.  Requires T * K < 2^31.
 */
int beam_moe_route(const void *x, const float *router_w, int64_t T,
                   const beam_moe_cfg *cfg, int32_t *topk_ids, float *topk_w,
                   float *scores, int32_t *counts, int32_t *offsets,
                   int32_t *row_of, void *stream);

/*
 * How the router logits of a batch of T tokens are computed (the pages pin
 * only "router in FP32": "Reflection Beam 1.0", section "Residual stream",
 * last paragraph).  Returns one of:
 *   BEAM_MOE_ROUTER_FMA_CHAIN  each logit is the FP32 fused multiply-add
 *                              chain over h = 0..H-1 from +0, i.e. exactly a
 *                              sequential FP32 dot product (T < 256);
 *   BEAM_MOE_ROUTER_TENSOR     tensor cores: router_w is split into three
 *                              bf16 parts whose sum is router_w exactly, so
 *                              every product x*w is exact, and the products
 *                              are summed in FP32 in the tensor cores' order
 *                              (T >= 256).  A logit then differs from the
 *                              sequential FP32 dot product only by FP32
 *                              accumulation rounding.
 * In both cases sigmoid(l) = 1/(1 + fp32(exp(-l))) is applied to the FP32
 * logit, and the selection uses those FP32 scores.  Returns
 * BEAM_MOE_ERR_INVALID_ARG for an invalid configuration or T < 0.
 */
#define BEAM_MOE_ROUTER_FMA_CHAIN 0
#define BEAM_MOE_ROUTER_TENSOR 1
int beam_moe_router_arith(int64_t T, const beam_moe_cfg *cfg);

/*
 * The whole layer forward (steps 1-7).
 *   x        [T,H] bf16, device
 *   router_w [H,E] fp32, device
 *   w_gate   [E,I,H] bf16, device (per expert: nn.Linear [out=I, in=H])
 *   w_up     [E,I,H] bf16, device
 *   w_down   [E,H,I] bf16, device (per expert: [out=H, in=I])
 *   out      [T,H] bf16, device, written
 * With cfg->wtype == BEAM_MOE_W_NVFP4 the three weight pointers are packed
 * E2M1 codes as produced by beam_moe_quantize_nvfp4 (w_gate/w_up: n_mat = E,
 * rows = I, cols = H; w_down: n_mat = E, rows = H, cols = I), and
 * cfg->w_*_sf / cfg->w_*_gs point at the matching block and global scales
 * (16-byte aligned).  The activations are then quantised to NVFP4 as well
 * (16-element blocks, global scale 1): x before the gate/up GEMM, h before
 * the down GEMM, and both expert GEMMs run on the FP4 tensor cores with
 * FP32 accumulation.  The router stays FP32 on the bf16 x.
 * Deterministic: the same inputs give bitwise the same output.
 */
int beam_moe_forward(const void *x, const float *router_w, const void *w_gate,
                     const void *w_up, const void *w_down, int64_t T,
                     const beam_moe_cfg *cfg, void *out, void *stream);

/*
 * beam_moe_forward with the activations in HOST memory: copies x_host
 * ([T,H] bf16, pinned for best speed) to the workspace, runs the layer and
 * copies the result back to out_host ([T,H] bf16).  Weights stay in device
 * memory.  Synchronises `stream` before returning, so out_host is ready.
 * Needs beam_moe_workspace_size(T) + 2*T*H*2 bytes of workspace.
 */
int beam_moe_forward_hostio(const void *x_host, const float *router_w,
                            const void *w_gate, const void *w_up,
                            const void *w_down, int64_t T,
                            const beam_moe_cfg *cfg, void *out_host,
                            void *stream);

/* Extra workspace bytes beam_moe_forward_hostio needs on top of
   beam_moe_workspace_size(). */
size_t beam_moe_hostio_extra_bytes(int64_t T, const beam_moe_cfg *cfg);

/*
 * beam_moe_forward for callers that cannot allocate device memory.  The
 * pages have no counterpart: this is a library convenience, not part of the
 * method.
 *
 * Who needs it: callers whose device memory is owned by someone else and who
 * cannot call cudaMalloc (a host application that forbids allocations after
 * start-up, a fixed inference arena, a plug-in without access to the
 * process's allocator).  They pass inputs and outputs only; the scratch
 * lives in a 24 MiB array compiled into the library, and this call makes no
 * allocation of any kind.
 *
 * Arguments are those of beam_moe_forward; cfg->workspace and
 * cfg->workspace_bytes are ignored.
 *  - Limit: beam_moe_workspace_size(T, cfg) must not exceed 24 MiB (at the
 *    Beam sizes: T <= 122 tokens); larger calls return BEAM_MOE_ERR_WORKSPACE
 *    with nothing enqueued.  Invalid configurations return
 *    BEAM_MOE_ERR_INVALID_ARG; T = 0 returns BEAM_MOE_OK.
 *  - Memory: the array sits in its own CUDA module.  Under lazy module
 *    loading (the CUDA default) a GPU holds the 24 MiB from the first call
 *    of this entry point on it until the process exits; under eager loading
 *    (CUDA_MODULE_LOADING=EAGER) every GPU on which the process creates a
 *    context holds it, even if this entry point is never called.
 *  - Set-up: the first call in each CUDA context (each device's primary
 *    context, and any context the caller makes current) looks up the
 *    array's device address (cudaGetSymbolAddress) with that context
 *    current and caches it under the context's id; make that first call
 *    before any stream capture.
 *  - Sharing: all calls share the one array and each call overwrites it, so
 *    calls that overlap on the GPU race; serialise them.  The device status
 *    word lives in the shared array and is not readable through
 *    beam_moe_read_status.
 */
int beam_moe_forward_noalloc(const void *x, const float *router_w,
                             const void *w_gate, const void *w_up,
                             const void *w_down, int64_t T,
                             const beam_moe_cfg *cfg, void *out, void *stream);

/*
 * NVFP4 weight quantisation (E2M1 values, one E4M3 scale per 16 consecutive
 * elements of a row, one FP32 global scale per matrix).
 *   w        [n_mat, rows, cols] bf16, device; rows % 128 == 0, cols % 64 == 0
 *   packed   [n_mat, rows, cols/2] uint8, device, out (two codes per byte,
 *            element 2j in the low nibble, bit 3 of a code = sign)
 *   block_sf [n_mat, rows/128, cols/64, 512] uint8, device, out (E4M3
 *            bits): the scale of elements [16b, 16b+16) of row r is byte
 *            16*(r % 32) + 4*((r % 128) / 32) + b % 4 of tile
 *            (r / 128, b / 4), so the 512 scales of one 128 x 64 weight tile
 *            are contiguous, rows in the order the FP4 tensor cores' scale
 *            copy takes them
 *   global_sf[n_mat] fp32, device, out
 * Recipe (the pages name the format only: "most parameters in 4 bits"; the
 * recipe is a reading): gs = amax|W| / (6*448) per matrix (1 if all zero);
 * per block sf = e4m3((amax16 / 6) / gs); q = e2m1(v / (sf * gs)), 0 when
 * sf = 0; round to nearest even, saturating.  Dequantised value: q * sf * gs.
 * All pointers 16-byte aligned.  Two kernel launches on `stream`.
 */
int beam_moe_quantize_nvfp4(const void *w, int64_t n_mat, int64_t rows,
                            int64_t cols, void *packed, void *block_sf,
                            float *global_sf, void *stream);

/*
 * Dense SwiGLU MLP, the feed-forward block of Beam's first three decoder
 * layers ("Reflection Beam 1.0", section "Architecture: hybrid attention,
 * grouped experts, constant-scale residual stream": the first 3 of the 52
 * layers use a dense SwiGLU MLP, the other 49 the MoE block).  The pages
 * give no intermediate size for it: cfg->inter is the caller's.
 *   out[t] = bf16( (silu(x[t] . Wg^T) * (x[t] . Wu^T)) . Wd^T )
 * with FP32 accumulation and the SiLU*up product in FP32 (h is rounded to
 * bf16 as the operand of the second GEMM, as in the MoE experts).
 *   x      [T,H] bf16, device        w_gate, w_up [I,H] bf16, device
 *   w_down [H,I] bf16, device        out [T,H] bf16, device, written
 * Uses cfg->hidden (H), cfg->inter (I), cfg->workspace/workspace_bytes
 * (>= beam_moe_dense_workspace_size) and cfg->wait_timeout_ns; the routing
 * fields are ignored.  Requirements: H and I multiples of 128, bf16 weights
 * (BEAM_MOE_ERR_UNSUPPORTED for NVFP4), 16-byte aligned pointers, out not
 * overlapping x.  Asynchronous on `stream`; T = 0 is a no-op; device errors
 * land in the workspace status word (beam_moe_read_status).  Deterministic.
 */
size_t beam_moe_dense_workspace_size(int64_t T, const beam_moe_cfg *cfg);
int beam_moe_dense_forward(const void *x, const void *w_gate, const void *w_up,
                           const void *w_down, int64_t T, const beam_moe_cfg *cfg,
                           void *out, void *stream);

/*
 * One MoE sublayer of the decoder with its norms and residual update
 * ("Reflection Beam 1.0", section "Residual stream: a constant scale with
 * depth-dependent weights": the input embedding is step 1; at step k the
 * sublayer output is added with weight 1/sqrt(k) and the stream kept with
 * weight sqrt((k-1)/k); every sublayer is normalised before and after, and
 * normalisations run in FP32).  Readings where the pages are silent: the
 * norm is RMSNorm with a per-channel gain; the sum of squares is
 * accumulated in FP64 and rounded to FP32 once as a mean; r = 1/sqrt(mean +
 * eps) in FP32; the stream is bf16.
 *   x      = bf16( (s * r_s) * norm_pre )            the MoE layer's input
 *   o      = the layer's FP32 combine of the K expert rows (no bf16 rounding)
 *   z      = (o * r_o) * norm_post
 *   s_out  = bf16( a * s + b * z ),  a = sqrt((step-1)/step), b = 1/sqrt(step)
 *   stream_in  [T,H] bf16, device (the residual stream at step-1)
 *   norm_pre, norm_post [H] fp32, device;  eps in [0, 1]
 *   stream_out [T,H] bf16, device, written; may be stream_in (in place), must
 *              not partly overlap it
 * Routing and experts as beam_moe_forward on x, with any expert format of
 * cfg->wtype (bf16, NVFP4 or MXFP8 weights and their scales, as for
 * beam_moe_forward; the quantised formats quantise x and h the same way, and
 * o is their FP32 combine); H <= 8192 (else BEAM_MOE_ERR_UNSUPPORTED).
 * Workspace: beam_moe_block_workspace_size.  step >= 1.  Asynchronous;
 * deterministic.
 */
size_t beam_moe_block_workspace_size(int64_t T, const beam_moe_cfg *cfg);
int beam_moe_block_forward(const void *stream_in, int step, const float *norm_pre,
                           const float *norm_post, float eps, const float *router_w,
                           const void *w_gate, const void *w_up, const void *w_down,
                           int64_t T, const beam_moe_cfg *cfg, void *stream_out,
                           void *stream);

/*
 * MXFP8 weight quantisation (E4M3 values, one power-of-two scale per 32
 * consecutive elements of a row).  The pages only say an FP8 checkpoint
 * exists ("Reflection Beam 1.0", section "Mixture of Experts", checkpoint
 * paragraph); the recipe is a reading, the OCP microscaling rule: shared
 * exponent E = floor(log2(amax32)) - 8 clamped to [-127, 127] (-127 for an
 * all-zero block), q = e4m3_rn_satfinite(v / 2^E), scale byte E + 127.
 *   w        [n_mat, rows, cols] bf16, device; rows % 128 == 0, cols % 128 == 0
 *   codes    [n_mat, rows, cols] uint8 (E4M3 bits), device, out
 *   block_sf [n_mat, rows/128, cols/128, 512] uint8, device, out: the scale
 *            byte of elements [32b, 32b+32) of row r is byte
 *            16*(r % 32) + 4*((r % 128) / 32) + b % 4 of tile (r/128, b/4)
 * With cfg->wtype == BEAM_MOE_W_MXFP8, beam_moe_forward takes these codes as
 * the weight pointers and cfg->w_*_sf as the matching scales (the global
 * scale pointers are unused); x and h are quantised to MXFP8 the same way
 * and the expert GEMMs run on the FP8 tensor cores (kind::mxf8f6f4).
 * All pointers 16-byte aligned.  One kernel launch on `stream`.
 */
int beam_moe_quantize_mxfp8(const void *w, int64_t n_mat, int64_t rows,
                            int64_t cols, void *codes, void *block_sf,
                            void *stream);

/*
 * Activation quantisation: FP32 rows quantised with the rule the layer
 * applies to x and h when wtype is NVFP4 or MXFP8 (global scale 1), for
 * callers that want the layer's activation codes outside the layer.
 *   NVFP4: codes [rows, cols/2] (two E2M1 codes per byte, even element in
 *          the low nibble), sf [rows, cols/16] E4M3 bytes; cols % 16 == 0.
 *          Per 16-block: sf = e4m3_rn_satfinite(amax/6), q = e2m1_rn_satfinite(v/sf)
 *          (0 where sf == 0).
 *   MXFP8: codes [rows, cols] E4M3 bytes, sf [rows, cols/32] scale bytes
 *          E + 127; cols % 32 == 0.  The rule of beam_moe_quantize_mxfp8.
 *   x [rows, cols] float32, device, 16-byte aligned; codes 16-byte aligned.
 * Returns BEAM_MOE_ERR_INVALID_ARG for any other wtype or a bad size or
 * pointer (nothing is launched then).  One kernel launch on `stream`.
 */
int beam_moe_quantize_act(int wtype, const float *x, int64_t rows,
                          int64_t cols, void *codes, void *sf, void *stream);

/*
 * Synchronise `stream`, read the device status word of cfg->workspace and
 * clear it.  Returns BEAM_MOE_OK, BEAM_MOE_ERR_TIMEOUT or BEAM_MOE_ERR_DEVICE
 * (or BEAM_MOE_ERR_CUDA if the synchronisation itself failed).
 * The status word is not sticky across calls: the first kernel of every
 * call that uses the workspace (route, forward, block, dense) clears it, so
 * a caller that wants a call's status must read it after that call and
 * before enqueueing the next call on the same workspace.
 */
int beam_moe_read_status(const beam_moe_cfg *cfg, void *stream);

/* Static text for a return code. */
const char *beam_moe_status_string(int code);

/* Number of kernels the library has launched from the calling host thread. */
int64_t beam_moe_launch_count(void);

/*
 * Per-kernel timing hook for benchmarks.  With n > 0, each kernel the
 * library launches from the calling host thread is bracketed by
 * cudaEventRecord(start[i]) and cudaEventRecord(stop[i]) on its stream, i
 * being the kernel's stage: 0 router scores, 1 selection, 2 histogram,
 * 3 scan, 4 permute, 5 gate/up GEMM, 6 down GEMM, 7 combine, 8 NVFP4
 * quantisation of h (NVFP4 layers only), 9 pre-norm (beam_moe_block_forward
 * only).  Events are cudaEvent_t handles passed as void*, owned by the caller
 * and alive while set; n = 0 turns the hook off.  Returns
 * BEAM_MOE_ERR_INVALID_ARG for n < 0, n > 10 or NULL arrays.
 */
int beam_moe_set_kernel_events(void *const *start, void *const *stop, int n);

/* Number of streaming multiprocessors of the current device (0 if none). */
int beam_moe_device_sms(void);

#ifdef __cplusplus
}
#endif

#endif /* BEAM_MOE_H */
