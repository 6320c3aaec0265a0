"""torch-facing wrapper of the C ABI: one Beam MoE layer with resident weights.

Marshalling only (shapes, dtypes, device pointers, the workspace tensor); all
arithmetic runs in libbeam_moe.so.
"""
from __future__ import annotations

import torch

from . import binding as B


def _stream_handle(stream) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def quantize_nvfp4(w: torch.Tensor, stream=None):
    """NVFP4-quantise bf16 matrices [n_mat, rows, cols] on the GPU.

    Returns (packed [n_mat, rows, cols/2] uint8, block scales (flat uint8, the
    tiled layout of beam_moe_quantize_nvfp4), global scales [n_mat] fp32)."""
    if w.dtype != torch.bfloat16 or w.dim() != 3 or not w.is_cuda or not w.is_contiguous():
        raise ValueError("w must be a contiguous CUDA bf16 [n_mat, rows, cols] tensor")
    n_mat, rows, cols = w.shape
    packed = torch.empty((n_mat, rows, cols // 2), dtype=torch.uint8, device=w.device)
    sf = torch.empty(n_mat * rows * (cols // 16), dtype=torch.uint8, device=w.device)
    gs = torch.empty(n_mat, dtype=torch.float32, device=w.device)
    B.check(B.beam_moe_quantize_nvfp4(w.data_ptr(), n_mat, rows, cols, packed.data_ptr(),
                                      sf.data_ptr(), gs.data_ptr(), _stream_handle(stream)),
            "beam_moe_quantize_nvfp4")
    return packed, sf, gs


def quantize_mxfp8(w: torch.Tensor, stream=None):
    """MXFP8-quantise bf16 matrices [n_mat, rows, cols] on the GPU.

    Returns (E4M3 codes [n_mat, rows, cols] uint8, block scales (flat uint8,
    the tiled layout of beam_moe_quantize_mxfp8))."""
    if w.dtype != torch.bfloat16 or w.dim() != 3 or not w.is_cuda or not w.is_contiguous():
        raise ValueError("w must be a contiguous CUDA bf16 [n_mat, rows, cols] tensor")
    n_mat, rows, cols = w.shape
    codes = torch.empty((n_mat, rows, cols), dtype=torch.uint8, device=w.device)
    sf = torch.empty(n_mat * rows * (cols // 32), dtype=torch.uint8, device=w.device)
    B.check(B.beam_moe_quantize_mxfp8(w.data_ptr(), n_mat, rows, cols, codes.data_ptr(),
                                      sf.data_ptr(), _stream_handle(stream)),
            "beam_moe_quantize_mxfp8")
    return codes, sf


def quantize_activations(x: torch.Tensor, wtype: int, stream=None):
    """Quantise FP32 activation rows [rows, cols] with the layer's activation
    rule (global scale 1).  wtype B.BEAM_MOE_W_NVFP4: (codes [rows, cols/2]
    two per byte, E4M3 scales [rows, cols/16]); B.BEAM_MOE_W_MXFP8: (E4M3
    codes [rows, cols], scale bytes [rows, cols/32])."""
    if x.dtype != torch.float32 or x.dim() != 2 or not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous CUDA float32 [rows, cols] tensor")
    rows, cols = x.shape
    mx8 = wtype == B.BEAM_MOE_W_MXFP8
    codes = torch.empty((rows, cols if mx8 else cols // 2), dtype=torch.uint8, device=x.device)
    sf = torch.empty((rows, cols // (32 if mx8 else 16)), dtype=torch.uint8, device=x.device)
    B.check(B.beam_moe_quantize_act(wtype, x.data_ptr(), rows, cols, codes.data_ptr(),
                                    sf.data_ptr(), _stream_handle(stream)),
            "beam_moe_quantize_act")
    return codes, sf


class BeamMoE:
    """Resident-weight layer.  Weights: w_gate/w_up [E,I,H] bf16, w_down [E,H,I]
    bf16, router_w [H,E] fp32, all contiguous on one CUDA device.  For NVFP4
    weights use BeamMoE.nvfp4()."""

    def __init__(self, router_w, w_gate, w_up, w_down, n_groups=8, topk_groups=4, top_k=8,
                 routed_scale=2.5, wait_timeout_ns=0, debug_flags=0):
        E, I, H = w_gate.shape
        for t, shape, dt in ((router_w, (H, E), torch.float32), (w_gate, (E, I, H), torch.bfloat16),
                             (w_up, (E, I, H), torch.bfloat16), (w_down, (E, H, I), torch.bfloat16)):
            if tuple(t.shape) != shape or t.dtype != dt or not t.is_cuda or not t.is_contiguous():
                raise ValueError(f"expected contiguous CUDA {dt} of shape {shape}")
        self._setup(router_w, w_gate, w_up, w_down, E, I, H, n_groups, topk_groups, top_k,
                    routed_scale, wait_timeout_ns, debug_flags)

    def _setup(self, router_w, w_gate, w_up, w_down, E, I, H, n_groups, topk_groups, top_k,
               routed_scale, wait_timeout_ns, debug_flags, wtype=B.BEAM_MOE_W_BF16):
        self.router_w, self.w_gate, self.w_up, self.w_down = router_w, w_gate, w_up, w_down
        self.H, self.I, self.E = H, I, E
        self.cfg = B.make_cfg(H, I, E, n_groups, topk_groups, top_k, routed_scale, wtype)
        self.cfg.wait_timeout_ns = wait_timeout_ns
        self.cfg.debug_flags = debug_flags
        self.device = w_gate.device
        self._ws = None

    @classmethod
    def nvfp4(cls, router_w, q_gate, q_up, q_down, n_groups=8, topk_groups=4, top_k=8,
              routed_scale=2.5, wait_timeout_ns=0):
        """Layer with NVFP4 experts; q_* = quantize_nvfp4(w_*)."""
        self = cls.__new__(cls)
        E, I, H2 = q_gate[0].shape
        H = H2 * 2
        self._setup(router_w, q_gate[0], q_up[0], q_down[0], E, I, H, n_groups, topk_groups,
                    top_k, routed_scale, wait_timeout_ns, 0, B.BEAM_MOE_W_NVFP4)
        self._scales = (q_gate, q_up, q_down)  # keep them alive
        self.cfg.w_gate_sf, self.cfg.w_up_sf, self.cfg.w_down_sf = (
            q[1].data_ptr() for q in (q_gate, q_up, q_down))
        self.cfg.w_gate_gs, self.cfg.w_up_gs, self.cfg.w_down_gs = (
            q[2].data_ptr() for q in (q_gate, q_up, q_down))
        return self

    @classmethod
    def mxfp8(cls, router_w, q_gate, q_up, q_down, n_groups=8, topk_groups=4, top_k=8,
              routed_scale=2.5, wait_timeout_ns=0):
        """Layer with MXFP8 experts; q_* = quantize_mxfp8(w_*)."""
        self = cls.__new__(cls)
        E, I, H = q_gate[0].shape
        self._setup(router_w, q_gate[0], q_up[0], q_down[0], E, I, H, n_groups, topk_groups,
                    top_k, routed_scale, wait_timeout_ns, 0, B.BEAM_MOE_W_MXFP8)
        self._scales = (q_gate, q_up, q_down)  # keep them alive
        self.cfg.w_gate_sf, self.cfg.w_up_sf, self.cfg.w_down_sf = (
            q[1].data_ptr() for q in (q_gate, q_up, q_down))
        return self

    @property
    def top_k(self):
        return self.cfg.top_k

    def workspace(self, T: int, extra: int = 0) -> torch.Tensor:
        need = B.beam_moe_workspace_size(T, self.cfg)
        if need == 0:
            raise ValueError("invalid layer configuration")
        need += extra
        if self._ws is None or self._ws.numel() < need:
            self._ws = torch.empty(need, dtype=torch.uint8, device=self.device)
        self.cfg.workspace = self._ws.data_ptr()
        self.cfg.workspace_bytes = self._ws.numel()
        return self._ws

    def _check_x(self, x):
        if x.dtype != torch.bfloat16 or x.dim() != 2 or x.shape[1] != self.H or not x.is_contiguous():
            raise ValueError("x must be contiguous bf16 [T, H]")

    def route(self, x, want_scores=True, stream=None):
        self._check_x(x)
        T, K, E = x.shape[0], self.top_k, self.E
        dev = x.device
        out = dict(
            ids=torch.empty((T, K), dtype=torch.int32, device=dev),
            w=torch.empty((T, K), dtype=torch.float32, device=dev),
            scores=torch.empty((T, E), dtype=torch.float32, device=dev) if want_scores else None,
            counts=torch.empty(E, dtype=torch.int32, device=dev),
            offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
            row_of=torch.empty((T, K), dtype=torch.int32, device=dev),
        )
        self.workspace(T)
        p = lambda t: t.data_ptr() if t is not None else None
        B.check(B.beam_moe_route(x.data_ptr(), self.router_w.data_ptr(), T, self.cfg,
                                 p(out["ids"]), p(out["w"]), p(out["scores"]), p(out["counts"]),
                                 p(out["offsets"]), p(out["row_of"]), _stream_handle(stream)),
                "beam_moe_route")
        return out

    def forward(self, x, out=None, stream=None):
        self._check_x(x)
        T = x.shape[0]
        if out is None:
            out = torch.empty_like(x)
        self.workspace(T)
        B.check(B.beam_moe_forward(x.data_ptr(), self.router_w.data_ptr(), self.w_gate.data_ptr(),
                                   self.w_up.data_ptr(), self.w_down.data_ptr(), T, self.cfg,
                                   out.data_ptr(), _stream_handle(stream)), "beam_moe_forward")
        return out

    def block_forward(self, s, step, norm_pre, norm_post, eps=1e-6, out=None, stream=None):
        """The MoE sublayer at residual step `step` with its pre-/post-norms:
        returns bf16(sqrt((step-1)/step) * s + rmsnorm(layer(rmsnorm(s) *
        norm_pre)) * norm_post / sqrt(step)).  out may be s (in place)."""
        self._check_x(s)
        for g in (norm_pre, norm_post):
            if (g.dtype != torch.float32 or tuple(g.shape) != (self.H,) or not g.is_cuda
                    or not g.is_contiguous()):
                raise ValueError("norm gains must be contiguous CUDA fp32 [H]")
        T = s.shape[0]
        if out is None:
            out = torch.empty_like(s)
        need = B.beam_moe_block_workspace_size(T, self.cfg)
        self.workspace(T, max(0, need - B.beam_moe_workspace_size(T, self.cfg)))
        B.check(B.beam_moe_block_forward(s.data_ptr(), int(step), norm_pre.data_ptr(),
                                         norm_post.data_ptr(), float(eps), self.router_w.data_ptr(),
                                         self.w_gate.data_ptr(), self.w_up.data_ptr(),
                                         self.w_down.data_ptr(), T, self.cfg, out.data_ptr(),
                                         _stream_handle(stream)), "beam_moe_block_forward")
        return out

    def forward_host(self, x_host, out_host, stream=None):
        """x_host/out_host: CPU bf16 [T,H] tensors (pinned for speed)."""
        if x_host.is_cuda or out_host.is_cuda:
            raise ValueError("host tensors expected")
        self._check_x(x_host)
        T = x_host.shape[0]
        self.workspace(T, B.beam_moe_hostio_extra_bytes(T, self.cfg))
        B.check(B.beam_moe_forward_hostio(x_host.data_ptr(), self.router_w.data_ptr(),
                                          self.w_gate.data_ptr(), self.w_up.data_ptr(),
                                          self.w_down.data_ptr(), T, self.cfg, out_host.data_ptr(),
                                          _stream_handle(stream)), "beam_moe_forward_hostio")
        return out_host

    def status(self, stream=None) -> int:
        return B.beam_moe_read_status(self.cfg, _stream_handle(stream))


class DenseSwiGLU:
    """Dense SwiGLU MLP with resident bf16 weights: w_gate/w_up [I,H],
    w_down [H,I], contiguous on one CUDA device."""

    def __init__(self, w_gate, w_up, w_down, wait_timeout_ns=0):
        I, H = w_gate.shape
        for t, shape in ((w_gate, (I, H)), (w_up, (I, H)), (w_down, (H, I))):
            if (tuple(t.shape) != shape or t.dtype != torch.bfloat16 or not t.is_cuda
                    or not t.is_contiguous()):
                raise ValueError(f"expected contiguous CUDA bf16 of shape {shape}")
        self.w_gate, self.w_up, self.w_down = w_gate, w_up, w_down
        self.H, self.I = H, I
        self.cfg = B.beam_moe_cfg()
        self.cfg.hidden, self.cfg.inter = H, I
        self.cfg.wtype = B.BEAM_MOE_W_BF16
        self.cfg.wait_timeout_ns = wait_timeout_ns
        self.device = w_gate.device
        self._ws = None

    def workspace(self, T: int) -> torch.Tensor:
        need = B.beam_moe_dense_workspace_size(T, self.cfg)
        if need == 0:
            raise ValueError("invalid layer configuration")
        if self._ws is None or self._ws.numel() < need:
            self._ws = torch.empty(need, dtype=torch.uint8, device=self.device)
        self.cfg.workspace = self._ws.data_ptr()
        self.cfg.workspace_bytes = self._ws.numel()
        return self._ws

    def forward(self, x, out=None, stream=None):
        if x.dtype != torch.bfloat16 or x.dim() != 2 or x.shape[1] != self.H or not x.is_contiguous():
            raise ValueError("x must be contiguous bf16 [T, H]")
        T = x.shape[0]
        if out is None:
            out = torch.empty_like(x)
        self.workspace(T)
        B.check(B.beam_moe_dense_forward(x.data_ptr(), self.w_gate.data_ptr(), self.w_up.data_ptr(),
                                         self.w_down.data_ptr(), T, self.cfg, out.data_ptr(),
                                         _stream_handle(stream)), "beam_moe_dense_forward")
        return out

    def status(self, stream=None) -> int:
        return B.beam_moe_read_status(self.cfg, _stream_handle(stream))

