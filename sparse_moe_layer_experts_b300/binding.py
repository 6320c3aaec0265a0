"""ctypes binding of libbeam_moe.so (the C ABI declared in include/beam_moe.h).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  torch supplies device memory and streams.  If the library is missing
or cannot be loaded, importing the functions raises; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libbeam_moe.so")

BEAM_MOE_OK = 0
BEAM_MOE_ERR_INVALID_ARG = -1
BEAM_MOE_ERR_UNSUPPORTED = -2
BEAM_MOE_ERR_CUDA = -3
BEAM_MOE_ERR_WORKSPACE = -4
BEAM_MOE_ERR_TIMEOUT = -5
BEAM_MOE_ERR_DEVICE = -6

BEAM_MOE_ROUTER_FMA_CHAIN = 0
BEAM_MOE_ROUTER_TENSOR = 1

BEAM_MOE_W_BF16 = 0
BEAM_MOE_W_NVFP4 = 1
BEAM_MOE_W_MXFP8 = 2
BEAM_MOE_DEBUG_DROP_ONE_LOAD = 0x1


class beam_moe_cfg(ctypes.Structure):
    _fields_ = [
        ("hidden", ctypes.c_int),
        ("inter", ctypes.c_int),
        ("n_experts", ctypes.c_int),
        ("n_groups", ctypes.c_int),
        ("topk_groups", ctypes.c_int),
        ("top_k", ctypes.c_int),
        ("routed_scale", ctypes.c_float),
        ("wtype", ctypes.c_int),
        ("w_gate_sf", ctypes.c_void_p),
        ("w_up_sf", ctypes.c_void_p),
        ("w_down_sf", ctypes.c_void_p),
        ("w_gate_gs", ctypes.c_void_p),
        ("w_up_gs", ctypes.c_void_p),
        ("w_down_gs", ctypes.c_void_p),
        ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_size_t),
        ("wait_timeout_ns", ctypes.c_int64),
        ("debug_flags", ctypes.c_uint),
    ]


class BeamMoeError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {beam_moe_status_string(code)} ({code})")
        self.code = code


_lib = None


def lib():
    """Load libbeam_moe.so (raises if it is absent: no fallback path exists)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing; build it with "
                              "`python -m sparse_moe_layer_experts_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
        vp, i64, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t
        cfgp = ctypes.POINTER(beam_moe_cfg)
        L.beam_moe_cfg_init_beam.argtypes = [cfgp]
        L.beam_moe_cfg_init_beam.restype = None
        L.beam_moe_workspace_size.argtypes = [i64, cfgp]
        L.beam_moe_workspace_size.restype = sz
        L.beam_moe_hostio_extra_bytes.argtypes = [i64, cfgp]
        L.beam_moe_hostio_extra_bytes.restype = sz
        L.beam_moe_router_arith.argtypes = [i64, cfgp]
        L.beam_moe_router_arith.restype = ctypes.c_int
        L.beam_moe_route.argtypes = [vp, vp, i64, cfgp, vp, vp, vp, vp, vp, vp, vp]
        L.beam_moe_route.restype = ctypes.c_int
        L.beam_moe_forward.argtypes = [vp, vp, vp, vp, vp, i64, cfgp, vp, vp]
        L.beam_moe_forward.restype = ctypes.c_int
        L.beam_moe_forward_hostio.argtypes = [vp, vp, vp, vp, vp, i64, cfgp, vp, vp]
        L.beam_moe_forward_hostio.restype = ctypes.c_int
        L.beam_moe_quantize_nvfp4.argtypes = [vp, i64, i64, i64, vp, vp, vp, vp]
        L.beam_moe_quantize_nvfp4.restype = ctypes.c_int
        L.beam_moe_quantize_mxfp8.argtypes = [vp, i64, i64, i64, vp, vp, vp]
        L.beam_moe_quantize_mxfp8.restype = ctypes.c_int
        L.beam_moe_quantize_act.argtypes = [ctypes.c_int, vp, i64, i64, vp, vp, vp]
        L.beam_moe_quantize_act.restype = ctypes.c_int
        L.beam_moe_read_status.argtypes = [cfgp, vp]
        L.beam_moe_read_status.restype = ctypes.c_int
        L.beam_moe_status_string.argtypes = [ctypes.c_int]
        L.beam_moe_status_string.restype = ctypes.c_char_p
        L.beam_moe_launch_count.argtypes = []
        L.beam_moe_launch_count.restype = i64
        L.beam_moe_set_kernel_events.argtypes = [ctypes.POINTER(vp), ctypes.POINTER(vp),
                                                 ctypes.c_int]
        L.beam_moe_set_kernel_events.restype = ctypes.c_int
        L.beam_moe_device_sms.argtypes = []
        L.beam_moe_device_sms.restype = ctypes.c_int
        L.beam_moe_dense_workspace_size.argtypes = [i64, cfgp]
        L.beam_moe_dense_workspace_size.restype = sz
        L.beam_moe_dense_forward.argtypes = [vp, vp, vp, vp, i64, cfgp, vp, vp]
        L.beam_moe_dense_forward.restype = ctypes.c_int
        L.beam_moe_block_workspace_size.argtypes = [i64, cfgp]
        L.beam_moe_block_workspace_size.restype = sz
        L.beam_moe_block_forward.argtypes = [vp, ctypes.c_int, vp, vp, ctypes.c_float, vp, vp, vp,
                                             vp, i64, cfgp, vp, vp]
        L.beam_moe_block_forward.restype = ctypes.c_int
        _lib = L
    return _lib


# ---------------------------------------------------------------- raw C calls
# Same names and argument order as the C ABI.  Pointers are ints (e.g.
# tensor.data_ptr()) or None; `stream` is a cudaStream_t as an int.

def beam_moe_cfg_init_beam(cfg: beam_moe_cfg) -> None:
    lib().beam_moe_cfg_init_beam(ctypes.byref(cfg))


def beam_moe_workspace_size(T: int, cfg: beam_moe_cfg) -> int:
    return int(lib().beam_moe_workspace_size(T, ctypes.byref(cfg)))


def beam_moe_router_arith(T: int, cfg: beam_moe_cfg) -> int:
    return int(lib().beam_moe_router_arith(T, ctypes.byref(cfg)))


def beam_moe_hostio_extra_bytes(T: int, cfg: beam_moe_cfg) -> int:
    return int(lib().beam_moe_hostio_extra_bytes(T, ctypes.byref(cfg)))


def beam_moe_route(x, router_w, T, cfg, topk_ids, topk_w, scores, counts, offsets, row_of,
                   stream) -> int:
    return lib().beam_moe_route(x, router_w, T, ctypes.byref(cfg), topk_ids, topk_w, scores,
                                counts, offsets, row_of, stream)


def beam_moe_forward(x, router_w, w_gate, w_up, w_down, T, cfg, out, stream) -> int:
    return lib().beam_moe_forward(x, router_w, w_gate, w_up, w_down, T, ctypes.byref(cfg), out,
                                  stream)


def beam_moe_forward_hostio(x_host, router_w, w_gate, w_up, w_down, T, cfg, out_host,
                            stream) -> int:
    return lib().beam_moe_forward_hostio(x_host, router_w, w_gate, w_up, w_down, T,
                                         ctypes.byref(cfg), out_host, stream)


def beam_moe_dense_workspace_size(T: int, cfg: beam_moe_cfg) -> int:
    return int(lib().beam_moe_dense_workspace_size(T, ctypes.byref(cfg)))


def beam_moe_dense_forward(x, w_gate, w_up, w_down, T, cfg, out, stream) -> int:
    return lib().beam_moe_dense_forward(x, w_gate, w_up, w_down, T, ctypes.byref(cfg), out, stream)


def beam_moe_block_workspace_size(T: int, cfg: beam_moe_cfg) -> int:
    return int(lib().beam_moe_block_workspace_size(T, ctypes.byref(cfg)))


def beam_moe_block_forward(stream_in, step, norm_pre, norm_post, eps, router_w, w_gate, w_up,
                           w_down, T, cfg, stream_out, stream) -> int:
    return lib().beam_moe_block_forward(stream_in, step, norm_pre, norm_post, eps, router_w, w_gate,
                                        w_up, w_down, T, ctypes.byref(cfg), stream_out, stream)


def beam_moe_quantize_nvfp4(w, n_mat, rows, cols, packed, block_sf, global_sf, stream) -> int:
    return lib().beam_moe_quantize_nvfp4(w, n_mat, rows, cols, packed, block_sf, global_sf,
                                         stream)


def beam_moe_quantize_mxfp8(w, n_mat, rows, cols, codes, block_sf, stream) -> int:
    return lib().beam_moe_quantize_mxfp8(w, n_mat, rows, cols, codes, block_sf, stream)


def beam_moe_quantize_act(wtype, x, rows, cols, codes, sf, stream) -> int:
    return lib().beam_moe_quantize_act(wtype, x, rows, cols, codes, sf, stream)


def beam_moe_read_status(cfg: beam_moe_cfg, stream) -> int:
    return lib().beam_moe_read_status(ctypes.byref(cfg), stream)


def beam_moe_status_string(code: int) -> str:
    return lib().beam_moe_status_string(code).decode()


def beam_moe_launch_count() -> int:
    return int(lib().beam_moe_launch_count())


def beam_moe_set_kernel_events(starts, stops) -> int:
    """starts/stops: sequences of cudaEvent_t handles (ints); empty turns off."""
    n = len(starts)
    arr = ctypes.c_void_p * max(n, 1)
    return int(lib().beam_moe_set_kernel_events(arr(*starts), arr(*stops), n))


KERNEL_STAGES = ("router_scores", "select", "hist", "scan", "permute", "gateup_gemm",
                 "down_gemm", "combine", "quantize_h", "prenorm")


def beam_moe_device_sms() -> int:
    return int(lib().beam_moe_device_sms())


def check(code: int, what: str) -> None:
    if code != BEAM_MOE_OK:
        raise BeamMoeError(code, what)


def make_cfg(H, I, E, G, topk_groups, top_k, scale=2.5, wtype=BEAM_MOE_W_BF16) -> beam_moe_cfg:
    c = beam_moe_cfg()
    c.hidden, c.inter, c.n_experts, c.n_groups = H, I, E, G
    c.topk_groups, c.top_k, c.routed_scale, c.wtype = topk_groups, top_k, scale, wtype
    return c


def beam_moe_forward_noalloc(x, router_w, w_gate, w_up, w_down, T, cfg, out, stream) -> int:
    """The layer forward with the library's built-in scratch (no workspace,
    no allocation); for callers that cannot allocate device memory."""
    f = lib().beam_moe_forward_noalloc
    if f.argtypes is None:
        vp = ctypes.c_void_p
        f.argtypes = [vp, vp, vp, vp, vp, ctypes.c_int64, ctypes.POINTER(beam_moe_cfg), vp, vp]
        f.restype = ctypes.c_int
    return f(x, router_w, w_gate, w_up, w_down, T, ctypes.byref(cfg), out, stream)
