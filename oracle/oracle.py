"""numpy front end of the plain C oracle (``beam_moe_oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers.  Nothing in the GPU library
imports this module, and this module imports nothing from the GPU library.

The C source states the method and every reading taken where the Beam pages
are silent.  This file only marshals numpy arrays to it (bf16 tensors travel as
their uint16 bit patterns).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "beam_moe_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

# -ffp-contract=off: no expression is fused unless the source calls fmaf.
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
          "-fno-fast-math"]


def build(force: bool = False) -> str:
    """Compile the oracle shared library next to its source."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        p = ctypes.c_void_p
        i64 = ctypes.c_int64
        i32 = ctypes.c_int
        f32 = ctypes.c_float
        L.oracle_num_threads.restype = i32
        L.oracle_router_scores.argtypes = [p, p, i64, i32, i32, p, p]
        L.oracle_router_scores.restype = None
        L.oracle_select.argtypes = [p, i64, i32, i32, i32, i32, f32, p, p]
        L.oracle_select.restype = i32
        L.oracle_dispatch.argtypes = [p, i64, i32, i32, p, p, p, p]
        L.oracle_dispatch.restype = i32
        L.oracle_expert_row.argtypes = [p, p, p, p, i32, i32, p]
        L.oracle_expert_row.restype = None
        L.oracle_forward.argtypes = [p, p, p, p, p, i64, i32, i32, i32, i32, i32, i32,
                                     f32, p, i64, p, p, p, p, p]
        L.oracle_forward.restype = i32
        L.oracle_dense_forward.argtypes = [p, p, p, p, i64, i32, i32, p, i64, p]
        L.oracle_dense_forward.restype = i32
        L.oracle_block_forward.argtypes = [p, i32, p, p, f32, p, p, p, p, i64, i32, i32, i32,
                                           i32, i32, i32, f32, p, i64, p, p]
        L.oracle_block_forward.restype = i32
        L.oracle_rmsnorm_bf16.argtypes = [p, p, f32, i64, i32, p]
        L.oracle_rmsnorm_bf16.restype = None
        L.oracle_mx_shared_exp.argtypes = [f32]
        L.oracle_mx_shared_exp.restype = i32
        L.oracle_quantize_mxfp8.argtypes = [p, i64, i64, i64, p, p]
        L.oracle_quantize_mxfp8.restype = i32
        L.oracle_fake_quant_mxfp8_rows.argtypes = [p, i64, i64]
        L.oracle_fake_quant_mxfp8_rows.restype = None
        L.oracle_forward_mxfp8.argtypes = [p, p, p, p, p, p, p, p, i64, i32, i32, i32, i32, i32,
                                           i32, f32, p, i64, p, p, p, p, p]
        L.oracle_forward_mxfp8.restype = i32
        L.oracle_e2m1_value.argtypes = [i32]
        L.oracle_e2m1_value.restype = f32
        L.oracle_e2m1_code.argtypes = [f32]
        L.oracle_e2m1_code.restype = i32
        L.oracle_e4m3_value.argtypes = [i32]
        L.oracle_e4m3_value.restype = f32
        L.oracle_e4m3_code.argtypes = [f32]
        L.oracle_e4m3_code.restype = i32
        L.oracle_quantize_nvfp4.argtypes = [p, i64, i64, i64, p, p, p]
        L.oracle_quantize_nvfp4.restype = i32
        L.oracle_fake_quant_rows.argtypes = [p, i64, i64]
        L.oracle_fake_quant_rows.restype = None
        L.oracle_forward_nvfp4.argtypes = [p, p, p, p, p, p, p, p, p, p, p, i64, i32, i32, i32, i32,
                                           i32, i32, f32, p, i64, p, p, p, p, p]
        L.oracle_block_tail.argtypes = [p, i32, p, f32, p, i64, i32, p, i64, p]
        L.oracle_block_tail.restype = i32
        L.oracle_forward_nvfp4.restype = i32
        _lib = L
    return _lib


def _c(a: np.ndarray, dtype) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        raise TypeError(f"expected {dtype}, got {a.dtype}")
    return a


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def num_threads() -> int:
    return int(lib().oracle_num_threads())


def router_scores(x_bits: np.ndarray, router_w: np.ndarray):
    """FP32 logits and sigmoid scores, [T,E] each."""
    x_bits = _c(x_bits, np.uint16)
    router_w = _c(router_w, np.float32)
    T, H = x_bits.shape
    H2, E = router_w.shape
    assert H == H2
    logits = np.empty((T, E), np.float32)
    scores = np.empty((T, E), np.float32)
    lib().oracle_router_scores(_ptr(x_bits), _ptr(router_w), T, H, E, _ptr(logits), _ptr(scores))
    return logits, scores


def select(scores: np.ndarray, n_groups: int, topk_groups: int, top_k: int, scale: float):
    """Group-limited top-k on given scores -> (ids [T,K] int32, w [T,K] fp32)."""
    scores = _c(scores, np.float32)
    T, E = scores.shape
    ids = np.empty((T, top_k), np.int32)
    w = np.empty((T, top_k), np.float32)
    rc = lib().oracle_select(_ptr(scores), T, E, n_groups, topk_groups, top_k,
                             float(scale), _ptr(ids), _ptr(w))
    if rc != 0:
        raise ValueError("oracle_select rejected the configuration or the scores")
    return ids, w


def dispatch(ids: np.ndarray, n_experts: int):
    """(counts [E], offsets [E+1], row_of [T,K], row_src [T*K]) for ids [T,K]."""
    ids = _c(ids, np.int32)
    T, K = ids.shape
    counts = np.empty(n_experts, np.int32)
    offsets = np.empty(n_experts + 1, np.int32)
    row_of = np.empty((T, K), np.int32)
    row_src = np.empty(T * K, np.int32)
    rc = lib().oracle_dispatch(_ptr(ids), T, K, n_experts, _ptr(counts), _ptr(offsets),
                               _ptr(row_of), _ptr(row_src))
    if rc != 0:
        raise ValueError("expert id out of range")
    return counts, offsets, row_of, row_src


def expert_row(x_row_bits, wg_bits, wu_bits, wd_bits):
    """One SwiGLU expert on one token row -> y [H] float64."""
    x_row_bits = _c(x_row_bits, np.uint16)
    wg_bits = _c(wg_bits, np.uint16)
    wu_bits = _c(wu_bits, np.uint16)
    wd_bits = _c(wd_bits, np.uint16)
    I, H = wg_bits.shape
    y = np.empty(H, np.float64)
    lib().oracle_expert_row(_ptr(x_row_bits), _ptr(wg_bits), _ptr(wu_bits), _ptr(wd_bits),
                            H, I, _ptr(y))
    return y


def _scores_in(scores, T, E):
    """Given router scores [T,E] fp32 (or None: the oracle's router runs)."""
    if scores is None:
        return None
    scores = _c(scores, np.float32)
    if scores.shape != (T, E):
        raise ValueError(f"scores must be [T,E] = {(T, E)}")
    return scores


def forward(x_bits, router_w, wg_bits, wu_bits, wd_bits, n_groups, topk_groups, top_k,
            scale, tokens=None, scores=None, combine=False):
    """Layer output for `tokens` (all when None).  With `scores` ([T,E] fp32)
    the given router scores replace the router step (selection onward).

    Returns (out_bits [n,H] uint16, ids [n,K] int32, w [n,K] fp32), and with
    combine=True also the FP32 combine o [n,H] before the bf16 rounding.
    """
    x_bits = _c(x_bits, np.uint16)
    router_w = _c(router_w, np.float32)
    wg_bits = _c(wg_bits, np.uint16)
    wu_bits = _c(wu_bits, np.uint16)
    wd_bits = _c(wd_bits, np.uint16)
    T, H = x_bits.shape
    E, I, H2 = wg_bits.shape
    assert H2 == H and wu_bits.shape == (E, I, H) and wd_bits.shape == (E, H, I)
    assert router_w.shape == (H, E)
    tok = None if tokens is None else _c(np.asarray(tokens, np.int64), np.int64)
    n = T if tok is None else tok.shape[0]
    out = np.empty((n, H), np.uint16)
    ids = np.empty((n, top_k), np.int32)
    w = np.empty((n, top_k), np.float32)
    sc = _scores_in(scores, T, E)  # kept alive for the call
    o = np.empty((n, H), np.float32) if combine else None
    rc = lib().oracle_forward(_ptr(x_bits), _ptr(router_w), _ptr(wg_bits), _ptr(wu_bits),
                              _ptr(wd_bits), T, H, I, E, n_groups, topk_groups, top_k,
                              float(scale), _ptr(tok), n, _ptr(out), _ptr(ids), _ptr(w),
                              _ptr(sc), _ptr(o))
    if rc != 0:
        raise ValueError("oracle_forward failed (bad configuration or token index)")
    return (out, ids, w, o) if combine else (out, ids, w)


def dense_forward(x_bits, wg_bits, wu_bits, wd_bits, tokens=None):
    """Dense SwiGLU MLP (x [T,H], wg/wu [I,H], wd [H,I], bf16 bits) for
    `tokens` (all when None) -> out bits [n,H] uint16."""
    x_bits = _c(x_bits, np.uint16)
    wg_bits = _c(wg_bits, np.uint16)
    wu_bits = _c(wu_bits, np.uint16)
    wd_bits = _c(wd_bits, np.uint16)
    T, H = x_bits.shape
    I, H2 = wg_bits.shape
    assert H2 == H and wu_bits.shape == (I, H) and wd_bits.shape == (H, I)
    tok = None if tokens is None else _c(np.asarray(tokens, np.int64), np.int64)
    n = T if tok is None else tok.shape[0]
    out = np.empty((n, H), np.uint16)
    rc = lib().oracle_dense_forward(_ptr(x_bits), _ptr(wg_bits), _ptr(wu_bits), _ptr(wd_bits),
                                    T, H, I, _ptr(tok), n, _ptr(out))
    if rc != 0:
        raise ValueError("oracle_dense_forward failed (bad token index)")
    return out


def block_forward(s_bits, step, gamma_pre, gamma_post, eps, router_w, wg_bits, wu_bits, wd_bits,
                  n_groups, topk_groups, top_k, scale, tokens=None, scores=None):
    """MoE sublayer with pre-norm, post-norm and the constant-scale residual
    at step `step`: the new stream rows (bf16 bits [n,H]) for `tokens`.
    With `scores` ([T,E] fp32, the router scores of the pre-normed x) the
    given scores replace the router step."""
    s_bits = _c(s_bits, np.uint16)
    gp = _c(gamma_pre, np.float32)
    gq = _c(gamma_post, np.float32)
    router_w = _c(router_w, np.float32)
    wg_bits = _c(wg_bits, np.uint16)
    wu_bits = _c(wu_bits, np.uint16)
    wd_bits = _c(wd_bits, np.uint16)
    T, H = s_bits.shape
    E, I, _ = wg_bits.shape
    assert gp.shape == (H,) and gq.shape == (H,) and router_w.shape == (H, E)
    tok = None if tokens is None else _c(np.asarray(tokens, np.int64), np.int64)
    n = T if tok is None else tok.shape[0]
    out = np.empty((n, H), np.uint16)
    sc = _scores_in(scores, T, E)  # kept alive for the call
    rc = lib().oracle_block_forward(_ptr(s_bits), int(step), _ptr(gp), _ptr(gq), float(eps),
                                    _ptr(router_w), _ptr(wg_bits), _ptr(wu_bits), _ptr(wd_bits),
                                    T, H, I, E, n_groups, topk_groups, top_k, float(scale),
                                    _ptr(tok), n, _ptr(out), _ptr(sc))
    if rc != 0:
        raise ValueError("oracle_block_forward failed (bad configuration, step or token)")
    return out


def block_tail(s_bits, step, gamma_post, eps, o, tokens=None):
    """The fused block's post-norm and residual on a given FP32 layer combine
    o [n,H] (rows of `tokens`, all when None): bf16 bits [n,H]."""
    s_bits = _c(s_bits, np.uint16)
    gq = _c(gamma_post, np.float32)
    o = _c(o, np.float32)
    T, H = s_bits.shape
    tok = None if tokens is None else _c(np.asarray(tokens, np.int64), np.int64)
    n = T if tok is None else tok.shape[0]
    assert o.shape == (n, H) and gq.shape == (H,)
    out = np.empty((n, H), np.uint16)
    rc = lib().oracle_block_tail(_ptr(s_bits), int(step), _ptr(gq), float(eps), _ptr(o), T, H,
                                 _ptr(tok), n, _ptr(out))
    if rc != 0:
        raise ValueError("oracle_block_tail failed (bad step or token)")
    return out


def rmsnorm_bf16(s_bits, gamma, eps):
    """x = bf16(rmsnorm(s) * gamma) row by row (bf16 bits in and out)."""
    s_bits = _c(s_bits, np.uint16)
    g = _c(gamma, np.float32)
    T, H = s_bits.shape
    x = np.empty((T, H), np.uint16)
    lib().oracle_rmsnorm_bf16(_ptr(s_bits), _ptr(g), float(eps), T, H, _ptr(x))
    return x


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


# ------------------------------------------------------------------- NVFP4

def e2m1_value(code: int) -> float:
    return float(lib().oracle_e2m1_value(int(code)))


def e2m1_code(v: float) -> int:
    return int(lib().oracle_e2m1_code(float(v)))


def e4m3_value(code: int) -> float:
    return float(lib().oracle_e4m3_value(int(code)))


def e4m3_code(v: float) -> int:
    return int(lib().oracle_e4m3_code(float(v)))


def quantize_nvfp4(w_bits: np.ndarray):
    """bf16 bits [n_mat, rows, cols] -> (codes [n_mat,rows,cols] u8 one per byte,
    sf [n_mat,rows,cols/16] u8 E4M3, gs [n_mat] f32)."""
    w_bits = _c(w_bits, np.uint16)
    n_mat, rows, cols = w_bits.shape
    codes = np.empty((n_mat, rows, cols), np.uint8)
    sf = np.empty((n_mat, rows, cols // 16), np.uint8)
    gs = np.empty(n_mat, np.float32)
    if lib().oracle_quantize_nvfp4(_ptr(w_bits), n_mat, rows, cols, _ptr(codes), _ptr(sf),
                                   _ptr(gs)) != 0:
        raise ValueError("cols must be a multiple of 16")
    return codes, sf, gs


def fake_quant_rows(v: np.ndarray) -> np.ndarray:
    """Quantise-dequantise fp32 rows [n, k] with global scale 1 (activations)."""
    v = np.array(v, np.float32, copy=True, order="C")
    lib().oracle_fake_quant_rows(_ptr(v), v.shape[0], v.shape[1])
    return v


def dequantize_nvfp4(codes, sf, gs) -> np.ndarray:
    """float64 values q * sf * gs of oracle-layout NVFP4 tensors."""
    e2 = np.array([e2m1_value(c) for c in range(16)], np.float64)
    e4 = np.array([e4m3_value(c) for c in range(256)], np.float64)
    v = e2[codes] * np.repeat(e4[sf], 16, axis=-1)
    return v * np.asarray(gs, np.float64).reshape((-1,) + (1,) * (codes.ndim - 1))


def forward_nvfp4(x_bits, router_w, q_gate, q_up, q_down, n_groups, topk_groups, top_k,
                  scale, tokens=None, scores=None, combine=False):
    """NVFP4 layer for `tokens`; q_* = (codes, sf, gs) from quantize_nvfp4;
    `scores` as in forward()."""
    x_bits = _c(x_bits, np.uint16)
    router_w = _c(router_w, np.float32)
    (gc, gsf, ggs), (uc, usf, ugs), (dc, dsf, dgs) = [
        (_c(c, np.uint8), _c(f, np.uint8), _c(g, np.float32)) for c, f, g in
        (q_gate, q_up, q_down)]
    T, H = x_bits.shape
    E, I, H2 = gc.shape
    assert H2 == H and dc.shape == (E, H, I)
    tok = None if tokens is None else _c(np.asarray(tokens, np.int64), np.int64)
    n = T if tok is None else tok.shape[0]
    out = np.empty((n, H), np.uint16)
    ids = np.empty((n, top_k), np.int32)
    w = np.empty((n, top_k), np.float32)
    sc = _scores_in(scores, T, E)  # kept alive for the call
    o = np.empty((n, H), np.float32) if combine else None
    rc = lib().oracle_forward_nvfp4(_ptr(x_bits), _ptr(router_w), _ptr(gc), _ptr(gsf), _ptr(ggs),
                                    _ptr(uc), _ptr(usf), _ptr(ugs), _ptr(dc), _ptr(dsf),
                                    _ptr(dgs), T, H, I, E, n_groups, topk_groups, top_k,
                                    float(scale), _ptr(tok), n, _ptr(out), _ptr(ids), _ptr(w),
                                    _ptr(sc), _ptr(o))
    if rc != 0:
        raise ValueError("oracle_forward_nvfp4 failed")
    return (out, ids, w, o) if combine else (out, ids, w)


# ---------------------------------------------------------------- MXFP8

def mx_shared_exp(amax: float) -> int:
    """floor(log2(amax)) - 8 clamped to [-127, 127]; -127 for amax = 0."""
    return int(lib().oracle_mx_shared_exp(float(amax)))


def quantize_mxfp8(w_bits: np.ndarray):
    """bf16 bits [n_mat, rows, cols] -> (E4M3 codes [n_mat, rows, cols] uint8,
    UE8M0 scales [n_mat, rows, cols/32] uint8)."""
    w_bits = _c(w_bits, np.uint16)
    n_mat, rows, cols = w_bits.shape
    codes = np.empty((n_mat, rows, cols), np.uint8)
    sf = np.empty((n_mat, rows, cols // 32), np.uint8)
    rc = lib().oracle_quantize_mxfp8(_ptr(w_bits), n_mat, rows, cols, _ptr(codes), _ptr(sf))
    if rc != 0:
        raise ValueError("cols must be a multiple of 32")
    return codes, sf


def fake_quant_mxfp8_rows(v: np.ndarray) -> np.ndarray:
    """Rows of FP32 values -> their MXFP8 values (a copy)."""
    v = np.array(v, np.float32, copy=True, order="C")
    lib().oracle_fake_quant_mxfp8_rows(_ptr(v), v.shape[0], v.shape[1])
    return v


def dequantize_mxfp8(codes, sf) -> np.ndarray:
    """E4M3 codes and UE8M0 scales -> float64 values."""
    codes = np.asarray(codes, np.uint8)
    mag_e = (codes >> 3) & 15
    mag_m = (codes & 7).astype(np.float64)
    mag = np.where(mag_e == 0, mag_m * 2.0 ** -9, (1.0 + mag_m / 8.0) * 2.0 ** (mag_e.astype(np.float64) - 7))
    val = np.where(codes & 0x80, -mag, mag)
    scale = 2.0 ** (np.repeat(np.asarray(sf, np.float64), 32, axis=-1) - 127)
    return val * scale


def forward_mxfp8(x_bits, router_w, q_gate, q_up, q_down, n_groups, topk_groups, top_k, scale,
                  tokens=None, scores=None, combine=False):
    """Layer output with MXFP8 experts; q_* = quantize_mxfp8(w_*) (codes, sf);
    `scores` as in forward()."""
    x_bits = _c(x_bits, np.uint16)
    router_w = _c(router_w, np.float32)
    T, H = x_bits.shape
    E, I, _ = q_gate[0].shape
    gc, gsf = (_c(a, np.uint8) for a in q_gate)
    uc, usf = (_c(a, np.uint8) for a in q_up)
    dc, dsf = (_c(a, np.uint8) for a in q_down)
    tok = None if tokens is None else _c(np.asarray(tokens, np.int64), np.int64)
    n = T if tok is None else tok.shape[0]
    out = np.empty((n, H), np.uint16)
    ids = np.empty((n, top_k), np.int32)
    w = np.empty((n, top_k), np.float32)
    sc = _scores_in(scores, T, E)  # kept alive for the call
    o = np.empty((n, H), np.float32) if combine else None
    rc = lib().oracle_forward_mxfp8(_ptr(x_bits), _ptr(router_w), _ptr(gc), _ptr(gsf), _ptr(uc),
                                    _ptr(usf), _ptr(dc), _ptr(dsf), T, H, I, E, n_groups,
                                    topk_groups, top_k, float(scale), _ptr(tok), n, _ptr(out),
                                    _ptr(ids), _ptr(w), _ptr(sc), _ptr(o))
    if rc != 0:
        raise ValueError("oracle_forward_mxfp8 failed")
    return (out, ids, w, o) if combine else (out, ids, w)

