"""Shared helpers of the GPU parity tests."""
import numpy as np
import torch

from sparse_moe_layer_experts_b300 import synth

# Per-token relative L2 bound of the bf16 layer against the oracle.
REL_L2_TOL = 1e-2


def host_inputs(d, experts=None):
    """Host copies for the oracle.  With `experts`, only those experts'
    weights are copied; the rest of the host weight arrays stay zero pages."""
    out = dict(x=synth.to_bits(d["x"]), router_w=synth.to_f32(d["router_w"]))
    for k in ("w_gate", "w_up", "w_down"):
        t = d[k]
        if experts is None:
            out[k] = synth.to_bits(t)
        else:
            a = np.zeros(tuple(t.shape), np.uint16)
            for e in sorted(set(int(v) for v in experts)):
                a[e] = synth.to_bits(t[e])
            out[k] = a
    return out


def rel_l2_per_token(got_bits, ref_bits):
    f = lambda b: (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(
        np.float64)
    g, r = f(got_bits), f(ref_bits)
    num = np.linalg.norm(g - r, axis=-1)
    den = np.linalg.norm(r, axis=-1)
    return num / np.maximum(den, 1e-30)


def out_bits(t: torch.Tensor):
    return synth.to_bits(t)


def sample_tokens(T, row_src, offsets, n_random, seed=0):
    """First/last token, seeded random tokens, and the first and last row of
    every few expert segments (tile edges)."""
    rng = np.random.default_rng(seed)
    toks = {0, T - 1}
    toks.update(int(v) for v in rng.choice(T, size=min(n_random, T), replace=False))
    E = len(offsets) - 1
    for e in range(0, E, max(1, E // 8)):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi > lo:
            toks.add(int(row_src[lo]))
            toks.add(int(row_src[hi - 1]))
    return sorted(toks)
