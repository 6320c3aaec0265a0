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


def sample_tokens(T, row_src, offsets, n_random, seed=0, chunk_rows=None, n_hot=1):
    """Tokens whose layer outputs a full-size test compares with the oracle.

    - token 0 and token T-1;
    - the first and last row of EVERY non-empty expert segment (the ragged
      edges of each expert's token tiles);
    - with chunk_rows: the first and last row of every token chunk of the
      n_hot most loaded experts.  An expert of n rows is cut into
      ceil(n / chunk_rows) near-equal chunks, chunk c starting at row
      floor(c * n / nc) of the segment (the grouped GEMMs' token tiles);
    - n_random seeded random tokens (all tokens when n_random >= T).
    Returns a sorted list of distinct token indices; no cap is applied."""
    rng = np.random.default_rng(seed)
    toks = {0, T - 1}
    if n_random >= T:
        toks.update(range(T))
    else:
        toks.update(int(v) for v in rng.choice(T, size=n_random, replace=False))
    offsets = np.asarray(offsets, np.int64)
    counts = offsets[1:] - offsets[:-1]
    for e in np.nonzero(counts)[0]:
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        toks.add(int(row_src[lo]))
        toks.add(int(row_src[hi - 1]))
    if chunk_rows:
        for e in np.argsort(-counts, kind="stable")[:n_hot]:
            n = int(counts[e])
            if n == 0:
                continue
            nc = -(-n // chunk_rows)
            base = int(offsets[e])
            for c in range(nc):
                first = c * n // nc
                last = (c + 1) * n // nc - 1
                toks.add(int(row_src[base + first]))
                toks.add(int(row_src[base + last]))
    return sorted(toks)


def chunk_rows_of(T, K, E, fmt="bf16"):
    """Token-chunk height of the grouped GEMMs the library runs for this
    batch: decode-size batches (T*K <= 16*E rows) use 32-row chunks, larger
    ones 256 rows (bf16) or 128 rows (NVFP4, MXFP8).  Used only to choose
    which rows to sample."""
    if T * K <= 16 * E:
        return 32
    return 256 if fmt == "bf16" else 128


# Random tokens every full-size test checks on top of the segment and chunk
# edges (the oracle runs about 25 tokens/s on 16 host cores).
N_RANDOM_FULL = 256
