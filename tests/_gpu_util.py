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


# ------------------------------------------------------------------ routing
#
# Router logits come from one of two FP32 evaluations (beam_moe_router_arith):
#  - the FMA chain (T < 256): the oracle's own arithmetic, so scores must match
#    the oracle bit for bit;
#  - the tensor cores (T >= 256): every product x*w is exact (x is bf16, the
#    FP32 router weight is split exactly into three bf16 parts), and the
#    products are added in FP32 in the tensor cores' order, over up to 8
#    ranges of h whose partial sums are then added in order.  Any FP32
#    summation of n exact terms with a longest chain of d roundings satisfies
#        |l - l_exact| <= ((1 + u)^d - 1) * sum|terms| ~ d * u * sum|x*w|
#    with u = 2^-23 even for round-toward-zero.  The chain here is at most
#    d = 3*H/16 + 16 + 8 (one accumulator addition per 16-deep MMA for each
#    of the three parts, up to 16 inside an MMA, up to 8 partial sums).
#    sigmoid has slope <= 1/4, and the FP32 exp/add/divide of the score add
#    at most 4 * 2^-24.
# Given the same FP32 scores, the selection is a pure function of them, so the
# GPU's ids and weights must equal the oracle's selection on the GPU's scores
# bit for bit (the comparison rule for routing); the oracle's own scores may
# select differently only on near-ties, which are counted and must be rare.

def tc_score_bound(x_bits, router_w):
    """(exact fp64 sigmoid scores [T,E], per-element bound on |s_gpu - s_exact|)."""
    x = (np.asarray(x_bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(
        np.float64)
    w = np.asarray(router_w, np.float64)
    logits = x @ w                     # products exact in fp64; sum error ~2^-53 * A
    A = np.abs(x) @ np.abs(w)
    d = 3 * x.shape[1] // 16 + 16 + 8
    bound = d * 2.0 ** -23 * A / 4.0 + 4 * 2.0 ** -24
    return 1.0 / (1.0 + np.exp(-logits)), bound


def check_tc_scores(g_scores, x_bits, router_w):
    s_exact, bound = tc_score_bound(x_bits, router_w)
    err = np.abs(np.asarray(g_scores, np.float64) - s_exact)
    bad = int((err > bound).sum())
    assert bad == 0, f"{bad} tensor-core router scores outside the FP32 accumulation bound " \
                     f"(max err {err.max():.3e}, max err/bound {(err / bound).max():.3f})"
    return float(err.max()), float(np.sqrt((err ** 2).mean()))


def check_route(oracle_mod, sh, r, x_bits, router_w, arith):
    """Check the GPU routing outputs `r` (BeamMoE.route with scores) of a batch
    against the oracle.  Returns a dict with the checked ids, counts, offsets,
    row_src, the GPU scores and the set of near-tie tokens on which the
    oracle's own scores select differently."""
    from sparse_moe_layer_experts_b300 import binding as B
    g = {k: v.cpu().numpy() for k, v in r.items() if v is not None}
    _, s_o = oracle_mod.router_scores(x_bits, router_w)
    if arith == B.BEAM_MOE_ROUTER_FMA_CHAIN:
        n_diff = int((g["scores"].view(np.uint32) != s_o.view(np.uint32)).sum())
        assert n_diff == 0, f"{n_diff} scores differ from the oracle's"
    else:
        assert arith == B.BEAM_MOE_ROUTER_TENSOR
        check_tc_scores(g["scores"], x_bits, router_w)
    ids, w = oracle_mod.select(g["scores"], sh.G, sh.topk_groups, sh.top_k, sh.scale)
    assert np.array_equal(g["ids"], ids)
    assert np.array_equal(g["w"].view(np.uint32), w.view(np.uint32))
    counts, offsets, row_of, row_src = oracle_mod.dispatch(ids, sh.E)
    assert np.array_equal(g["counts"], counts)
    assert np.array_equal(g["offsets"], offsets)
    assert np.array_equal(g["row_of"], row_of)
    ids_o, _ = oracle_mod.select(s_o, sh.G, sh.topk_groups, sh.top_k, sh.scale)
    flipped = set(int(t) for t in np.nonzero((ids_o != ids).any(axis=1))[0])
    if arith == B.BEAM_MOE_ROUTER_FMA_CHAIN:
        assert not flipped
    else:
        assert len(flipped) <= max(4, sh.T // 1000), f"{len(flipped)} near-tie flips"
    return dict(ids=ids, w=w, counts=counts, offsets=offsets, row_src=row_src,
                scores=g["scores"], flipped=flipped)


def oracle_rows(fwd, toks, route, *args, **kw):
    """The oracle's layer rows for tokens `toks` (a list): its own router for
    every token whose selection agrees with the GPU's, and the GPU's checked
    scores for the near-tie tokens where two valid FP32 evaluations of the
    router select different experts."""
    res = fwd(*args, tokens=toks, **kw)
    ref = res[0] if isinstance(res, tuple) else res
    flip = [i for i, t in enumerate(toks) if t in route["flipped"]]
    if flip:
        sub = fwd(*args, tokens=[toks[i] for i in flip], scores=route["scores"], **kw)
        ref[flip] = sub[0] if isinstance(sub, tuple) else sub
    return ref


def router_arith(layer, T):
    from sparse_moe_layer_experts_b300 import binding as B
    a = B.beam_moe_router_arith(T, layer.cfg)
    assert a >= 0
    return a
