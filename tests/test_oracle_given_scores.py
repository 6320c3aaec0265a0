"""Pins for the oracle's given-scores form: the layer from the selection step
on, applied to FP32 router scores handed in by the caller.

The pages fix the selection, the combine weights, the experts and the combine
as functions of the FP32 scores ("Reflection Beam 1.0", section "Mixture of
Experts": sigmoid scores, group-limited top-8, normalised weights x 2.5), so
the layer given scores must (1) reproduce the router path bit for bit when
handed the router's own scores, and (2) with any other scores, equal the
composition select(scores) -> weighted SwiGLU experts built from pinned
pieces (exhaustive-search selection, numpy expert MLPs).
"""
import numpy as np
import pytest
import torch

from sparse_moe_layer_experts_b300 import synth
from tests import _brute


@pytest.fixture(scope="module")
def tiny():
    sh = synth.shape("tiny", T=24)
    d = synth.make_inputs(sh, seed=21, device="cpu")
    return sh, {k: (synth.to_bits(v) if v.dtype == torch.bfloat16 else synth.to_f32(v))
                for k, v in d.items()}


def _shuffled_scores(scores, seed):
    """Scores that route differently: each token's scores permuted over the
    experts, plus exact ties between the first two experts of group 0."""
    rng = np.random.default_rng(seed)
    s = np.array([row[rng.permutation(row.shape[0])] for row in scores], np.float32)
    s[:, 1] = s[:, 0]
    return s


def _np_swiglu(x, wg, wu, wd):
    g = x @ wg.T
    u = x @ wu.T
    return (g / (1.0 + np.exp(-g)) * u) @ wd.T


def test_bf16_own_scores_reproduce_router_path(oracle_mod, tiny):
    sh, d = tiny
    args = (d["x"], d["router_w"], d["w_gate"], d["w_up"], d["w_down"], sh.G, sh.topk_groups,
            sh.top_k, sh.scale)
    _, scores = oracle_mod.router_scores(d["x"], d["router_w"])
    a = oracle_mod.forward(*args)
    b = oracle_mod.forward(*args, scores=scores)
    for u, v in zip(a, b):
        assert np.array_equal(u.view(np.uint8), v.view(np.uint8))


def test_bf16_given_scores_compose(oracle_mod, tiny):
    sh, d = tiny
    _, scores = oracle_mod.router_scores(d["x"], d["router_w"])
    s = _shuffled_scores(scores, 0)
    # the router weight must not be read: pass a poisoned one
    rw_nan = np.full_like(d["router_w"], np.nan)
    tokens = [0, 5, 23]
    out, ids, w = oracle_mod.forward(d["x"], rw_nan, d["w_gate"], d["w_up"], d["w_down"], sh.G,
                                     sh.topk_groups, sh.top_k, sh.scale, tokens=tokens, scores=s)
    f = oracle_mod.bf16_bits_to_f32
    x = f(d["x"]).astype(np.float64)
    wg, wu, wd = (f(d[k]).astype(np.float64) for k in ("w_gate", "w_up", "w_down"))
    for r, t in enumerate(tokens):
        order, wb, _ = _brute.select(s[t], sh.G, sh.topk_groups, sh.top_k, sh.scale)
        assert ids[r].tolist() == order
        assert np.array_equal(w[r], np.asarray(wb, np.float32))
        ref = sum(float(wk) * _np_swiglu(x[t:t + 1], wg[e], wu[e], wd[e])[0]
                  for e, wk in zip(order, wb))
        got = f(out[r]).astype(np.float64)
        assert np.linalg.norm(got - ref) / np.linalg.norm(ref) < 4e-3, t


def test_quantised_and_block_own_scores_reproduce_router_path(oracle_mod, tiny):
    sh, d = tiny
    rw = d["router_w"]
    _, scores = oracle_mod.router_scores(d["x"], rw)
    qn = [oracle_mod.quantize_nvfp4(d[k]) for k in ("w_gate", "w_up", "w_down")]
    qm = [oracle_mod.quantize_mxfp8(d[k]) for k in ("w_gate", "w_up", "w_down")]
    cfg = (sh.G, sh.topk_groups, sh.top_k, sh.scale)
    for fwd, q in ((oracle_mod.forward_nvfp4, qn), (oracle_mod.forward_mxfp8, qm)):
        a = fwd(d["x"], rw, *q, *cfg)
        b = fwd(d["x"], rw, *q, *cfg, scores=scores)
        for u, v in zip(a, b):
            assert np.array_equal(u.view(np.uint8), v.view(np.uint8))
    gp, gq = (g.numpy() for g in synth.make_block_gains(sh.H, seed=3))
    xn = oracle_mod.rmsnorm_bf16(d["x"], gp, 1e-6)
    _, sn = oracle_mod.router_scores(xn, rw)
    blk = (d["x"], 9, gp, gq, 1e-6, rw, d["w_gate"], d["w_up"], d["w_down"], *cfg)
    assert np.array_equal(oracle_mod.block_forward(*blk),
                          oracle_mod.block_forward(*blk, scores=sn))


def test_quantised_given_scores_select_from_them(oracle_mod, tiny):
    # NVFP4 and MXFP8 layers on other scores pick exactly select(scores)'s
    # experts and weights, and the block's router step is replaced likewise.
    sh, d = tiny
    _, scores = oracle_mod.router_scores(d["x"], d["router_w"])
    s = _shuffled_scores(scores, 1)
    cfg = (sh.G, sh.topk_groups, sh.top_k, sh.scale)
    ids_ref, w_ref = oracle_mod.select(s, *cfg)
    qn = [oracle_mod.quantize_nvfp4(d[k]) for k in ("w_gate", "w_up", "w_down")]
    qm = [oracle_mod.quantize_mxfp8(d[k]) for k in ("w_gate", "w_up", "w_down")]
    for fwd, q in ((oracle_mod.forward_nvfp4, qn), (oracle_mod.forward_mxfp8, qm)):
        _, ids, w = fwd(d["x"], d["router_w"], *q, *cfg, scores=s)
        assert np.array_equal(ids, ids_ref)
        assert np.array_equal(w.view(np.uint32), w_ref.view(np.uint32))
        # and the bf16 layer's expert set differs, so the scores were used
        _, ids_own, _ = fwd(d["x"], d["router_w"], *q, *cfg)
        assert not np.array_equal(ids_own, ids_ref)


def test_given_scores_shape_is_checked(oracle_mod, tiny):
    sh, d = tiny
    with pytest.raises(ValueError):
        oracle_mod.forward(d["x"], d["router_w"], d["w_gate"], d["w_up"], d["w_down"], sh.G,
                           sh.topk_groups, sh.top_k, sh.scale,
                           scores=np.zeros((sh.T, sh.E + 1), np.float32))
