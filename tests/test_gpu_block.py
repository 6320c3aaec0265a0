"""Fused MoE block (pre-norm -> layer -> post-norm -> constant-scale
residual) on the GPU against the oracle, every token at small shapes and
sampled tokens at the prefill size; in-place equals out-of-place."""
import numpy as np
import pytest
import torch

from sparse_moe_layer_experts_b300 import synth
from sparse_moe_layer_experts_b300.layer import BeamMoE

from tests._gpu_util import (N_RANDOM_FULL, REL_L2_TOL, check_route, chunk_rows_of, host_inputs,
                             oracle_rows, out_bits, rel_l2_per_token, router_arith, sample_tokens)

pytestmark = pytest.mark.gpu


def _layer(sh, d):
    return BeamMoE(d["router_w"], d["w_gate"], d["w_up"], d["w_down"], n_groups=sh.G,
                   topk_groups=sh.topk_groups, top_k=sh.top_k, routed_scale=sh.scale)


def _oracle(oracle_mod, sh, h, gp, gq, step, eps, tokens=None, scores=None):
    return oracle_mod.block_forward(h["x"], step, gp.cpu().numpy(), gq.cpu().numpy(), eps,
                                    h["router_w"], h["w_gate"], h["w_up"], h["w_down"], sh.G,
                                    sh.topk_groups, sh.top_k, sh.scale, tokens=tokens,
                                    scores=scores)


@pytest.mark.parametrize("T,step", [(64, 9), (200, 9), (200, 1), (33, 1000)])
def test_block_all_tokens(oracle_mod, T, step):
    sh = synth.shape("tiny", T=T)
    d = synth.make_inputs(sh, seed=7, device="cuda")
    gp, gq = synth.make_block_gains(sh.H, seed=7, device="cuda")
    layer = _layer(sh, d)
    out = layer.block_forward(d["x"], step, gp, gq, 1e-6)
    torch.cuda.synchronize()
    assert layer.status() == 0
    ref = _oracle(oracle_mod, sh, host_inputs(d), gp, gq, step, 1e-6)
    rel = rel_l2_per_token(out_bits(out), ref)
    assert rel.max() <= REL_L2_TOL, (rel.max(), int(rel.argmax()))


def test_block_in_place_and_deterministic():
    sh = synth.shape("tiny", T=150)
    d = synth.make_inputs(sh, seed=8, device="cuda")
    gp, gq = synth.make_block_gains(sh.H, seed=8, device="cuda")
    layer = _layer(sh, d)
    a = layer.block_forward(d["x"], 5, gp, gq, 1e-6).clone()
    b = layer.block_forward(d["x"], 5, gp, gq, 1e-6).clone()
    s = d["x"].clone()
    layer.block_forward(s, 5, gp, gq, 1e-6, out=s)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert torch.equal(a.view(torch.int16), s.view(torch.int16))


@pytest.mark.slow
def test_block_prefill_sampled(oracle_mod):
    sh = synth.shape("prefill")
    d = synth.make_inputs(sh, seed=0, device="cuda")
    gp, gq = synth.make_block_gains(sh.H, seed=0, device="cuda")
    layer = _layer(sh, d)
    out = layer.block_forward(d["x"], 9, gp, gq, 1e-6)
    torch.cuda.synchronize()
    assert layer.status() == 0
    # the block routes the pre-normed stream; the library's router on the
    # oracle's pre-norm of it gives the routing to check (the pre-norm itself
    # is pinned on its own), and its expert segments choose the rows: their
    # edges, the chunk edges of the most loaded expert and 256 seeded random
    # tokens are compared
    h = host_inputs(d)
    xn = oracle_mod.rmsnorm_bf16(h["x"], gp.cpu().numpy(), 1e-6)
    r = layer.route(torch.from_numpy(xn.view(np.int16)).view(torch.bfloat16).cuda())
    route = check_route(oracle_mod, sh, r, xn, h["router_w"], router_arith(layer, sh.T))
    del r
    toks = sample_tokens(sh.T, route["row_src"], route["offsets"], n_random=N_RANDOM_FULL,
                         seed=1, chunk_rows=chunk_rows_of(sh.T, sh.top_k, sh.E))
    ref = oracle_rows(lambda *a, **k: _oracle(oracle_mod, sh, h, gp, gq, 9, 1e-6, **k), toks,
                      route)
    rel = rel_l2_per_token(out_bits(out)[toks], ref)
    assert rel.max() <= REL_L2_TOL, (rel.max(), toks[int(rel.argmax())], len(toks))


@pytest.mark.parametrize("fmt,tol", [("nvfp4", 2e-2), ("mxfp8", 1e-2)])
@pytest.mark.parametrize("T,step", [(64, 9), (300, 5)])
def test_block_quantised_experts_all_tokens(oracle_mod, fmt, tol, T, step):
    """The fused block with NVFP4 / MXFP8 experts on every token, against the
    oracle's pre-norm, the quantised layer oracle's FP32 combine on it, and
    the oracle's post-norm and residual (each pinned on its own).  The
    tolerances are those of the quantised layers."""
    from sparse_moe_layer_experts_b300.layer import quantize_mxfp8, quantize_nvfp4
    sh = synth.shape("tiny", T=T)
    d = synth.make_inputs(sh, seed=17, device="cuda")
    gp, gq = synth.make_block_gains(sh.H, seed=17, device="cuda")
    ws = ("w_gate", "w_up", "w_down")
    kw = dict(n_groups=sh.G, topk_groups=sh.topk_groups, top_k=sh.top_k, routed_scale=sh.scale)
    if fmt == "nvfp4":
        layer = BeamMoE.nvfp4(d["router_w"], *[quantize_nvfp4(d[k]) for k in ws], **kw)
        qo = [oracle_mod.quantize_nvfp4(synth.to_bits(d[k])) for k in ws]
        fwd = oracle_mod.forward_nvfp4
    else:
        layer = BeamMoE.mxfp8(d["router_w"], *[quantize_mxfp8(d[k]) for k in ws], **kw)
        qo = [oracle_mod.quantize_mxfp8(synth.to_bits(d[k])) for k in ws]
        fwd = oracle_mod.forward_mxfp8
    out = layer.block_forward(d["x"], step, gp, gq, 1e-6)
    torch.cuda.synchronize()
    assert layer.status() == 0
    h = host_inputs(d)
    gpn, gqn = gp.cpu().numpy(), gq.cpu().numpy()
    xn = oracle_mod.rmsnorm_bf16(h["x"], gpn, 1e-6)
    r = layer.route(torch.from_numpy(xn.view(np.int16)).view(torch.bfloat16).cuda())
    route = check_route(oracle_mod, sh, r, xn, h["router_w"], router_arith(layer, sh.T))
    cfg = (sh.G, sh.topk_groups, sh.top_k, sh.scale)
    o = fwd(xn, h["router_w"], *qo, *cfg, combine=True)[3]
    flip = sorted(route["flipped"])
    if flip:
        o[flip] = fwd(xn, h["router_w"], *qo, *cfg, tokens=flip, scores=route["scores"],
                      combine=True)[3]
    ref = oracle_mod.block_tail(h["x"], step, gqn, 1e-6, o)
    rel = rel_l2_per_token(out_bits(out), ref)
    assert rel.max() <= tol, (rel.max(), int(rel.argmax()))
