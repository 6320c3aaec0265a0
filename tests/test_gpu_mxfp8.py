"""MXFP8 experts on the GPU (kind::mxf8f6f4 tensor cores) against the oracle:
the weight quantiser bit for bit, the layer on every token at small shapes
(decode and prefill kernel shapes, ragged tails, several weight tiles) and
sampled tokens at the decode and prefill sizes."""
import numpy as np
import pytest
import torch

from sparse_moe_layer_experts_b300 import synth
from sparse_moe_layer_experts_b300.layer import BeamMoE, quantize_mxfp8

from tests._gpu_util import (N_RANDOM_FULL, check_route, chunk_rows_of, oracle_rows, out_bits,
                             rel_l2_per_token, router_arith, sample_tokens)

pytestmark = pytest.mark.gpu

# Both sides quantise x and h with the same rule; they differ by FP32 vs FP64
# accumulation and by h codes that land on the other side of a rounding
# boundary (each such code moves one element by up to 1/16 of its value).
MXFP8_TOL = 1e-2


def untile_scales(flat: np.ndarray, n_mat, rows, cols) -> np.ndarray:
    """tiled [n, rows/128, cols/128, 512] -> [n, rows, cols/32]; inside a tile
    row r = m0 + 32*m1 holds its 4 scales at byte 16*m0 + 4*m1."""
    t = flat.reshape(n_mat, rows // 128, cols // 128, 32, 4, 4)
    return t.transpose(0, 1, 4, 3, 2, 5).reshape(n_mat, rows, cols // 32)


def test_quantizer_bitexact(oracle_mod):
    g = torch.Generator(device="cuda").manual_seed(9)
    w = (torch.randn(3, 256, 384, generator=g, device="cuda")
         * torch.exp(torch.randn(3, 256, 1, generator=g, device="cuda") * 3)).to(torch.bfloat16)
    w[1, 5, 64:96] = 0.0
    codes, sf = quantize_mxfp8(w)
    torch.cuda.synchronize()
    c_o, s_o = oracle_mod.quantize_mxfp8(synth.to_bits(w))
    assert np.array_equal(codes.cpu().numpy(), c_o)
    assert np.array_equal(untile_scales(sf.cpu().numpy(), 3, 256, 384), s_o)


def _oracle_q(oracle_mod, d, experts=None):
    out = []
    for k in ("w_gate", "w_up", "w_down"):
        t = d[k]
        if experts is None:
            out.append(oracle_mod.quantize_mxfp8(synth.to_bits(t)))
        else:
            E, R, C = t.shape
            codes = np.zeros((E, R, C), np.uint8)
            sf = np.zeros((E, R, C // 32), np.uint8)
            for e in experts:
                c1, s1 = oracle_mod.quantize_mxfp8(synth.to_bits(t[e:e + 1]))
                codes[e], sf[e] = c1[0], s1[0]
            out.append((codes, sf))
    return out


def _layer(sh, d):
    q = [quantize_mxfp8(d[k]) for k in ("w_gate", "w_up", "w_down")]
    return BeamMoE.mxfp8(d["router_w"], *q, n_groups=sh.G, topk_groups=sh.topk_groups,
                         top_k=sh.top_k, routed_scale=sh.scale)


SMALL = {
    "tiny": synth.shape("tiny"),
    "tiny_T200": synth.shape("tiny", T=200),
    "medium": synth.LayerShape(T=1501, H=512, I=384, E=64, G=8, topk_groups=4, top_k=8),
    # H/128 odd: the weight-major MXFP8 down GEMM (the token-major down GEMM
    # pairs weight tiles, so it needs an even H/128)
    "odd_tiles": synth.LayerShape(T=3001, H=640, I=256, E=32, G=8, topk_groups=4, top_k=8),
}


@pytest.mark.parametrize("name", list(SMALL))
def test_mxfp8_forward_small_all_tokens(oracle_mod, name):
    sh = SMALL[name]
    d = synth.make_inputs(sh, seed=13, device="cuda")
    layer = _layer(sh, d)
    xb, rw = synth.to_bits(d["x"]), synth.to_f32(d["router_w"])
    route = check_route(oracle_mod, sh, layer.route(d["x"]), xb, rw, router_arith(layer, sh.T))
    out = layer.forward(d["x"])
    torch.cuda.synchronize()
    assert layer.status() == 0
    ref = oracle_rows(oracle_mod.forward_mxfp8, list(range(sh.T)), route, xb, rw,
                      *_oracle_q(oracle_mod, d), sh.G, sh.topk_groups, sh.top_k, sh.scale)
    rel = rel_l2_per_token(out_bits(out), ref)
    assert rel.max() <= MXFP8_TOL, (rel.max(), int(rel.argmax()))


def test_mxfp8_deterministic():
    sh = SMALL["medium"]
    d = synth.make_inputs(sh, seed=14, device="cuda")
    layer = _layer(sh, d)
    a = layer.forward(d["x"]).clone()
    b = layer.forward(d["x"]).clone()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.slow
@pytest.mark.parametrize("name", ["decode", "prefill"])
def test_mxfp8_full_size_sampled(oracle_mod, name):
    """Full-size MXFP8 layer against the oracle with the identical
    quantisation: routing of every token checked; outputs of every decode
    token, and
    at prefill size of the segment edges of every expert, the chunk edges of
    the most loaded expert and 256 seeded random tokens."""
    sh = synth.shape(name)
    d = synth.make_inputs(sh, seed=0, device="cuda")
    layer = _layer(sh, d)
    out = layer.forward(d["x"])
    r = layer.route(d["x"])
    torch.cuda.synchronize()
    assert layer.status() == 0
    xb, rw = synth.to_bits(d["x"]), synth.to_f32(d["router_w"])
    route = check_route(oracle_mod, sh, r, xb, rw, router_arith(layer, sh.T))
    del r
    toks = sample_tokens(sh.T, route["row_src"], route["offsets"], n_random=N_RANDOM_FULL,
                         chunk_rows=chunk_rows_of(sh.T, sh.top_k, sh.E, "mxfp8"))
    if name == "decode":
        assert toks == list(range(sh.T))
    q = _oracle_q(oracle_mod, d, experts=np.unique(route["ids"][toks]))
    ref = oracle_rows(oracle_mod.forward_mxfp8, toks, route, xb, rw, *q, sh.G, sh.topk_groups,
                      sh.top_k, sh.scale)
    rel = rel_l2_per_token(out_bits(out)[toks], ref)
    assert rel.max() <= MXFP8_TOL, (rel.max(), toks[int(rel.argmax())], len(toks))
