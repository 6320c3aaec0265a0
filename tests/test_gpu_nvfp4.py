"""GPU parity of the NVFP4 variant: the device quantiser bit-exact against the
oracle's, and the NVFP4 layer within a per-token relative L2 of 2e-2 of the
oracle that applies the same quantisation (weights, x and h)."""
import numpy as np
import pytest
import torch

from sparse_moe_layer_experts_b300 import synth
from sparse_moe_layer_experts_b300.layer import BeamMoE, quantize_nvfp4
from tests._gpu_util import (N_RANDOM_FULL, check_route, chunk_rows_of, oracle_rows, out_bits,
                             rel_l2_per_token, router_arith, sample_tokens)

pytestmark = pytest.mark.gpu

NVFP4_TOL = 2e-2


def unpack_codes(packed: np.ndarray) -> np.ndarray:
    """[..., cols/2] two codes per byte (even element low) -> [..., cols]."""
    lo, hi = packed & 0xF, packed >> 4
    return np.stack([lo, hi], axis=-1).reshape(*packed.shape[:-1], packed.shape[-1] * 2)


def untile_scales(flat: np.ndarray, n_mat, rows, cols) -> np.ndarray:
    """tiled [n, rows/128, cols/64, 512] -> [n, rows, cols/16].  Inside a tile,
    row r = m0 + 32*m1 holds its 4 scales at byte 16*m0 + 4*m1."""
    t = flat.reshape(n_mat, rows // 128, cols // 64, 32, 4, 4)  # .., m0, m1, kb
    return t.transpose(0, 1, 4, 3, 2, 5).reshape(n_mat, rows, cols // 16)


def test_quantizer_bitexact(oracle_mod):
    g = torch.Generator(device="cuda").manual_seed(7)
    w = torch.randn(4, 256, 320, generator=g, device="cuda")
    w[0] *= 0.02
    # wide dynamic range: E4M3 subnormal and saturated block scales
    w[1] *= torch.exp2(torch.randint(-24, 6, (256, 320), generator=g, device="cuda").float())
    w[2] = 0.0                      # all-zero matrix (global scale 1)
    w[3, 5, 16:48] = 0.0            # zero blocks
    w[3, 7, :16] = -0.0
    wb = w.to(torch.bfloat16).contiguous()
    packed, sf, gs = quantize_nvfp4(wb)
    torch.cuda.synchronize()
    codes, sf_o, gs_o = oracle_mod.quantize_nvfp4(synth.to_bits(wb))
    assert np.array_equal(gs.cpu().numpy().view(np.uint32), gs_o.view(np.uint32))
    assert np.array_equal(untile_scales(sf.cpu().numpy(), 4, 256, 320), sf_o)
    assert np.array_equal(unpack_codes(packed.cpu().numpy()), codes)


def _oracle_q(oracle_mod, d, experts=None):
    """Oracle quantisation of the layer's weights (only `experts` if given)."""
    out = []
    for k in ("w_gate", "w_up", "w_down"):
        t = d[k]
        E, R, C = t.shape
        codes = np.zeros((E, R, C), np.uint8)
        sf = np.zeros((E, R, C // 16), np.uint8)
        gs = np.ones(E, np.float32)
        sel = range(E) if experts is None else sorted(set(int(e) for e in experts))
        for e in sel:
            c1, s1, g1 = oracle_mod.quantize_nvfp4(synth.to_bits(t[e:e + 1]))
            codes[e], sf[e], gs[e] = c1[0], s1[0], g1[0]
        out.append((codes, sf, gs))
    return out


def _nvfp4_layer(sh, d):
    q = [quantize_nvfp4(d[k]) for k in ("w_gate", "w_up", "w_down")]
    return BeamMoE.nvfp4(d["router_w"], *q, n_groups=sh.G, topk_groups=sh.topk_groups,
                         top_k=sh.top_k, routed_scale=sh.scale)


SMALL = {
    "tiny": synth.shape("tiny"),
    "tiny_T200": synth.shape("tiny", T=200),
    "medium": synth.LayerShape(T=1501, H=512, I=384, E=64, G=8, topk_groups=4, top_k=8),
    # H/128 odd and K = H not a multiple of 256: a short last k-step in the
    # token-major NVFP4 gate/up, and the weight-major NVFP4 down GEMM (the
    # token-major down GEMM pairs weight tiles, so it needs an even H/128)
    "odd_tiles": synth.LayerShape(T=3001, H=640, I=256, E=32, G=8, topk_groups=4, top_k=8),
}


@pytest.mark.parametrize("name", list(SMALL))
def test_nvfp4_forward_small_all_tokens(oracle_mod, name):
    sh = SMALL[name]
    d = synth.make_inputs(sh, seed=11, device="cuda")
    layer = _nvfp4_layer(sh, d)
    xb, rw = synth.to_bits(d["x"]), synth.to_f32(d["router_w"])
    route = check_route(oracle_mod, sh, layer.route(d["x"]), xb, rw, router_arith(layer, sh.T))
    out = layer.forward(d["x"])
    torch.cuda.synchronize()
    assert layer.status() == 0
    q = _oracle_q(oracle_mod, d)
    ref = oracle_rows(oracle_mod.forward_nvfp4, list(range(sh.T)), route, xb, rw, *q, sh.G,
                      sh.topk_groups, sh.top_k, sh.scale)
    rel = rel_l2_per_token(out_bits(out), ref)
    assert rel.max() <= NVFP4_TOL, (rel.max(), int(rel.argmax()))


def test_nvfp4_deterministic():
    sh = SMALL["medium"]
    d = synth.make_inputs(sh, seed=12, device="cuda")
    layer = _nvfp4_layer(sh, d)
    a = layer.forward(d["x"]).clone()
    b = layer.forward(d["x"]).clone()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.slow
@pytest.mark.parametrize("name", ["nvfp4", "decode"])
def test_nvfp4_full_size_sampled(oracle_mod, name):
    """Full-size NVFP4 layer in the configuration the benchmark times, against
    the oracle with the identical quantisation: routing of every token
    checked; layer
    outputs of every token of the decode batch, and at T=8192 of token 0 and
    T-1, the first and last row of every non-empty expert segment, the first
    and last row of every token chunk of the most loaded expert, and 256
    seeded random tokens."""
    sh = synth.shape(name)
    d = synth.make_inputs(sh, seed=0, device="cuda")
    layer = _nvfp4_layer(sh, d)
    out = layer.forward(d["x"])
    r = layer.route(d["x"])
    torch.cuda.synchronize()
    assert layer.status() == 0
    xb, rw = synth.to_bits(d["x"]), synth.to_f32(d["router_w"])
    route = check_route(oracle_mod, sh, r, xb, rw, router_arith(layer, sh.T))
    del r
    toks = sample_tokens(sh.T, route["row_src"], route["offsets"], n_random=N_RANDOM_FULL,
                         chunk_rows=chunk_rows_of(sh.T, sh.top_k, sh.E, "nvfp4"))
    if name == "decode":
        assert toks == list(range(sh.T))
    q = _oracle_q(oracle_mod, d, experts=np.unique(route["ids"][toks]))
    ref = oracle_rows(oracle_mod.forward_nvfp4, toks, route, xb, rw, *q, sh.G, sh.topk_groups,
                      sh.top_k, sh.scale)
    rel = rel_l2_per_token(out_bits(out)[toks], ref)
    assert rel.max() <= NVFP4_TOL, (rel.max(), toks[int(rel.argmax())], len(toks))
