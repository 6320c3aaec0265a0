"""GPU parity: the CUDA library against the CPU oracle on the same seeded
inputs.  Routing: scores bit-exact where the FMA-chain router runs, within the
FP32 accumulation bound where the tensor-core router runs; ids, weights,
counts, offsets and permuted rows bit-exact given the same FP32 scores.  The
layer output within a per-token relative L2 of 1e-2."""
import numpy as np
import pytest
import torch

from sparse_moe_layer_experts_b300 import synth
from sparse_moe_layer_experts_b300.layer import BeamMoE
from tests._gpu_util import (N_RANDOM_FULL, REL_L2_TOL, check_route, chunk_rows_of, host_inputs,
                             oracle_rows, out_bits, rel_l2_per_token, router_arith,
                             sample_tokens)

pytestmark = pytest.mark.gpu

# small shapes that still span several tiles, chunks and ragged tails
SMALL = {
    "tiny": synth.shape("tiny"),
    "tiny_T1": synth.shape("tiny", T=1),
    "tiny_T7": synth.shape("tiny", T=7),
    "tiny_T200": synth.shape("tiny", T=200),
    "tiny_T1000": synth.shape("tiny", T=1000),
    "medium": synth.LayerShape(T=3001, H=512, I=384, E=64, G=8, topk_groups=4, top_k=8),
    "wide_groups": synth.LayerShape(T=777, H=256, I=256, E=96, G=4, topk_groups=2, top_k=6,
                                    scale=1.5),
    # decode-size router with E % 8 == 4 (a half-empty last expert group) and a
    # ragged last token group
    "e36_T50": synth.LayerShape(T=50, H=256, I=128, E=36, G=4, topk_groups=2, top_k=4),
    # the tensor-core router with a ragged last expert tile and token tile
    "e36_T300": synth.LayerShape(T=300, H=256, I=128, E=36, G=4, topk_groups=2, top_k=4),
}

# routing only, at the Beam expert count: the tensor-core router's 128- and
# 64-expert tiles (chosen by batch size) with a short hidden size
ROUTE_ONLY = {
    "e256_T16384": synth.LayerShape(T=16384, H=256, I=128, E=256, G=8, topk_groups=4, top_k=8),
    "e256_T8192": synth.LayerShape(T=8192, H=512, I=128, E=256, G=8, topk_groups=4, top_k=8),
}


def _layer(sh, d, **kw):
    return BeamMoE(d["router_w"], d["w_gate"], d["w_up"], d["w_down"], n_groups=sh.G,
                   topk_groups=sh.topk_groups, top_k=sh.top_k, routed_scale=sh.scale, **kw)


def _check_route(oracle_mod, sh, layer, d, hx):
    r = layer.route(d["x"])
    torch.cuda.synchronize()
    assert layer.status() == 0
    return check_route(oracle_mod, sh, r, hx["x"], hx["router_w"], router_arith(layer, sh.T))


@pytest.mark.parametrize("name", list(SMALL) + list(ROUTE_ONLY))
def test_route_small(oracle_mod, name):
    sh = SMALL.get(name) or ROUTE_ONLY[name]
    d = synth.make_inputs(sh, seed=0, device="cuda")
    hx = host_inputs(d)
    _check_route(oracle_mod, sh, _layer(sh, d), d, hx)


@pytest.mark.parametrize("name", list(SMALL))
def test_forward_small_all_tokens(oracle_mod, name):
    sh = SMALL[name]
    d = synth.make_inputs(sh, seed=1, device="cuda")
    hx = host_inputs(d)
    layer = _layer(sh, d)
    route = _check_route(oracle_mod, sh, layer, d, hx)
    out = layer.forward(d["x"])
    torch.cuda.synchronize()
    assert layer.status() == 0
    ref = oracle_rows(oracle_mod.forward, list(range(sh.T)), route, hx["x"], hx["router_w"],
                      hx["w_gate"], hx["w_up"], hx["w_down"], sh.G, sh.topk_groups, sh.top_k,
                      sh.scale)
    rel = rel_l2_per_token(out_bits(out), ref)
    assert rel.max() <= REL_L2_TOL, (rel.max(), int(rel.argmax()))


def test_forward_deterministic_and_hostio(oracle_mod):
    sh = SMALL["medium"]
    d = synth.make_inputs(sh, seed=2, device="cuda")
    layer = _layer(sh, d)
    a = layer.forward(d["x"]).clone()
    b = layer.forward(d["x"]).clone()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    # a second stream, and host buffers through the host-I/O entry point
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        c = layer.forward(d["x"], stream=s)
    s.synchronize()
    assert torch.equal(a.view(torch.int16), c.view(torch.int16))
    xh = d["x"].cpu().pin_memory()
    oh = torch.empty_like(xh).pin_memory()
    layer.forward_host(xh, oh)
    assert torch.equal(a.cpu().view(torch.int16), oh.view(torch.int16))


def test_timeout_reports_status_and_gpu_recovers(oracle_mod):
    sh = SMALL["tiny"]
    d = synth.make_inputs(sh, seed=3, device="cuda")
    bad = _layer(sh, d, wait_timeout_ns=50_000_000, debug_flags=1)
    bad.forward(d["x"])
    torch.cuda.synchronize()
    assert bad.status() == -5  # BEAM_MOE_ERR_TIMEOUT
    good = _layer(sh, d)
    out = good.forward(d["x"])
    torch.cuda.synchronize()
    assert good.status() == 0
    hx = host_inputs(d)
    ref, _, _ = oracle_mod.forward(hx["x"], hx["router_w"], hx["w_gate"], hx["w_up"],
                                   hx["w_down"], sh.G, sh.topk_groups, sh.top_k, sh.scale)
    assert rel_l2_per_token(out_bits(out), ref).max() <= REL_L2_TOL


# ------------------------------------------------------------- full sizes

@pytest.fixture(scope="module")
def beam_weights():
    sh = synth.shape("decode")
    w = synth.make_inputs(sh, seed=0, device="cuda", weights=True)
    yield {k: w[k] for k in ("w_gate", "w_up", "w_down")}
    del w
    torch.cuda.empty_cache()


@pytest.mark.slow
@pytest.mark.parametrize("name", ["decode", "prefill", "skewed", "nvfp4"])
def test_full_size_route_and_sampled_forward(oracle_mod, beam_weights, name):
    """Full-size workloads in the configuration the benchmark times: every
    token's routing checked; layer outputs of every token of the decode
    batch, and at the larger sizes of token 0 and T-1, the first and last row
    of every non-empty expert segment, the first and last row of every token
    chunk of the most loaded expert, and 256 seeded random tokens."""
    sh = synth.shape(name)
    d = synth.make_inputs(sh, seed=0, device="cuda", weights=False)
    d.update(beam_weights)
    layer = _layer(sh, d)
    hx_route = dict(x=synth.to_bits(d["x"]), router_w=synth.to_f32(d["router_w"]))
    route = _check_route(oracle_mod, sh, layer, d, hx_route)
    ids, counts = route["ids"], route["counts"]
    out = layer.forward(d["x"])
    torch.cuda.synchronize()
    assert layer.status() == 0
    toks = sample_tokens(sh.T, route["row_src"], route["offsets"], n_random=N_RANDOM_FULL,
                         chunk_rows=chunk_rows_of(sh.T, sh.top_k, sh.E))
    if name == "decode":
        assert toks == list(range(sh.T))
    hx = host_inputs(d, experts=np.unique(ids[toks]))
    ref = oracle_rows(oracle_mod.forward, toks, route, hx["x"], hx["router_w"], hx["w_gate"],
                      hx["w_up"], hx["w_down"], sh.G, sh.topk_groups, sh.top_k, sh.scale)
    rel = rel_l2_per_token(out_bits(out)[toks], ref)
    assert rel.max() <= REL_L2_TOL, (rel.max(), toks[int(rel.argmax())], len(toks))
    if name == "skewed":
        # the synthetic Zipf bias makes one expert hot
        assert counts.max() > 4 * counts.mean()
