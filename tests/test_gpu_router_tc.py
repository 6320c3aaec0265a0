"""The tensor-core router (batches of 256 tokens and more).

It splits the FP32 router weight into three bf16 parts and sums the exact
products on the tensor cores in FP32.  Two checks pin it beyond the bound
tests of the parity files:

 - Exact split: with one-hot token rows (a single nonzero x[t,h], a power of
   two), every logit is one exact product, whatever order the tensor cores
   add in, so scores must equal the oracle's bit for bit.  A lost or
   mis-scaled part of the split (hi, mid or lo) changes the low bits of
   every such logit.
 - The selection given the scores: ids and weights bit-exact against the
   oracle's selection on the same FP32 scores, with real group structure.
"""
import numpy as np
import pytest
import torch

from sparse_moe_layer_experts_b300 import binding as B
from sparse_moe_layer_experts_b300 import synth
from sparse_moe_layer_experts_b300.layer import BeamMoE
from tests._gpu_util import check_tc_scores

pytestmark = pytest.mark.gpu


def _router_only_layer(sh, router_w):
    w = torch.zeros(1, dtype=torch.bfloat16, device="cuda")
    layer = BeamMoE.__new__(BeamMoE)
    layer._setup(router_w, w, w, w, sh.E, sh.I, sh.H, sh.G, sh.topk_groups, sh.top_k, sh.scale,
                 0, 0)
    return layer


def _one_hot_inputs(T, H, E, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    # FP32 weights with full 24-bit significands over a wide range of
    # magnitudes (2^-40 .. 2^8), some exact zeros and negatives
    mag = torch.exp2(torch.randint(-40, 9, (H, E), generator=g).float())
    w = torch.randn(H, E, generator=g) * mag
    w[torch.rand(H, E, generator=g) < 0.02] = 0.0
    x = torch.zeros(T, H)
    t = torch.arange(T)
    pow2 = torch.tensor([1.0, -1.0, 0.5, -2.0, 4.0, -0.25])
    x[t, t % H] = pow2[(t // H) % len(pow2)]
    return x.to(torch.bfloat16), w


@pytest.mark.parametrize("T,H,E", [(16384, 512, 256), (8192, 256, 256), (300, 256, 36),
                                   (1000, 640, 64)])
def test_one_hot_rows_give_exact_scores(oracle_mod, T, H, E):
    G = max(4, E // 32)  # at most 32 experts per group
    sh = synth.LayerShape(T=T, H=H, I=128, E=E, G=G, topk_groups=2, top_k=4)
    x, w = _one_hot_inputs(T, H, E, seed=T + H + E)
    layer = _router_only_layer(sh, w.cuda().contiguous())
    assert B.beam_moe_router_arith(T, layer.cfg) == B.BEAM_MOE_ROUTER_TENSOR
    r = layer.route(x.cuda().contiguous())
    torch.cuda.synchronize()
    assert layer.status() == 0
    g = r["scores"].cpu().numpy()
    _, s_o = oracle_mod.router_scores(synth.to_bits(x), w.numpy())
    n_diff = int((g.view(np.uint32) != s_o.view(np.uint32)).sum())
    assert n_diff == 0, f"{n_diff} of {g.size} scores differ"


def test_random_rows_within_bound_and_selection_exact(oracle_mod):
    # Beam sizes, prefill batch: every score within the FP32 accumulation
    # bound of the fp64 reference; the selection exact given those scores
    sh = synth.shape("prefill")
    d = synth.make_inputs(sh, seed=3, device="cuda", weights=False)
    layer = _router_only_layer(sh, d["router_w"])
    r = layer.route(d["x"])
    torch.cuda.synchronize()
    assert layer.status() == 0
    g = r["scores"].cpu().numpy()
    err_max, err_rms = check_tc_scores(g, synth.to_bits(d["x"]), synth.to_f32(d["router_w"]))
    print(f"tensor-core router: max |s - s_exact| {err_max:.3e}, rms {err_rms:.3e}")
    ids, w = oracle_mod.select(g, sh.G, sh.topk_groups, sh.top_k, sh.scale)
    assert np.array_equal(r["ids"].cpu().numpy(), ids)
    assert np.array_equal(r["w"].cpu().numpy().view(np.uint32), w.view(np.uint32))


def test_deterministic_across_calls_and_streams():
    sh = synth.shape("nvfp4")
    d = synth.make_inputs(sh, seed=4, device="cuda", weights=False)
    layer = _router_only_layer(sh, d["router_w"])
    a = layer.route(d["x"])["scores"].clone()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        b = layer.route(d["x"], stream=s)["scores"].clone()
    s.synchronize()
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def _route_both(layer, x):
    a = layer.route(x, want_scores=True)    # every score evaluated and written
    b = layer.route(x, want_scores=False)   # only the scores the selection needs
    torch.cuda.synchronize()
    assert layer.status() == 0
    for k in ("ids", "w", "counts", "offsets", "row_of"):
        ua, ub = a[k].cpu().numpy(), b[k].cpu().numpy()
        assert np.array_equal(ua.view(np.uint32), ub.view(np.uint32)), k
    return a


@pytest.mark.parametrize("case", ["prefill", "one_hot", "zero_x", "saturated", "e36", "g4_24"])
def test_lazy_sigmoid_selection_equals_full(oracle_mod, case):
    """The selection without written scores evaluates the sigmoid only for
    each group's two largest logits and the top-K candidates, falling back
    to every candidate on a plateau of the FP32 sigmoid or tied logits.  It
    must select exactly what the full evaluation selects, and that must be
    the oracle's selection on the same scores."""
    if case == "prefill":
        sh = synth.shape("prefill")
        d = synth.make_inputs(sh, seed=9, device="cuda", weights=False)
        x, w = d["x"], d["router_w"]
    elif case == "one_hot":
        sh = synth.LayerShape(T=4096, H=512, I=128, E=256, G=8, topk_groups=4, top_k=8)
        xc, wc = _one_hot_inputs(sh.T, sh.H, sh.E, seed=5)
        x, w = xc.cuda().contiguous(), wc.cuda().contiguous()
    elif case == "zero_x":
        # every logit 0: every score 0.5, all ties resolved by index
        sh = synth.LayerShape(T=512, H=256, I=128, E=256, G=8, topk_groups=4, top_k=8)
        x = torch.zeros(sh.T, sh.H, dtype=torch.bfloat16, device="cuda")
        w = torch.randn(sh.H, sh.E, device="cuda") * 0.02
    elif case == "saturated":
        # logits of +-20..60: most scores round to exactly 1.0 or to tiny values
        sh = synth.LayerShape(T=1024, H=256, I=128, E=256, G=8, topk_groups=4, top_k=8)
        g = torch.Generator(device="cuda").manual_seed(3)
        x = torch.randn(sh.T, sh.H, generator=g, device="cuda").to(torch.bfloat16)
        w = torch.randn(sh.H, sh.E, generator=g, device="cuda") * 2.5
    elif case == "e36":
        sh = synth.LayerShape(T=700, H=256, I=128, E=36, G=4, topk_groups=2, top_k=4)
        d = synth.make_inputs(sh, seed=2, device="cuda", weights=False)
        x, w = d["x"], d["router_w"]
    else:  # groups of 24 experts: the group stage's non-shuffle branch
        sh = synth.LayerShape(T=900, H=256, I=128, E=96, G=4, topk_groups=2, top_k=6, scale=1.5)
        d = synth.make_inputs(sh, seed=4, device="cuda", weights=False)
        x, w = d["x"], d["router_w"]
    layer = _router_only_layer(sh, w)
    assert B.beam_moe_router_arith(sh.T, layer.cfg) == B.BEAM_MOE_ROUTER_TENSOR
    a = _route_both(layer, x)
    g = a["scores"].cpu().numpy()
    ids, wts = oracle_mod.select(g, sh.G, sh.topk_groups, sh.top_k, sh.scale)
    assert np.array_equal(a["ids"].cpu().numpy(), ids)
    assert np.array_equal(a["w"].cpu().numpy().view(np.uint32), wts.view(np.uint32))


@pytest.mark.parametrize("T", [255, 256, 300, 1000, 2304])
def test_beam_router_around_the_threshold_and_eight_way_split(oracle_mod, T):
    """Beam sizes (H=5120, E=256) at small batches: T=255 takes the FMA-chain
    router (scores bit-exact); from T=256 the tensor cores with the hidden
    dimension split 8 ways (one or a few 256-token tiles leave most SMs
    free), checked against the FP32 accumulation bound, the selection
    bit-exact given the scores, and the near-tie count."""
    from tests._gpu_util import check_route
    sh = synth.shape("decode", T=T)
    d = synth.make_inputs(sh, seed=T, device="cuda", weights=False)
    layer = _router_only_layer(sh, d["router_w"])
    arith = B.beam_moe_router_arith(T, layer.cfg)
    assert arith == (B.BEAM_MOE_ROUTER_TENSOR if T >= 256 else B.BEAM_MOE_ROUTER_FMA_CHAIN)
    r = layer.route(d["x"])
    torch.cuda.synchronize()
    assert layer.status() == 0
    check_route(oracle_mod, sh, r, synth.to_bits(d["x"]), synth.to_f32(d["router_w"]), arith)
    # the lazy selection (no scores written) agrees
    _route_both(layer, d["x"])
