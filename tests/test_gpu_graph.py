"""The layer forward is a fixed sequence of kernel launches on one stream with
no allocation and no host synchronisation, so it can be captured once in a
CUDA graph and replayed.  Replays on new inputs (copied into the captured
input buffer) must give the bytes an eager call gives, for the bf16, NVFP4
and MXFP8 layers at decode and prefill sizes."""
import pytest
import torch

from sparse_moe_layer_experts_b300 import synth
from sparse_moe_layer_experts_b300.layer import BeamMoE, quantize_mxfp8, quantize_nvfp4

pytestmark = pytest.mark.gpu

SHAPES = {
    "decode": synth.LayerShape(T=16, H=512, I=384, E=64, G=8, topk_groups=4, top_k=8),
    "prefill": synth.LayerShape(T=700, H=512, I=512, E=64, G=8, topk_groups=4, top_k=8),
}


def _layer(fmt, sh, d):
    kw = dict(n_groups=sh.G, topk_groups=sh.topk_groups, top_k=sh.top_k, routed_scale=sh.scale)
    if fmt == "bf16":
        return BeamMoE(d["router_w"], d["w_gate"], d["w_up"], d["w_down"], **kw)
    qf, mk = (quantize_nvfp4, BeamMoE.nvfp4) if fmt == "nvfp4" else (quantize_mxfp8, BeamMoE.mxfp8)
    q = [qf(d[k]) for k in ("w_gate", "w_up", "w_down")]
    return mk(d["router_w"], *q, **kw)


@pytest.mark.parametrize("fmt", ["bf16", "nvfp4", "mxfp8"])
@pytest.mark.parametrize("size", list(SHAPES))
def test_graph_replay_matches_eager(fmt, size):
    sh = SHAPES[size]
    d = synth.make_inputs(sh, seed=21, device="cuda")
    layer = _layer(fmt, sh, d)
    x = d["x"].clone()
    out = torch.empty_like(x)
    layer.forward(x, out)  # warm-up: workspace, kernel attributes
    torch.cuda.synchronize()

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        layer.forward(x, out)

    gen = torch.Generator(device="cuda").manual_seed(22)
    for _ in range(2):
        x_new = torch.randn(x.shape, generator=gen, device="cuda").to(torch.bfloat16)
        x.copy_(x_new)
        g.replay()
        torch.cuda.synchronize()
        assert layer.status() == 0
        eager = layer.forward(x_new.clone())
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
