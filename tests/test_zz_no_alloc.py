"""The allocation-free entry point (beam_moe_forward_noalloc).

Callers that cannot allocate device memory (their allocator belongs to a host
application or a fixed arena) use this call: it takes inputs and outputs only
and keeps its scratch in a fixed array inside the library.  These checks call
it through the C ABI and compare it with beam_moe_forward, the entry point
that takes a caller-allocated workspace, on two calls in a row with different
inputs (the second call must not be disturbed by what the first left in the
shared scratch).

This file is collected last on purpose, so that a run stopping at the first
failure has run every other test first.
"""
import pytest
import torch

from sparse_moe_layer_experts_b300 import binding as B
from sparse_moe_layer_experts_b300 import synth
from sparse_moe_layer_experts_b300.layer import BeamMoE
from tests._gpu_util import REL_L2_TOL, out_bits, rel_l2_per_token

pytestmark = pytest.mark.gpu


def _noalloc(layer, x):
    out = torch.empty_like(x)
    rc = B.beam_moe_forward_noalloc(x.data_ptr(), layer.router_w.data_ptr(),
                                    layer.w_gate.data_ptr(), layer.w_up.data_ptr(),
                                    layer.w_down.data_ptr(), x.shape[0], layer.cfg,
                                    out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == B.BEAM_MOE_OK, B.beam_moe_status_string(rc)
    return out


def _compare(layer, xs):
    got = [_noalloc(layer, x) for x in xs]          # two calls in a row
    torch.cuda.synchronize()
    for x, g in zip(xs, got):
        ref = layer.forward(x)                      # caller-allocated workspace
        torch.cuda.synchronize()
        assert layer.status() == 0
        # Both entry points run the same deterministic kernels on the same
        # inputs, so the outputs must agree byte for byte; anything the first
        # call left in the shared scratch must not change the second.
        n_diff = int((g.view(torch.int16) != ref.view(torch.int16)).sum())
        assert n_diff == 0, f"{n_diff} output values differ from beam_moe_forward"
        # the tolerance of the parity tests holds a fortiori
        assert rel_l2_per_token(out_bits(g), out_bits(ref)).max() <= REL_L2_TOL


@pytest.mark.parametrize("name,T2", [("tiny", 37), ("decode", 32)])
def test_noalloc_matches_workspace_entry_point(name, T2):
    sh = synth.shape(name)
    d = synth.make_inputs(sh, seed=5, device="cuda")
    layer = BeamMoE(d["router_w"], d["w_gate"], d["w_up"], d["w_down"], n_groups=sh.G,
                    topk_groups=sh.topk_groups, top_k=sh.top_k, routed_scale=sh.scale)
    x2 = synth.make_inputs(synth.shape(name, T=T2), seed=6, device="cuda", weights=False)["x"]
    _compare(layer, [d["x"], x2])
    del d, layer
    torch.cuda.empty_cache()


def test_noalloc_rejects_batches_beyond_its_scratch():
    c = B.beam_moe_cfg()
    B.beam_moe_cfg_init_beam(c)
    before = B.beam_moe_launch_count()
    # 128 Beam tokens need ~25 MiB of scratch, above the 24 MiB array
    rc = B.beam_moe_forward_noalloc(16, 16, 16, 16, 16, 128, c, 16, None)
    assert rc == B.BEAM_MOE_ERR_WORKSPACE
    c.top_k = 0
    assert B.beam_moe_forward_noalloc(16, 16, 16, 16, 16, 8, c, 16, None) == \
        B.BEAM_MOE_ERR_INVALID_ARG
    assert B.beam_moe_launch_count() == before
