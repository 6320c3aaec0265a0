"""Dense SwiGLU layer (Beam's first three decoder layers) on the GPU against
the oracle: every token at small shapes (several weight tiles and token
chunks, ragged tails, the decode-size path), sampled tokens at the benchmark
size."""
import numpy as np
import pytest
import torch

from sparse_moe_layer_experts_b300 import synth
from sparse_moe_layer_experts_b300.layer import DenseSwiGLU

from tests._gpu_util import REL_L2_TOL, out_bits, rel_l2_per_token

pytestmark = pytest.mark.gpu

SMALL = [
    dict(T=200, H=256, I=384),     # prefill path: 1 full + 1 ragged 256-row chunk
    dict(T=700, H=384, I=256),     # 3 chunks, ragged tail, 3 down-GEMM tiles
    dict(T=16, H=256, I=128),      # decode-size path
    dict(T=1, H=128, I=128),       # one token
]


def _oracle(oracle_mod, d, tokens=None):
    return oracle_mod.dense_forward(synth.to_bits(d["x"]), synth.to_bits(d["w_gate"]),
                                    synth.to_bits(d["w_up"]), synth.to_bits(d["w_down"]),
                                    tokens=tokens)


@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "T{T}_H{H}_I{I}".format(**s))
def test_dense_all_tokens(oracle_mod, shape):
    d = synth.make_dense_inputs(seed=3, device="cuda", **shape)
    layer = DenseSwiGLU(d["w_gate"], d["w_up"], d["w_down"])
    out = layer.forward(d["x"])
    torch.cuda.synchronize()
    assert layer.status() == 0
    rel = rel_l2_per_token(out_bits(out), _oracle(oracle_mod, d))
    assert rel.max() <= REL_L2_TOL, (rel.max(), int(rel.argmax()))


def test_dense_deterministic_and_zero_tokens():
    d = synth.make_dense_inputs(T=300, H=256, I=256, seed=4, device="cuda")
    layer = DenseSwiGLU(d["w_gate"], d["w_up"], d["w_down"])
    a = layer.forward(d["x"]).clone()
    b = layer.forward(d["x"]).clone()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    empty = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    assert layer.forward(empty).shape == (0, 256)


@pytest.mark.slow
def test_dense_full_size_sampled(oracle_mod):
    """The benchmark workload (T=4096, H=5120, I=20480) on sampled tokens:
    first, last, chunk edges and seeded random rows."""
    sh = synth.DENSE_CONFIGS["dense"]
    d = synth.make_dense_inputs(seed=0, device="cuda", **sh)
    layer = DenseSwiGLU(d["w_gate"], d["w_up"], d["w_down"])
    out = layer.forward(d["x"])
    torch.cuda.synchronize()
    assert layer.status() == 0
    T = sh["T"]
    rng = np.random.default_rng(0)
    toks = sorted({0, T - 1, 255, 256, 2047, 2048} | set(int(v) for v in rng.choice(T, 8, replace=False)))
    rel = rel_l2_per_token(out_bits(out)[toks], _oracle(oracle_mod, d, toks))
    assert rel.max() <= REL_L2_TOL, (rel.max(), toks[int(rel.argmax())])
