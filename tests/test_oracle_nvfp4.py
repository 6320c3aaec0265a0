"""Pins for the oracle's NVFP4 pieces: code tables and roundings against the
format definitions and torch's float8_e4m3fn, exact round trips of
representable matrices, error bounds, and the NVFP4 layer against a numpy
composition of the pinned quantiser."""
import os

import numpy as np
import pytest
import torch

from sparse_moe_layer_experts_b300 import synth
from tests import _brute

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _fixture():
    d = {}
    for line in open(os.path.join(GOLDEN, "nvfp4_rounding.txt")):
        line = line.strip()
        if line and not line.startswith("#"):
            k, *v = line.split()
            d[k] = [float(x) for x in v]
    return d


def test_e2m1_table_and_rounding(oracle_mod):
    fx = _fixture()
    table = [oracle_mod.e2m1_value(c) for c in range(16)]
    assert table == fx["e2m1_table"]
    assert all(np.signbit(oracle_mod.e2m1_value(c)) == (c >= 8) for c in range(16))
    got = [oracle_mod.e2m1_value(oracle_mod.e2m1_code(v)) for v in fx["e2m1_round_in"]]
    assert got == fx["e2m1_round_out"]
    assert np.signbit(got[fx["e2m1_round_in"].index(-0.1)])


def test_e4m3_rounding_fixture(oracle_mod):
    fx = _fixture()
    got = [oracle_mod.e4m3_value(oracle_mod.e4m3_code(v)) for v in fx["e4m3_round_in"]]
    assert got == fx["e4m3_round_out"]


def test_e4m3_against_torch_float8(oracle_mod):
    # decoding: every finite non-negative code
    codes = torch.arange(0, 0x7F, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float32).tolist()
    assert [oracle_mod.e4m3_value(c) for c in range(0x7F)] == ref
    # encoding: random values in range, plus every midpoint between codes
    rng = np.random.default_rng(0)
    vals = np.concatenate([
        np.exp(rng.uniform(np.log(2.0 ** -12), np.log(448.0), 3000)),
        (np.array(ref[:-1]) + np.array(ref[1:])) / 2.0]).astype(np.float32)
    want = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).tolist()
    got = [oracle_mod.e4m3_code(float(v)) for v in vals]
    assert got == want


def _representable_matrix(rng, rows, cols, gs):
    """A bf16 matrix whose NVFP4 quantisation is lossless, with global scale gs."""
    e2 = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    sfv = [2.0 ** rng.integers(-6, 8) * (1 + rng.integers(0, 8) / 8) for _ in range(rows * cols // 16)]
    sfv = np.array(sfv).reshape(rows, cols // 16)
    q = e2[rng.integers(0, 8, (rows, cols))] * rng.choice([-1.0, 1.0], (rows, cols))
    q.reshape(rows, cols // 16, 16)[:, :, 0] = 6.0  # the block maximum is 6 * sf
    sfv[0, 0] = 448.0  # the matrix maximum is 6 * 448 * gs
    v = q * np.repeat(sfv, 16, axis=1) * gs
    t = torch.from_numpy(v.astype(np.float32))
    assert torch.equal(t.to(torch.bfloat16).to(torch.float32), t)  # exact in bf16
    return t.to(torch.bfloat16)


def test_quantize_round_trip_is_exact(oracle_mod):
    rng = np.random.default_rng(1)
    mats = [_representable_matrix(rng, 8, 64, gs) for gs in (2.0 ** -9, 2.0 ** -12, 1.0)]
    w = torch.stack(mats)
    codes, sf, gs = oracle_mod.quantize_nvfp4(synth.to_bits(w))
    assert gs.tolist() == [2.0 ** -9, 2.0 ** -12, 1.0]
    back = oracle_mod.dequantize_nvfp4(codes, sf, gs)
    assert np.array_equal(back, w.to(torch.float64).numpy())


def test_quantize_error_bound_and_zero_blocks(oracle_mod):
    g = torch.Generator().manual_seed(2)
    w = (torch.randn(2, 32, 128, generator=g) * 0.02).to(torch.bfloat16)
    w[1, 3, 16:32] = 0.0  # an all-zero block
    codes, sf, gs = oracle_mod.quantize_nvfp4(synth.to_bits(w))
    amax = w.abs().amax(dim=(1, 2)).float().numpy()
    assert np.array_equal(gs, (amax / np.float32(2688.0)).astype(np.float32))
    back = oracle_mod.dequantize_nvfp4(codes, sf, gs)
    v = w.to(torch.float64).numpy()
    e4 = np.array([oracle_mod.e4m3_value(c) for c in range(256)])
    unit = np.repeat(e4[sf], 16, axis=-1) * gs.reshape(-1, 1, 1)
    # nearest E2M1 value: error at most half the widest gap (between 4 and 6)
    # in units of the block scale, plus E4M3 rounding of the scale itself
    assert (np.abs(v - back) <= unit * 1.0 + 1e-12).all()
    assert (codes[1, 3, 16:32] == 0).all() and sf[1, 3, 1] == 0


def test_fake_quant_rows_matches_quantizer_with_unit_scale(oracle_mod):
    g = torch.Generator().manual_seed(3)
    x = torch.randn(4, 64, generator=g).to(torch.bfloat16)
    fq = oracle_mod.fake_quant_rows(x.float().numpy())
    # the same numbers through the matrix quantiser forced to gs = 1: append a
    # row whose maximum is 6 * 448 so that amax / 2688 = 1
    big = torch.cat([x, torch.full((1, 64), 6.0 * 448.0).to(torch.bfloat16)])
    codes, sf, gs = oracle_mod.quantize_nvfp4(synth.to_bits(big[None]))
    assert gs[0] == 1.0
    ref = oracle_mod.dequantize_nvfp4(codes, sf, gs)[0, :4]
    assert np.array_equal(fq.astype(np.float64), ref)


def test_nvfp4_layer_against_numpy_composition(oracle_mod):
    sh = synth.shape("tiny")
    d = synth.make_inputs(sh, seed=4, device="cpu")
    xb = synth.to_bits(d["x"])
    rw = synth.to_f32(d["router_w"])
    q = [oracle_mod.quantize_nvfp4(synth.to_bits(d[k])) for k in ("w_gate", "w_up", "w_down")]
    tokens = list(range(0, sh.T, 5))
    out, ids, w = oracle_mod.forward_nvfp4(xb, rw, *q, sh.G, sh.topk_groups, sh.top_k, sh.scale,
                                           tokens=tokens)
    _, scores = oracle_mod.router_scores(xb, rw)
    wg, wu, wd = (oracle_mod.dequantize_nvfp4(*qq) for qq in q)
    xq = oracle_mod.fake_quant_rows(oracle_mod.bf16_bits_to_f32(xb)).astype(np.float64)
    f = oracle_mod.bf16_bits_to_f32
    for r, t in enumerate(tokens):
        order, wb, _ = _brute.select(scores[t], sh.G, sh.topk_groups, sh.top_k, sh.scale)
        assert ids[r].tolist() == order
        ref = np.zeros(sh.H)
        for e, wk in zip(order, wb):
            gg = wg[e] @ xq[t]
            uu = wu[e] @ xq[t]
            hh = oracle_mod.fake_quant_rows((gg / (1 + np.exp(-gg)) * uu)[None])[0]
            ref += float(wk) * (wd[e] @ hh.astype(np.float64))
        got = f(out[r]).astype(np.float64)
        assert np.linalg.norm(got - ref) / np.linalg.norm(ref) < 1e-2, t
