"""Pins for the oracle's MXFP8 pieces (E4M3 values, one power-of-two scale
per 32 elements; the OCP microscaling rule as the reading of the pages'
unspecified FP8 checkpoint): the shared-exponent rule against numpy's
log2, codes against torch's float8_e4m3fn encoder, exact round trips,
saturation, and the MXFP8 layer against a numpy composition."""
import numpy as np
import torch

from sparse_moe_layer_experts_b300 import synth
from tests import _brute


def test_shared_exponent_rule(oracle_mod):
    rng = np.random.default_rng(1)
    vals = np.concatenate([np.exp(rng.uniform(np.log(1e-30), np.log(1e30), 2000)),
                           2.0 ** np.arange(-126, 127), [1.9, 448.0, 511.0, 3e-45]]).astype(np.float32)
    want = np.clip(np.floor(np.log2(vals.astype(np.float64))) - 8, -127, 127).astype(int)
    got = np.array([oracle_mod.mx_shared_exp(float(v)) for v in vals])
    assert np.array_equal(got, want)
    assert oracle_mod.mx_shared_exp(0.0) == -127


def _torch_mx(w):
    """Independent MXFP8 quantisation of a float32 [rows, cols] matrix with
    torch's E4M3 encoder (round to nearest even, saturating)."""
    rows, cols = w.shape
    blk = w.reshape(rows, cols // 32, 32).astype(np.float64)
    amax = np.abs(blk).max(axis=2)
    with np.errstate(divide="ignore"):
        e = np.where(amax > 0, np.clip(np.floor(np.log2(amax)) - 8, -127, 127), -127).astype(int)
    scaled = blk * 2.0 ** (-e[..., None])
    t = torch.from_numpy(np.clip(scaled, -448, 448).astype(np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy().reshape(rows, cols), (e + 127).astype(np.uint8)


def test_quantizer_against_torch_e4m3(oracle_mod):
    g = torch.Generator().manual_seed(3)
    w = (torch.randn(3, 64, 256, generator=g) * torch.exp(torch.randn(3, 64, 1, generator=g) * 3)
         ).to(torch.bfloat16)
    w[0, 0, :32] = 0.0  # an all-zero block
    codes, sf = oracle_mod.quantize_mxfp8(synth.to_bits(w))
    for m in range(3):
        wc, ws = _torch_mx(w[m].float().numpy())
        # zeros: the oracle keeps the sign of -0.0 like the encoder
        assert np.array_equal(codes[m], wc)
        assert np.array_equal(sf[m], ws)
    assert sf[0, 0, 0] == 0 and (codes[0, 0, :32] == 0).all()


def test_round_trip_of_representable_values_is_exact(oracle_mod):
    rng = np.random.default_rng(2)
    e4 = torch.arange(0, 0x7F, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    rows, cols = 8, 128
    vals = rng.choice(e4[8:], size=(rows, cols)) * rng.choice([-1.0, 1.0], size=(rows, cols))
    exps = rng.integers(-20, 20, size=(rows, cols // 32))
    for r in range(rows):
        for b in range(cols // 32):
            vals[r, b * 32] = 256.0  # block max 256 -> shared exponent exactly exps
    w = (vals * 2.0 ** np.repeat(exps, 32, axis=1)).astype(np.float32)
    wb = torch.from_numpy(w).to(torch.bfloat16)
    assert torch.equal(wb.float(), torch.from_numpy(w))  # representable in bf16
    codes, sf = oracle_mod.quantize_mxfp8(synth.to_bits(wb)[None])
    back = oracle_mod.dequantize_mxfp8(codes[0], sf[0])
    assert np.array_equal(back, w.astype(np.float64))


def test_saturation_between_448_and_512(oracle_mod):
    # amax = 1.9: exponent -8, 1.9 * 256 = 486.4 saturates to 448
    v = np.zeros((1, 1, 32), np.float32)
    v[0, 0, 0] = 1.9
    v[0, 0, 1] = -1.9
    codes, sf = oracle_mod.quantize_mxfp8(synth.to_bits(torch.from_numpy(v).to(torch.bfloat16)))
    assert sf[0, 0, 0] == 127 - 8
    assert codes[0, 0, 0] == 0x7E and codes[0, 0, 1] == 0xFE


def test_mxfp8_layer_against_numpy_composition(oracle_mod):
    sh = synth.shape("tiny")
    d = synth.make_inputs(sh, seed=6, device="cpu")
    xb = synth.to_bits(d["x"])
    rw = synth.to_f32(d["router_w"])
    q = [oracle_mod.quantize_mxfp8(synth.to_bits(d[k])) for k in ("w_gate", "w_up", "w_down")]
    tokens = list(range(0, sh.T, 5))
    out, ids, w = oracle_mod.forward_mxfp8(xb, rw, *q, sh.G, sh.topk_groups, sh.top_k, sh.scale,
                                           tokens=tokens)
    _, scores = oracle_mod.router_scores(xb, rw)
    wg, wu, wd = (oracle_mod.dequantize_mxfp8(*qq) for qq in q)
    f = oracle_mod.bf16_bits_to_f32
    xq = oracle_mod.fake_quant_mxfp8_rows(f(xb)).astype(np.float64)
    for r, t in enumerate(tokens):
        order, wb, _ = _brute.select(scores[t], sh.G, sh.topk_groups, sh.top_k, sh.scale)
        assert ids[r].tolist() == order
        ref = np.zeros(sh.H)
        for e, wk in zip(order, wb):
            gg = wg[e] @ xq[t]
            uu = wu[e] @ xq[t]
            hh = oracle_mod.fake_quant_mxfp8_rows((gg / (1 + np.exp(-gg)) * uu)[None])[0]
            ref += float(wk) * (wd[e] @ hh.astype(np.float64))
        got = f(out[r]).astype(np.float64)
        assert np.linalg.norm(got - ref) / np.linalg.norm(ref) < 1e-2, t
