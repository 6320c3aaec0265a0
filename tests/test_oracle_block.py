"""Pins for the oracle's fused MoE block: pre-norm -> MoE -> post-norm ->
constant-scale residual ("Reflection Beam 1.0", section "Residual stream":
the input embedding is step 1, step k adds the sublayer output with weight
1/sqrt(k) and keeps the stream with weight sqrt((k-1)/k); sublayers are
normalised before and after, in FP32).  Each test checks the oracle against
something other than itself: numpy norms, an invariant, a closed form, or
the separately pinned MoE layer oracle."""
import numpy as np
import torch

from sparse_moe_layer_experts_b300 import synth


def _f32(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def _inputs(seed=5, T=24, H=256, I=128, E=32):
    sh = synth.shape("tiny", T=T, H=H, I=I, E=E)
    d = synth.make_inputs(sh, seed=seed)
    g = torch.Generator().manual_seed(seed + 100)
    gp = (1.0 + 0.1 * torch.randn(H, generator=g)).numpy().astype(np.float32)
    gq = (1.0 + 0.1 * torch.randn(H, generator=g)).numpy().astype(np.float32)
    return sh, d, gp, gq


def test_prenorm_matches_numpy_rmsnorm(oracle_mod):
    sh, d, gp, _ = _inputs()
    s = synth.to_bits(d["x"])
    x = _f32(oracle_mod.rmsnorm_bf16(s, gp, 1e-6)).astype(np.float64)
    sv = _f32(s).astype(np.float64)
    ref = sv / np.sqrt((sv ** 2).mean(axis=1, keepdims=True) + 1e-6) * gp
    # FP32 steps then one bf16 rounding: within one bf16 ulp of the exact value
    assert (np.abs(x - ref) <= np.abs(ref) * 2 ** -7 + 1e-30).all()


def test_prenorm_is_scale_invariant(oracle_mod):
    # with eps = 0, rmsnorm(2 s) == rmsnorm(s) exactly (powers of two are exact)
    sh, d, gp, _ = _inputs()
    s = synth.to_bits(d["x"])
    s2 = synth.to_bits(d["x"] * 2)
    assert np.array_equal(oracle_mod.rmsnorm_bf16(s, gp, 0.0), oracle_mod.rmsnorm_bf16(s2, gp, 0.0))


def test_block_step_one_is_the_normalised_sublayer(oracle_mod):
    # k = 1: a = 0, b = 1, so s' = bf16(rmsnorm(o) * 1); with eps = 0 its RMS
    # is 1 up to the bf16 rounding of each element
    sh, d, gp, _ = _inputs()
    ones = np.ones(sh.H, np.float32)
    out = oracle_mod.block_forward(synth.to_bits(d["x"]), 1, gp, ones, 0.0, synth.to_f32(d["router_w"]),
                                   synth.to_bits(d["w_gate"]), synth.to_bits(d["w_up"]),
                                   synth.to_bits(d["w_down"]), sh.G, sh.topk_groups, sh.top_k, sh.scale)
    rms = np.sqrt((_f32(out).astype(np.float64) ** 2).mean(axis=1))
    assert np.all(np.abs(rms - 1.0) <= 2 ** -8)


def test_block_composes_pinned_parts(oracle_mod):
    # numpy composition: pinned pre-norm -> pinned MoE layer oracle -> numpy
    # post-norm and residual weights
    sh, d, gp, gq = _inputs()
    k, eps = 9, 1e-6
    s = synth.to_bits(d["x"])
    args = (synth.to_f32(d["router_w"]), synth.to_bits(d["w_gate"]), synth.to_bits(d["w_up"]),
            synth.to_bits(d["w_down"]), sh.G, sh.topk_groups, sh.top_k, sh.scale)
    out = oracle_mod.block_forward(s, k, gp, gq, eps, *args)
    x = oracle_mod.rmsnorm_bf16(s, gp, eps)
    y, _, _ = oracle_mod.forward(x, *args)
    yv = _f32(y).astype(np.float64)
    z = yv / np.sqrt((yv ** 2).mean(axis=1, keepdims=True) + eps) * gq
    ref = np.sqrt((k - 1) / k) * _f32(s).astype(np.float64) + z / np.sqrt(k)
    got = _f32(out).astype(np.float64)
    rel = np.linalg.norm(got - ref, axis=1) / np.linalg.norm(ref, axis=1)
    assert rel.max() <= 2e-3, rel.max()


def test_block_large_step_keeps_the_stream(oracle_mod):
    # k -> large: a -> 1, b -> 0; the stream passes through up to b*|z|
    sh, d, gp, gq = _inputs()
    k = 1 << 20
    s = synth.to_bits(d["x"])
    out = oracle_mod.block_forward(s, k, gp, gq, 1e-6, synth.to_f32(d["router_w"]),
                                   synth.to_bits(d["w_gate"]), synth.to_bits(d["w_up"]),
                                   synth.to_bits(d["w_down"]), sh.G, sh.topk_groups, sh.top_k, sh.scale,
                                   tokens=[0, 5, 23])
    # per row: ||s' - s|| <= bf16 rounding (2^-8 ||s||) + b ||z||, and
    # ||z|| <= sqrt(H) max|gamma_post| because rmsnorm(o) has unit RMS
    sv = _f32(s[[0, 5, 23]]).astype(np.float64)
    got = _f32(out).astype(np.float64)
    dev = np.linalg.norm(got - sv, axis=1)
    bound = 2 ** -8 * np.linalg.norm(sv, axis=1) + 2 ** -10 * np.sqrt(sh.H) * np.abs(gq).max()
    assert np.all(dev <= bound) and np.all(dev > 0)


def test_block_tail_composes_to_the_block(oracle_mod):
    # pre-norm -> layer (its FP32 combine) -> tail == the block oracle, bit
    # for bit; and the combine rounds to the layer's bf16 output
    sh = synth.shape("tiny", T=40)
    d = synth.make_inputs(sh, seed=31, device="cpu")
    h = {k: (synth.to_bits(v) if v.dtype == torch.bfloat16 else synth.to_f32(v))
         for k, v in d.items()}
    gp, gq = (g.numpy() for g in synth.make_block_gains(sh.H, seed=31))
    for step, toks in ((9, None), (1, [3, 0, 39]), (400, [7])):
        blk = oracle_mod.block_forward(h["x"], step, gp, gq, 1e-6, h["router_w"], h["w_gate"],
                                       h["w_up"], h["w_down"], sh.G, sh.topk_groups, sh.top_k,
                                       sh.scale, tokens=toks)
        xn = oracle_mod.rmsnorm_bf16(h["x"], gp, 1e-6)
        out, _, _, o = oracle_mod.forward(xn, h["router_w"], h["w_gate"], h["w_up"], h["w_down"],
                                          sh.G, sh.topk_groups, sh.top_k, sh.scale, tokens=toks,
                                          combine=True)
        assert np.array_equal(out, torch.from_numpy(o).to(torch.bfloat16).view(torch.int16)
                              .numpy().view(np.uint16))
        tail = oracle_mod.block_tail(h["x"], step, gq, 1e-6, o, tokens=toks)
        assert np.array_equal(tail, blk), step


def test_quantised_layers_expose_their_combine(oracle_mod):
    sh = synth.shape("tiny", T=16)
    d = synth.make_inputs(sh, seed=32, device="cpu")
    xb, rw = synth.to_bits(d["x"]), synth.to_f32(d["router_w"])
    for quant, fwd in ((oracle_mod.quantize_nvfp4, oracle_mod.forward_nvfp4),
                       (oracle_mod.quantize_mxfp8, oracle_mod.forward_mxfp8)):
        q = [quant(synth.to_bits(d[k])) for k in ("w_gate", "w_up", "w_down")]
        out, ids, w = fwd(xb, rw, *q, sh.G, sh.topk_groups, sh.top_k, sh.scale)
        out2, ids2, w2, o = fwd(xb, rw, *q, sh.G, sh.topk_groups, sh.top_k, sh.scale,
                                combine=True)
        assert np.array_equal(out, out2) and np.array_equal(ids, ids2)
        assert np.array_equal(out, torch.from_numpy(o).to(torch.bfloat16).view(torch.int16)
                              .numpy().view(np.uint16))
