"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each test ties one oracle function to the pages' rule through an independent
route: a hand-worked example, exhaustive search, a library routine, a closed
form or an invariant.
"""
import math
import os

import numpy as np
import pytest
import torch

from sparse_moe_layer_experts_b300 import synth
from tests import _brute

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_fixture(name):
    d = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            d[key] = vals
    return d


def _bits(a_f32):
    """fp32 numpy -> bf16 bit patterns (values already exact in bf16)."""
    return torch.from_numpy(np.asarray(a_f32, np.float32)).to(torch.bfloat16).view(
        torch.int16).numpy().view(np.uint16)


@pytest.fixture(scope="module")
def tiny():
    sh = synth.shape("tiny")
    d = synth.make_inputs(sh, seed=0, device="cpu")
    return sh, {k: (synth.to_bits(v) if v.dtype == torch.bfloat16 else synth.to_f32(v))
                for k, v in d.items()}


# ------------------------------------------------------------------ routing

def test_hand_routing_example(oracle_mod):
    fx = _read_fixture("routing_hand_example.txt")
    s = np.array([float(v) for v in fx["scores"]], np.float32)[None, :]
    ids, w = oracle_mod.select(s, int(fx["n_groups"][0]), int(fx["topk_groups"][0]),
                               int(fx["top_k"][0]), float(fx["scale"][0]))
    assert ids[0].tolist() == [int(v) for v in fx["ids"]]
    assert w[0].tolist() == [float(v) for v in fx["weights"]]


def test_selection_matches_exhaustive_search(oracle_mod, tiny):
    sh, d = tiny
    _, scores = oracle_mod.router_scores(d["x"], d["router_w"])
    ids, w = oracle_mod.select(scores, sh.G, sh.topk_groups, sh.top_k, sh.scale)
    for t in range(0, sh.T, 4):  # 16 tokens: 70 group subsets x 12870 expert subsets each
        order, wb, _ = _brute.select(scores[t], sh.G, sh.topk_groups, sh.top_k, sh.scale)
        assert ids[t].tolist() == order, t
        assert w[t].tolist() == [float(v) for v in wb], t


@pytest.mark.parametrize("case", ["all_equal", "group_ties", "pair_ties"])
def test_selection_ties_exhaustive(oracle_mod, case):
    rng = np.random.default_rng(7)
    E, G = 32, 8
    if case == "all_equal":
        s = np.full(E, 0.5, np.float32)
    elif case == "group_ties":
        # every group has the same top-2 sum but different members
        s = rng.permutation(np.tile(np.array([0.6, 0.4, 0.1, 0.05], np.float32), G))
        s = s.reshape(G, 4)
        s = np.stack([np.sort(r)[::-1][[0, 1, 2, 3]] for r in s]).reshape(-1)
        s = s.astype(np.float32)
    else:
        # many exactly-equal scores straddling the selection boundary
        s = rng.choice(np.array([0.25, 0.5, 0.75], np.float32), size=E)
    ids, w = oracle_mod.select(s[None, :], G, 4, 8, 2.5)
    order, wb, _ = _brute.select(s, G, 4, 8, 2.5)
    assert ids[0].tolist() == order
    assert w[0].tolist() == [float(v) for v in wb]
    if case == "all_equal":
        assert order == list(range(8))  # groups 0,1 kept by index; lowest experts


def test_selection_invariants_full_width(oracle_mod):
    rng = np.random.default_rng(3)
    T, E, G, TG, K = 512, 256, 8, 4, 8
    logits = rng.normal(0, 1.4, size=(T, E)).astype(np.float32)
    s = (1.0 / (1.0 + np.exp(-logits.astype(np.float64)))).astype(np.float32)
    ids, w = oracle_mod.select(s, G, TG, K, 2.5)
    gsize = E // G
    for t in range(T):
        row = ids[t]
        assert len(set(row.tolist())) == K
        # the kept groups are the best TG by top-2 sum
        gs = np.array([np.sort(s[t, g * gsize:(g + 1) * gsize])[-2:].sum(dtype=np.float32)
                       for g in range(G)])
        kept = sorted(np.lexsort((np.arange(G), -gs))[:TG].tolist())
        assert set((row // gsize).tolist()) <= set(kept)
        # slot order: score descending, id ascending on ties
        key = [(-float(s[t, e]), int(e)) for e in row]
        assert key == sorted(key)
        # every chosen expert beats every unchosen candidate
        cand = [e for g in kept for e in range(g * gsize, (g + 1) * gsize) if e not in row]
        worst = min(row.tolist(), key=lambda e: (s[t, e], -e))
        for e in cand:
            assert (s[t, e], -e) < (s[t, worst], -worst)
        assert abs(float(w[t].astype(np.float64).sum()) - 2.5) <= 2.5 * 8 * 2 ** -23 * 4
        assert (w[t] > 0).all()


def test_single_group_is_plain_topk(oracle_mod):
    rng = np.random.default_rng(11)
    T, E, K = 64, 64, 6
    s = rng.random((T, E)).astype(np.float32)
    s[:, 5] = s[:, 9]  # a tie pair
    ids, _ = oracle_mod.select(s, 1, 1, K, 1.0)
    for t in range(T):
        ref = np.lexsort((np.arange(E), -s[t].astype(np.float64)))[:K]
        assert ids[t].tolist() == ref.tolist()


def test_select_rejects_bad_config(oracle_mod):
    s = np.full((1, 32), 0.5, np.float32)
    with pytest.raises(ValueError):
        oracle_mod.select(s, 5, 2, 4, 2.5)  # 32 % 5 != 0
    with pytest.raises(ValueError):
        oracle_mod.select(s, 8, 2, 9, 2.5)  # 9 > 2 groups * 4
    with pytest.raises(ValueError):
        oracle_mod.select(np.full((1, 32), np.nan, np.float32), 8, 4, 8, 2.5)


def test_router_scores_against_float64_matmul(oracle_mod, tiny):
    sh, d = tiny
    logits, scores = oracle_mod.router_scores(d["x"], d["router_w"])
    x64 = oracle_mod.bf16_bits_to_f32(d["x"]).astype(np.float64)
    w64 = d["router_w"].astype(np.float64)
    ref = x64 @ w64
    # forward error of an H-term FP32 dot product (fused steps): H*u*sum|x*w|
    bound = sh.H * 2 ** -24 * (np.abs(x64) @ np.abs(w64)) * 1.01
    assert (np.abs(logits - ref) <= bound).all()
    sig = 1.0 / (1.0 + np.exp(-logits.astype(np.float64)))
    assert (np.abs(scores - sig) <= 4 * 2 ** -24 * sig).all()


def test_router_sigmoid_exact_points(oracle_mod):
    # x . W = 0 exactly -> sigmoid(0) = 0.5 exactly
    x = _bits(np.array([[1.0, -1.0, 2.0]], np.float32))
    w = np.array([[0.5], [0.5], [0.0]], np.float32)
    logits, scores = oracle_mod.router_scores(x, w)
    assert logits[0, 0] == 0.0 and scores[0, 0] == 0.5


def test_router_is_sequential_fma_chain(oracle_mod):
    # 1 + 2^-24 - 1 in ascending order: the first fma gives 1, the second
    # 1 + 2^-24 rounds to 1 (tie to even), the third gives 0.  A pairwise or
    # reversed sum would keep the 2^-24 term.
    x = _bits(np.array([[1.0, 1.0, 1.0]], np.float32))
    w = np.array([[1.0], [2.0 ** -24], [-1.0]], np.float32)
    logits, _ = oracle_mod.router_scores(x, w)
    assert logits[0, 0] == 0.0
    w2 = np.array([[-1.0], [2.0 ** -24], [1.0]], np.float32)
    logits2, _ = oracle_mod.router_scores(x, w2)
    assert logits2[0, 0] == 2.0 ** -24
    # each step is one fused multiply-add: (1+2^-7)(1+2^-23) - (1+2^-7) keeps
    # the 2^-30 term that a rounded product would drop.
    x3 = _bits(np.array([[1.0078125, 1.0078125]], np.float32))
    w3 = np.array([[-1.0], [1.0 + 2.0 ** -23]], np.float32)
    logits3, _ = oracle_mod.router_scores(x3, w3)
    assert logits3[0, 0] == 2.0 ** -23 + 2.0 ** -30


# ----------------------------------------------------------------- dispatch

def test_dispatch_against_stable_argsort(oracle_mod):
    rng = np.random.default_rng(5)
    T, K, E = 300, 8, 32
    ids = np.stack([rng.choice(E, K, replace=False) for _ in range(T)]).astype(np.int32)
    counts, offsets, row_of, row_src = oracle_mod.dispatch(ids, E)
    assert counts.tolist() == np.bincount(ids.reshape(-1), minlength=E).tolist()
    assert offsets.tolist() == [0] + np.cumsum(counts).tolist()
    order = np.argsort(ids.reshape(-1), kind="stable")  # expert-major, then (t,k) order
    expect_row_of = np.empty(T * K, np.int64)
    expect_row_of[order] = np.arange(T * K)
    assert row_of.reshape(-1).tolist() == expect_row_of.tolist()
    assert row_src.tolist() == (order // K).tolist()


# ------------------------------------------------------------- expert + layer

def test_hand_swiglu_example(oracle_mod):
    fx = _read_fixture("swiglu_hand_example.txt")
    H, I = int(fx["H"][0]), int(fx["I"][0])
    f = lambda k: np.array([float(v) for v in fx[k]], np.float32)
    x = _bits(f("x").reshape(1, H))
    wg = _bits(f("w_gate").reshape(1, I, H))
    wu = _bits(f("w_up").reshape(1, I, H))
    wd = _bits(f("w_down").reshape(1, H, I))
    rw = f("router_w").reshape(H, 1)
    y = oracle_mod.expert_row(x[0], wg[0], wu[0], wd[0])
    assert np.allclose(y, f("y_exact").astype(np.float64), rtol=1e-7, atol=0)
    out, ids, w = oracle_mod.forward(x, rw, wg, wu, wd, 1, 1, 1, 1.0)
    assert ids.tolist() == [[0]] and w.tolist() == [[1.0]]
    assert oracle_mod.bf16_bits_to_f32(out[0]).tolist() == f("out_bf16").tolist()


def _np_swiglu(x, wg, wu, wd):
    g = x @ wg.T
    u = x @ wu.T
    h = g / (1.0 + np.exp(-g)) * u
    return h @ wd.T


def test_single_expert_layer_is_dense_swiglu(oracle_mod):
    # E=1, one group, top-1, scale 1: the layer is one plain SwiGLU MLP.
    g = torch.Generator().manual_seed(21)
    T, H, I = 16, 96, 64
    x = torch.randn(T, H, generator=g).to(torch.bfloat16)
    wg = (torch.randn(1, I, H, generator=g) * 0.1).to(torch.bfloat16)
    wu = (torch.randn(1, I, H, generator=g) * 0.1).to(torch.bfloat16)
    wd = (torch.randn(1, H, I, generator=g) * 0.1).to(torch.bfloat16)
    rw = torch.randn(H, 1, generator=g).numpy()
    xb, gb, ub, db = (synth.to_bits(t) for t in (x, wg, wu, wd))
    out, ids, w = oracle_mod.forward(xb, rw, gb, ub, db, 1, 1, 1, 1.0)
    assert (ids == 0).all() and (w == 1.0).all()
    ref = _np_swiglu(x.double().numpy(), wg[0].double().numpy(), wu[0].double().numpy(),
                     wd[0].double().numpy())
    got = oracle_mod.bf16_bits_to_f32(out).astype(np.float64)
    # bf16 output rounding: half an ulp of 8 significant bits, plus FP32 h
    assert (np.abs(got - ref) <= np.abs(ref) * 2 ** -8 + 1e-6).all()


def test_dense_forward_is_swiglu_mlp(oracle_mod):
    # The dense layer against an independent numpy SwiGLU, and equal to the
    # single-expert layer row for row.
    g = torch.Generator().manual_seed(23)
    T, H, I = 12, 128, 96
    x = torch.randn(T, H, generator=g).to(torch.bfloat16)
    wg = (torch.randn(I, H, generator=g) * 0.1).to(torch.bfloat16)
    wu = (torch.randn(I, H, generator=g) * 0.1).to(torch.bfloat16)
    wd = (torch.randn(H, I, generator=g) * 0.1).to(torch.bfloat16)
    xb, gb, ub, db = (synth.to_bits(t) for t in (x, wg, wu, wd))
    out = oracle_mod.dense_forward(xb, gb, ub, db)
    ref = _np_swiglu(x.double().numpy(), wg.double().numpy(), wu.double().numpy(),
                     wd.double().numpy())
    got = oracle_mod.bf16_bits_to_f32(out).astype(np.float64)
    assert (np.abs(got - ref) <= np.abs(ref) * 2 ** -8 + 1e-6).all()
    moe, _, _ = oracle_mod.forward(xb, np.ones((H, 1), np.float32), gb[None], ub[None], db[None],
                                   1, 1, 1, 1.0)
    assert np.array_equal(moe, out)
    sub = oracle_mod.dense_forward(xb, gb, ub, db, tokens=[3, 0, 11])
    assert np.array_equal(sub, out[[3, 0, 11]])


def test_layer_is_weighted_sum_of_expert_mlps(oracle_mod, tiny):
    # Independent composition: exhaustive-search routing + numpy expert MLPs.
    sh, d = tiny
    _, scores = oracle_mod.router_scores(d["x"], d["router_w"])
    tokens = list(range(0, sh.T, 8))
    out, ids, w = oracle_mod.forward(d["x"], d["router_w"], d["w_gate"], d["w_up"],
                                     d["w_down"], sh.G, sh.topk_groups, sh.top_k, sh.scale,
                                     tokens=tokens)
    f = oracle_mod.bf16_bits_to_f32
    x = f(d["x"]).astype(np.float64)
    wg, wu, wd = (f(d[k]).astype(np.float64) for k in ("w_gate", "w_up", "w_down"))
    for r, t in enumerate(tokens):
        order, wb, _ = _brute.select(scores[t], sh.G, sh.topk_groups, sh.top_k, sh.scale)
        assert ids[r].tolist() == order
        ref = sum(float(wk) * _np_swiglu(x[t:t + 1], wg[e], wu[e], wd[e])[0]
                  for e, wk in zip(order, wb))
        got = f(out[r]).astype(np.float64)
        rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
        assert rel < 4e-3, (t, rel)


def test_routed_scale_is_linear(oracle_mod, tiny):
    # Doubling the routed scale doubles every weight and every output exactly.
    sh, d = tiny
    args = (d["x"], d["router_w"], d["w_gate"], d["w_up"], d["w_down"], sh.G,
            sh.topk_groups, sh.top_k)
    o1, _, w1 = oracle_mod.forward(*args, 2.5, tokens=[0, 1, 2])
    o2, _, w2 = oracle_mod.forward(*args, 5.0, tokens=[0, 1, 2])
    assert (w2 == 2 * w1).all()
    f = oracle_mod.bf16_bits_to_f32
    assert (f(o2) == 2 * f(o1)).all()


def test_expert_params_closed_form():
    # Each expert: gate + up + down = 3 * H * I parameters; the pages give
    # "about 39M" per expert at H=5120, I=2560, 256 experts in each of 49 layers
    # and 98.4% of 501.3B parameters in experts.
    sh = synth.shape("decode")
    per_expert = 3 * sh.H * sh.I
    assert per_expert == 39_321_600
    assert math.isclose(49 * 256 * per_expert / 501.3e9, 0.984, abs_tol=5e-4)
