"""Seeded synthetic inputs for the Beam MoE layer workloads.

This module draws random tensors of the shapes, dtypes and value
distributions of the benchmark workloads.  It holds none of the layer's
arithmetic; both the GPU path and the CPU oracle take their inputs from here.

Recipe (base seed ``seed``; one sub-seed per tensor, in this order):
  x        [T,H]    N(0,1) drawn in FP32, rounded to bf16 (RNE)     sub-seed 0
  router_w [H,E]    N(0,0.02) FP32                                  sub-seed 1
  w_gate   [E,I,H]  N(0,0.02) drawn in FP32, rounded to bf16        sub-seed 2
  w_up     [E,I,H]  same                                            sub-seed 3
  w_down   [E,H,I]  same                                            sub-seed 4
  skewed routing only: a random rank permutation of the experts     sub-seed 5

Skewed routing shifts every token's router logit of expert e by
b_e = 0.5 * ln(p_r(e)), p_r = r^-1.1 / sum_{j<=E} j^-1.1 (a Zipf law over the
expert's rank r).  The layer itself has no bias term, so the shift is carried
by the inputs: hidden channel 0 of every token is set to 1.0 and router row 0
is set to b.  The logit of expert e then contains exactly 1.0 * b_e.

Dense SwiGLU layers (Beam's first three decoder layers) draw
  x        [T,H]    N(0,1) bf16                                     sub-seed 10
  w_gate   [I,H]    N(0,0.02) bf16                                  sub-seed 11
  w_up     [I,H]    same                                            sub-seed 12
  w_down   [H,I]    same                                            sub-seed 13
The pages give no intermediate size for the dense layers; the "dense"
workload takes I = 8 * 2560 = 20480, the FFN width one MoE layer's eight
active experts add up to.

The fused block's RMS-norm gains are 1 + 0.1 N(0,1) in FP32 (norm_pre
sub-seed 20, norm_post sub-seed 21).

Tensors are drawn on ``device``.  CPU and CUDA generators produce different
streams, so a test draws each tensor once and hands the same tensor to both
sides.
"""
from __future__ import annotations

import dataclasses

import torch

CONFIGS = {
    # name: (T, H, I, E, n_groups, topk_groups, top_k, routing)
    "tiny": dict(T=64, H=256, I=128, E=32, G=8, topk_groups=4, top_k=8, routing="random"),
    "decode": dict(T=32, H=5120, I=2560, E=256, G=8, topk_groups=4, top_k=8, routing="random"),
    "prefill": dict(T=4096, H=5120, I=2560, E=256, G=8, topk_groups=4, top_k=8,
                    routing="random"),
    "skewed": dict(T=16384, H=5120, I=2560, E=256, G=8, topk_groups=4, top_k=8,
                   routing="zipf"),
    "nvfp4": dict(T=8192, H=5120, I=2560, E=256, G=8, topk_groups=4, top_k=8,
                  routing="random"),
    # the decode batch with MXFP8 experts
    "mxfp8": dict(T=32, H=5120, I=2560, E=256, G=8, topk_groups=4, top_k=8, routing="random"),
}

DENSE_CONFIGS = {
    "dense": dict(T=4096, H=5120, I=20480),
}

ROUTED_SCALE = 2.5


@dataclasses.dataclass
class LayerShape:
    T: int
    H: int
    I: int
    E: int
    G: int
    topk_groups: int
    top_k: int
    routing: str = "random"
    scale: float = ROUTED_SCALE


def shape(name: str, **overrides) -> LayerShape:
    d = dict(CONFIGS[name])
    d.update(overrides)
    return LayerShape(**d)


def _gen(device, seed: int, sub: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1000 + sub)
    return g


def _normal_bf16(shape_, std, gen, device, chunk_rows=None):
    """N(0, std^2) drawn in FP32 and rounded to bf16, drawn in row chunks."""
    out = torch.empty(shape_, dtype=torch.bfloat16, device=device)
    flat = out.view(shape_[0], -1)
    step = chunk_rows or shape_[0]
    for r0 in range(0, shape_[0], step):
        r1 = min(shape_[0], r0 + step)
        tmp = torch.randn((r1 - r0, flat.shape[1]), generator=gen, device=device,
                          dtype=torch.float32)
        if std != 1.0:
            tmp.mul_(std)
        flat[r0:r1].copy_(tmp)
        del tmp
    return out


def zipf_logit_bias(E: int, seed: int, device="cpu", s: float = 1.1) -> torch.Tensor:
    """Per-expert logit shift 0.5*ln(p_rank) for a Zipf(s) law over random ranks."""
    g = _gen("cpu", seed, 5)
    perm = torch.randperm(E, generator=g)
    ranks = torch.empty(E, dtype=torch.float64)
    ranks[perm] = torch.arange(1, E + 1, dtype=torch.float64)
    z = sum(j ** -s for j in range(1, E + 1))
    p = ranks.pow(-s) / z
    return (0.5 * p.log()).to(torch.float32).to(device)


def make_inputs(sh: LayerShape, seed: int = 0, device="cpu", weights=True):
    """Return a dict of the layer's inputs drawn per the module recipe."""
    dev = torch.device(device)
    chunk = 8 if sh.E * sh.I * sh.H > (1 << 26) else None
    x = _normal_bf16((sh.T, sh.H), 1.0, _gen(dev, seed, 0), dev)
    rw = torch.randn((sh.H, sh.E), generator=_gen(dev, seed, 1), device=dev,
                     dtype=torch.float32).mul_(0.02)
    if sh.routing == "zipf":
        x[:, 0] = 1.0
        rw[0, :] = zipf_logit_bias(sh.E, seed, dev)
    d = dict(x=x, router_w=rw)
    if weights:
        d["w_gate"] = _normal_bf16((sh.E, sh.I, sh.H), 0.02, _gen(dev, seed, 2), dev, chunk)
        d["w_up"] = _normal_bf16((sh.E, sh.I, sh.H), 0.02, _gen(dev, seed, 3), dev, chunk)
        d["w_down"] = _normal_bf16((sh.E, sh.H, sh.I), 0.02, _gen(dev, seed, 4), dev, chunk)
    return d


def make_dense_inputs(T: int, H: int, I: int, seed: int = 0, device="cpu"):
    """x [T,H], w_gate/w_up [I,H], w_down [H,I] per the module recipe."""
    dev = torch.device(device)
    chunk = 1024 if I * H > (1 << 26) else None
    return dict(
        x=_normal_bf16((T, H), 1.0, _gen(dev, seed, 10), dev),
        w_gate=_normal_bf16((I, H), 0.02, _gen(dev, seed, 11), dev, chunk),
        w_up=_normal_bf16((I, H), 0.02, _gen(dev, seed, 12), dev, chunk),
        w_down=_normal_bf16((H, I), 0.02, _gen(dev, seed, 13), dev, chunk),
    )


def make_block_gains(H: int, seed: int = 0, device="cpu"):
    """(norm_pre, norm_post) gains [H] fp32 per the module recipe."""
    dev = torch.device(device)
    return tuple(torch.randn(H, generator=_gen(dev, seed, sub), device=dev,
                             dtype=torch.float32).mul_(0.1).add_(1.0) for sub in (20, 21))


def to_bits(t: torch.Tensor):
    """bf16 tensor -> numpy uint16 bit patterns (host copy)."""
    assert t.dtype == torch.bfloat16
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view("uint16")


def to_f32(t: torch.Tensor):
    assert t.dtype == torch.float32
    return t.detach().contiguous().cpu().numpy()


def expected_distinct_experts(T: int, E: int, K: int) -> float:
    """E[#experts with >=1 token] for uniform random routing (context only)."""
    return E * (1.0 - (1.0 - K / E) ** T)

