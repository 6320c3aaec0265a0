"""Host-side checks of the benchmark's roofline arithmetic and of the token
sampler the full-size parity tests use (no GPU needed)."""
import importlib.util
import os

import numpy as np

from sparse_moe_layer_experts_b300 import synth
from tests._gpu_util import chunk_rows_of, sample_tokens

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_algorithmic_bytes_and_flops_closed_forms():
    b = _bench()
    sh = synth.shape("decode")
    a = b.workload_algorithmic(sh, n_active=163)
    H, I, E, T, K = sh.H, sh.I, sh.E, sh.T, sh.top_k
    per_expert_gu = 2 * I * H * 2            # gate + up, bf16
    assert per_expert_gu == 52_428_800
    assert a["gateup_gemm"]["bytes"] == 163 * per_expert_gu + T * K * H * 2 + T * K * I * 2
    assert a["down_gemm"]["bytes"] == 163 * H * I * 2 + T * K * I * 2 + T * K * H * 2
    assert a["gateup_gemm"]["flops"] == 2 * T * K * H * 2 * I
    # layer: weights of the active experts + router + x and out
    assert a["layer"]["bytes"] == 163 * 3 * H * I * 2 + H * E * 4 + 2 * T * H * 2
    assert a["layer"]["flops"] == 2 * T * H * E + 6 * T * K * H * I
    # NVFP4 at prefill size: 0.5625 B per weight and per activation, h written quantised
    sh4 = synth.shape("nvfp4")
    a4 = b.workload_algorithmic(sh4, n_active=256, fmt="nvfp4")
    R = sh4.T * K
    assert a4["gateup_gemm"]["bytes"] == int(int(256 * 2 * I * H * 0.5625) + R * H * 0.5625 +
                                             R * I * 0.5625)
    # per-token expert work: 8 experts x 3 GEMMs x 2 H I (the survey's closed form)
    assert a4["layer"]["flops"] - 2 * sh4.T * H * E == sh4.T * 629_145_600


def test_tensor_peak_sources():
    b = _bench()
    peaks = {"bf16_tflops": 1800.0, "hbm_gbs": 6400.0}
    v, src = b.tensor_peak("bf16", peaks, None)
    assert v == 1800.0 and "bf16" in src
    v, src = b.tensor_peak("nvfp4", peaks, {"nvfp4_tflops": 5000.0, "shape": "s", "reps": 1})
    assert v == 5000.0 and "cuBLASLt" in src
    v, src = b.tensor_peak("nvfp4", peaks, {"nvfp4_tflops": None})
    assert v == 1800.0 * 13.5 / 2.25 and "nominal" in src
    v, _ = b.tensor_peak("mxfp8", peaks, None)
    assert v == 1800.0 * 4.5 / 2.25


def test_sampler_covers_every_segment_edge_and_hot_chunks():
    rng = np.random.default_rng(0)
    T, K, E = 3000, 8, 64
    ids = np.stack([rng.choice(E, K, replace=False) for _ in range(T)]).astype(np.int32)
    # skew: half the tokens route to expert 5 in slot 0 (if not routed there already)
    for t in range(T // 2):
        if 5 not in ids[t]:
            ids[t, 0] = 5

    def dispatch(ids, E):
        rows = sorted((int(e), t) for t in range(ids.shape[0]) for e in ids[t])
        counts = np.bincount(ids.reshape(-1), minlength=E)
        return np.array([t for _, t in rows]), np.concatenate([[0], np.cumsum(counts)]), counts

    row_src, offsets, counts = dispatch(ids, E)
    toks = set(sample_tokens(T, row_src, offsets, n_random=16, chunk_rows=64))
    assert {0, T - 1} <= toks
    for e in range(E):
        if counts[e]:
            assert row_src[offsets[e]] in toks and row_src[offsets[e + 1] - 1] in toks
    hot = int(np.argmax(counts))
    n = counts[hot]
    nc = -(-n // 64)
    for c in range(nc):
        assert row_src[offsets[hot] + c * n // nc] in toks
        assert row_src[offsets[hot] + (c + 1) * n // nc - 1] in toks
    # every token of a small batch when n_random >= T
    rs32, off32, _ = dispatch(ids[:32], E)
    assert sample_tokens(32, rs32, off32, n_random=32) == list(range(32))
    assert chunk_rows_of(32, 8, 256) == 32 and chunk_rows_of(4096, 8, 256) == 256
    assert chunk_rows_of(8192, 8, 256, "nvfp4") == 128
