#!/usr/bin/env python
"""Beam MoE layer forward throughput on B300 (tokens/s), with roofline.

One step = one whole layer forward (router, selection, dispatch, gate/up and
down grouped GEMMs, combine) over one batch of T synthetic tokens whose
activations are already resident in HBM.  The expert weights (20 GB bf16)
are larger than L2, so no L2 flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config all|decode|...]
  python bench.py --impl reference ...   # the CPU oracle, timed on host cores

The default (--config all) times the decode batch (the headline line) and,
in the same process with the same resident expert weights, the prefill,
skewed-routing and NVFP4 workloads, each reported under the line's
"configs" key with its own clocks, roofline, end-to-end leg and CPU sample.

Multi-GPU (torchrun): every rank runs an independent replica on its own batch
(the layer is per-token independent; no collective on the data path).
Prints one JSON line on rank 0.
"""
from __future__ import annotations

import argparse
import hashlib
import datetime
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "Beam MoE-layer tokens/s at 1 B300; % of HBM (decode) / tensor (prefill) roofline"
UNIT = "tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
# fused-block runs: the first MoE sublayer of the decoder is step 9 of the
# residual stream (embedding 1, then attention and MLP of layers 0-2 and
# the attention of layer 3)
BLOCK_STEP = 9
BLOCK_EPS = 1e-6
# ratio of nominal dense fp4 to bf16 tensor rates
NVFP4_OVER_BF16 = 13.5 / 2.25
# ratio of nominal dense fp8 to bf16 tensor rates
FP8_OVER_BF16 = 4.5 / 2.25


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="all",
                    choices=["all", "tiny", "decode", "prefill", "skewed", "nvfp4", "mxfp8",
                             "dense"],
                    help="'all' (default): decode (the headline line) plus prefill, skewed "
                         "and NVFP4 under the line's 'configs' key, in one process")
    ap.add_argument("--cpu-tokens", type=int, default=16,
                    help="tokens of the batch the CPU oracle baseline computes")
    ap.add_argument("--override", default="",
                    help="shape overrides for profiling runs, e.g. T=512,E=32 (not a bench line)")
    ap.add_argument("--route-only", action="store_true",
                    help="profiling mode: time only the routing kernels (no expert weights "
                         "are allocated); prints a diagnostic line, not a bench line")
    ap.add_argument("--block", action="store_true",
                    help="time the fused block (pre-norm, MoE, post-norm, residual at step 9) "
                         "instead of the bare layer")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-library-peaks", action="store_true",
                    help="skip timing cuBLASLt's FP4/FP8 GEMMs (their peaks then come from the "
                         "bf16 peak times the nominal ratio)")
    return ap.parse_args()


def parse_override(text):
    out = {}
    for item in filter(None, text.split(",")):
        k, v = item.split("=")
        out[k.strip()] = int(v)
    return out


# ------------------------------------------------------------- distributed

def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() and args.impl == "ours" else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, world: int, device=None) -> float:
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------- helpers

class ClockSampler:
    """nvidia-smi clock / throttle-reason samples during the timed region.

    The sampler starts before the caller's timed region and waits (bounded)
    for its first sample; mark_start()/mark_stop() bracket the region, and
    only samples whose nvidia-smi timestamp falls inside it are summarised
    (the nearest later sample when the region is shorter than the interval)."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    INTERVAL_MS = 20

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index
        self.lines = []
        self.t0 = self.t1 = None

    def _reader(self):
        for line in self.proc.stdout:
            if line.strip():
                self.lines.append(line)

    def __enter__(self):
        import threading
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.INTERVAL_MS)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True, bufsize=1)
        except (OSError, ValueError):
            self.proc = None
            return self
        self.thread = threading.Thread(target=self._reader, daemon=True)
        self.thread.start()
        t_end = time.time() + 5.0
        while not self.lines and time.time() < t_end and self.proc.poll() is None:
            time.sleep(0.01)
        return self

    def mark_start(self):
        self.t0 = datetime.datetime.now()

    def mark_stop(self):
        self.t1 = datetime.datetime.now()

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(2 * self.INTERVAL_MS / 1000.0)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.proc.wait()
            self.thread.join(timeout=5)
        return False

    def summary(self):
        rows = []
        for line in list(self.lines):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f")
                rows.append((ts, float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sel = rows
        if self.t0 is not None and self.t1 is not None:
            slack = datetime.timedelta(milliseconds=self.INTERVAL_MS)
            sel = [r for r in rows if self.t0 - slack <= r[0] <= self.t1 + slack]
            if not sel:
                later = [r for r in rows if r[0] >= self.t0]
                sel = later[:1] or rows[-1:]
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = set()
        for r in sel:
            for n, v in zip(names, r[3]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(r[1] for r in sel), "sm_max_mhz": sel[-1][2],
                "reasons": sorted(reasons), "samples": len(sel)}


KERNEL_SOURCES = {
    "router_scores": ("router.cu", "router_tc.cu", "router_math.cuh", "common.cuh"),
    "select": ("router.cu", "router_math.cuh", "common.cuh"),
    "hist": ("dispatch.cu", "common.cuh"),
    "scan": ("dispatch.cu", "common.cuh"),
    "permute": ("dispatch.cu", "common.cuh", "nvfp4.cuh"),
    "combine": ("dispatch.cu", "common.cuh"),
    "gateup_gemm": ("grouped_gemm.cu", "gemm_common.cuh", "common.cuh"),
    "down_gemm": ("grouped_gemm.cu", "grouped_gemm_pair.cu", "gemm_common.cuh", "common.cuh"),
}
FP4_GEMM_SOURCES = ("grouped_gemm_fp4.cu", "grouped_gemm_tm.cu", "blockscaled.cuh",
                    "gemm_common.cuh", "common.cuh", "nvfp4.cuh")


def weight_format(config: str) -> str:
    """The expert format a benchmark config runs: bf16, nvfp4 or mxfp8."""
    return config if config in ("nvfp4", "mxfp8") else "bf16"


def kernel_source_sha(kernel: str, nvfp4: bool = False) -> str:
    """Hash of the source files a kernel is built from."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "sparse_moe_layer_experts_b300", "csrc")
    files = FP4_GEMM_SOURCES if (nvfp4 and kernel.endswith("_gemm")) else KERNEL_SOURCES[kernel]
    for name in files:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary
    (profiles/dram_traffic.json), if it was taken on the kernel's current
    sources; else None."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(workload, {}).get(kernel)
    if not e or e.get("source_sha") != kernel_source_sha(kernel, workload in ("nvfp4", "mxfp8")):
        return None
    return e.get("bytes_per_launch")


def token_major(sh, fmt: str) -> bool:
    """NVFP4 / MXFP8 layers at prefill size (more than 16 rows per expert on
    average) run the token-major GEMMs, whose gate/up writes h quantised."""
    return fmt != "bf16" and sh.T * sh.top_k > 16 * sh.E


def workload_algorithmic(sh, n_active: int, fmt: str = "bf16"):
    """Algorithmic bytes / FLOPs per launch of each kernel (compulsory traffic
    of the kernel's own inputs and outputs; expert weights of active experts
    only).  NVFP4 weights and activations: 0.5 B per code + 1/16 B of block
    scale.  At decode size an NVFP4 / MXFP8 h leaves gate/up in FP32 for the
    quantize_h pass; at prefill size gate/up writes it quantised."""
    T, H, I, E, K = sh.T, sh.H, sh.I, sh.E, sh.top_k
    R = T * K
    # bytes per element: NVFP4 0.5 + 1/16 of scale, MXFP8 1 + 1/32
    wb = {"bf16": 2, "nvfp4": 0.5625, "mxfp8": 1.03125}[fmt]
    ab = wb                             # activation operand bytes per element
    # h as written by gate/up
    hb = 2 if fmt == "bf16" else (wb if token_major(sh, fmt) else 4)
    w_gu = int(n_active * 2 * I * H * wb)
    w_d = int(n_active * H * I * wb)
    return {
        "router_scores": dict(bytes=T * H * 2 + H * E * 4 + T * E * 4, flops=2 * T * H * E),
        "select": dict(bytes=T * E * 4 + R * 8, flops=0),
        "hist": dict(bytes=R * 8 + ((T + 255) // 256) * E * 4, flops=0),
        "scan": dict(bytes=((T + 255) // 256) * E * 8, flops=0),
        "permute": dict(bytes=int(T * H * 2 + R * H * ab), flops=0),
        "gateup_gemm": dict(bytes=int(w_gu + R * H * ab + R * I * hb), flops=2 * R * H * 2 * I),
        "down_gemm": dict(bytes=int(w_d + R * I * ab + R * H * 2), flops=2 * R * I * H),
        "combine": dict(bytes=R * H * 2 + T * H * 2 + R * 8, flops=2 * R * H),
        "quantize_h": dict(bytes=int(R * I * (4 + 0.5625)), flops=0),
        "prenorm": dict(bytes=2 * T * H * 2 + H * 4, flops=0),
        "layer": dict(bytes=w_gu + w_d + H * E * 4 + 2 * T * H * 2,
                      flops=2 * T * H * E + 6 * R * H * I),
    }


# ------------------------------------------------------------------ oracle

def host_sample(sh, d, toks):
    """Host copies for the oracle: x, router and the weights of the experts
    the sampled tokens route to (the rest stay zero pages)."""
    import numpy as np
    from oracle import oracle
    from sparse_moe_layer_experts_b300 import synth
    xh = synth.to_bits(d["x"])
    rw = synth.to_f32(d["router_w"])
    _, s = oracle.router_scores(xh[toks], rw)
    ids, _ = oracle.select(s, sh.G, sh.topk_groups, sh.top_k, sh.scale)
    host = dict(x=xh, router_w=rw, experts=sorted(set(ids.reshape(-1).tolist())))
    for k in ("w_gate", "w_up", "w_down"):
        a = np.zeros(tuple(d[k].shape), np.uint16)
        for e in sorted(set(ids.reshape(-1).tolist())):
            a[e] = synth.to_bits(d[k][e])
        host[k] = a
    return host


def oracle_quantize_sample(host, fmt):
    """The oracle's quantised experts of the sample (weights are quantised
    ahead of the layer, on both arms, so this stays outside the timing)."""
    from oracle import oracle
    if fmt == "bf16":
        return None
    q = []
    for k in ("w_gate", "w_up", "w_down"):
        w = host[k]
        blk = 32 if fmt == "mxfp8" else 16
        codes = np.zeros(w.shape, np.uint8)
        sf = np.zeros(w.shape[:-1] + (w.shape[-1] // blk,), np.uint8)
        gs = np.ones(w.shape[0], np.float32)
        for e in host["experts"]:
            if fmt == "mxfp8":
                c1, s1 = oracle.quantize_mxfp8(w[e:e + 1])
            else:
                c1, s1, g1 = oracle.quantize_nvfp4(w[e:e + 1])
                gs[e] = g1[0]
            codes[e], sf[e] = c1[0], s1[0]
        q.append((codes, sf) if fmt == "mxfp8" else (codes, sf, gs))
    return q


def oracle_step(sh, host, toks, fmt="bf16", q=None):
    """One timed oracle pass over the sampled tokens (q: the quantised
    experts for the NVFP4 and MXFP8 formats)."""
    from oracle import oracle
    t0 = time.perf_counter()
    if fmt == "mxfp8":
        oracle.forward_mxfp8(host["x"], host["router_w"], *q, sh.G, sh.topk_groups, sh.top_k,
                             sh.scale, tokens=toks)
    elif fmt == "nvfp4":
        oracle.forward_nvfp4(host["x"], host["router_w"], *q, sh.G, sh.topk_groups, sh.top_k,
                             sh.scale, tokens=toks)
    else:
        oracle.forward(host["x"], host["router_w"], host["w_gate"], host["w_up"],
                       host["w_down"], sh.G, sh.topk_groups, sh.top_k, sh.scale, tokens=toks)
    return time.perf_counter() - t0


def cpu_oracle_run(sh, d, n_tokens, seed=0, fmt="bf16"):
    """Time the CPU oracle on `n_tokens` seeded tokens of the batch."""
    import numpy as np
    from oracle import oracle
    rng = np.random.default_rng(seed)
    toks = sorted(rng.choice(sh.T, size=min(n_tokens, sh.T), replace=False).tolist())
    host = host_sample(sh, d, toks)
    dt = oracle_step(sh, host, toks, fmt, oracle_quantize_sample(host, fmt))
    return len(toks) / dt, min(oracle.num_threads(), len(toks)), len(toks), dt


# -------------------------------------------------------------------- arms

def run_reference(args, world, rank):
    """The CPU oracle as the reference arm (rank 0 only): each step computes
    a fixed seeded sample of the batch's tokens on the host cores."""
    if rank != 0:
        return
    import numpy as np
    import torch
    from oracle import oracle
    from sparse_moe_layer_experts_b300 import synth
    if args.config == "dense":
        run_reference_dense(args)
        return
    name = DEFAULT_SET[0] if args.config == "all" else args.config
    sh = synth.shape(name)
    # the inputs are drawn exactly as the GPU arm draws them
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    d = synth.make_inputs(sh, seed=0, device=dev, weights=True)
    ntok = min(args.cpu_tokens, sh.T)
    toks = sorted(np.random.default_rng(0).choice(sh.T, size=ntok, replace=False).tolist())
    host = host_sample(sh, d, toks)
    del d
    fmt = weight_format(name)
    q = oracle_quantize_sample(host, fmt)
    times = [oracle_step(sh, host, toks, fmt, q) for _ in range(args.warmup + args.steps)]
    total = sum(times[args.warmup:])
    value = ntok * args.steps / total
    cores = min(oracle.num_threads(), ntok)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 0,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32/f64", "data": "synthetic",
        "config": {"workload": f"{name}: T={sh.T} tokens, hidden {sh.H}, intermediate {sh.I}, "
                               f"{sh.E} experts in {sh.G} groups, top-{sh.topk_groups} groups, "
                               f"top-{sh.top_k}, {fmt} experts",
                   "sample": f"{ntok} seeded tokens of the batch per step"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{ntok} seeded tokens per step, {args.steps} steps"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_reference_dense(args):
    """Reference arm of the dense workload: the oracle's dense SwiGLU on a
    seeded sample of the batch's tokens per step."""
    import numpy as np
    import torch
    from oracle import oracle
    from sparse_moe_layer_experts_b300 import synth
    sh = dict(synth.DENSE_CONFIGS["dense"])
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    d = synth.make_dense_inputs(sh["T"], sh["H"], sh["I"], seed=0, device=dev)
    xb, gb, ub, db = (synth.to_bits(d[k]) for k in ("x", "w_gate", "w_up", "w_down"))
    del d
    ntok = min(args.cpu_tokens, sh["T"])
    toks = sorted(np.random.default_rng(0).choice(sh["T"], size=ntok, replace=False).tolist())
    times = []
    for _ in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        oracle.dense_forward(xb, gb, ub, db, tokens=toks)
        times.append(time.perf_counter() - t0)
    total = sum(times[args.warmup:])
    value = ntok * args.steps / total
    print(json.dumps({
        "impl": "reference",
        "metric": "Beam dense SwiGLU layer tokens/s at 1 B300 (first three decoder layers)",
        "value": value, "unit": UNIT, "n_gpus": 0, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32/f64", "data": "synthetic",
        "config": {"workload": f"dense: T={sh['T']} tokens, hidden {sh['H']}, "
                               f"intermediate {sh['I']}",
                   "sample": f"{ntok} seeded tokens of the batch per step"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": min(oracle.num_threads(), ntok),
                         "kind": "oracle", "sample": f"{ntok} seeded tokens per step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


# Workloads a default run measures, in this order; the first is the headline
# (the decode batch, whose step streams the active experts' weights).
DEFAULT_SET = ("decode", "prefill", "skewed", "nvfp4")
# the skewed workload's target: the hottest expert takes about 8x the mean load
SKEW_TARGET = 8.0


def make_layer(name, sh, weights, qcache, dev, rank):
    """Resident layer of one workload (its own router and batch; the expert
    weights are shared across the Beam-size workloads and quantised once)."""
    from sparse_moe_layer_experts_b300 import synth
    from sparse_moe_layer_experts_b300.layer import BeamMoE, quantize_mxfp8, quantize_nvfp4
    fmt = weight_format(name)
    d = synth.make_inputs(sh, seed=0, device=dev, weights=False)
    if rank > 0:  # each replica routes its own batch
        d["x"] = synth.make_inputs(sh, seed=rank, device=dev, weights=False)["x"]
    d.update(weights)
    kw = dict(n_groups=sh.G, topk_groups=sh.topk_groups, top_k=sh.top_k, routed_scale=sh.scale)
    if fmt == "mxfp8":
        if "mxfp8" not in qcache:
            qcache["mxfp8"] = [quantize_mxfp8(weights[k]) for k in ("w_gate", "w_up", "w_down")]
        layer = BeamMoE.mxfp8(d["router_w"], *qcache["mxfp8"], **kw)
    elif fmt == "nvfp4":
        if "nvfp4" not in qcache:
            qcache["nvfp4"] = [quantize_nvfp4(weights[k]) for k in ("w_gate", "w_up", "w_down")]
        layer = BeamMoE.nvfp4(d["router_w"], *qcache["nvfp4"], **kw)
    else:
        layer = BeamMoE(d["router_w"], weights["w_gate"], weights["w_up"], weights["w_down"], **kw)
    return layer, d


def tensor_peak(fmt, peaks, lib_peaks):
    """(dense tensor peak in TFLOP/s for the path's MMA type, its source).
    bf16: the measured cuBLAS rate.  NVFP4 / MXFP8: the cuBLASLt
    block-scaled GEMM measured in this run when that ran, else the bf16 rate
    times the nominal dense ratio (13.5/2.25 for FP4, 4.5/2.25 for FP8)."""
    if fmt == "bf16":
        return peaks["bf16_tflops"], "measured bf16 cuBLAS GEMM (MEASURED_PEAKS.json)"
    key = f"{fmt}_tflops"
    if lib_peaks and lib_peaks.get(key):
        return lib_peaks[key], (f"measured in this run: cuBLASLt {fmt} block-scaled GEMM "
                                f"{lib_peaks['shape']} via torch._scaled_mm, best of "
                                f"{lib_peaks['reps']}")
    ratio = NVFP4_OVER_BF16 if fmt == "nvfp4" else FP8_OVER_BF16
    return peaks["bf16_tflops"] * ratio, ("bf16 measured (MEASURED_PEAKS.json) x nominal dense "
                                          + ("13.5/2.25" if fmt == "nvfp4" else "4.5/2.25"))


def measure_library_peaks(dev, reps=20, warm_s=0.5):
    """Dense FP4 and FP8 tensor peaks of this GPU as the vendor library
    reaches them: cuBLASLt's block-scaled GEMMs (NVFP4: E2M1 with an E4M3
    scale per 16; MXFP8: E4M3 with a UE8M0 scale per 32) on 8192^3 through
    torch._scaled_mm, best of `reps` CUDA-event timings after `warm_s`
    seconds of back-to-back warm-up calls.  Returns None entries for formats
    the installed torch cannot run."""
    import torch
    M = N = K = 8192
    out = {"shape": f"{M}x{N}x{K}", "reps": reps, "nvfp4_tflops": None, "mxfp8_tflops": None}

    def best_ms(fn):
        t_end = time.time() + warm_s
        while time.time() < t_end:
            for _ in range(5):
                fn()
            torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        best = float("inf")
        for _ in range(reps):
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            best = min(best, e0.elapsed_time(e1))
        return best

    flops = 2.0 * M * N * K
    try:
        g = torch.Generator(device=dev).manual_seed(0)
        a = torch.randint(0, 256, (M, K // 2), dtype=torch.uint8, device=dev, generator=g)
        b = torch.randint(0, 256, (N, K // 2), dtype=torch.uint8, device=dev, generator=g)
        one = 0x38  # 1.0 in E4M3
        sa = torch.full((M, K // 16), one, dtype=torch.uint8, device=dev)
        sb = torch.full((N, K // 16), one, dtype=torch.uint8, device=dev)
        a4, b4 = a.view(torch.float4_e2m1fn_x2), b.view(torch.float4_e2m1fn_x2)
        sa4, sb4 = sa.view(torch.float8_e4m3fn), sb.view(torch.float8_e4m3fn)
        fn = lambda: torch._scaled_mm(a4, b4.t(), sa4, sb4, out_dtype=torch.bfloat16)
        out["nvfp4_tflops"] = flops / best_ms(fn) / 1e9
        del a, b, sa, sb
    except Exception as ex:  # noqa: BLE001 - reported, not fatal
        out["nvfp4_error"] = repr(ex)[:200]
    try:
        g = torch.Generator(device=dev).manual_seed(1)
        a = torch.randn(M, K, device=dev, generator=g).to(torch.float8_e4m3fn)
        b = torch.randn(N, K, device=dev, generator=g).to(torch.float8_e4m3fn)
        sa = torch.full((M, K // 32), 127, dtype=torch.uint8, device=dev).view(torch.float8_e8m0fnu)
        sb = torch.full((N, K // 32), 127, dtype=torch.uint8, device=dev).view(torch.float8_e8m0fnu)
        fn = lambda: torch._scaled_mm(a, b.t(), sa, sb, out_dtype=torch.bfloat16)
        out["mxfp8_tflops"] = flops / best_ms(fn) / 1e9
        del a, b, sa, sb
    except Exception as ex:  # noqa: BLE001
        out["mxfp8_error"] = repr(ex)[:200]
    torch.cuda.empty_cache()
    return out


def measure(name, sh, layer, d, args, world, rank, local, dev, peaks, lib_peaks):
    """Time one workload: warm-up, K timed steps (device events on the launch
    stream, per-kernel events through the library's hook, clocks sampled in
    the region), the host-I/O end-to-end leg, and the roofline figures."""
    import torch
    from sparse_moe_layer_experts_b300 import binding as B
    from sparse_moe_layer_experts_b300 import synth
    fmt = weight_format(name)
    x = d["x"]
    out = torch.empty_like(x)
    if args.block:
        gp, gq = synth.make_block_gains(sh.H, seed=0, device=dev)
        step_fn = lambda: layer.block_forward(x, BLOCK_STEP, gp, gq, BLOCK_EPS, out=out)
    else:
        step_fn = lambda: layer.forward(x, out)
    r = layer.route(x, want_scores=False)
    counts = r["counts"].cpu().numpy()
    del r
    n_active = int((counts > 0).sum())
    stream = torch.cuda.current_stream()

    for _ in range(args.warmup):
        step_fn()
    torch.cuda.synchronize()
    if layer.status() != 0:
        raise SystemExit(f"{name}: device status word reports an error during warm-up")

    # per-kernel events: one (start, stop) pair per stage per step
    nst = len(B.KERNEL_STAGES)
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(nst)] for _ in range(args.steps)]
    for pair in ev:  # torch creates the CUDA event on its first record
        for e0, e1 in pair:
            e0.record(stream)
            e1.record(stream)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = B.beam_moe_launch_count()
    torch.cuda.synchronize()
    barrier(world)
    with ClockSampler(local) as clk:
        clk.mark_start()
        start.record(stream)
        for i in range(args.steps):
            B.check(B.beam_moe_set_kernel_events([e[0].cuda_event for e in ev[i]],
                                                 [e[1].cuda_event for e in ev[i]]), "events")
            step_fn()
        stop.record(stream)
        torch.cuda.synchronize()
        clk.mark_stop()
    B.beam_moe_set_kernel_events([], [])
    barrier(world)
    launches = B.beam_moe_launch_count() - launches0
    ms = start.elapsed_time(stop)
    ms_max = max_over_ranks(ms, world, dev)
    if layer.status() != 0:
        raise SystemExit(f"{name}: device status word reports an error in the timed region")
    # stages the path launched: their events were recorded inside the timed
    # region (the others keep their setup records from before `start`)
    ran = [start.elapsed_time(ev[-1][j][0]) >= 0.0 for j in range(nst)]
    per_kernel_ms = {kn: sum(ev[i][j][0].elapsed_time(ev[i][j][1]) for i in range(args.steps))
                     / args.steps for j, kn in enumerate(B.KERNEL_STAGES) if ran[j]}
    del ev

    # end to end through the host-I/O entry point (pinned host buffers)
    e2e = None
    if not args.no_e2e:
        xh = x.cpu().pin_memory()
        oh = torch.empty_like(xh).pin_memory()
        if args.block:  # host copies around the block call, through torch
            def host_step():
                x.copy_(xh, non_blocking=True)
                step_fn()
                oh.copy_(out, non_blocking=True)
                torch.cuda.synchronize()
        else:
            host_step = lambda: layer.forward_host(xh, oh)
        for _ in range(max(1, args.warmup)):
            host_step()
        barrier(world)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            host_step()
        dt = max_over_ranks(time.perf_counter() - t0, world, dev)
        nbytes = sh.T * sh.H * 2
        e2e = {"value": world * sh.T * args.steps / dt, "unit": UNIT,
               "h2d_bytes_per_step": nbytes, "d2h_bytes_per_step": nbytes}
        del xh, oh

    value = world * sh.T * args.steps / (ms_max / 1e3)
    t_peak, t_peak_src = tensor_peak(fmt, peaks, lib_peaks)
    alg = workload_algorithmic(sh, n_active, fmt)
    dom = max(per_kernel_ms, key=per_kernel_ms.get)
    a = alg[dom]
    t_dom = per_kernel_ms[dom] / 1e3
    t_bw = a["bytes"] / (peaks["hbm_gbs"] * 1e9)
    t_fl = a["flops"] / (t_peak * 1e12) if a["flops"] else 0.0
    if t_fl > t_bw:
        achieved = a["flops"] / t_dom / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": t_peak,
                "unit": "TFLOP/s", "frac": achieved / t_peak}
        roof["peak_source"] = t_peak_src
    else:
        achieved = a["bytes"] / t_dom / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"]}
        roof["peak_source"] = "measured HBM copy (MEASURED_PEAKS.json)" \
            if peaks.get("_src") == "measured" else "fallback"
    roof["traffic"] = ncu_traffic(dom, name)
    roof["kernel"] = dom
    roof["algorithmic_bytes_per_launch"] = a["bytes"]
    roof["algorithmic_flops_per_launch"] = a["flops"]
    lay = alg["layer"]
    t_step = ms_max / args.steps / 1e3
    layer_roof = {
        "hbm_frac": lay["bytes"] / t_step / 1e9 / peaks["hbm_gbs"],
        "tensor_frac": lay["flops"] / t_step / 1e12 / t_peak,
        "tensor_peak": t_peak, "tensor_peak_source": t_peak_src,
        "attainable_frac": max(lay["bytes"] / (peaks["hbm_gbs"] * 1e9),
                               lay["flops"] / (t_peak * 1e12)) / t_step,
    }
    if fmt == "bf16":
        sus = peaks.get("bf16_tflops_sustained")
        if sus:
            layer_roof["tensor_frac_of_sustained"] = lay["flops"] / t_step / 1e12 / sus
            layer_roof["attainable_frac_sustained"] = max(
                lay["bytes"] / (peaks["hbm_gbs"] * 1e9), lay["flops"] / (sus * 1e12)) / t_step
    elif fmt == "nvfp4":
        layer_roof["tensor_frac_of_nominal_ratio_peak"] = (
            lay["flops"] / t_step / 1e12 / (peaks["bf16_tflops"] * NVFP4_OVER_BF16))

    load = float(counts.max() / counts.mean())
    config = {"workload": f"{name}{'(' + args.override + ')' if args.override else ''}: "
                          f"T={sh.T} tokens, hidden {sh.H}, intermediate {sh.I}, {sh.E} experts "
                          f"in {sh.G} groups, top-{sh.topk_groups} groups, top-{sh.top_k}, "
                          f"{fmt} experts"
                          + (f"; fused block: RMS pre-norm, the layer, RMS post-norm, "
                             f"residual step {BLOCK_STEP}" if args.block else ""),
              "tokens_per_step_per_gpu": sh.T, "active_experts": n_active,
              "max_expert_load_over_mean": load,
              "l2": "no flush: expert weights read per step exceed the 126 MB L2",
              "parallelism": f"replicas x{world}"}
    if sh.routing == "zipf":
        config["skew_target_load_over_mean"] = SKEW_TARGET
    res = {"value": value, "unit": UNIT, "ms_per_step": ms_max / args.steps,
           "dtype": DTYPES[fmt], "config": config, "roofline": roof,
           "layer_roofline": layer_roof, "kernels_ms": per_kernel_ms, "e2e": e2e,
           "gpu_launches": launches, "clocks": clk.summary()}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, cores, n, dt = cpu_oracle_run(sh, d, args.cpu_tokens, fmt=fmt)
        res["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
                               "sample": f"{n} seeded tokens of the {name} batch ({dt:.1f} s)"}
    else:
        res["cpu_baseline"] = None
    return res


DTYPES = {"bf16": "bf16",
          "nvfp4": "nvfp4 weights+activations, fp4 MMA (kind::mxf4nvf4), f32 accumulate",
          "mxfp8": "mxfp8 weights+activations, fp8 MMA (kind::mxf8f6f4), f32 accumulate"}


def run_ours(args, world, rank, local):
    import torch
    from sparse_moe_layer_experts_b300 import build as build_mod
    from sparse_moe_layer_experts_b300 import synth

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (there is no CPU fallback)")
    build_mod.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    names = list(DEFAULT_SET) if args.config == "all" else [args.config]
    shapes = {n: synth.shape(n, **parse_override(args.override)) for n in names}
    sh0 = shapes[names[0]]
    weights = synth.make_inputs(sh0, seed=0, device=dev, weights=True)
    weights = {k: weights[k] for k in ("w_gate", "w_up", "w_down")}
    peaks, peak_src = load_peaks()
    peaks["_src"] = peak_src
    lib_peaks = None
    if any(weight_format(n) != "bf16" for n in names) and not args.no_library_peaks:
        lib_peaks = measure_library_peaks(dev)
    qcache = {}
    results = {}
    for n in names:
        sh = shapes[n]
        assert (sh.H, sh.I, sh.E) == (sh0.H, sh0.I, sh0.E), "workloads share the expert weights"
        layer, d = make_layer(n, sh, weights, qcache, dev, rank)
        results[n] = measure(n, sh, layer, d, args, world, rank, local, dev, peaks, lib_peaks)
        del layer, d
        torch.cuda.empty_cache()

    if rank == 0:
        head = results[names[0]]
        line = {"metric": METRIC, "value": head["value"], "unit": UNIT, "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": head["dtype"],
                "data": "synthetic (seeded N(0,1) activations, N(0,0.02) bf16 weights)"}
        for k in ("config", "roofline", "layer_roofline", "kernels_ms", "cpu_baseline", "e2e",
                  "gpu_launches", "clocks"):
            line[k] = head[k]
        if len(names) > 1:
            line["configs"] = {n: results[n] for n in names[1:]}
        if lib_peaks is not None:
            line["library_tensor_peaks"] = lib_peaks
        print(json.dumps(line), flush=True)


def run_route_only(args):
    """Diagnostic: the routing kernels alone on the configured batch."""
    import torch
    from sparse_moe_layer_experts_b300 import binding as B
    from sparse_moe_layer_experts_b300 import build as build_mod
    from sparse_moe_layer_experts_b300 import synth
    from sparse_moe_layer_experts_b300.layer import BeamMoE
    build_mod.build()
    name = DEFAULT_SET[0] if args.config == "all" else args.config
    sh = synth.shape(name, **parse_override(args.override))
    d = synth.make_inputs(sh, seed=0, device="cuda", weights=False)
    w = torch.zeros(1, dtype=torch.bfloat16, device="cuda")
    layer = BeamMoE.__new__(BeamMoE)
    layer._setup(d["router_w"], w, w, w, sh.E, sh.I, sh.H, sh.G, sh.topk_groups, sh.top_k,
                 sh.scale, 0, 0)
    for _ in range(args.warmup):
        layer.route(d["x"], want_scores=False)
    torch.cuda.synchronize()
    names = B.KERNEL_STAGES[:4]
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in names] for _ in range(args.steps)]
    for pair in ev:
        for e0, e1 in pair:
            e0.record()
            e1.record()
    torch.cuda.synchronize()
    for i in range(args.steps):
        B.check(B.beam_moe_set_kernel_events([e[0].cuda_event for e in ev[i]],
                                             [e[1].cuda_event for e in ev[i]]), "events")
        layer.route(d["x"], want_scores=False)
    torch.cuda.synchronize()
    B.beam_moe_set_kernel_events([], [])
    ms = {n: sum(ev[i][j][0].elapsed_time(ev[i][j][1]) for i in range(args.steps)) / args.steps
          for j, n in enumerate(names)}
    gflop = 2 * sh.T * sh.H * sh.E / 1e9
    print(json.dumps({"route_only": True, "config": name, "T": sh.T, "kernels_ms": ms,
                      "router_tflops": gflop / ms["router_scores"]}), flush=True)


def run_dense(args, world, rank, local):
    """Dense SwiGLU layer (Beam's first three decoder layers) through
    beam_moe_dense_forward: a second workload of the same GEMM kernels."""
    import torch
    from sparse_moe_layer_experts_b300 import binding as B, synth
    from sparse_moe_layer_experts_b300.layer import DenseSwiGLU
    from oracle import oracle
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    sh = dict(synth.DENSE_CONFIGS["dense"])
    sh.update(parse_override(args.override))
    T, H, I = sh["T"], sh["H"], sh["I"]
    d = synth.make_dense_inputs(T, H, I, seed=rank, device=dev)
    layer = DenseSwiGLU(d["w_gate"], d["w_up"], d["w_down"])
    x, out = d["x"], torch.empty_like(d["x"])
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        layer.forward(x, out)
    torch.cuda.synchronize()
    nst = len(B.KERNEL_STAGES)
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(nst)] for _ in range(args.steps)]
    for pair in ev:
        for e0, e1 in pair:
            e0.record(stream)
            e1.record(stream)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = B.beam_moe_launch_count()
    torch.cuda.synchronize()
    barrier(world)
    with ClockSampler(local) as clk:
        clk.mark_start()
        start.record(stream)
        for i in range(args.steps):
            B.check(B.beam_moe_set_kernel_events([e[0].cuda_event for e in ev[i]],
                                                 [e[1].cuda_event for e in ev[i]]), "events")
            layer.forward(x, out)
        stop.record(stream)
        torch.cuda.synchronize()
        clk.mark_stop()
    B.beam_moe_set_kernel_events([], [])
    barrier(world)
    launches = B.beam_moe_launch_count() - launches0
    ms_max = max_over_ranks(start.elapsed_time(stop), world, dev)
    if layer.status() != 0:
        raise SystemExit("device status word reports an error in the timed region")
    used = {"scan": "setup", "gateup_gemm": "gateup_gemm", "down_gemm": "down_gemm"}
    per_kernel_ms = {used[name]: sum(ev[i][j][0].elapsed_time(ev[i][j][1])
                                     for i in range(args.steps)) / args.steps
                     for j, name in enumerate(B.KERNEL_STAGES) if name in used}
    value = world * T * args.steps / (ms_max / 1e3)
    peaks, peak_src = load_peaks()
    flops = {"gateup_gemm": 4.0 * T * H * I, "down_gemm": 2.0 * T * H * I}
    dom = max(flops, key=lambda k: per_kernel_ms[k])
    achieved = flops[dom] / (per_kernel_ms[dom] / 1e3) / 1e12
    roof = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"],
            "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"], "traffic": None,
            "kernel": dom, "peak_source": f"{peak_src} (MEASURED_PEAKS.json)",
            "algorithmic_flops_per_launch": flops[dom]}
    t_step = ms_max / args.steps / 1e3
    layer_roof = {"tensor_frac": 6.0 * T * H * I / t_step / 1e12 / peaks["bf16_tflops"],
                  "hbm_frac": (3.0 * H * I * 2 + 2 * T * H * 2) / t_step / 1e9 / peaks["hbm_gbs"]}
    e2e = None
    if not args.no_e2e:
        xh = x.cpu().pin_memory()
        oh = torch.empty_like(xh).pin_memory()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            xd = xh.to(dev, non_blocking=True)
            layer.forward(xd, out)
            oh.copy_(out, non_blocking=True)
            torch.cuda.synchronize()
        dt = max_over_ranks(time.perf_counter() - t0, world, dev)
        e2e = {"value": world * T * args.steps / dt, "unit": UNIT,
               "h2d_bytes_per_step": T * H * 2, "d2h_bytes_per_step": T * H * 2}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        toks = list(range(0, T, max(1, T // args.cpu_tokens)))[:args.cpu_tokens]
        xb, gb, ub, db = (synth.to_bits(d[k]) for k in ("x", "w_gate", "w_up", "w_down"))
        t0 = time.perf_counter()
        oracle.dense_forward(xb, gb, ub, db, tokens=toks)
        dtc = time.perf_counter() - t0
        cpu = {"value": len(toks) / dtc, "unit": UNIT, "cores": oracle.num_threads(),
               "kind": "oracle", "sample": f"{len(toks)} seeded tokens of the dense batch ({dtc:.1f} s)"}
    if rank == 0:
        print(json.dumps({
            "metric": "Beam dense SwiGLU layer tokens/s at 1 B300 (first three decoder layers)",
            "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_max / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) activations, N(0,0.02) bf16 weights)",
            "config": {"workload": f"dense: T={T} tokens, hidden {H}, intermediate {I}",
                       "tokens_per_step_per_gpu": T,
                       "l2": "no flush: the 0.63 GB of weights read per step exceed the 126 MB L2",
                       "parallelism": f"replicas x{world}"},
            "roofline": roof, "layer_roofline": layer_roof, "kernels_ms": per_kernel_ms,
            "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches, "clocks": clk.summary(),
        }), flush=True)


def main():
    args = parse_args()
    if args.route_only:
        run_route_only(args)
        return
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
    elif args.config == "dense":
        run_dense(args, world, rank, local)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
