"""Benchmark of the fused input projection on GB300.

One step = one fp_forward over one batch of synthetic input: the whole path
(strided load, fused GEMM, bias, activation, rotary embedding, head-major
split) on the Walrus-shaped channels-first workload by default.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]
                    [--pass forward|backward]

With --pass backward a step is one fp_backward (gradients of x, W and b from
seeded upstream gradients) and the line reports its own metric.

Prints one JSON line (rank 0). Under torchrun each rank projects its own copy
of the workload (weak scaling, no data-path collective); the step time is the
max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import fpsynth  # noqa: E402

METRIC = "fused-proj TFLOP/s & tokens/s on 1 GB300; % of min(TC peak, HBM) roofline"
DEFAULT_WORKLOAD = "walrus_bf16"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# GB300 data-sheet figures: dense bf16 tensor throughput and HBM3e bandwidth
NOMINAL = {"bf16_tflops": 2250.0, "hbm_gbs": 8000.0}
# the sources each kind of ncu summary under profiles/ was taken on: a summary
# whose recorded hash no longer matches is stale and its traffic is not used
KERNEL_SOURCES = {
    "gemm": ["ff_input_projection_gb300/csrc/gemm_tc.cu",
             "ff_input_projection_gb300/csrc/epilogue.cuh",
             "ff_input_projection_gb300/csrc/tc_ptx.cuh"],
    "simt": ["ff_input_projection_gb300/csrc/gemm_simt.cu",
             "ff_input_projection_gb300/csrc/epilogue.cuh"],
    "attention": ["ff_input_projection_gb300/csrc/attention.cu",
                  "ff_input_projection_gb300/csrc/epilogue.cuh",
                  "ff_input_projection_gb300/csrc/tc_ptx.cuh"],
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(fpsynth.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="time only the chosen workload (no per_config key)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--cluster", type=int, default=2, choices=[1, 2],
                    help="tensor-core path: CTA pairs sharing weight tiles (2) or single CTAs (1)")
    ap.add_argument("--group-m", type=int, default=0,
                    help="tensor-core tile rasterisation: M-tiles per group (0: the library's default)")
    ap.add_argument("--tile-n", type=int, default=0, choices=[0, 192, 256],
                    help="tensor-core tile width without rotation (0: the library's choice)")
    ap.add_argument("--pass", dest="which", default="forward",
                    choices=["forward", "backward", "attention", "library-gemm"],
                    help="time fp_forward (default), fp_backward (gradients of x, W, b), or "
                         "fp_attention over the UNet projection's outputs, or the workload's "
                         "plain GEMM through this library and through cuBLAS")
    return ap.parse_args()


def algorithmic(w: fpsynth.Workload):
    esz = 2 if w.dtype == "bf16" else 4
    n_out = w.M * w.N
    bytes_ = (w.M * w.C + w.C * w.N + (w.N if w.bias else 0) + n_out) * esz
    return w.flops, bytes_


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


def kernel_hash(kind: str = "gemm") -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kind]:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch of the workload's dominant kernel from a committed
    ncu summary (tensor-core GEMM, FFMA GEMM or attention), if it was taken on
    the current kernel sources (else None)."""
    paths = [(os.path.join(ROOT, "profiles", f"{k}_{workload}.md"), kind)
             for k, kind in (("tc_gemm", "gemm"), ("simt_gemm", "simt"), ("attention", "attention"))]
    paths = [q for q in paths if os.path.exists(q[0])]
    if not paths:
        return None
    path, kind = paths[0]
    text = open(path).read()
    mh = re.search(r"kernel_hash:\s*([0-9a-f]+)", text)
    mt = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not mh or not mt or mh.group(1) != kernel_hash(kind):
        return None
    return float(mt.group(1))


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_uuid: str):
        self.uuid = device_uuid
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.uuid, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self):
        rows = []
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), parts[4:8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, flags in rows for i, fl in enumerate(flags)
                          if fl.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons,
                "samples": len(rows)}


def cpu_baseline(w: fpsynth.Workload, inp, seconds: float):
    """The oracle, as it stands, on a bounded sample of token rows."""
    import oracle
    cores = os.cpu_count() or 1
    rng = np.random.default_rng(0)
    n = 8
    t0 = time.perf_counter()
    done_rows = 0
    elapsed = 0.0
    while True:
        rows = np.sort(rng.choice(w.M, size=min(n, w.M), replace=False))
        t = time.perf_counter()
        oracle.forward_workload(w, inp, rows=rows, threads=cores)
        dt = time.perf_counter() - t
        done_rows += len(rows)
        elapsed += dt
        if elapsed >= seconds or time.perf_counter() - t0 > 3 * seconds:
            break
        rate = len(rows) / max(dt, 1e-6)
        n = int(max(8, min(rate * (seconds - elapsed), 4 * n, w.M)))
    flops = 2.0 * done_rows * w.C * w.N
    return {"value": flops / elapsed / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "tokens_per_s": done_rows / elapsed,
            "sample": f"{done_rows} token rows drawn from the {w.M} of {w.name} (all {w.N} "
                      f"fused columns each), fp64, {elapsed:.1f} s"}


def run_reference(args, rank, world):
    if rank != 0:
        return
    w = fpsynth.WORKLOADS[args.workload]
    inp = fpsynth.make_inputs(w)
    import oracle
    cores = os.cpu_count() or 1
    # per step: a fixed sample of rows sized so the whole run takes a few minutes
    per_step_rows = max(1, min(w.M, int(os.environ.get("FP_REF_ROWS", "64"))))
    rng = np.random.default_rng(1)
    rows = np.sort(rng.choice(w.M, size=per_step_rows, replace=False))
    for _ in range(args.warmup):
        oracle.forward_workload(w, inp, rows=rows[:8], threads=cores)
    times = []
    for _ in range(args.steps):
        t = time.perf_counter()
        oracle.forward_workload(w, inp, rows=rows, threads=cores)
        times.append(time.perf_counter() - t)
        if sum(times) > 150:
            break
    total = sum(times)
    flops = 2.0 * per_step_rows * len(times) * w.C * w.N
    value = flops / total / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": len(times), "warmup": args.warmup, "ms_per_step": 1e3 * total / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": w.name, "x": list(w.x_shape), "C": w.C, "F": w.F,
                       "heads": w.heads, "head_dim": w.head_dim, "N": w.N, "tokens": w.M},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": f"{per_step_rows} token rows of {w.M} per step"},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


PER_CONFIG = ["bert_ff_bf16", "bert_qkv_bf16", "llm_qkv_rope_bf16", "unet_qkv_bf16",
              "unet_qkv_fp32", "gqa_rope_toy_bf16", "tiny_fp32"]
MAX_SETS = 64


def to_device_fn(torch, dev, dtype):
    def to_dev(a):
        if a is None:
            return None
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16) \
            if dtype == "bf16" else torch.from_numpy(np.ascontiguousarray(a))
        return t.to(dev)
    return to_dev


def ffma_peak_tflops(sm_count: int, mhz: float) -> float:
    """FP32 FFMA peak: SMs x 128 FP32 lanes x 2 FLOP per FMA x SM clock."""
    return sm_count * 128 * 2 * mhz * 1e6 / 1e12


def roofline(w, ms, pk, pk_src, sm_count, flops=None, bytes_=None):
    """Roofline of one timed configuration: bf16 against the tensor or HBM bound
    (whichever takes longer at the measured peaks), f32 (TF32 off) against the
    FFMA peak. frac_nominal: the same achieved figure over the data-sheet peak."""
    if flops is None:
        flops, bytes_ = algorithmic(w)
    t = ms * 1e-3
    if w.dtype == "bf16":
        tensor_time = flops / (pk["bf16_tflops"] * 1e12)
        hbm_time = bytes_ / (pk["hbm_gbs"] * 1e9)
        if tensor_time >= hbm_time:
            r = {"bound": "tensor", "achieved": flops / t / 1e12, "peak": pk["bf16_tflops"],
                 "unit": "TFLOP/s", "peak_source": f"{pk_src} (cuBLAS bf16 burst)",
                 "nominal_peak": NOMINAL["bf16_tflops"]}
        else:
            r = {"bound": "hbm", "achieved": bytes_ / t / 1e9, "peak": pk["hbm_gbs"],
                 "unit": "GB/s", "peak_source": f"{pk_src} (copy)",
                 "nominal_peak": NOMINAL["hbm_gbs"]}
    else:
        mhz = float(pk.get("sm_max_mhz") or 2070.0)
        r = {"bound": "alu", "achieved": flops / t / 1e12, "peak": ffma_peak_tflops(sm_count, mhz),
             "unit": "TFLOP/s",
             "peak_source": f"derived: {sm_count} SMs x 128 FP32 lanes x 2 FLOP x {mhz:.0f} MHz",
             "nominal_peak": ffma_peak_tflops(sm_count, mhz)}
    r["frac"] = r["achieved"] / r["peak"]
    r["frac_nominal"] = r["achieved"] / r["nominal_peak"]
    return r


class ForwardRun:
    """One forward configuration set up for timing: input and output sets
    rotated so that one pass over them exceeds twice the L2."""

    def __init__(self, torch, fpx, dev, w, *, explicit_pos=False, cluster=2, group_m=0,
                 tile_n=0):
        self.torch, self.w, self.dev = torch, w, dev
        inp = fpsynth.make_inputs(w)
        self.inp = inp
        to_dev = to_device_fn(torch, dev, w.dtype)
        esz = 2 if w.dtype == "bf16" else 4
        self.in_bytes = (w.M * w.C + w.C * w.N + (w.N if w.bias else 0)) * esz
        self.out_bytes = w.M * w.N * esz
        per_set = self.in_bytes + self.out_bytes
        self.n_sets = int(min(MAX_SETS, max(2, np.ceil(2 * L2_BYTES / per_set))))
        self.xs = [to_dev(inp["x"]) for _ in range(self.n_sets)]
        self.Ws = [to_dev(inp["W"]) for _ in range(self.n_sets)]
        self.bs = [to_dev(inp["b"]) for _ in range(self.n_sets)]
        self.proj = fpx.FusedProjection(w.C, w.F, w.heads, w.head_dim, w.act, w.rope_base,
                                        w.n_query_groups, w.rope_n_elem, w.k_transposed)
        self.proj.set_option(fpx.FP_OPT_CLUSTER, cluster)
        if group_m:
            self.proj.set_option(fpx.FP_OPT_GROUP_M, group_m)
        if tile_n:
            self.proj.set_option(fpx.FP_OPT_TILE_N, tile_n)
        self.proj.reserve(w.T)
        self.pos = torch.arange(w.T, dtype=torch.int32, device=dev) if explicit_pos else None
        self.stream = torch.cuda.Stream(device=dev)
        with torch.cuda.stream(self.stream):
            self.outs = [self.proj.forward(self.xs[0], self.Ws[0], self.bs[0], self.pos,
                                           channel_dim=w.channel_dim, n_batch_dims=w.n_batch_dims,
                                           stream=self.stream.cuda_stream)
                         for _ in range(self.n_sets)]
        self.fpx = fpx

    def step(self, i):
        j = i % self.n_sets
        w = self.w
        return self.proj.forward(self.xs[j], self.Ws[j], self.bs[j], self.pos,
                                 channel_dim=w.channel_dim, n_batch_dims=w.n_batch_dims,
                                 out=self.outs[j], stream=self.stream.cuda_stream)

    def l2_note(self):
        tot = self.n_sets * (self.in_bytes + self.out_bytes)
        cap = " (capped)" if self.n_sets == MAX_SETS and tot < 2 * L2_BYTES else ""
        return (f"inputs and outputs rotate over {self.n_sets} sets{cap} "
                f"({tot / 1e6:.0f} MB; L2 129 MB)")

    def time(self, steps, warmup, uuid, dist=None):
        """Mean ms per step over `steps` steps replayed from a CUDA graph, after
        `warmup` eager steps; clocks sampled during the timed region."""
        torch, fpx = self.torch, self.fpx
        with torch.cuda.stream(self.stream):
            for i in range(max(3, warmup)):
                self.step(i)
        torch.cuda.synchronize(self.dev)
        fpx.check(self.proj.device_status(self.stream.cuda_stream))
        self.launches_per_step = self.proj.last_launch_count
        G = max(d for d in range(1, min(steps, 64) + 1) if steps % d == 0)
        graph = None
        try:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=self.stream):
                for i in range(G):
                    self.step(i)
            with torch.cuda.stream(self.stream):
                graph.replay()
            torch.cuda.synchronize(self.dev)
        except Exception as exc:  # capture unsupported here: time the eager loop instead
            graph = None
            self.timing_note = f"eager (graph capture failed: {type(exc).__name__})"
        else:
            self.timing_note = f"CUDA graph of {G} steps replayed {steps // G} times"
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        if dist:
            dist.barrier()
        torch.cuda.synchronize(self.dev)
        # graph.replay() launches on torch's current stream: make that the timed stream
        with ClockSampler(uuid) as clk, torch.cuda.stream(self.stream):
            ev0.record(self.stream)
            if graph is not None:
                for _ in range(steps // G):
                    graph.replay()
            else:
                for i in range(steps):
                    self.step(i)
            ev1.record(self.stream)
            torch.cuda.synchronize(self.dev)
        if dist:
            dist.barrier()
        fpx.check(self.proj.device_status(self.stream.cuda_stream))
        self.clocks = clk.summary()
        return ev0.elapsed_time(ev1) / steps

    def close(self):
        self.proj.close()
        del self.xs, self.Ws, self.bs, self.outs
        self.torch.cuda.empty_cache()


def steps_for(run, target_s=0.25, lo=20, hi=4000):
    """Steps whose timed region lasts about target_s, from a short eager trial."""
    torch = run.torch
    with torch.cuda.stream(run.stream):
        run.step(0)
        torch.cuda.synchronize(run.dev)
        t = time.perf_counter()
        for i in range(5):
            run.step(i)
        torch.cuda.synchronize(run.dev)
    per = max((time.perf_counter() - t) / 5, 1e-6)
    n = int(min(hi, max(lo, target_s / per)))
    return max(lo, n // 20 * 20)


def time_attention(torch, fpx, dev, uuid, pk, pk_src, sm_count):
    """fp_attention over the outputs of the diffusion-UNet projection (k emitted
    pre-transposed): per_config entry with its own timing, clocks and roofline."""
    w = fpsynth.WORKLOADS["unet_qkv_bf16"].scaled(k_transposed=True)
    inp = fpsynth.make_inputs(w)
    to_dev = to_device_fn(torch, dev, "bf16")
    proj = fpx.FusedProjection(w.C, w.F, w.heads, w.head_dim, w.act, w.rope_base, 0, 0, True)
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        _, q, kT, v = proj.forward(to_dev(inp["x"]), to_dev(inp["W"]), None, None,
                                   channel_dim=w.channel_dim, n_batch_dims=w.n_batch_dims,
                                   stream=stream.cuda_stream)
    torch.cuda.synchronize(dev)
    per_set = 4 * q.numel() * 2
    n_sets = int(min(MAX_SETS, max(2, np.ceil(2 * L2_BYTES / per_set))))
    sets = [(q.clone(), kT.clone(), v.clone(), torch.empty_like(q)) for _ in range(n_sets)]
    B, T = w.Bb, w.T

    def step(i):
        a, b, c, o = sets[i % n_sets]
        proj.attention(a, b, c, batch=B, out=o, stream=stream.cuda_stream)

    with torch.cuda.stream(stream):
        for i in range(5):
            step(i)
    torch.cuda.synchronize(dev)
    fpx.check(proj.device_status(stream.cuda_stream))
    steps = 200
    G = 20
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for i in range(G):
            step(i)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        graph.replay()
    torch.cuda.synchronize(dev)
    with ClockSampler(uuid) as clk, torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(steps // G):
            graph.replay()
        ev1.record(stream)
        torch.cuda.synchronize(dev)
    fpx.check(proj.device_status(stream.cuda_stream))
    ms = ev0.elapsed_time(ev1) / steps
    BH = B * w.heads
    flops = 4 * BH * T * T * w.head_dim
    bytes_ = 4 * BH * T * w.head_dim * 2
    roof = roofline(w, ms, pk, pk_src, sm_count, flops, bytes_)
    entry = {"workload": "unet_attention_bf16", "pass": "attention", "ms_per_step": ms,
             "tflops": flops / (ms * 1e-3) / 1e12, "tokens_per_s": BH * T / (ms * 1e-3),
             "steps": steps, "timing": f"CUDA graph of {G} steps replayed {steps // G} times",
             "gpu_launches_per_step": proj.last_launch_count, "dtype": "bf16",
             "shape": {"batch_heads": BH, "T_q": T, "T_k": T, "head_dim": w.head_dim,
                       "k": "pre-transposed [B*heads, head_dim, T] from fp_forward"},
             "flops_per_step": flops,
             "l2": f"q, k, v, out rotate over {n_sets} sets ({n_sets * per_set / 1e6:.0f} MB)",
             "roofline": {k: roof[k] for k in ("bound", "achieved", "peak", "unit", "frac",
                                               "frac_nominal", "peak_source")},
             "clocks": clk.summary()}
    entry["roofline"]["traffic"] = recorded_traffic("unet_attention_bf16")
    proj.close()
    del sets
    torch.cuda.empty_cache()
    return entry


def config_entry(w, ms, roof, clocks, steps, timing, launches, extra=None):
    e = {"workload": w.name, "ms_per_step": ms, "tflops": 2.0 * w.M * w.C * w.N / (ms * 1e-3) / 1e12,
         "tokens_per_s": w.M / (ms * 1e-3), "steps": steps, "timing": timing,
         "gpu_launches_per_step": launches, "dtype": w.dtype,
         "roofline": {k: roof[k] for k in ("bound", "achieved", "peak", "unit", "frac",
                                           "frac_nominal", "peak_source")},
         "clocks": clocks}
    if not (extra and extra.get("pass") == "backward"):
        e["roofline"]["traffic"] = recorded_traffic(w.name)
    if extra:
        e.update(extra)
    return e


def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, rank, world)
    if args.which == "backward":
        return main_backward(args, rank, world, local)
    if args.which == "library-gemm":
        return main_library_gemm(args, local)
    if args.which == "attention":
        return main_attention(local)

    import torch
    import ff_input_projection_gb300 as fpx
    from ff_input_projection_gb300 import _build
    from ff_input_projection_gb300.shard import max_over_ranks
    _build.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        uuid = str(local)
    sm_count = torch.cuda.get_device_properties(dev).multi_processor_count
    pk, pk_src = peaks()

    w = fpsynth.WORKLOADS[args.workload]
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    flops, alg_bytes = algorithmic(w)
    run = ForwardRun(torch, fpx, dev, w, cluster=args.cluster, group_m=args.group_m,
                     tile_n=args.tile_n)
    ms = run.time(args.steps, args.warmup, uuid, dist)
    ms = max_over_ranks(ms, dev)
    total_flops = flops * world
    value = total_flops / (ms * 1e-3) / 1e12
    tokens_per_s = w.M * world / (ms * 1e-3)
    clocks = run.clocks

    # ---- end to end through the public API with pinned host buffers: one
    # fp_forward_host call per step (x uploaded, outputs downloaded, in chunks
    # the library overlaps with the compute)
    proj, outs, stream = run.proj, run.outs[0], run.stream
    hx = torch.empty(run.xs[0].shape, dtype=tdt, pin_memory=True)
    hx.copy_(run.xs[0].cpu())
    host_outs = tuple(None if o is None else torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
                      for o in outs)
    h2d = hx.numel() * hx.element_size()
    d2h = sum(o.numel() * o.element_size() for o in host_outs if o is not None)
    e2e_steps = max(3, min(args.steps, 30))

    def e2e_step():
        proj.forward_host(hx, run.Ws[0], run.bs[0], None, channel_dim=w.channel_dim,
                          n_batch_dims=w.n_batch_dims, out=host_outs, stream=stream.cuda_stream)

    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e2e_step()
        torch.cuda.synchronize(dev)
        if dist:
            dist.barrier()
        ev0.record(stream)
        for _ in range(e2e_steps):
            e2e_step()
        ev1.record(stream)
        torch.cuda.synchronize(dev)
    e2e_ms = ev0.elapsed_time(ev1) / e2e_steps
    e2e_ms = max_over_ranks(e2e_ms, dev)
    roof = roofline(w, ms, pk, pk_src, sm_count)
    roof["traffic"] = recorded_traffic(w.name)
    roof["kernel_hash"] = kernel_hash("simt" if w.dtype == "f32" else "gemm")
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if w.dtype == "bf16" else "f32", "data": "synthetic",
        "tokens_per_s": tokens_per_s,
        "config": {"workload": w.name, "x": list(w.x_shape), "channel_dim": w.channel_dim,
                   "C": w.C, "F": w.F, "heads": w.heads, "head_dim": w.head_dim, "N": w.N,
                   "tokens": w.M, "act": fpsynth.ACT_NAMES[w.act], "rope_base": w.rope_base,
                   "bias": w.bias, "parallelism": f"replicas x{world}",
                   "cta_cluster": args.cluster, "tile_n": args.tile_n or "auto", "l2": run.l2_note(), "timing": run.timing_note},
        "gpu_launches": run.launches_per_step * args.steps,
        "roofline": roof,
        "clocks": clocks,
        "e2e": {"value": total_flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "call": "fp_forward_host"},
    }
    run.close()

    # ---- every other configuration, each with its own timing, clocks and roofline
    if not args.no_per_config and world == 1 and rank == 0:
        per = []
        names = [(n, False) for n in PER_CONFIG if n != w.name] + [(w.name, True)]
        for name, explicit_pos in names:
            cw = fpsynth.WORKLOADS[name]
            if explicit_pos and cw.rope_base <= 0:
                continue
            r = ForwardRun(torch, fpx, dev, cw, explicit_pos=explicit_pos, cluster=args.cluster,
                           tile_n=args.tile_n)
            n = steps_for(r)
            cms = r.time(n, 5, uuid)
            extra = {"positions": "caller int32 [T] (rotary table rebuilt every call)"} \
                if explicit_pos else None
            per.append(config_entry(cw, cms, roofline(cw, cms, pk, pk_src, sm_count), r.clocks, n,
                                    r.timing_note, r.launches_per_step, extra))
            r.close()
        if w.dtype == "bf16":
            bms, bclk, bn, blaunch = time_backward_run(torch, fpx, dev, w, uuid)
            bfl, bby = backward_algorithmic(w)
            e = config_entry(w, bms, roofline(w, bms, pk, pk_src, sm_count, bfl, bby),
                             bclk, bn, "eager loop of fp_backward calls", blaunch,
                             {"pass": "backward", "flops_per_step": bfl})
            e["tflops"] = bfl / (bms * 1e-3) / 1e12
            per.append(e)
        per.append(time_attention(torch, fpx, dev, uuid, pk, pk_src, sm_count))
        line["per_config"] = per
    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(w, run.inp, args.cpu_seconds)
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def backward_algorithmic(w: fpsynth.Workload):
    """FLOPs of one backward: the ff pre-activation recomputed (2 M C F), dx = G W^T
    and dW = X^T G (2 M N C each); bytes: x, W, b and the upstream gradients read
    once, dx, dW (fp32) and db (fp32) written once."""
    flops = 2 * w.M * w.C * (w.F + 2 * w.N)
    bytes_ = (w.M * w.C + w.C * w.N + (w.N if w.bias else 0) + w.M * w.N + w.M * w.C) * 2 \
        + (w.C * w.N + (w.N if w.bias else 0)) * 4
    return flops, bytes_


class BackwardRun:
    """fp_backward on one workload, set up for timing: input and upstream
    gradient sets rotated so that one pass over them exceeds twice the L2."""

    def __init__(self, torch, fpx, dev, w):
        self.torch, self.fpx, self.dev, self.w = torch, fpx, dev, w
        self.inp = inp = fpsynth.make_inputs(w)
        self.grads = grads = fpsynth.make_grads(w)
        to_dev = to_device_fn(torch, dev, "bf16")
        self.in_bytes = (w.M * w.C + w.C * w.N + w.M * w.N) * 2
        self.n_sets = max(1, int(np.ceil(2 * L2_BYTES / self.in_bytes)))
        self.sets = [(to_dev(inp["x"]), to_dev(inp["W"]), to_dev(inp["b"]),
                      tuple(to_dev(grads[k]) for k in ("ff", "q", "k", "v")))
                     for _ in range(self.n_sets)]
        self.proj = fpx.FusedProjection(w.C, w.F, w.heads, w.head_dim, w.act, w.rope_base,
                                        w.n_query_groups, w.rope_n_elem, w.k_transposed)
        self.proj.reserve(w.T)
        self.stream = torch.cuda.Stream(device=dev)
        x0 = self.sets[0][0]
        L = fpx.make_layout(x0.shape, x0.stride(), w.channel_dim, w.n_batch_dims, fpx.FP_BF16)
        st, ws_bytes = fpx.fp_backward_workspace_size(self.proj.plan, L)
        fpx.check(st)
        self.ws = torch.empty((ws_bytes,), dtype=torch.uint8, device=dev)
        self.dx = torch.empty_strided(x0.shape, x0.stride(), dtype=torch.bfloat16, device=dev)

    def step(self, i):
        x, W, b, g = self.sets[i % self.n_sets]
        w = self.w
        return self.proj.backward(x, W, b, g, None, channel_dim=w.channel_dim,
                                  n_batch_dims=w.n_batch_dims, dx=self.dx, workspace=self.ws,
                                  stream=self.stream.cuda_stream)

    def time(self, steps, warmup, uuid, dist=None):
        torch, fpx = self.torch, self.fpx
        with torch.cuda.stream(self.stream):
            for i in range(max(3, warmup)):
                self.step(i)
        torch.cuda.synchronize(self.dev)
        fpx.check(self.proj.device_status(self.stream.cuda_stream))
        self.launches_per_step = self.proj.last_launch_count
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        if dist:
            dist.barrier()
        torch.cuda.synchronize(self.dev)
        with ClockSampler(uuid) as clk, torch.cuda.stream(self.stream):
            ev0.record(self.stream)
            for i in range(steps):
                self.step(i)
            ev1.record(self.stream)
            torch.cuda.synchronize(self.dev)
        if dist:
            dist.barrier()
        fpx.check(self.proj.device_status(self.stream.cuda_stream))
        self.clocks = clk.summary()
        return ev0.elapsed_time(ev1) / steps

    def close(self):
        self.proj.close()
        del self.sets, self.ws, self.dx
        self.torch.cuda.empty_cache()


def time_backward_run(torch, fpx, dev, w, uuid, steps=100):
    r = BackwardRun(torch, fpx, dev, w)
    ms = r.time(steps, 5, uuid)
    out = (ms, r.clocks, steps, r.launches_per_step)
    r.close()
    return out


def main_backward(args, rank, world, local):
    import torch
    import ff_input_projection_gb300 as fpx
    from ff_input_projection_gb300 import _build
    from ff_input_projection_gb300.shard import max_over_ranks
    _build.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    w = fpsynth.WORKLOADS[args.workload]
    if w.dtype != "bf16":
        raise SystemExit("the backward takes bf16 workloads")
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        uuid = str(local)
    sm_count = torch.cuda.get_device_properties(dev).multi_processor_count
    flops, alg_bytes = backward_algorithmic(w)
    run = BackwardRun(torch, fpx, dev, w)
    ms = max_over_ranks(run.time(args.steps, args.warmup, uuid, dist), dev)
    value = flops * world / (ms * 1e-3) / 1e12
    proj, stream, dx, ws = run.proj, run.stream, run.dx, run.ws

    # end to end: upstream gradients and x from pinned host memory, dx, dW, db
    # back, one fp_backward_host call per step (copies pipelined in chunks)
    x0, W0, b0, g0 = run.sets[0]
    hx = torch.empty(x0.shape, dtype=torch.bfloat16, pin_memory=True)
    hx.copy_(x0.cpu())
    hg = [None if g is None else torch.empty(g.shape, dtype=g.dtype, pin_memory=True) for g in g0]
    for h, g in zip(hg, g0):
        if h is not None:
            h.copy_(g.cpu())
    hdx = torch.empty(x0.shape, dtype=torch.bfloat16, pin_memory=True)
    hdW = torch.empty((w.C, w.N), dtype=torch.float32, pin_memory=True)
    hdb = torch.empty((w.N,), dtype=torch.float32, pin_memory=True) if w.bias else None
    h2d = hx.numel() * 2 + sum(h.numel() * 2 for h in hg if h is not None)
    d2h = hdx.numel() * 2 + hdW.numel() * 4 + (hdb.numel() * 4 if hdb is not None else 0)
    e2e_steps = max(3, min(args.steps, 20))

    def e2e_step():
        proj.backward_host(hx, W0, b0, tuple(hg), None, channel_dim=w.channel_dim,
                           n_batch_dims=w.n_batch_dims, out=(hdx, hdW, hdb),
                           stream=stream.cuda_stream)

    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e2e_step()
        torch.cuda.synchronize(dev)
        ev0.record(stream)
        for _ in range(e2e_steps):
            e2e_step()
        ev1.record(stream)
        torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(ev0.elapsed_time(ev1) / e2e_steps, dev)

    pk, pk_src = peaks()
    roof = roofline(w, ms, pk, pk_src, sm_count, flops, alg_bytes)
    roof["traffic"] = None
    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return
    line = {
        "metric": "fused-proj backward TFLOP/s & tokens/s on 1 GB300; % of TC roofline",
        "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "tokens_per_s": w.M * world / (ms * 1e-3),
        "config": {"workload": w.name, "pass": "backward", "x": list(w.x_shape),
                   "channel_dim": w.channel_dim, "C": w.C, "F": w.F, "heads": w.heads,
                   "head_dim": w.head_dim, "N": w.N, "tokens": w.M,
                   "act": fpsynth.ACT_NAMES[w.act], "bias": w.bias,
                   "flops_per_step": flops, "parallelism": f"replicas x{world}",
                   "l2": f"inputs rotate over {run.n_sets} sets "
                         f"({run.n_sets * run.in_bytes / 1e6:.0f} MB) > L2 129 MB",
                   "timing": "eager loop of fp_backward calls"},
        "gpu_launches": run.launches_per_step * args.steps,
        "roofline": roof,
        "clocks": run.clocks,
        "e2e": {"value": flops * world / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "call": "fp_backward_host"},
    }
    if not args.no_cpu_baseline and world == 1:
        import oracle
        cores = os.cpu_count() or 1
        rng = np.random.default_rng(0)
        el, done = 0.0, 0
        while el < args.cpu_seconds and done < 64 * w.M:
            rows = np.sort(rng.choice(w.M, size=min(64, w.M), replace=False))
            t = time.perf_counter()
            oracle.backward_workload(w, run.inp, run.grads, rows=rows, threads=cores)
            el += time.perf_counter() - t
            done += len(rows)
        fl = 2.0 * done * w.C * (w.F + w.N)
        line["cpu_baseline"] = {"value": fl / el / 1e12, "unit": "TFLOP/s", "cores": cores,
                                "kind": "oracle",
                                "sample": f"dx of {done} token rows drawn from the {w.M} (ff "
                                          f"recompute + G W^T per row), fp64, {el:.1f} s"}
    run.close()
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def main_attention(local):
    """The attention consumer alone (its per_config entry), for profiling."""
    import torch
    import ff_input_projection_gb300 as fpx
    from ff_input_projection_gb300 import _build
    _build.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        uuid = str(local)
    pk, pk_src = peaks()
    sm_count = torch.cuda.get_device_properties(dev).multi_processor_count
    print(json.dumps(time_attention(torch, fpx, dev, uuid, pk, pk_src, sm_count)), flush=True)


def main_library_gemm(args, local):
    """Context line, not the headline: the workload's contraction as a plain
    bf16 GEMM [M, C] x [C, N] (channels-last x, no bias, activation, rotation or
    head split) through fp_forward and through torch.matmul (cuBLAS), both on
    the same rotated operand sets, CUDA-graph replays timed with CUDA events."""
    import torch
    import ff_input_projection_gb300 as fpx
    from ff_input_projection_gb300 import _build
    _build.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = fpsynth.WORKLOADS[args.workload]
    if w.dtype != "bf16":
        raise SystemExit("the library comparison takes bf16 workloads")
    M, C, N = w.M, w.C, w.N
    per_set = (M * C + C * N + M * N) * 2
    n_sets = int(min(MAX_SETS, max(2, np.ceil(2 * L2_BYTES / per_set))))
    gen = torch.Generator(device=dev).manual_seed(1)
    xs = [torch.randn(M, C, device=dev, generator=gen).to(torch.bfloat16) for _ in range(n_sets)]
    Ws = [(torch.randn(C, N, device=dev, generator=gen) * C ** -0.5).to(torch.bfloat16)
          for _ in range(n_sets)]
    ys = [torch.empty(M, N, device=dev, dtype=torch.bfloat16) for _ in range(n_sets)]
    proj = fpx.FusedProjection(C, N, 0, 0, "none", 0.0)
    stream = torch.cuda.Stream(device=dev)

    def ours(i):
        j = i % n_sets
        proj.forward(xs[j].view(1, M, C), Ws[j], None, None, channel_dim=2,
                     out=(ys[j], None, None, None), stream=stream.cuda_stream)

    def cublas(i):
        j = i % n_sets
        torch.matmul(xs[j], Ws[j], out=ys[j])

    def timed(step, steps):
        with torch.cuda.stream(stream):
            for i in range(max(3, args.warmup)):
                step(i)
        torch.cuda.synchronize(dev)
        G = max(d for d in range(1, min(steps, 64) + 1) if steps % d == 0)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for i in range(G):
                step(i)
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            graph.replay()
            torch.cuda.synchronize(dev)
            ev0.record(stream)
            for _ in range(steps // G):
                graph.replay()
            ev1.record(stream)
        torch.cuda.synchronize(dev)
        return ev0.elapsed_time(ev1) / steps

    steps = max(20, args.steps // 20 * 20)
    ms_ours = timed(ours, steps)
    fpx.check(proj.device_status(stream.cuda_stream))
    ms_cb = timed(cublas, steps)
    ref = torch.matmul(xs[0], Ws[0])
    ours(0)
    torch.cuda.synchronize(dev)
    err = (ys[0].float() - ref.float()).abs().max().item()
    flops = 2.0 * M * C * N
    print(json.dumps({
        "metric": "plain bf16 GEMM, this library against cuBLAS (context, not the headline)",
        "workload": w.name, "shape_MxCxN": [M, C, N], "steps": steps,
        "ours_us": ms_ours * 1e3, "cublas_us": ms_cb * 1e3,
        "ours_tflops": flops / (ms_ours * 1e-3) / 1e12,
        "cublas_tflops": flops / (ms_cb * 1e-3) / 1e12,
        "ours_over_cublas_time": ms_ours / ms_cb, "max_abs_diff_vs_cublas": err,
        "l2": f"operands rotate over {n_sets} sets ({n_sets * per_set / 1e6:.0f} MB; L2 129 MB)",
    }), flush=True)
    proj.close()


if __name__ == "__main__":
    main()
