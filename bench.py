#!/usr/bin/env python
"""Benchmark of the block-quantized GEMV/GEMM library on GB300.

Headline (one JSON line on stdout, rank 0):
  metric  Q4_K GEMV weight GB/s (and % of HBM peak); 7B-shape decode tok/s
  step    one pass of the hot path over 64 distinct Q4_K 4096x4096 weight
          matrices at batch 1 (outlier-weighted weights): per matrix, the
          activation quantize (fp32 -> Q8_K) and the GEMV.  64 x 9.44 MB of
          weights per step is larger than L2, so no step is served from L2.
  value   weight bytes streamed per second over the timed steps (device
          resident inputs; CUDA-event timing of a CUDA graph of the step).
Also in the line: roofline of the GEMV kernel (with its ncu DRAM traffic
when the kernel source matches the committed capture), the one-launch
streaming point, the unfused step, the end-to-end figure with host buffers,
the 7B-shape decode (tok/s), the batch sweep on 14336x4096 through both
kernel families, the 512-column prefill GEMM, the quantized KV cache
(scores and append), the Q6_K and Q5_K GEMVs (dependent launches and one streaming
launch), the 512x1024 Q4_0 GEMV (latency), the CPU oracle baseline (all
cores and one core), the
number of library kernel launches in the timed region, and the SM clocks
sampled during it.

  python bench.py [--gpus N --steps K --warmup W] [--impl reference] [--quick]
                  [--only prefill|sweep|decode|stream|kv|kv_q4_0|q6k|q5k|q4_0|q0_gemm] [--no-cpu]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

GEMV_ROWS = GEMV_COLS = 4096
COPIES = 64
Q4K_ROW_BYTES = GEMV_COLS // 256 * 144


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=4000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", default="gq", choices=["gq", "reference"])
    p.add_argument("--quick", action="store_true", help="headline only (no sweeps)")
    p.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    p.add_argument("--only", choices=["prefill", "sweep", "decode", "stream", "kv", "kv_q4_0", "q6k", "q5k", "q4_0",
                                      "q0_gemm"],
                   default=None,
                   help="run one secondary workload alone and print its result (profiling)")
    return p.parse_args()


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d.get("bf16_tflops", 1900.0)), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, 1900.0, "fallback"


def kernel_traffic(kernel: str):
    """Per-launch DRAM bytes of `kernel` from the committed ncu summary, if
    the kernel source has not changed since it was captured."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)[kernel]
        src = os.path.join(ROOT, d["source"])
        h = hashlib.sha256(open(src, "rb").read()).hexdigest()
        return d["bytes_per_launch"] if h == d["sha256"] else None
    except (OSError, KeyError, ValueError):
        return None


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [s.strip() for s in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        # samples taken under load: clocks near their maximum or power well above idle
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "samples": len(rows), "reasons": reasons}


def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return
        run_reference(args)
        return
    run_gpu(args, world, rank)


class Ranks:
    """Replica bookkeeping for `--gpus N` (one process per GPU, no data-path
    collective): a barrier, and the max over ranks of a duration -- the job
    took as long as its slowest rank.  `dist` is torch.distributed after
    init_process_group (nccl on GPUs, gloo in the CPU tests), or None for one
    process; reductions run on `device`."""

    def __init__(self, dist=None, device="cpu"):
        self.dist = dist
        self.device = device

    def barrier(self):
        if self.dist is not None:
            self.dist.barrier()

    def max(self, v: float) -> float:
        if self.dist is None:
            return v
        import torch
        t = torch.tensor([v], device=self.device, dtype=torch.float64)
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX)
        return float(t.item())


def whole_job_rate(units_per_rank: float, world: int, seconds_max: float) -> float:
    """Units per second of the whole job: every rank did units_per_rank in
    its own time, and the slowest rank's time (max over ranks) counts."""
    return world * units_per_rank / seconds_max


# ---------------------------------------------------------------- CPU oracle

METRIC = "Q4_K GEMV weight GB/s (% of HBM peak); 7B-shape decode tok/s"


def headline_config(world: int) -> dict:
    """The headline workload, named identically by the GPU arm and the
    reference (CPU oracle) arm."""
    return {"workload": "Q4_K x Q8_K GEMV 4096x4096 batch 1, row-std spread + 0.1% outliers; "
                        "step = 64 distinct weight matrices, each with its activation quantize",
            "rows": GEMV_ROWS, "cols": GEMV_COLS, "batch": 1, "matrices_per_step": COPIES,
            "weight_bytes_per_step": COPIES * GEMV_ROWS * Q4K_ROW_BYTES,
            "l2": "inputs larger than L2 (604 MB of weights per step)",
            "parallelism": f"replicas x{world}"}


def oracle_gemv_sample():
    import oracle as orc
    from block_quantized_gb300 import inputs
    W, x = inputs.gemv_q4_k(0)
    Wq = orc.quantize(orc.Q4_K, W)
    return orc, Wq, x


def run_cpu_baseline(seconds=10.0, seconds_one=4.0):
    """The oracle, as it stands, on the host cores: act-quantize + GEMV of the
    4096x4096 Q4_K matrix, repeated for about `seconds` on all cores, then for
    about `seconds_one` on one core; and the act-quantize alone."""
    orc, Wq, x = oracle_gemv_sample()
    nt = orc.max_threads()

    def timed(threads, budget):
        n = 0
        t0 = time.perf_counter()
        while True:
            xq = orc.quantize(orc.Q8_K, x)
            orc.matmul_ref(orc.Q4_K, Wq, xq, GEMV_ROWS, GEMV_COLS, 1, threads)
            n += 1
            dt = time.perf_counter() - t0
            if dt >= budget:
                return n, dt

    n, dt = timed(nt, seconds)
    n1, dt1 = timed(1, seconds_one)
    nq = 0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < 0.5:
        orc.quantize(orc.Q8_K, x)
        nq += 1
    tq = (time.perf_counter() - t0) / nq
    return {"value": n * Wq.nbytes / dt / 1e9, "unit": "GB/s", "cores": nt, "kind": "oracle",
            "cpu_model": cpu_model(),
            "sample": f"{n} x (Q8_K act-quant + Q4_K GEMV 4096x4096, batch 1) in {dt:.1f} s",
            "single_core": {"value": n1 * Wq.nbytes / dt1 / 1e9, "unit": "GB/s", "cores": 1,
                            "sample": f"{n1} x the same in {dt1:.1f} s"},
            "act_quantize_us": tq * 1e6}


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo), for the
    baselines' records."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu model")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def _time_call(fn, budget):
    """Median-free simple rate: repeat fn for about `budget` seconds; seconds
    per call."""
    n = 0
    t0 = time.perf_counter()
    while True:
        fn()
        n += 1
        dt = time.perf_counter() - t0
        if dt >= budget:
            return dt / n


def run_cpu_configs(budget=0.25):
    """The oracle, as it stands, timed on the host cores for the other
    workloads, each on a bounded row sample scaled to the full shape (the
    product's cost is linear in the rows): the 7B-shape decode token (every
    layer matrix and the Q8_0 head, with their activation quantizes), the
    14336x4096 batch sweep, and the 28672x8192x512 prefill.  One core and all
    cores."""
    import oracle as orc
    from block_quantized_gb300 import inputs
    nt = orc.max_threads()
    g = inputs.rng(11)
    cache = {}

    def sample(wtype, rows, cols):
        key = (wtype, rows, cols)
        if key not in cache:
            cache[key] = orc.quantize(wtype, inputs.normal(g, (rows, cols), 0.02))
        return cache[key]

    def act(atype, batch, cols):
        return orc.quantize(atype, inputs.normal(g, (batch, cols)))

    out = {"cores_all": nt, "cpu_model": cpu_model()}
    # 7B decode token: rows sampled per matrix
    R = 256
    layer = [("wq", 4096, 4096), ("wk", 4096, 4096), ("wv", 4096, 4096), ("wo", 4096, 4096),
             ("w1", 11008, 4096), ("w3", 11008, 4096), ("w2", 4096, 11008)]
    xq = {c: act(orc.Q8_K, 1, c) for c in (4096, 11008)}
    xh = act(orc.Q8_0, 1, 4096)
    xf = {c: inputs.normal(g, (c,)) for c in (4096, 11008)}
    dec = {}
    for label, threads in (("all_cores", nt), ("one_core", 1)):
        t_layer = 0.0
        for _, rows, cols in layer:
            W = sample(orc.Q4_K, R, cols)
            t = _time_call(lambda: orc.matmul_ref(orc.Q4_K, W, xq[cols], R, cols, 1, threads), budget)
            t_layer += t * rows / R
        # four activation quantizes per layer (attention, o, ffn, down)
        tq = sum(_time_call(lambda: orc.quantize(orc.Q8_K, xf[c]), budget / 4) for c in (4096, 4096, 4096, 11008))
        Wh = sample(orc.Q8_0, R, 4096)
        t_head = _time_call(lambda: orc.matmul_ref(orc.Q8_0, Wh, xh, R, 4096, 1, threads), budget) * 32000 / R
        t_tok = 32 * (t_layer + tq) + t_head
        dec[label] = {"tok_s": 1.0 / t_tok, "ms_per_token": t_tok * 1e3,
                      "cores": threads}
    dec["sample"] = (f"{R} rows of each layer matrix and of the 32000x4096 Q8_0 head, scaled by rows; "
                     "32 layers + head; the act-quantize of the four layer inputs included")
    out["decode_7b"] = dec
    # batch sweep 14336 x 4096
    R4 = 256
    W4 = sample(orc.Q4_K, R4, 4096)
    sweep = {}
    for b in (1, 2, 4, 8, 16, 32, 64):
        xb = act(orc.Q8_K, b, 4096)
        row = {}
        for label, threads in (("all_cores", nt), ("one_core", 1)):
            t = _time_call(lambda: orc.matmul_ref(orc.Q4_K, W4, xb, R4, 4096, b, threads), budget / 2)
            t_full = t * 14336 / R4
            row[label] = {"us": t_full * 1e6, "tops": 2.0 * 14336 * 4096 * b / t_full / 1e12}
        sweep[str(b)] = row
    out["batch_sweep_14336x4096"] = {"results": sweep,
                                     "sample": f"{R4} of the 14336 rows, scaled by rows"}
    # prefill 28672 x 8192 x 512
    R5 = 32
    W5 = sample(orc.Q4_K, R5, 8192)
    x5 = act(orc.Q8_K, 512, 8192)
    pre = {}
    for label, threads in (("all_cores", nt), ("one_core", 1)):
        t = _time_call(lambda: orc.matmul_ref(orc.Q4_K, W5, x5, R5, 8192, 512, threads), budget)
        t_full = t * 28672 / R5
        pre[label] = {"ms": t_full * 1e3, "tops": 2.0 * 28672 * 8192 * 512 / t_full / 1e12}
    pre["sample"] = f"{R5} of the 28672 rows x 512 columns, scaled by rows"
    out["prefill_28672x8192x512"] = pre
    return out


def run_cpu_q6k(seconds=3.0, wtype=None):
    """The oracle, as it stands, on all host cores for the Q6_K (or Q5_K)
    workload: Q8_K act-quant + GEMV of the 4096x4096 matrix, repeated for
    about `seconds`."""
    import oracle as orc
    from block_quantized_gb300 import inputs
    wt = orc.Q6_K if wtype is None else wtype
    W, _ = inputs.gemv_q4_k(0)
    Wq = orc.quantize(wt, W)
    x = inputs.normal(inputs.rng(2), (GEMV_COLS,))
    nt = orc.max_threads()
    n = 0
    t0 = time.perf_counter()
    while True:
        xq = orc.quantize(orc.Q8_K, x)
        orc.matmul_ref(wt, Wq, xq, GEMV_ROWS, GEMV_COLS, 1, nt)
        n += 1
        dt = time.perf_counter() - t0
        if dt >= seconds:
            break
    return {"value": n * Wq.nbytes / dt / 1e9, "unit": "GB/s", "cores": nt, "kind": "oracle",
            "sample": f"{n} x (Q8_K act-quant + {orc.TYPE_NAMES[wt]} GEMV 4096x4096, batch 1) in {dt:.1f} s"}


def run_cpu_q4_0(seconds=1.0):
    """The oracle on one core for the 512x1024 Q4_0 x Q8_0 GEMV (batch 1):
    Q8_0 act-quant + GEMV, repeated for about `seconds`."""
    import oracle as orc
    from block_quantized_gb300 import inputs
    W, x = inputs.gemv_q4_0(0)
    Wq = orc.quantize(orc.Q4_0, W)
    n = 0
    t0 = time.perf_counter()
    while True:
        xq = orc.quantize(orc.Q8_0, x)
        orc.matmul_ref(orc.Q4_0, Wq, xq, 512, 1024, 1, 1)
        n += 1
        dt = time.perf_counter() - t0
        if dt >= seconds:
            break
    return {"us_per_gemv": dt / n * 1e6, "cores": 1, "kind": "oracle",
            "sample": f"{n} x (Q8_0 act-quant + Q4_0 GEMV 512x1024, batch 1) in {dt:.1f} s"}


def run_reference(args):
    orc, Wq, x = oracle_gemv_sample()
    nt = orc.max_threads()

    def step():
        xq = orc.quantize(orc.Q8_K, x)
        orc.matmul_ref(orc.Q4_K, Wq, xq, GEMV_ROWS, GEMV_COLS, 1, nt)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    value = args.steps * Wq.nbytes / dt / 1e9
    sample = ("per step: Q8_K act-quant + Q4_K GEMV 4096x4096 batch 1, one of the 64 matrices of the "
              "workload's step (a bounded sample of it)")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": headline_config(args.gpus),
        "timing": "host perf_counter around the oracle on the CPU cores",
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": nt, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


# ---------------------------------------------------------------------- GPU

def run_gpu(args, world, rank):
    import numpy as np
    import torch

    from block_quantized_gb300 import gq, inputs

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    gq.load(build_if_missing=True)
    dev = torch.device("cuda", local)
    hbm_peak, bf16_peak, peak_src = measured_peaks()

    ranks = Ranks(dist, dev)

    def barrier():
        ranks.barrier()
        torch.cuda.synchronize()

    max_over_ranks = ranks.max

    s = torch.cuda.Stream(device=dev)

    def capture(fn):
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            fn()  # warm (module load, attribute cache) outside capture
            torch.cuda.synchronize()
            with torch.cuda.graph(graph, stream=s):
                fn()
        torch.cuda.synchronize()
        return graph

    def time_graph(graph, steps, warmup, clocks=None):
        with torch.cuda.stream(s):
            for _ in range(warmup):
                graph.replay()
            barrier()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            if clocks:
                clocks.start()
            e0.record(s)
            for _ in range(steps):
                graph.replay()
            e1.record(s)
            torch.cuda.synchronize()
            clk = clocks.stop() if clocks else None
            barrier()
        return max_over_ranks(e0.elapsed_time(e1) / 1e3), clk

    if args.only:
        fn = {"prefill": lambda: bench_prefill(gq, inputs, torch, np, dev, s, capture, time_graph, bf16_peak),
              "sweep": lambda: bench_batch_sweep(gq, inputs, torch, np, dev, s, capture, time_graph),
              "decode": lambda: bench_decode(gq, inputs, torch, np, dev, s, capture, time_graph, world),
              "stream": lambda: bench_stream(gq, inputs, torch, np, dev, s, capture, time_graph, hbm_peak,
                                             args.steps),
              "kv": lambda: bench_kv(gq, torch, dev, capture, time_graph, hbm_peak),
              "kv_q4_0": lambda: bench_kv(gq, torch, dev, capture, time_graph, hbm_peak, types=("q4_0",)),
              "q6k": lambda: bench_q6k(gq, inputs, torch, np, dev, capture, time_graph, hbm_peak,
                                       cpu=rank == 0 and world == 1 and not args.no_cpu),
              "q5k": lambda: bench_q6k(gq, inputs, torch, np, dev, capture, time_graph, hbm_peak,
                                       cpu=rank == 0 and world == 1 and not args.no_cpu, wtype=gq.Q5_K),
              "q4_0": lambda: bench_q4_0(gq, inputs, torch, np, dev, capture, time_graph,
                                         cpu=rank == 0 and world == 1 and not args.no_cpu),
              "q0_gemm": lambda: bench_q0_gemm(gq, inputs, torch, np, dev, capture, time_graph, bf16_peak)}
        if rank == 0:
            print(json.dumps({"only": args.only, "result": fn[args.only]()}))
        else:
            fn[args.only]()
        return

    # ---- headline workload: 64 distinct Q4_K 4096x4096 matrices per step
    W, x0 = inputs.gemv_q4_k(0)
    Wq1 = gq.quantize(gq.Q4_K, torch.from_numpy(W).to(dev))
    del W
    Wall = Wq1.reshape(1, -1).repeat(COPIES, 1)          # [64, 4096 * 2304] distinct copies
    g = inputs.rng(1)
    X = torch.from_numpy(np.concatenate([x0[None], inputs.normal(g, (COPIES - 1, GEMV_COLS))])).to(dev)
    XQ = torch.empty(COPIES, GEMV_COLS // 256 * 276, dtype=torch.uint8, device=dev)
    Y = torch.empty(COPIES, GEMV_ROWS, dtype=torch.float32, device=dev)
    w_bytes = GEMV_ROWS * Q4K_ROW_BYTES

    FLAGS = gq.FLAG_W_STATIC  # model weights: written once, never by a kernel in flight

    def step_body():
        # the hot path per matrix: fp32 activations -> Q8_K (in-kernel) -> GEMV
        for i in range(COPIES):
            gq.gq_matmul_f32(gq.Q4_K, Wall[i], X[i], Y[i], GEMV_ROWS, GEMV_COLS, 1, FLAGS)

    def step_unfused():
        for i in range(COPIES):
            gq.gq_quantize_rows_async(gq.Q8_K, X[i], XQ[i], GEMV_COLS)
            gq.gq_matmul_ex(gq.Q4_K, Wall[i], XQ[i], Y[i], GEMV_ROWS, GEMV_COLS, 1,
                            gq.PATH_GEMV, FLAGS)

    step_graph = capture(step_body)
    sampler = ClockSampler(local)
    t_total, clk = time_graph(step_graph, args.steps, max(3, args.warmup), sampler)
    ms_step = t_total / args.steps * 1e3
    value = whole_job_rate(args.steps * COPIES * w_bytes, world, t_total) / 1e9
    if not torch.isfinite(Y).all():
        raise RuntimeError("non-finite GEMV output")

    # the step is nothing but launches of the fused GEMV kernel, so its
    # per-launch duration is the step time over the launches in it
    per_launch = t_total / (args.steps * COPIES)
    alg_bytes = w_bytes + GEMV_COLS * 4 + GEMV_ROWS * 4
    achieved = alg_bytes / per_launch / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                "frac": achieved / hbm_peak, "traffic": kernel_traffic("gemv_q4k_fused"),
                "kernel": "gemv_kernel<Q4_K, NB=1, fused fp32 activations>",
                "peak_source": peak_src, "launch_us": per_launch * 1e6,
                "alg_bytes_per_launch": alg_bytes,
                "note": "dependent back-to-back launches of one 9.44 MB matrix each"}

    # the unfused pair (standalone act-quant kernel + GEMV) for comparison
    k_steps = max(50, args.steps // 4)
    t_u, _ = time_graph(capture(step_unfused), k_steps, 5)
    unfused = {"value": world * k_steps * COPIES * w_bytes / t_u / 1e9, "unit": "GB/s",
               "us_per_matrix": t_u / (k_steps * COPIES) * 1e6}

    # streaming capability: the same 64 matrices as one tall GEMV launch
    def tall():
        gq.gq_matmul_f32(gq.Q4_K, Wall, X[0], Yt, GEMV_ROWS * COPIES, GEMV_COLS, 1, FLAGS)
    Yt = torch.empty(1, GEMV_ROWS * COPIES, dtype=torch.float32, device=dev)
    t_t, _ = time_graph(capture(tall), k_steps, 5)
    streaming = {"achieved": COPIES * w_bytes / (t_t / k_steps) / 1e9, "unit": "GB/s",
                 "frac": COPIES * w_bytes / (t_t / k_steps) / 1e9 / hbm_peak,
                 "workload": "one launch over 262144 x 4096 Q4_K rows (604 MB)"}

    # ---- end to end with host buffers: pinned H2D of each x, D2H of each y
    Xh = X.cpu().pin_memory()
    Yh = torch.empty(COPIES, GEMV_ROWS, dtype=torch.float32).pin_memory()
    Xd = torch.empty_like(X)

    def e2e_body():
        Xd.copy_(Xh, non_blocking=True)
        for i in range(COPIES):
            gq.gq_matmul_f32(gq.Q4_K, Wall[i], Xd[i], Y[i], GEMV_ROWS, GEMV_COLS, 1, FLAGS)
        Yh.copy_(Y, non_blocking=True)

    e2e_graph = capture(e2e_body)
    e2e_steps = max(20, args.steps // 4)
    t_e2e, _ = time_graph(e2e_graph, e2e_steps, 3)
    e2e = {"value": world * e2e_steps * COPIES * w_bytes / t_e2e / 1e9, "unit": "GB/s",
           "h2d_bytes_per_step": COPIES * GEMV_COLS * 4, "d2h_bytes_per_step": COPIES * GEMV_ROWS * 4,
           "how": "CUDA graph of the public calls: one pinned H2D of the 64 activation vectors, "
                  "64 x gq_matmul_f32, one D2H of the 64 outputs"}
    del Wall, Xh, Yh, Yt

    def leg(fn, *a, **k):
        # a secondary workload that raises is reported in the line as an
        # error; the headline figures above stand
        try:
            return fn(*a, **k)
        except Exception as e:  # noqa: BLE001
            return {"error": f"{type(e).__name__}: {e}"}

    extras = {}
    if not args.quick:
        cpu_leg = rank == 0 and world == 1 and not args.no_cpu
        extras["decode"] = leg(bench_decode, gq, inputs, torch, np, dev, s, capture, time_graph, world)
        extras["batch_sweep"] = leg(bench_batch_sweep, gq, inputs, torch, np, dev, s, capture, time_graph)
        extras["prefill"] = leg(bench_prefill, gq, inputs, torch, np, dev, s, capture, time_graph, bf16_peak)
        extras["kv_cache"] = leg(bench_kv, gq, torch, dev, capture, time_graph, hbm_peak)
        extras["q6k"] = leg(bench_q6k, gq, inputs, torch, np, dev, capture, time_graph, hbm_peak, cpu=cpu_leg)
        extras["q5k"] = leg(bench_q6k, gq, inputs, torch, np, dev, capture, time_graph, hbm_peak, cpu=cpu_leg,
                            wtype=gq.Q5_K)
        extras["q4_0_512x1024"] = leg(bench_q4_0, gq, inputs, torch, np, dev, capture, time_graph, cpu=cpu_leg)
        extras["q0_gemm"] = leg(bench_q0_gemm, gq, inputs, torch, np, dev, capture, time_graph, bf16_peak)

    cpu = cpu_configs = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = run_cpu_baseline()
        if not args.quick:
            cpu_configs = leg(run_cpu_configs)

    if rank == 0:
        line = {
            "metric": METRIC,
            "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": max(3, args.warmup), "ms_per_step": ms_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "int8xint4->int32,fp32",
            "data": "synthetic",
            "config": headline_config(world),
            "timing": "CUDA graph, CUDA events",
            "pct_of_hbm_peak": value / hbm_peak * 100.0,
            "roofline": roofline,
            "roofline_streaming": streaming,
            "unfused_step": unfused,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": args.steps * COPIES,
            "clocks": clk,
        }
        line.update(extras)
        line["cpu_baseline_configs"] = cpu_configs
        # the headline figures of every workload once more, last, in a few
        # hundred bytes: records that keep only the end of the line keep these
        line["summary"] = summary_keys(line)
        print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()


def summary_keys(line: dict) -> dict:
    """A compact digest of the line's workloads (rounded), emitted as its last
    key."""
    def get(d, *path):
        for k in path:
            if not isinstance(d, dict) or k not in d:
                return None
            d = d[k]
        return d

    def r(v, n=3):
        return None if v is None else round(float(v), n)

    out = {"gemv_4096_gbps": r(line.get("value"), 1), "gemv_4096_frac": r(get(line, "roofline", "frac")),
           "gemv_4096_launch_us": r(get(line, "roofline", "launch_us")),
           "stream_frac": r(get(line, "roofline_streaming", "frac")),
           "decode_tok_s": r(get(line, "decode", "tok_s"), 1),
           "decode_fused_weights_tok_s": r(get(line, "decode", "fused_weights", "tok_s"), 1),
           "decode_head_us": r(get(line, "decode", "head_q8_0", "us_per_token"), 1),
           "prefill_ms": r(get(line, "prefill", "results", "mma", "ms"), 4),
           "prefill_tops": r(get(line, "prefill", "results", "mma", "tops"), 1),
           "prefill_frac": r(get(line, "prefill", "results", "mma", "roofline", "frac"))}
    sweep = get(line, "batch_sweep", "results")
    if isinstance(sweep, dict):
        out["sweep_us_gemv_mma_skinny"] = {b: [r(get(v, "gemv", "us"), 1), r(get(v, "mma", "us"), 1),
                                               r(get(v, "skinny", "us"), 1)] for b, v in sweep.items()}
        tc_wins = [int(b) for b, v in sweep.items() if v.get("faster") in ("mma", "skinny")]
        out["sweep_crossover_batch"] = min(tc_wins) if tc_wins else None
    for t in ("q4_0", "q8_0"):
        out[f"prefill_{t}_tops"] = r(get(line, "q0_gemm", t, "prefill_28672x8192x512", "mma", "tops"), 1)
        out[f"prefill_{t}_frac"] = r(get(line, "q0_gemm", t, "prefill_28672x8192x512", "mma", "roofline", "frac"))
        sw0 = get(line, "q0_gemm", t, "sweep_14336x4096")
        if isinstance(sw0, dict):
            out[f"sweep_{t}_us_gemv_mma_skinny"] = {
                b: [r(get(v, "gemv", "us"), 1), r(get(v, "mma", "us"), 1), r(get(v, "skinny", "us"), 1)]
                for b, v in sw0.items()}
    out["q6k_frac"] = r(get(line, "q6k", "frac"))
    out["q5k_frac"] = r(get(line, "q5k", "frac"))
    out["q5k_stream_frac"] = r(get(line, "q5k", "streaming", "frac"))
    out["kv_q8_0_frac"] = r(get(line, "kv_cache", "q8_0", "frac"))
    out["cpu_oracle_gbps_all_cores"] = r(get(line, "cpu_baseline", "value"))
    out["cpu_oracle_decode_tok_s"] = r(get(line, "cpu_baseline_configs", "decode_7b", "all_cores", "tok_s"), 4)
    return out


def bench_stream(gq, inputs, torch, np, dev, s, capture, time_graph, hbm_peak, steps):
    """Streaming capability of the fused Q4_K GEMV: one launch over 64
    concatenated 4096x4096 matrices (262144 x 4096, 604 MB), timed over
    back-to-back launches."""
    W, x0 = inputs.gemv_q4_k(0)
    Wq1 = gq.quantize(gq.Q4_K, torch.from_numpy(W).to(dev))
    del W
    Wall = Wq1.reshape(1, -1).repeat(COPIES, 1)
    x = torch.from_numpy(x0).to(dev)
    y = torch.empty(1, GEMV_ROWS * COPIES, dtype=torch.float32, device=dev)

    def body():
        gq.gq_matmul_f32(gq.Q4_K, Wall, x, y, GEMV_ROWS * COPIES, GEMV_COLS, 1, gq.FLAG_W_STATIC)

    k = max(2, min(steps, 50))
    t, _ = time_graph(capture(body), k, 2)
    gbs = Wall.numel() / (t / k) / 1e9
    del Wall
    torch.cuda.empty_cache()
    return {"workload": "one launch over 262144 x 4096 Q4_K rows (604 MB)", "us": t / k * 1e6,
            "weight_gbps": gbs, "frac": gbs / hbm_peak}


def bench_q4_0(gq, inputs, torch, np, dev, capture, time_graph, cpu=False):
    """The 512x1024 Q4_0 x Q8_0 GEMV at batch 1 (295 KB of weights, resident
    in L2, so latency-bound: time reported, not graded against a roofline):
    back-to-back dependent launches on a pre-quantized vector, and with the
    activation quantize fused into each launch."""
    rows, cols, n = 512, 1024, 256
    W, x = inputs.gemv_q4_0(0)
    Wq = gq.quantize(gq.Q4_0, torch.from_numpy(W).to(dev))
    xd = torch.from_numpy(x).to(dev)
    xq = gq.quantize(gq.Q8_0, xd)
    y = torch.empty(1, rows, dtype=torch.float32, device=dev)

    def chain():
        for _ in range(n):
            gq.gq_matmul(gq.Q4_0, Wq, xq, y, rows, cols, 1)

    def chain_fused():
        for _ in range(n):
            gq.gq_matmul_f32(gq.Q4_0, Wq, xd, y, rows, cols, 1, gq.FLAG_W_STATIC)

    k = 50
    t, _ = time_graph(capture(chain), k, 3)
    tf, _ = time_graph(capture(chain_fused), k, 3)
    if not torch.isfinite(y).all():
        raise RuntimeError("non-finite Q4_0 GEMV output")
    return {"workload": "Q4_0 x Q8_0 GEMV 512x1024 batch 1 (weights resident in L2)",
            "us_per_gemv": t / (k * n) * 1e6, "us_per_gemv_fused_quantize": tf / (k * n) * 1e6,
            "weight_bytes": Wq.numel(), "cpu_baseline": run_cpu_q4_0() if cpu else None}


def bench_q6k(gq, inputs, torch, np, dev, capture, time_graph, hbm_peak, cpu=False, wtype=None):
    """Q6_K (or, with wtype, Q5_K) x Q8_K GEMV on the 4096x4096 row-spread +
    outlier weights: 64 distinct copies (203 / 185 MB, larger than L2) as
    dependent back-to-back launches on pre-quantized activations (weights
    marked static, as the headline's; also without the flag, and from fp32
    activations quantized inside the kernel), and the same bytes as one tall
    launch (262144 x 4096 rows)."""
    wt = gq.Q6_K if wtype is None else wtype
    name = "Q6_K" if wt == gq.Q6_K else "Q5_K"
    W, _ = inputs.gemv_q4_k(0)
    Wq1 = gq.quantize(wt, torch.from_numpy(W).to(dev))
    del W
    Wall = Wq1.reshape(1, -1).repeat(COPIES, 1)
    X = torch.from_numpy(inputs.normal(inputs.rng(2), (COPIES, GEMV_COLS))).to(dev)
    XQ = gq.quantize(gq.Q8_K, X)
    Y = torch.empty(COPIES, GEMV_ROWS, dtype=torch.float32, device=dev)
    Yt = torch.empty(1, GEMV_ROWS * COPIES, dtype=torch.float32, device=dev)
    w_bytes = Wq1.numel()

    def chain():
        # model weights: written once, never by a kernel in flight
        for i in range(COPIES):
            gq.gq_matmul_ex(wt, Wall[i], XQ[i], Y[i], GEMV_ROWS, GEMV_COLS, 1, gq.PATH_AUTO, gq.FLAG_W_STATIC)

    def chain_plain():
        for i in range(COPIES):
            gq.gq_matmul(wt, Wall[i], XQ[i], Y[i], GEMV_ROWS, GEMV_COLS, 1)

    def chain_fused():
        # fp32 activations quantized to Q8_K inside the GEMV (no separate pass)
        for i in range(COPIES):
            gq.gq_matmul_f32(wt, Wall[i], X[i], Y[i], GEMV_ROWS, GEMV_COLS, 1, gq.FLAG_W_STATIC)

    def tall():
        gq.gq_matmul(wt, Wall, XQ[0], Yt, GEMV_ROWS * COPIES, GEMV_COLS, 1)

    k = 200
    t_c, _ = time_graph(capture(chain), k, 5)
    t_p, _ = time_graph(capture(chain_plain), k, 5)
    t_f, _ = time_graph(capture(chain_fused), k, 5)
    # small batches through gq_matmul's own choice: up to eight vectors share
    # one pass of the GEMV over each matrix; Q5_K takes the warp-level
    # tensor-core kernel from batch 16 on these 4096 rows
    Yb = torch.empty(32, GEMV_ROWS, dtype=torch.float32, device=dev)
    batch_us = {}
    for nb in (2, 4, 8, 16, 32):
        def chain_b():
            for i in range(COPIES):
                gq.gq_matmul_ex(wt, Wall[i], XQ[:nb], Yb, GEMV_ROWS, GEMV_COLS, nb, gq.PATH_AUTO,
                                gq.FLAG_W_STATIC)
        t_b, _ = time_graph(capture(chain_b), 50, 3)
        batch_us[str(nb)] = t_b / (50 * COPIES) * 1e6
    t_t, _ = time_graph(capture(tall), 50, 3)
    if not (torch.isfinite(Y).all() and torch.isfinite(Yt).all()):
        raise RuntimeError(f"non-finite {name} GEMV output")
    per = t_c / (k * COPIES)
    alg = w_bytes + GEMV_COLS // 256 * 276 + GEMV_ROWS * 4
    tall_s = t_t / 50
    del Wall, XQ
    torch.cuda.empty_cache()
    return {"workload": f"{name} x Q8_K GEMV 4096x4096 batch 1, 64 distinct matrices "
                        f"({COPIES * w_bytes / 1e6:.0f} MB)",
            "cpu_baseline": run_cpu_q6k(wtype=wt) if cpu else None,
            "kernel": f"gemv_{name.lower().replace('_', '')}_kernel (whole-row bulk copies, per-warp ring)",
            "traffic": kernel_traffic("gemv_" + name.lower().replace("_", "")),
            "launch_us": per * 1e6, "alg_bytes_per_launch": alg, "weight_gbps": w_bytes / per / 1e9,
            "achieved": alg / per / 1e9, "frac": alg / per / 1e9 / hbm_peak,
            "launch_us_without_w_static": t_p / (k * COPIES) * 1e6,
            "batch_launch_us": batch_us,
            "fused_f32": {"launch_us": t_f / (k * COPIES) * 1e6,
                          "frac": (w_bytes + GEMV_COLS * 4 + GEMV_ROWS * 4) / (t_f / (k * COPIES)) / 1e9
                          / hbm_peak},
            "streaming": {"workload": f"one launch over 262144 x 4096 {name} rows "
                                      f"({COPIES * w_bytes / 1e6:.0f} MB)",
                          "us": tall_s * 1e6, "weight_gbps": COPIES * w_bytes / tall_s / 1e9,
                          "frac": COPIES * w_bytes / tall_s / 1e9 / hbm_peak}}


def bench_kv(gq, torch, dev, capture, time_graph, hbm_peak, types=("q8_0", "q4_0")):
    """Quantized KV cache at 7B shape: 32 heads x 4096 positions x 128, keys
    as Q8_0 and as Q4_0.  Scores of one query against every cached key,
    rotated over 16 layer caches (larger than L2) and timed back to back; and
    the append of one position (all heads)."""
    n_heads, capacity, head_dim, layers = 32, 4096, 128, 16
    out = {"workload": f"{n_heads} heads x {capacity} positions x {head_dim}, {layers} layer caches"}
    g = torch.Generator(device=dev).manual_seed(5)
    q = torch.randn(n_heads, head_dim, device=dev, generator=g)
    x = torch.randn(n_heads, head_dim, device=dev, generator=g)
    for name, t in (("q8_0", gq.Q8_0), ("q4_0", gq.Q4_0)):
        if name not in types:
            continue
        caches = [gq.kv_cache(t, n_heads, capacity, head_dim, dev) for _ in range(layers)]
        keys = torch.randn(capacity, n_heads, head_dim, device=dev, generator=g)
        for p in range(capacity):
            gq.gq_kv_append(t, keys[p], caches[0], n_heads, head_dim, capacity, p)
        for c in caches[1:]:
            c.copy_(caches[0])
        del keys
        sc = torch.empty(n_heads, capacity, dtype=torch.float32, device=dev)

        def body():
            for c in caches:
                gq.gq_kv_scores(t, c, q, sc, n_heads, head_dim, capacity, capacity)

        t_s, _ = time_graph(capture(body), 20, 3)
        per = t_s / (20 * layers)
        kbytes = caches[0].numel()

        def app():
            for i, c in enumerate(caches):
                gq.gq_kv_append(t, x, c, n_heads, head_dim, capacity, i)

        t_a, _ = time_graph(capture(app), 20, 3)
        out[name] = {"scores_us": per * 1e6, "key_bytes": kbytes, "key_gbps": kbytes / per / 1e9,
                     "frac": kbytes / per / 1e9 / hbm_peak, "append_us": t_a / (20 * layers) * 1e6,
                     "traffic": kernel_traffic("kv_scores_" + name)}
        del caches
        torch.cuda.empty_cache()
    return out


def bench_decode(gq, inputs, torch, np, dev, s, capture, time_graph, world):
    """7B-shape decode: 32 layers x (wq, wk, wv, wo, w1, w3, w2) Q4_K GEMVs
    with their activation quantizes, then the Q8_0 output head; one token =
    one pass.  Layer weights are 32 device copies of one generated layer.
    Timed three ways: with the standalone act-quant kernel before each group
    of products sharing an input; with the act-quant fused into every GEMV;
    and fused, with wq|wk|wv and w1|w3 stored as concatenated matrices so
    each group sharing an input is one launch."""
    ws, _ = inputs.decode_weights(0)
    layer = {}
    for name, r, c in inputs.DECODE_LAYER:
        layer[name] = gq.quantize(gq.Q4_K, torch.from_numpy(ws[name]).to(dev))
    hname, hr, hc = inputs.DECODE_HEAD
    head = gq.quantize(gq.Q8_0, torch.from_numpy(ws[hname]).to(dev))
    del ws
    L = inputs.DECODE_LAYERS
    layers = [{k: v.clone() for k, v in layer.items()} for _ in range(L)]
    del layer
    g = inputs.rng(2)
    xin = {k: torch.from_numpy(inputs.normal(g, (c,))).to(dev)
           for k, c in (("attn", 4096), ("o", 4096), ("ffn", 4096), ("down", 11008), ("head", 4096))}
    xq = {k: torch.empty(v.numel() // 256 * 276, dtype=torch.uint8, device=dev) for k, v in xin.items()}
    xq["head"] = torch.empty(4096 // 32 * 34, dtype=torch.uint8, device=dev)
    outs = {name: torch.empty(r, dtype=torch.float32, device=dev) for name, r, c in inputs.DECODE_LAYER}
    yh = torch.empty(hr, dtype=torch.float32, device=dev)
    F = gq.FLAG_W_STATIC
    G = gq.PATH_GEMV

    def token_unfused():
        for lw in layers:
            gq.gq_quantize_rows_async(gq.Q8_K, xin["attn"], xq["attn"], 4096)
            for nm in ("wq", "wk", "wv"):
                gq.gq_matmul_ex(gq.Q4_K, lw[nm], xq["attn"], outs[nm], 4096, 4096, 1, G, F)
            gq.gq_quantize_rows_async(gq.Q8_K, xin["o"], xq["o"], 4096)
            gq.gq_matmul_ex(gq.Q4_K, lw["wo"], xq["o"], outs["wo"], 4096, 4096, 1, G, F)
            gq.gq_quantize_rows_async(gq.Q8_K, xin["ffn"], xq["ffn"], 4096)
            gq.gq_matmul_ex(gq.Q4_K, lw["w1"], xq["ffn"], outs["w1"], 11008, 4096, 1, G, F)
            gq.gq_matmul_ex(gq.Q4_K, lw["w3"], xq["ffn"], outs["w3"], 11008, 4096, 1, G, F)
            gq.gq_quantize_rows_async(gq.Q8_K, xin["down"], xq["down"], 11008)
            gq.gq_matmul_ex(gq.Q4_K, lw["w2"], xq["down"], outs["w2"], 4096, 11008, 1, G, F)
        gq.gq_quantize_rows_async(gq.Q8_0, xin["head"], xq["head"], 4096)
        gq.gq_matmul_ex(gq.Q8_0, head, xq["head"], yh, hr, hc, 1, G, F)

    def token_fused():
        for lw in layers:
            for nm, x in (("wq", "attn"), ("wk", "attn"), ("wv", "attn"), ("wo", "o"),
                          ("w1", "ffn"), ("w3", "ffn"), ("w2", "down")):
                r, c = lw[nm].shape[0], xin[x].numel()
                gq.gq_matmul_f32(gq.Q4_K, lw[nm], xin[x], outs[nm], r, c, 1, F)
        gq.gq_matmul_f32(gq.Q8_0, head, xin["head"], yh, hr, hc, 1, F)

    # the same weights stored as fused matrices -- wq|wk|wv (12288 rows) and
    # w1|w3 (22016 rows) concatenated by rows -- so each group sharing an input
    # is one launch: 4 products per layer
    fused_w = [{"qkv": torch.cat([lw["wq"], lw["wk"], lw["wv"]]), "wo": lw["wo"],
                "w13": torch.cat([lw["w1"], lw["w3"]]), "w2": lw["w2"]} for lw in layers]
    y_qkv = torch.empty(3 * 4096, dtype=torch.float32, device=dev)
    y_13 = torch.empty(2 * 11008, dtype=torch.float32, device=dev)

    def token_grouped():
        for lw in fused_w:
            gq.gq_matmul_f32(gq.Q4_K, lw["qkv"], xin["attn"], y_qkv, 3 * 4096, 4096, 1, F)
            gq.gq_matmul_f32(gq.Q4_K, lw["wo"], xin["o"], outs["wo"], 4096, 4096, 1, F)
            gq.gq_matmul_f32(gq.Q4_K, lw["w13"], xin["ffn"], y_13, 2 * 11008, 4096, 1, F)
            gq.gq_matmul_f32(gq.Q4_K, lw["w2"], xin["down"], outs["w2"], 4096, 11008, 1, F)
        gq.gq_matmul_f32(gq.Q8_0, head, xin["head"], yh, hr, hc, 1, F)

    bytes_tok = sum(v.numel() for v in layers[0].values()) * L + head.numel()
    res = {"weight_bytes_per_token": bytes_tok, "tokens_timed": 40,
           "workload": "7B shapes: 32 x (4 x 4096x4096, 2 x 11008x4096, 4096x11008) Q4_K + "
                       "32000x4096 Q8_0 head, batch 1"}
    for name, fn, launches in (("unfused", token_unfused, 32 * 11 + 2), ("fused", token_fused, 32 * 7 + 1),
                               ("fused_weights", token_grouped, 32 * 4 + 1)):
        t, _ = time_graph(capture(fn), 40, 3)
        per_tok = t / 40
        res[name] = {"tok_s": world / per_tok, "ms_per_token": per_tok * 1e3,
                     "weight_gbps": bytes_tok / per_tok / 1e9, "launches_per_token": launches}
    res["tok_s"] = max(res["unfused"]["tok_s"], res["fused"]["tok_s"], res["fused_weights"]["tok_s"])

    # the Q8_0 output head alone (139 MB, larger than L2), fused act-quantize,
    # as dependent launches: its share of a token
    def head_chain():
        for _ in range(8):
            gq.gq_matmul_f32(gq.Q8_0, head, xin["head"], yh, hr, hc, 1, F)
    t_h, _ = time_graph(capture(head_chain), 10, 2)
    per_head = t_h / 80
    res["head_q8_0"] = {"us_per_token": per_head * 1e6, "weight_gbps": head.numel() / per_head / 1e9,
                        "share_of_token": per_head / res["fused_weights"]["ms_per_token"] * 1e3}
    del layers, head, fused_w
    torch.cuda.empty_cache()
    return res


def bench_batch_sweep(gq, inputs, torch, np, dev, s, capture, time_graph):
    """Q4_K 14336x4096 at batch 1..64 through the three kernel families: the
    GEMV, the tcgen05 kernel (its activation pack kernel included) and the
    warp-level tensor-core kernel (weights rotated over 8 copies, 264 MB > L2)."""
    rows, cols, copies = 14336, 4096, 8
    W, X = inputs.gemm_q4_k(0, rows, cols, 64)
    Wq = gq.quantize(gq.Q4_K, torch.from_numpy(W).to(dev))
    del W
    Wc = Wq.reshape(1, -1).repeat(copies, 1)
    Xq = gq.quantize(gq.Q8_K, torch.from_numpy(X).to(dev))
    Y = torch.empty(64, rows, dtype=torch.float32, device=dev)
    wsb = torch.empty(gq.gq_matmul_workspace_bytes(gq.Q4_K, rows, cols, 64), dtype=torch.uint8, device=dev)
    wbytes = Wq.numel()
    out = {}
    for b in (1, 2, 4, 8, 16, 32, 64):
        res = {}
        for pname, path in (("gemv", gq.PATH_GEMV), ("mma", gq.PATH_MMA), ("skinny", gq.PATH_SKINNY)):
            def body():
                for i in range(copies):
                    gq.gq_matmul_ws(gq.Q4_K, Wc[i], Xq, Y, rows, cols, b, path, gq.FLAG_W_STATIC,
                                    wsb, wsb.numel())
            steps = 20
            t, _ = time_graph(capture(body), steps, 3)
            per = t / (steps * copies)
            res[pname] = {"us": per * 1e6, "weight_gbps": wbytes / per / 1e9,
                          "tops": 2.0 * rows * cols * b / per / 1e12}
            if pname == "skinny" and b == 16:
                res[pname]["traffic"] = kernel_traffic("skinny_q4k_b16")
        res["faster"] = min(("gemv", "mma", "skinny"), key=lambda k: res[k]["us"])
        out[str(b)] = res
    del Wc, Wq, Xq, Y, wsb
    torch.cuda.empty_cache()
    return {"rows": rows, "cols": cols, "results": out}


def bench_prefill(gq, inputs, torch, np, dev, s, capture, time_graph, bf16_peak):
    """Q4_K 28672x8192 weights x 512 Q8_K columns (70B FFN shape)."""
    rows, cols, batch = 28672, 8192, 512
    W, X = inputs.gemm_q4_k(0, rows, cols, batch)
    Wq = gq.quantize(gq.Q4_K, torch.from_numpy(W).to(dev))
    del W
    Xq = gq.quantize(gq.Q8_K, torch.from_numpy(X).to(dev))
    Y = torch.empty(batch, rows, dtype=torch.float32, device=dev)
    wsb = torch.empty(gq.gq_matmul_workspace_bytes(gq.Q4_K, rows, cols, batch), dtype=torch.uint8, device=dev)
    res = {}
    for pname, path, steps in (("mma", gq.PATH_MMA, 20), ("gemv", gq.PATH_GEMV, 3)):
        def body():
            gq.gq_matmul_ws(gq.Q4_K, Wq, Xq, Y, rows, cols, batch, path, gq.FLAG_W_STATIC, wsb, wsb.numel())
        t, _ = time_graph(capture(body), steps, 2)
        per = t / steps
        tops = 2.0 * rows * cols * batch / per / 1e12
        res[pname] = {"ms": per * 1e3, "tops": tops}
    # gq_matmul itself (no workspace): the warp-level kernel over 64-column chunks
    def body_nows():
        gq.gq_matmul(gq.Q4_K, Wq, Xq, Y, rows, cols, batch)
    t, _ = time_graph(capture(body_nows), 5, 2)
    res["gq_matmul_no_workspace"] = {"ms": t / 5 * 1e3, "tops": 2.0 * rows * cols * batch / (t / 5) / 1e12}
    res["mma"]["roofline"] = {"bound": "tensor", "achieved": res["mma"]["tops"], "peak": bf16_peak,
                              "unit": "TFLOP/s", "frac": res["mma"]["tops"] / bf16_peak,
                              "traffic": kernel_traffic("mma_q4k"),
                              "note": "int ops counted as 2 per multiply-add; fp16 tensor kind"}
    del Wq, Xq, Y, wsb
    torch.cuda.empty_cache()
    return {"rows": rows, "cols": cols, "batch": batch, "results": res}


def bench_q0_gemm(gq, inputs, torch, np, dev, capture, time_graph, bf16_peak):
    """Q4_0 / Q8_0 weights x Q8_0 columns on the tensor-core kernel that
    needs no workspace (what gq_matmul runs from batch 16): the prefill shape
    28672x8192 x 512 against the GEMV, and 14336x4096 at batch 4..64 (weights
    rotated over copies larger than L2) against the GEMV and the warp-level
    kernel."""
    out = {}
    big = inputs.gemm_q4_k(0, 28672, 8192, 512)
    mid = inputs.gemm_q4_k(0, 14336, 4096, 64)
    for name, wt in (("q4_0", gq.Q4_0), ("q8_0", gq.Q8_0)):
        rows, cols, batch = 28672, 8192, 512
        Wq = gq.quantize(wt, torch.from_numpy(big[0]).to(dev))
        Xq = gq.quantize(gq.Q8_0, torch.from_numpy(big[1]).to(dev))
        Y = torch.empty(batch, rows, dtype=torch.float32, device=dev)
        res = {}
        for pname, path, steps in (("mma", gq.PATH_MMA, 20), ("gemv", gq.PATH_GEMV, 3)):
            def body():
                gq.gq_matmul_path(wt, Wq, Xq, Y, rows, cols, batch, path)
            t, _ = time_graph(capture(body), steps, 2)
            per = t / steps
            res[pname] = {"ms": per * 1e3, "tops": 2.0 * rows * cols * batch / per / 1e12}
        res["mma"]["roofline"] = {"bound": "tensor", "achieved": res["mma"]["tops"], "peak": bf16_peak,
                                  "unit": "TFLOP/s", "frac": res["mma"]["tops"] / bf16_peak,
                                  "traffic": kernel_traffic("mma_q0_" + name) if name == "q4_0" else None,
                                  "note": "int ops counted as 2 per multiply-add; fp16 tensor kind"}
        del Wq, Xq, Y
        rows, cols = 14336, 4096
        Wq = gq.quantize(wt, torch.from_numpy(mid[0]).to(dev))
        copies = max(2, int(np.ceil(300e6 / Wq.numel())))
        Wc = Wq.reshape(1, -1).repeat(copies, 1)
        Xq = gq.quantize(gq.Q8_0, torch.from_numpy(mid[1]).to(dev))
        Y = torch.empty(64, rows, dtype=torch.float32, device=dev)
        sweep = {}
        for b in (4, 8, 16, 32, 64):
            r = {}
            for pname, path in (("gemv", gq.PATH_GEMV), ("mma", gq.PATH_MMA), ("skinny", gq.PATH_SKINNY)):
                def body():
                    for i in range(copies):
                        gq.gq_matmul_ex(wt, Wc[i], Xq, Y, rows, cols, b, path, gq.FLAG_W_STATIC)
                t, _ = time_graph(capture(body), 10, 3)
                per = t / (10 * copies)
                r[pname] = {"us": per * 1e6, "weight_gbps": Wq.numel() / per / 1e9}
                if pname == "skinny" and b == 16 and name == "q4_0":
                    r[pname]["traffic"] = kernel_traffic("skinny_q0_q4_0_b16")
            r["faster"] = min(("gemv", "mma", "skinny"), key=lambda k: r[k]["us"])
            sweep[str(b)] = r
        del Wc, Wq, Xq, Y
        torch.cuda.empty_cache()
        out[name] = {"prefill_28672x8192x512": res, "sweep_14336x4096": sweep}
    return out


if __name__ == "__main__":
    main()
