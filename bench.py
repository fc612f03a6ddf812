"""Benchmark: decode GEMV on Q5_K weights, N = K = 4096, M in {1, 2, 4}, fused residual.

One step = the three GEMV calls (M = 1, 2, 4; bf16 activations, bf16 residual,
bf16 output) on three different copies of the weight, so every call streams its
11,534,336 weight bytes from HBM: the copies rotate over more than twice the L2
size.  Steps are captured in CUDA graphs and replayed; the timed region is
exactly K steps, bracketed by a barrier and a device synchronization, timed
with CUDA events on the launching stream.

Printed JSON line (rank 0): value = weight GB/s over the whole job, plus
  e2e         the same steps fed from pinned host buffers (x and residual copied
              in, y copied out inside the timed region);
  roofline    the GEMV kernel's algorithmic bytes per launch / average launch
              time, against the measured HBM copy bandwidth;
  cpu_baseline the CPU oracle (int8-path restatement) on a bounded sample;
  clocks      SM clock and throttle reasons sampled during the timed region;
  prefill     tensor-core GEMM figures for the prefill shapes (context).
`--impl reference` times the CPU oracle instead (the reference arm).
Multi-GPU runs (torchrun) are independent replicas: every rank runs the same
workload on its own GPU and value sums over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

N, K = 4096, 4096
MS = (1, 2, 4)
QTYPE = 13  # Q5_K
ROW_BYTES = K // 256 * 176
W_BYTES = N * ROW_BYTES                      # 11,534,336
METRIC = "decode GEMV weight GB/s (% of HBM peak); prefill GEMM TFLOPS (% of TC peak)"
WORKLOAD = "q5_k_gemv_4096x4096_residual_m1_m2_m4"


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# ------------------------------------------------------------------ CPU arm (the oracle)

def cpu_oracle_run(steps: int, rows: int):
    """Run the CPU oracle's int8-path GEMV over `rows` weight rows for each M in
    MS, `steps` times; returns (seconds, weight bytes processed, threads)."""
    import gguf_synth as syn
    from oracle import gguf_oracle as O
    rs = syn.rng(1001)
    w = syn.weight_blocks(rs, QTYPE, rows, K)
    xs = {m: O.bf16_bits_to_f32(syn.normal(rs, (m, K), "bf16")) for m in MS}
    rr = {m: O.bf16_bits_to_f64(syn.normal(rs, (m, rows), "bf16")) for m in MS}
    t0 = time.perf_counter()
    for _ in range(steps):
        for m in MS:
            O.gemv_int8_path(w, QTYPE, rows, K, xs[m], rr[m])
    dt = time.perf_counter() - t0
    return dt, steps * len(MS) * rows * ROW_BYTES, 1


def cpu_baseline(sample_steps: int = 12):
    dt, nbytes, threads = cpu_oracle_run(sample_steps, N)
    return {"value": nbytes / dt / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{sample_steps} step(s) of the full workload: Q5_K 4096x4096 at M=1,2,4 "
                      f"through the numpy int8-path oracle, single thread ({dt:.1f} s)"}


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    steps = max(1, args.steps)
    for _ in range(max(0, min(args.warmup, 1))):
        cpu_oracle_run(1, 512)
    dt, nbytes, threads = cpu_oracle_run(steps, 1024)
    value = nbytes / dt / 1e9
    per_step = dt / steps
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws, "steps": steps,
        "warmup": args.warmup, "ms_per_step": per_step * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int8", "data": "synthetic",
        "config": {"workload": WORKLOAD, "N": N, "K": K, "M": list(MS), "qtype": "Q5_K",
                   "sample_rows": 1024},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": f"each step: 1024 of the 4096 weight rows at M=1,2,4 through the numpy "
                                   f"int8-path oracle, single thread"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [c.strip() for c in line.split(",")]))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)

    def summary(self, t0, t1):
        rows = [r for t, r in self.rows if t0 - 0.05 <= t <= t1 + 0.05 and len(r) >= 9]
        if not rows:
            rows = [r for _, r in self.rows if len(r) >= 9]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": num(rows[0][2]),
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------ GPU arm

def kernel_source_hash():
    h = hashlib.sha256()
    with open(os.path.join(ROOT, "gguf_quant_weight_gb300", "csrc", "gemv.cu"), "rb") as f:
        h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic():
    """DRAM bytes per GEMV launch from the committed ncu summary, if it was
    taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", "gemv_q5k_4096x4096.traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    if d.get("gemv_source_sha256_16") != kernel_source_hash():
        return None
    return d.get("dram_bytes_per_launch")


def run_gpu(args):
    import torch
    import gguf_quant_weight_gb300 as g
    import gguf_synth as syn

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    g.load_library()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    copies = max(3 * 2, int(np.ceil(2.2 * l2 / W_BYTES)))
    copies = (copies + 2) // 3 * 3
    rs = syn.rng(1001)
    w0 = syn.weight_blocks(rs, QTYPE, N, K).reshape(-1)
    W = torch.from_numpy(w0).to(dev).repeat(copies).view(copies, -1)
    xs = {m: torch.from_numpy(syn.normal(rs, (m, K), "bf16")).to(dev).view(torch.bfloat16) for m in MS}
    rsd = {m: torch.from_numpy(syn.normal(rs, (m, N), "bf16")).to(dev).view(torch.bfloat16) for m in MS}
    ys = {m: torch.empty((m, N), dtype=torch.bfloat16, device=dev) for m in MS}
    stream = torch.cuda.Stream(device=dev)
    # one graph replay walks every copy exactly once (3 calls per step), so a
    # copy is reused only after all the others: never an L2 hit
    per_graph = copies // 3
    state = {"c": 0}

    def step(xsrc=None, rsrc=None, ydst=None):
        for m in MS:
            if xsrc is not None:
                xs[m].copy_(xsrc[m], non_blocking=True)
                rsd[m].copy_(rsrc[m], non_blocking=True)
            g.gguf_mm_gemv(W[state["c"] % copies], QTYPE, 0, N, K, xs[m], g.GGUF_DT_BF16, m, rsd[m], ys[m],
                           g.GGUF_DT_BF16, stream=stream)
            if ydst is not None:
                ydst[m].copy_(ys[m], non_blocking=True)
            state["c"] += 1

    def capture(nsteps, **kw):
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(graph, stream=stream):
                for _ in range(nsteps):
                    step(**kw)
        return graph

    def replay(graphs_counts):
        for gr, cnt in graphs_counts:
            for _ in range(cnt):
                gr.replay()

    with torch.cuda.stream(stream):
        for _ in range(3):
            step()
        stream.synchronize()
    full, rem = divmod(args.steps, per_graph)
    g_full = capture(per_graph) if full else None
    g_rem = capture(rem) if rem else None
    plan = [(g_full, full)] if full else []
    if rem:
        plan.append((g_rem, 1))
    # warm-up steps (graph replays of the same launches)
    wfull, wrem = divmod(max(args.warmup, 3), per_graph)
    with torch.cuda.stream(stream):
        for _ in range(wfull):
            (g_full or capture(per_graph)).replay()
        if wrem:
            capture(wrem).replay()
    stream.synchronize()

    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    smi_index = vis.split(",")[local].strip() if vis else str(local)
    clocks = ClockSampler(smi_index)
    clocks.start()
    time.sleep(0.3)

    def timed(plan_):
        if ws > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        t_host0 = time.time()
        with torch.cuda.stream(stream):
            e0.record(stream)
            replay(plan_)
            e1.record(stream)
        e1.synchronize()
        torch.cuda.synchronize(dev)
        if ws > 1:
            torch.distributed.barrier()
        return e0.elapsed_time(e1) / 1e3, t_host0, time.time()

    sec, th0, th1 = timed(plan)
    clk = clocks.summary(th0, th1)

    # end to end: pinned host inputs copied in and outputs copied out every step
    hx = {m: xs[m].cpu().pin_memory() for m in MS}
    hr = {m: rsd[m].cpu().pin_memory() for m in MS}
    hy = {m: torch.empty((m, N), dtype=torch.bfloat16).pin_memory() for m in MS}
    e_full = capture(per_graph, xsrc=hx, rsrc=hr, ydst=hy) if full else None
    e_rem = capture(rem, xsrc=hx, rsrc=hr, ydst=hy) if rem else None
    eplan = ([(e_full, full)] if full else []) + ([(e_rem, 1)] if rem else [])
    with torch.cuda.stream(stream):
        (e_full or e_rem).replay()
    stream.synchronize()
    esec, _, _ = timed(eplan)
    clocks.stop()

    h2d = sum(m * K * 2 + m * N * 2 for m in MS)
    d2h = sum(m * N * 2 for m in MS)
    status = g.gguf_mm_check_errors(stream)
    if status != 0:
        raise RuntimeError(f"device status {status}")

    # max over ranks; value sums the replicas
    t = torch.tensor([sec, esec], dtype=torch.float64, device=dev)
    if ws > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    sec, esec = float(t[0]), float(t[1])
    steps = args.steps
    weight_bytes = steps * len(MS) * W_BYTES * ws
    value = weight_bytes / sec / 1e9
    e2e = weight_bytes / esec / 1e9
    hbm, tc, tc_sus, peak_kind = peaks()
    algo = sum(W_BYTES + m * K * 2 + 2 * m * N * 2 for m in MS) / len(MS)   # weights + x + residual + y
    launches = steps * len(MS)
    achieved = algo * launches / (sec * ws / ws) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws, "steps": steps, "warmup": args.warmup,
        "ms_per_step": sec / steps * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int8", "data": "synthetic",
        "config": {"workload": WORKLOAD, "N": N, "K": K, "M": list(MS), "qtype": "Q5_K",
                   "residual": True, "activations": "bf16", "output": "bf16",
                   "l2": f"weights rotate over {copies} copies ({copies * W_BYTES / 1e6:.0f} MB > 2x L2)",
                   "parallelism": f"replicas x{ws}"},
        "hbm_frac_of_" + peak_kind: value / ws / hbm,
        "e2e": {"value": e2e, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm, "traffic": recorded_traffic(), "peak_kind": peak_kind,
                     "kernel": "gemv_direct_kernel", "algorithmic_bytes_per_launch": algo},
        "gpu_launches": launches,
        "clocks": {"sm_mhz": clk["sm_mhz"], "sm_max_mhz": clk["sm_max_mhz"], "reasons": clk["reasons"]},
    }
    if rank == 0:
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline()
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
