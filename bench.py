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


# ------------------------------------------------------------------ ranks

def max_over_ranks(values, device):
    """Each timed duration, maxed over the ranks of the process group (a
    barrier-bracketed region ends when its slowest rank ends)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor(values, dtype=torch.float64, device=device)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t]


def job_gbs(steps, world_size, seconds):
    """Whole-job weight GB/s: every rank (an independent replica) streams
    steps x |MS| weight matrices in the same max-over-ranks time."""
    return steps * len(MS) * W_BYTES * world_size / seconds / 1e9


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


def time_graph(fn, reps, stream, calls):
    """Mean device time of one call: `calls` calls captured in a CUDA graph,
    replayed `reps` times (after two untimed replays)."""
    import torch
    with torch.cuda.stream(stream):
        for i in range(2):
            fn(i)
        stream.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            for i in range(calls):
                fn(i)
        gr.replay()
        gr.replay()
        stream.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            gr.replay()
        e1.record(stream)
        e1.synchronize()
    return e0.elapsed_time(e1) / 1e3 / (reps * calls)


def prefill_figures(dev, stream, tc_peak, hbm_peak, only=None):
    """Figures for the other workloads (context for the second half of the
    metric): the small Q6_K GEMV, the Q6_K / Q5_K and Q8_0 prefill GEMMs and the
    MoE expert GEMM; weights rotate over copies larger than L2.  `only`: a
    regular expression; just the entries whose key it matches are run."""
    import re
    import torch
    import gguf_quant_weight_gb300 as g
    import gguf_synth as syn
    out = {}
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size

    def want(key):
        return only is None or re.search(only, key) is not None

    def copies_of(arr):
        c = max(2, int(np.ceil(2.2 * l2 / arr.size)))
        return torch.from_numpy(arr.reshape(-1)).to(dev).repeat(c).view(c, -1), c

    # Q6_K GEMV 256x1024, M = 1, f32 activations and output (no residual)
    key = "q6_k_gemv_256x1024_m1_f32"
    if want(key):
        N, K = 256, 1024
        w = syn.weight_blocks(syn.rng(1005), 14, N, K)
        W, c = copies_of(w)
        x = torch.from_numpy(syn.normal(syn.rng(1006), (1, K), "f32")).to(dev)
        y = torch.empty((1, N), dtype=torch.float32, device=dev)
        wsb = g.gguf_mm_workspace_size(g.GGUF_OP_GEMV, 14, N, K, 1)
        ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
        t = time_graph(lambda i: g.gguf_mm_gemv(W[i % c], 14, 0, N, K, x, g.GGUF_DT_F32, 1, None, y, g.GGUF_DT_F32,
                                                ws, wsb, stream=stream), 5, stream, c)
        out[key] = {"us": t * 1e6, "weight_gbs": w.size / t / 1e9, "hbm_frac": w.size / t / 1e9 / hbm_peak}

    # Q6_K (planes and raw blocks) and Q5_K prefill, 14336x4096
    rs = syn.rng(1002)
    for qt, name, layout, ms in ((14, "q6_k_planes", 1, (8, 64, 128, 256, 512, 2048)),
                                 (13, "q5_k", 0, (8, 64, 128, 256, 512, 2048)),
                                 (14, "q6_k", 0, (512, 2048))):
        N, K = 14336, 4096
        # M = 8 sits on the border of the two paths: both are timed
        runs = [(M, path, tag) for M in ms for path, tag in ((g.GGUF_PATH_FUSED, "fused"), (g.GGUF_PATH_GEMV, "gemv"))
                if (path == g.GGUF_PATH_FUSED or M <= 8) and want(f"{name}_14336x4096_m{M}_{tag}")]
        if not runs:
            continue
        w = syn.weight_blocks(rs, qt, N, K)
        W, c = copies_of(w)
        if layout:   # regroup every copy into the QL | QH | SC | D planes on the GPU
            P = torch.empty_like(W)
            for i in range(c):
                g.gguf_repack_q6k_planes(W[i], P[i], N * K // 256, 0, stream=stream)
            stream.synchronize()
            W = P
        for M, path, tag in runs:
            x = torch.from_numpy(syn.normal(rs, (M, K), "bf16")).to(dev).view(torch.bfloat16)
            y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            wsb = g.gguf_mm_workspace_size(g.GGUF_OP_GEMM, qt, N, K, M)
            ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
            t = time_graph(lambda i: g.gguf_mm_gemm(W[i % c], qt, layout, N, K, x, g.GGUF_DT_BF16, M, None, y,
                                                    g.GGUF_DT_BF16, ws, wsb, path, stream=stream), 5, stream, c)
            tf = 2 * M * N * K / t / 1e12
            out[f"{name}_14336x4096_m{M}_{tag}"] = {"us": t * 1e6, "tflops": tf, "tc_frac": tf / tc_peak,
                                                    "weight_gbs": W[0].numel() / t / 1e9}

    # Q8_0 2048x8192: fused vs decode-once (K-padded f16) + dense GEMM
    N, K = 2048, 8192
    ms = [M for M in (128, 512, 4096) if want(f"q8_0_2048x8192_m{M}_fused") or
          want(f"q8_0_2048x8192_m{M}_dense_after_decode_once")]
    if ms or want("q8_0_2048x8192_decode_once"):
        w = syn.weight_blocks(syn.rng(1003), 8, N, K)
        W, c = copies_of(w)
        ld = K + 64
        wd = torch.empty((N, ld), dtype=torch.float16, device=dev)
        g.gguf_dequant_padded(W[0], 8, 0, N, K, wd, g.GGUF_DT_F16, ld, stream=stream)
        cd = max(2, int(np.ceil(2.2 * l2 / (wd.numel() * 2))))
        WD = wd.unsqueeze(0).repeat(cd, 1, 1)
        if want("q8_0_2048x8192_decode_once"):
            t_dec = time_graph(lambda i: g.gguf_dequant_padded(W[i % c], 8, 0, N, K, wd, g.GGUF_DT_F16, ld,
                                                               stream=stream), 5, stream, c)
            out["q8_0_2048x8192_decode_once"] = {"us": t_dec * 1e6, "gbs": (w.size + N * ld * 2) / t_dec / 1e9}
        for M in ms:
            x = torch.from_numpy(syn.normal(rs, (M, K), "bf16")).to(dev).view(torch.bfloat16)
            y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            wsb = g.gguf_mm_workspace_size(g.GGUF_OP_GEMM, 8, N, K, M)
            ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
            fl = 2 * M * N * K
            if want(f"q8_0_2048x8192_m{M}_fused"):
                t = time_graph(lambda i: g.gguf_mm_gemm(W[i % c], 8, 0, N, K, x, g.GGUF_DT_BF16, M, None, y,
                                                        g.GGUF_DT_BF16, ws, wsb, g.GGUF_PATH_FUSED, stream=stream),
                               5, stream, c)
                out[f"q8_0_2048x8192_m{M}_fused"] = {"us": t * 1e6, "tflops": fl / t / 1e12,
                                                     "tc_frac": fl / t / 1e12 / tc_peak}
            if want(f"q8_0_2048x8192_m{M}_dense_after_decode_once"):
                t2 = time_graph(lambda i: g.gguf_dense_gemm(WD[i % cd], g.GGUF_DT_F16, ld, N, K, x, g.GGUF_DT_BF16, M,
                                                            None, y, g.GGUF_DT_BF16, ws, wsb, stream=stream),
                                5, stream, cd)
                out[f"q8_0_2048x8192_m{M}_dense_after_decode_once"] = {"us": t2 * 1e6, "tflops": fl / t2 / 1e12,
                                                                         "tc_frac": fl / t2 / 1e12 / tc_peak}

    # MoE: 128 experts top-8, Q4_K 768x2048; ids rotate over 8 Zipf(1.1) draws.
    # T = 32..512 is the prefill batch; T = 1, 4, 16 the decode form (one int8
    # GEMV per routed row), timed against the routed path as well
    E, N, K, top_k = 128, 768, 2048, 8
    ts = [T for T in (1, 4, 16, 32, 64, 256, 512) if want(f"q4_k_moe_128x768x2048_top8_t{T}")]
    if ts:
        wE = syn.weight_blocks(syn.rng(1004), 12, E * N, K)
        WE, c = copies_of(wE)
    per_expert = N * (K // 256) * 144
    for T in ts:
        id_sets = [syn.zipf_ids(syn.rng(2000 + T + j), T, E, top_k, 1.1) for j in range(8)]
        IDS = [torch.from_numpy(a).to(dev) for a in id_sets]
        touched = float(np.mean([len(np.unique(a)) for a in id_sets])) * per_expert
        x = torch.from_numpy(syn.normal(rs, (T, K), "bf16")).to(dev).view(torch.bfloat16)
        y = torch.empty((T, top_k, N), dtype=torch.bfloat16, device=dev)
        wsb = g.gguf_mm_workspace_size(g.GGUF_OP_ID, 12, N, K, T, E, top_k)
        ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
        calls = 8 * c
        fl = 2 * top_k * T * N * K
        rec = {}
        # comparison arms (the switches are read when a call is made, so while
        # the graph is captured): the decode form off (T <= 16), and every
        # tile's MMAs at the full tile width instead of the tile-skip (T >= 32)
        arms = [("default", {})]
        arms.append(("routed_path", {"GGUF_MM_MOE_MV": "0"}) if T * top_k <= 128 else
                    ("full_width_tiles", {"GGUF_MM_MOE_FULL_TILES": "1"}))
        for arm, env in arms:
            os.environ.update(env)
            try:
                t = time_graph(lambda i: g.gguf_mm_id(WE[i % c], 12, E, N, K, x, g.GGUF_DT_BF16, T, IDS[i % 8], top_k,
                                                      None, y, g.GGUF_DT_BF16, ws, wsb, stream=stream), 3, stream, calls)
            finally:
                for k in env:
                    os.environ.pop(k, None)
            if arm == "default":
                rec.update({"us": t * 1e6, "tflops": fl / t / 1e12, "tc_frac": fl / t / 1e12 / tc_peak,
                            "touched_gbs": touched / t / 1e9, "hbm_frac": touched / t / 1e9 / hbm_peak,
                            "experts_touched": touched / per_expert})
            else:
                rec["us_" + arm] = t * 1e6
        out[f"q4_k_moe_128x768x2048_top8_t{T}"] = rec
    return out


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
    wsz = {m: g.gguf_mm_workspace_size(g.GGUF_OP_GEMV, QTYPE, N, K, m) for m in MS}
    wss = {m: torch.empty(wsz[m], dtype=torch.uint8, device=dev) for m in MS}
    stream = torch.cuda.Stream(device=dev)
    # A decode step runs every layer at one M, so each M is timed as its own
    # chain of calls: `steps` calls at M = 1, then at M = 2, then at M = 4 (the
    # same calls and bytes as `steps` rounds of one call per M).  A graph walks
    # the weight copies in order ten times (a decode step's graph holds every
    # layer's calls; ten walks keep the replay's own start-up off the per-call
    # time), so a copy is reused only after all the others: never an L2 hit.
    per_graph = 10 * copies
    state = {"c": 0}

    def call(m, xsrc=None, rsrc=None, ydst=None):
        if xsrc is not None:
            xs[m].copy_(xsrc[m], non_blocking=True)
            rsd[m].copy_(rsrc[m], non_blocking=True)
        g.gguf_mm_gemv(W[state["c"] % copies], QTYPE, 0, N, K, xs[m], g.GGUF_DT_BF16, m, rsd[m], ys[m],
                       g.GGUF_DT_BF16, wss[m], wsz[m], stream=stream)
        if ydst is not None:
            ydst[m].copy_(ys[m], non_blocking=True)
        state["c"] += 1

    def capture(m, ncalls, **kw):
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(graph, stream=stream):
                for _ in range(ncalls):
                    call(m, **kw)
        return graph

    def make_plan(ncalls, **kw):
        # [(graph, replays)] covering ncalls calls of each M, M by M
        out = []
        full, rem = divmod(ncalls, per_graph)
        for m in MS:
            if full:
                out.append((capture(m, per_graph, **kw), full))
            if rem:
                out.append((capture(m, rem, **kw), 1))
        return out

    def replay(graphs_counts):
        for gr, cnt in graphs_counts:
            for _ in range(cnt):
                gr.replay()

    with torch.cuda.stream(stream):
        for m in MS:
            for _ in range(3):
                call(m)
        stream.synchronize()
    plan = make_plan(args.steps)
    # warm-up calls (graph replays of the same launches)
    with torch.cuda.stream(stream):
        replay(make_plan(max(args.warmup, 3)))
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
    eplan = make_plan(args.steps, xsrc=hx, rsrc=hr, ydst=hy)
    with torch.cuda.stream(stream):
        for gr, _ in eplan:
            gr.replay()
    stream.synchronize()
    esec, _, _ = timed(eplan)
    clocks.stop()

    h2d = sum(m * K * 2 + m * N * 2 for m in MS)
    d2h = sum(m * N * 2 for m in MS)
    status = g.gguf_mm_check_errors(stream)
    if status != 0:
        raise RuntimeError(f"device status {status}")

    # max over ranks; value sums the replicas
    sec, esec = max_over_ranks([sec, esec], dev)
    steps = args.steps
    value = job_gbs(steps, ws, sec)
    e2e = job_gbs(steps, ws, esec)
    hbm, tc, tc_sus, peak_kind = peaks()
    algo = sum(W_BYTES + m * K * 2 + 2 * m * N * 2 for m in MS) / len(MS)   # weights + x + residual + y
    calls = steps * len(MS)
    achieved = algo * calls / sec / 1e9   # per call: every kernel of gguf_mm_gemv, chained
    # kernels per call: the tile kernel alone at M = 1; the activation quantizer
    # plus the pair kernel at M = 2, 4 (the library's plan for this shape)
    launches = steps * sum(1 if m == 1 else 2 for m in MS)
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws, "steps": steps, "warmup": args.warmup,
        "ms_per_step": sec / steps * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int8", "data": "synthetic",
        "config": {"workload": WORKLOAD, "N": N, "K": K, "M": list(MS), "qtype": "Q5_K",
                   "residual": True, "activations": "bf16", "output": "bf16",
                   "l2": f"weights rotate over {copies} copies ({copies * W_BYTES / 1e6:.0f} MB > 2x L2)",
                   "order": "each M as its own chain of calls (a decode step runs every layer at one M)",
                   "graph_calls": per_graph,
                   "parallelism": f"replicas x{ws}"},
        "hbm_frac_of_" + peak_kind: value / ws / hbm,
        "e2e": {"value": e2e, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm, "traffic": recorded_traffic(), "peak_kind": peak_kind,
                     "kernel": "gguf_mm_gemv: gemv_tile_kernel (M=1); act_quant_kernel + gemv_pair_kernel (M=2,4)",
                     "algorithmic_bytes_per_launch": algo},
        "gpu_launches": launches,
        "clocks": {"sm_mhz": clk["sm_mhz"], "sm_max_mhz": clk["sm_max_mhz"], "reasons": clk["reasons"]},
    }
    if rank == 0:
        if not args.no_prefill:
            line["prefill"] = prefill_figures(dev, stream, tc, hbm, args.prefill_only)
            line["prefill"]["peak_tflops"] = tc
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
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--prefill-only", default=None, metavar="REGEX",
                    help="run only the prefill figures whose key matches (e.g. q6_k_planes_14336x4096_m512)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
