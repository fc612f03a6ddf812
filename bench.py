"""Benchmark: decode GEMV on Q5_K weights, N = K = 4096, M in {1, 2, 4}, fused residual.

One step = the three GEMV calls (M = 1, 2, 4; bf16 activations, bf16 residual,
bf16 output) on three different copies of the weight, so every call streams its
11,534,336 weight bytes from HBM: the copies rotate over more than twice the L2
size.  A decode step runs every layer at one M, so each M is a chain of calls
(`steps` calls at M = 1, then at M = 2, then at M = 4).  The timed region is
exactly those calls, captured in CUDA graphs, bracketed by a barrier and a
device synchronization, timed with CUDA events on the launching stream.

Printed JSON line (rank 0): value = weight GB/s over the whole job, plus
  per_m       us per call and weight GB/s at each M (graphs of 270 calls);
  e2e         the same calls made eagerly from the host through the C ABI's
              host-buffer entry (gguf_mm_gemv_host): x and the residual
              copied in from pinned host memory and y copied out, every call;
  roofline    the GEMV kernel's algorithmic bytes per launch / its mean
              launch time in the timed region, against the measured HBM copy
              bandwidth;
  cpu_baseline the CPU oracle (int8-path restatement) on a bounded sample, at
              all host cores (row shards in spawned processes) and at one;
  clocks      SM clock and throttle reasons sampled during the timed region;
  prefill     tensor-core figures for the other workloads, last in the line:
              [us, TFLOPS, fraction of the measured bf16 peak] (GEMVs:
              [us, GB/s, fraction of HBM]).
`--impl reference` times the CPU oracle instead (the reference arm);
`--crossover` times the decode GEMV against the fused GEMM for M = 1..16.
Multi-GPU runs (torchrun) are independent replicas: every rank runs the same
workload on its own GPU and value sums over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import multiprocessing as mproc
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
GRAPH_CALLS = 270


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return (float(d["hbm_gbs"]), float(d["bf16_tflops"]),
                float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured")
    return 6800.0, 1900.0, 1700.0, "fallback"


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# ------------------------------------------------------------------ CPU arm (the oracle)

def _oracle_shard(job):
    """Worker: the oracle's int8-path GEMV over `rows` weight rows (a shard of
    the workload), for each M, `steps` times.  Returns its own seconds."""
    rows, steps, seed = job
    import gguf_synth as syn
    from oracle import gguf_oracle as O
    rs = syn.rng(seed)
    w = syn.weight_blocks(rs, QTYPE, rows, K)
    xs = {m: O.bf16_bits_to_f32(syn.normal(rs, (m, K), "bf16")) for m in MS}
    rr = {m: O.bf16_bits_to_f64(syn.normal(rs, (m, rows), "bf16")) for m in MS}
    t0 = time.perf_counter()
    for _ in range(steps):
        for m in MS:
            O.gemv_int8_path(w, QTYPE, rows, K, xs[m], rr[m])
    return time.perf_counter() - t0


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


class OraclePool:
    """A pool of spawned processes (started before any GPU work), one thread each."""

    def __init__(self, procs: int):
        self.procs = procs
        self.pool = None
        if procs > 1:
            os.environ.setdefault("OMP_NUM_THREADS", "1")
            self.pool = mproc.get_context("spawn").Pool(procs)
            self.pool.map(_oracle_shard, [(8, 1, 1001)] * procs)   # imports done before timing

    def run(self, rows: int, steps: int):
        """Wall seconds for `rows` weight rows x `steps` steps of the three M,
        sharded over the pool's processes; returns (seconds, weight bytes, threads)."""
        if self.pool is None:
            dt = _oracle_shard((rows, steps, 1001))
            return dt, steps * len(MS) * rows * ROW_BYTES, 1
        shard = -(-rows // self.procs)
        jobs = [(min(shard, rows - i * shard), steps, 1001 + i) for i in range(self.procs) if i * shard < rows]
        t0 = time.perf_counter()
        self.pool.map(_oracle_shard, jobs)
        dt = time.perf_counter() - t0
        return dt, steps * len(MS) * rows * ROW_BYTES, len(jobs)

    def close(self):
        if self.pool is not None:
            self.pool.close()
            self.pool.join()


def cpu_baseline(pool: OraclePool):
    dt1, b1, _ = OraclePool(1).run(N // 4, 16)       # one thread: a quarter of the rows, 16 steps (~2 s)
    dtn, bn, used = pool.run(N, 24)                  # all cores: 24 steps of the whole workload (~12 s of CPU)
    return {"value": round(bn / dtn / 1e9, 4), "unit": "GB/s", "cores": used, "kind": "oracle",
            "single_thread_value": round(b1 / dt1 / 1e9, 4),
            "sample": f"numpy int8-path oracle on the Q5_K 4096x4096 M=1,2,4 calls: all {used} host cores "
                      f"(row shards in spawned processes) {bn // (3 * ROW_BYTES * N)} step(s) of the full "
                      f"workload in {dtn:.1f} s; one thread 1024 rows x 16 steps in {dt1:.1f} s"}


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    pool = OraclePool(host_cores())
    try:
        steps = max(1, args.steps)
        if args.warmup > 0:
            pool.run(256, 1)
        dt, nbytes, used = pool.run(1024, steps)
    finally:
        pool.close()
    value = nbytes / dt / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws, "steps": steps,
        "warmup": args.warmup, "ms_per_step": dt / steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int8", "data": "synthetic",
        "config": {"workload": WORKLOAD, "N": N, "K": K, "M": list(MS), "qtype": "Q5_K", "sample_rows": 1024},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": used, "kind": "oracle",
                         "sample": f"each step: 1024 of the 4096 weight rows at M=1,2,4 through the numpy "
                                   f"int8-path oracle, sharded over {used} host processes"},
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
    """DRAM bytes per GEMV launch per M from the committed ncu summary, if it
    was taken on the current kernel source."""
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
    replayed `reps` times (after two untimed replays); median over replays."""
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
        ts = []
        for _ in range(reps):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            gr.replay()
            e1.record(stream)
            e1.synchronize()
            ts.append(e0.elapsed_time(e1) / 1e3 / calls)
    return float(np.median(ts))


_CUDART = None


def upload_graph(graph, stream) -> bool:
    """cudaGraphUpload of a captured graph: its first launch then pays no
    upload inside a timed region.  False if the runtime or handle is unavailable."""
    global _CUDART
    import ctypes
    try:
        exec_handle = graph.raw_cuda_graph_exec()
    except (AttributeError, RuntimeError):
        return False
    if _CUDART is None:
        for name in ("libcudart.so.13", "libcudart.so.12", "libcudart.so"):
            try:
                _CUDART = ctypes.CDLL(name)
                break
            except OSError:
                continue
        if _CUDART is None:
            return False
    h = exec_handle if isinstance(exec_handle, int) else int(exec_handle)
    return _CUDART.cudaGraphUpload(ctypes.c_void_p(h), ctypes.c_void_p(stream.cuda_stream)) == 0


def _r(x, nd=1):
    return round(float(x), nd)


def prefill_figures(dev, stream, tc_peak, hbm_peak, only=None):
    """Figures for the other workloads (context for the second half of the
    metric).  Returns (compact dict for the JSON line, full detail dict).
    Weights rotate over copies larger than L2.  `only`: a regular expression
    over the detail keys.  Compact keys: q8s_mM / q8sdense_mM = Q8_0 2048 x 8192
    fused / dense after decode-once, [us, TFLOP/s, fraction of the tensor peak];
    q4_, q5_, q6_ (raw Q6_K), q6p_ (Q6_K planes), q8_mM = 14336 x 4096, same
    triple; moe_tT = [us, touched-expert GB/s, fraction of HBM, TFLOP/s]."""
    import re
    import torch
    import gguf_quant_weight_gb300 as g
    import gguf_synth as syn
    compact, detail = {}, {}
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size

    def want(key):
        return only is None or re.search(only, key) is not None

    def copies_of(arr):
        c = max(2, int(np.ceil(2.2 * l2 / arr.size)))
        return torch.from_numpy(arr.reshape(-1)).to(dev).repeat(c).view(c, -1), c

    # Q6_K GEMV 256x1024, M = 1, f32 activations and output (no residual)
    key = "q6_k_gemv_256x1024_m1_f32"
    if want(key):
        n, k = 256, 1024
        w = syn.weight_blocks(syn.rng(1005), 14, n, k)
        W, c = copies_of(w)
        x = torch.from_numpy(syn.normal(syn.rng(1006), (1, k), "f32")).to(dev)
        y = torch.empty((1, n), dtype=torch.float32, device=dev)
        wsb = g.gguf_mm_workspace_size(g.GGUF_OP_GEMV, 14, n, k, 1)
        ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
        t = time_graph(lambda i: g.gguf_mm_gemv(W[i % c], 14, 0, n, k, x, g.GGUF_DT_F32, 1, None, y, g.GGUF_DT_F32,
                                                ws, wsb, stream=stream), 5, stream, c)
        detail[key] = {"us": t * 1e6, "weight_gbs": w.size / t / 1e9, "hbm_frac": w.size / t / 1e9 / hbm_peak}
        compact["q6gemv"] = [_r(t * 1e6, 2), _r(w.size / t / 1e9), _r(w.size / t / 1e9 / hbm_peak, 3)]

    # Q8_0 2048x8192: fused vs decode-once (K-padded f16) + dense GEMM
    n, k = 2048, 8192
    ms = [M for M in (128, 512, 4096) if want(f"q8_0_2048x8192_m{M}")]
    if ms:
        rs = syn.rng(1003)
        w = syn.weight_blocks(rs, 8, n, k)
        W, c = copies_of(w)
        ld = k + 64
        wd = torch.empty((n, ld), dtype=torch.float16, device=dev)
        g.gguf_dequant_padded(W[0], 8, 0, n, k, wd, g.GGUF_DT_F16, ld, stream=stream)
        cd = max(2, int(np.ceil(2.2 * l2 / (wd.numel() * 2))))
        WD = wd.unsqueeze(0).repeat(cd, 1, 1)
        t_dec = time_graph(lambda i: g.gguf_dequant_padded(W[i % c], 8, 0, n, k, wd, g.GGUF_DT_F16, ld,
                                                           stream=stream), 5, stream, c)
        detail["q8_0_2048x8192_decode_once"] = {"us": t_dec * 1e6, "gbs": (w.size + n * ld * 2) / t_dec / 1e9}
        compact["q8_decode_once"] = [_r(t_dec * 1e6), _r((w.size + n * ld * 2) / t_dec / 1e9)]
        for M in ms:
            x = torch.from_numpy(syn.normal(rs, (M, k), "bf16")).to(dev).view(torch.bfloat16)
            y = torch.empty((M, n), dtype=torch.bfloat16, device=dev)
            wsb = max(g.gguf_mm_workspace_size(g.GGUF_OP_GEMM, 8, n, k, M),
                      g.gguf_mm_workspace_size(g.GGUF_OP_DENSE, 8, n, k, M))
            ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
            fl = 2 * M * n * k
            t = time_graph(lambda i: g.gguf_mm_gemm(W[i % c], 8, 0, n, k, x, g.GGUF_DT_BF16, M, None, y,
                                                    g.GGUF_DT_BF16, ws, wsb, g.GGUF_PATH_FUSED, stream=stream),
                           5, stream, c)
            t2 = time_graph(lambda i: g.gguf_dense_gemm(WD[i % cd], g.GGUF_DT_F16, ld, n, k, x, g.GGUF_DT_BF16, M,
                                                        None, y, g.GGUF_DT_BF16, ws, wsb, stream=stream),
                            5, stream, cd)
            detail[f"q8_0_2048x8192_m{M}_fused"] = {"us": t * 1e6, "tflops": fl / t / 1e12}
            detail[f"q8_0_2048x8192_m{M}_dense_after_decode_once"] = {"us": t2 * 1e6, "tflops": fl / t2 / 1e12}
            compact[f"q8s_m{M}"] = [_r(t * 1e6), _r(fl / t / 1e12), _r(fl / t / 1e12 / tc_peak, 3)]
            compact[f"q8sdense_m{M}"] = [_r(t2 * 1e6), _r(fl / t2 / 1e12), _r(fl / t2 / 1e12 / tc_peak, 3)]

    # MoE: 128 experts top-8, Q4_K 768x2048; ids rotate over 8 Zipf(1.1) draws.
    # T = 32..512 is the prefill batch; T = 1, 4, 16 the decode form (one int8
    # GEMV per routed row), timed against the routed path as well
    E, n, k, top_k = 128, 768, 2048, 8
    ts = [T for T in (1, 4, 16, 32, 64, 256, 512) if want(f"q4_k_moe_128x768x2048_top8_t{T}")]
    if ts:
        wE = syn.weight_blocks(syn.rng(1004), 12, E * n, k)
        WE, c = copies_of(wE)
    per_expert = n * (k // 256) * 144
    rs = syn.rng(1007)
    for T in ts:
        id_sets = [syn.zipf_ids(syn.rng(2000 + T + j), T, E, top_k, 1.1) for j in range(8)]
        IDS = [torch.from_numpy(a).to(dev) for a in id_sets]
        touched = float(np.mean([len(np.unique(a)) for a in id_sets])) * per_expert
        x = torch.from_numpy(syn.normal(rs, (T, k), "bf16")).to(dev).view(torch.bfloat16)
        y = torch.empty((T, top_k, n), dtype=torch.bfloat16, device=dev)
        wsb = g.gguf_mm_workspace_size(g.GGUF_OP_ID, 12, n, k, T, E, top_k)
        ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
        calls = 8 * c
        fl = 2 * top_k * T * n * k
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
                t = time_graph(lambda i: g.gguf_mm_id(WE[i % c], 12, E, n, k, x, g.GGUF_DT_BF16, T, IDS[i % 8],
                                                      top_k, None, y, g.GGUF_DT_BF16, ws, wsb, stream=stream),
                               3, stream, calls)
            finally:
                for kk in env:
                    os.environ.pop(kk, None)
            if arm == "default":
                rec.update({"us": t * 1e6, "tflops": fl / t / 1e12, "touched_gbs": touched / t / 1e9,
                            "hbm_frac": touched / t / 1e9 / hbm_peak, "experts_touched": touched / per_expert})
            else:
                rec["us_" + arm] = t * 1e6
        detail[f"q4_k_moe_128x768x2048_top8_t{T}"] = rec
        compact[f"moe_t{T}"] = [_r(rec["us"]), _r(rec["touched_gbs"]), _r(rec["hbm_frac"], 3), _r(rec["tflops"])]

    # the 14336 x 4096 prefill shapes; Q5_K and Q6_K planes at M = 512 and 2048 last
    runs = []
    for M in (8, 64, 128, 256):
        runs += [(14, "q6p", 1, M), (13, "q5", 0, M)]
    for M in (512, 2048):
        runs += [(12, "q4", 0, M), (8, "q8", 0, M), (14, "q6", 0, M)]
    for M in (512, 2048):
        runs += [(13, "q5", 0, M), (14, "q6p", 1, M)]
    n, k = 14336, 4096
    cache = {}
    rs = syn.rng(1002)
    for qt, name, layout, M in runs:
        full = f"{name}_14336x4096_m{M}"
        if not want(full):
            continue
        if (qt, layout) not in cache:
            w = syn.weight_blocks(syn.rng(1002 + qt), qt, n, k)
            W, c = copies_of(w)
            if layout:   # regroup every copy into the QL | QH | SC | D planes on the GPU
                P = torch.empty_like(W)
                for i in range(c):
                    g.gguf_repack_q6k_planes(W[i], P[i], n * k // 256, 0, stream=stream)
                stream.synchronize()
                W = P
            cache[(qt, layout)] = (W, c)
        W, c = cache[(qt, layout)]
        x = torch.from_numpy(syn.normal(rs, (M, k), "bf16")).to(dev).view(torch.bfloat16)
        y = torch.empty((M, n), dtype=torch.bfloat16, device=dev)
        wsb = g.gguf_mm_workspace_size(g.GGUF_OP_GEMM, qt, n, k, M)
        ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
        t = time_graph(lambda i: g.gguf_mm_gemm(W[i % c], qt, layout, n, k, x, g.GGUF_DT_BF16, M, None, y,
                                                g.GGUF_DT_BF16, ws, wsb, g.GGUF_PATH_FUSED, stream=stream),
                       5, stream, c)
        tf = 2 * M * n * k / t / 1e12
        detail[full] = {"us": t * 1e6, "tflops": tf, "tc_frac": tf / tc_peak, "weight_gbs": W[0].numel() / t / 1e9}
        compact[f"{name}_m{M}"] = [_r(t * 1e6), _r(tf), _r(tf / tc_peak, 3)]
    cache.clear()
    return compact, detail


def crossover(dev, stream, out_path, formats=None):
    """GEMV against the fused GEMM for M = 1..16, every format, at the decode
    shape (4096 x 4096) and the prefill shape (14336 x 4096): us per call in
    chains of calls on rotating weight copies (both paths forced).  `formats`:
    a regular expression over the format names (default: all)."""
    import torch
    import gguf_quant_weight_gb300 as g
    import gguf_synth as syn
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    table = {}
    for n, k in ((4096, 4096), (14336, 4096)):
        for qt, layout, name in ((13, 0, "Q5_K"), (12, 0, "Q4_K"), (14, 1, "Q6_K_planes"), (14, 0, "Q6_K"),
                                 (8, 0, "Q8_0"), (2, 0, "Q4_0"), (3, 0, "Q4_1"), (6, 0, "Q5_0"), (7, 0, "Q5_1"),
                                 (10, 0, "Q2_K"), (11, 0, "Q3_K")):
            if formats and not __import__("re").search(formats, name):
                continue
            w = syn.weight_blocks(syn.rng(7000 + qt), qt, n, k)
            c = max(2, int(np.ceil(2.2 * l2 / w.size)))
            W = torch.from_numpy(w.reshape(-1)).to(dev).repeat(c).view(c, -1)
            if layout:
                P = torch.empty_like(W)
                for i in range(c):
                    g.gguf_repack_q6k_planes(W[i], P[i], n * k // 256, 0, stream=stream)
                W = P
            stream.synchronize()
            row = {}
            for M in range(1, 17):
                x = torch.from_numpy(syn.normal(syn.rng(M), (M, k), "bf16")).to(dev).view(torch.bfloat16)
                y = torch.empty((M, n), dtype=torch.bfloat16, device=dev)
                wsb = g.gguf_mm_workspace_size(g.GGUF_OP_GEMM, qt, n, k, M)
                ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device=dev)
                cell = {}
                for path, tag in ((g.GGUF_PATH_GEMV, "gemv"), (g.GGUF_PATH_FUSED, "fused")):
                    if path == g.GGUF_PATH_GEMV and M > 8:
                        continue
                    calls = 10 * c
                    t = time_graph(lambda i: g.gguf_mm_gemm(W[i % c], qt, layout, n, k, x, g.GGUF_DT_BF16, M, None,
                                                            y, g.GGUF_DT_BF16, ws, wsb, path, stream=stream),
                                   3, stream, calls)
                    cell[tag] = round(t * 1e6, 2)
                row[M] = cell
            table[f"{name}_{n}x{k}"] = row
            print(name, n, k, json.dumps(row), flush=True)
            del W
            torch.cuda.empty_cache()
    if out_path:
        with open(out_path, "w") as f:
            json.dump(table, f, indent=1)
    return table


def run_gpu(args):
    ws, rank, local = dist_env()
    # the CPU pool first: spawned processes, before any GPU work in this one
    pool = OraclePool(host_cores()) if (rank == 0 and not args.no_cpu_baseline) else None
    import torch
    import gguf_quant_weight_gb300 as g
    import gguf_synth as syn

    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    g.load_library()
    stream = torch.cuda.Stream(device=dev)
    if args.crossover:
        crossover(dev, stream, args.crossover, args.crossover_formats)
        return
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
    kernels = {m: g.GEMV_KERNELS.get(g.gguf_mm_gemv_kernel(QTYPE, 0, N, K, m), "?") for m in MS}
    launches_per_call = {m: 1 if kernels[m] in ("rowlane", "tile") else 2 for m in MS}
    state = {"c": 0}

    def call(m):
        g.gguf_mm_gemv(W[state["c"] % copies], QTYPE, 0, N, K, xs[m], g.GGUF_DT_BF16, m, rsd[m], ys[m],
                       g.GGUF_DT_BF16, wss[m], wsz[m], stream=stream)
        state["c"] += 1

    def capture(seq):
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(graph, stream=stream):
                for m in seq:
                    call(m)
        return graph

    def make_plan(ncalls):
        """[(graph, replays)] for ncalls calls at each M, M by M (a copy is
        reused only after all the others: never an L2 hit).  One graph per M
        (up to 270 calls each): a graph that mixes the M's measured slower per
        call (7.35 us against 4.35 / 5.5 / 8.06 for M = 1 / 2 / 4 alone)."""
        out = []
        full, rem = divmod(ncalls, GRAPH_CALLS)
        for m in MS:
            if full:
                out.append((capture([m] * GRAPH_CALLS), full))
            if rem:
                out.append((capture([m] * rem), 1))
        return out

    def replay(plan_):
        for gr, cnt in plan_:
            for _ in range(cnt):
                gr.replay()

    with torch.cuda.stream(stream):
        for m in MS:
            for _ in range(3):
                call(m)
        stream.synchronize()
    plan = make_plan(args.steps)
    uploaded = all(upload_graph(gr, stream) for gr, _ in plan)   # no first-launch upload in the timed region
    with torch.cuda.stream(stream):
        replay(make_plan(max(args.warmup, 3)))
    stream.synchronize()

    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    smi_index = vis.split(",")[local].strip() if vis else str(local)
    clocks = ClockSampler(smi_index)
    clocks.start()
    time.sleep(0.3)

    def timed(body):
        if ws > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        t_host0 = time.time()
        with torch.cuda.stream(stream):
            e0.record(stream)
            body()
            e1.record(stream)
        e1.synchronize()
        torch.cuda.synchronize(dev)
        if ws > 1:
            torch.distributed.barrier()
        return e0.elapsed_time(e1) / 1e3, t_host0, time.time()

    sec, th0, th1 = timed(lambda: replay(plan))
    clk = clocks.summary(th0, th1)

    # end to end, eagerly through the C ABI: every call copies its inputs in
    # from pinned host memory, is launched from the host, and copies y out
    hx = {m: xs[m].cpu().pin_memory() for m in MS}
    hr = {m: rsd[m].cpu().pin_memory() for m in MS}
    hy = {m: torch.empty((m, N), dtype=torch.bfloat16).pin_memory() for m in MS}

    # the host leg holds raw pointers, as a C caller would (no tensor indexing per call)
    w_ptrs = [W[i].data_ptr() for i in range(copies)]
    host_args = {m: (hx[m].data_ptr(), xs[m].data_ptr(), hr[m].data_ptr(), rsd[m].data_ptr(), hy[m].data_ptr(),
                     ys[m].data_ptr(), wss[m].data_ptr(), wsz[m]) for m in MS}
    stream_ptr = stream.cuda_stream

    def call_host(m):
        # one C-ABI call: x and the residual copied in, the GEMV, y copied out
        xh, xd, rh, rd, yh, yd, wsp, wsn = host_args[m]
        g.gguf_mm_gemv_host(w_ptrs[state["c"] % copies], QTYPE, 0, N, K, xh, xd, g.GGUF_DT_BF16, m, rh, rd, yh, yd,
                            g.GGUF_DT_BF16, wsp, wsn, stream=stream_ptr)
        state["c"] += 1

    def eager_steps():
        for m in MS:
            for _ in range(args.steps):
                call_host(m)

    with torch.cuda.stream(stream):
        for m in MS:
            call_host(m)
    stream.synchronize()
    esec, _, _ = timed(eager_steps)
    clocks.stop()

    # each M on its own: graphs of 270 calls (reported beside the headline)
    per_m = {}
    for m in MS:
        t = time_graph(lambda i, m=m: call(m), 5, stream, GRAPH_CALLS)
        per_m[m] = t

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
    algo = {m: W_BYTES + m * K * 2 + 2 * m * N * 2 for m in MS}   # weights + x + residual + y
    algo_mean = sum(algo.values()) / len(MS)
    launches = steps * sum(launches_per_call[m] for m in MS)
    dominant = "gemv_rowlane_kernel" if all(kernels[m] == "rowlane" for m in MS) else "/".join(kernels.values())
    achieved = algo_mean * steps * len(MS) / sec / 1e9   # every launch of the timed region is this kernel
    traffic = recorded_traffic()
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws, "steps": steps, "warmup": args.warmup,
        "ms_per_step": sec / steps * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int8", "data": "synthetic",
        "config": {"workload": WORKLOAD, "N": N, "K": K, "M": list(MS), "qtype": "Q5_K",
                   "residual": True, "activations": "bf16", "output": "bf16",
                   "l2": f"weights rotate over {copies} copies ({copies * W_BYTES / 1e6:.0f} MB > 2x L2)",
                   "order": "each M a chain of calls", "graphs_uploaded_before_timing": uploaded,
                   "parallelism": f"replicas x{ws}"},
        "hbm_frac": round(value / ws / hbm, 4),
        "per_m": {str(m): [round(per_m[m] * 1e6, 3), round(W_BYTES / per_m[m] / 1e9, 1)] for m in MS},
        "e2e": {"value": e2e, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "path": "eager host calls of gguf_mm_gemv_host (x and residual copied in from pinned memory, "
                        "the GEMV, y copied out: one C-ABI call per step)"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(achieved / hbm, 4),
                     "traffic": None if traffic is None else round(sum(traffic[str(m)] for m in MS) / len(MS)),
                     "peak_kind": peak_kind, "kernel": dominant,
                     "algorithmic_bytes_per_launch": algo_mean},
        "gpu_launches": launches,
        "clocks": {"sm_mhz": clk["sm_mhz"], "sm_max_mhz": clk["sm_max_mhz"], "reasons": clk["reasons"]},
    }
    if rank == 0:
        if pool is not None:
            line["cpu_baseline"] = cpu_baseline(pool)
            pool.close()
        if not args.no_prefill:
            compact, detail = prefill_figures(dev, stream, tc, hbm, args.prefill_only)
            print("# prefill detail " + json.dumps({k: {kk: round(vv, 3) for kk, vv in v.items()}
                                                     for k, v in detail.items()}), flush=True)
            line["prefill"] = {"peak_tf": tc, **compact}
        print(json.dumps(line), flush=True)
    elif pool is not None:
        pool.close()
    if ws > 1:
        torch.distributed.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--prefill-only", default=None, metavar="REGEX",
                    help="run only the prefill figures whose key matches (e.g. q6p_14336x4096_m512)")
    ap.add_argument("--crossover", default=None, metavar="OUT.json",
                    help="time GEMV against fused GEMM for M = 1..16 instead, and write the table")
    ap.add_argument("--crossover-formats", default=None, metavar="REGEX",
                    help="with --crossover: only the formats whose name matches")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
