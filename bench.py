#!/usr/bin/env python3
"""Benchmark of the weight-only matmul C = A @ W^T on GB300.

Headline workload: the Q8_0 decode GEMV, M=1, N=4096, K=4096 (metric: achieved
HBM GB/s on the algorithmic bytes W + A + C, as a fraction of the measured
HBM peak). One step is one decode pass over a stack of R such weight matrices
(R copies whose total exceeds twice the L2), each multiplied by its own
activation row. For M = 1 the pass is one lq_gemv_chain call (the R GEMVs are
independent: each has its own A and C); the same pass as R separate
lq_matmul calls, and as a chain whose every problem waits for the previous
one, is reported under "workloads" too. Steps are captured as CUDA graphs
(eight steps back to back, and one for a remainder) and replayed, so the GPU
never waits on the host and, as in a decode loop, a step's kernels may start
streaming their weights while the previous step finishes. The other workload
families (the f16 / Q4_0 GEMVs, the LM head, the prefill GEMMs and the
M = 2 .. 64 crossover) are timed the same way under "workloads", each
entry "name [mode]": [value, unit, fraction of the measured peak, µs a
matmul], the prefill GEMMs last.

`--impl reference` times the CPU oracle on a bounded sample of the same
workload (rank 0 only) and prints the same JSON line with "impl": "reference".

Inputs are synthetic and seeded (synthetic.py); nothing is read from disk
except the measured peaks and the committed ncu summaries.
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import synthetic  # noqa: E402

HEADLINE = "gemv_q8_0_4096x4096"
GRAPH_STEPS = 8  # steps captured in one CUDA graph for the timed replays

KERNEL_OF_MODE = {"chain": "gemv_chain_kernel", "chain-dependent": "gemv_chain_kernel",
                  "calls": "gemv_stream_kernel", "argmax": "gemv_stream_kernel",
                  "argmax-unfused": "gemv_stream_kernel", "topk": "gemv_stream_kernel"}
METRIC = "decode GEMV achieved HBM GB/s (% of peak); prefill GEMM TFLOP/s (% peak)"
L2_BYTES = 129 * 2**20
FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS = 6800.0, 1900.0


# ---------------------------------------------------------------- helpers
def algorithmic_bytes(fmt, M, N, K) -> int:
    row = {"f16": 2 * K, "q8_0": K // 32 * 34, "q4_0": K // 32 * 18}[fmt]
    return N * row + 4 * M * K + 4 * M * N


def flops(M, N, K) -> int:
    return 2 * M * N * K


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return (float(p["hbm_gbs"]), float(p["bf16_tflops"]),
                float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), "measured")
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


def ncu_traffic(workload: str, kernel: str):
    """DRAM bytes per launch of the dominant kernel, from the committed ncu
    summary of this kernel and workload (profiles/<kernel>.<workload>.md, line
    'traffic_bytes_per_launch: <int>'); None when there is no summary or when
    a kernel source it lists ('source: <path> <sha256 prefix>') has changed
    since the capture."""
    for path in sorted(glob.glob(os.path.join(ROOT, "profiles", f"{kernel}.{workload}.md"))):
        with open(path) as f:
            text = f.read()
        m = re.search(r"traffic_bytes_per_launch:\s*(\d+)", text)
        if not m:
            continue
        for src, digest in re.findall(r"source:\s*(\S+)\s+([0-9a-f]{16})", text):
            try:
                with open(os.path.join(ROOT, src), "rb") as g:
                    if hashlib.sha256(g.read()).hexdigest()[:16] != digest:
                        return None
            except OSError:
                return None
        return int(m.group(1))
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.out = ""

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- workloads
class Workbench:
    """R device copies of one workload's packed weights (R chosen so that the
    copies together exceed twice the L2), R activation blocks and R outputs;
    step() runs the library's router once per copy."""

    def __init__(self, lq, w: synthetic.Workload, dev, copies=None, max_bytes=3 * 2**30,
                 mode="auto"):
        """mode: "calls" (one lq_matmul per copy), "chain" (one lq_gemv_chain
        over the independent copies), "chain-dependent" (every problem waits
        for the previous one), "argmax" (M = 1: one lq_gemv_argmax per copy,
        logits not stored), "argmax-unfused" (M = 1: lq_matmul into C, then
        lq_argmax_f32 on C), "topk" (M = 1: lq_gemv_topk with k = 50), "tc" /
        "batch" (M > 1: separate calls forced onto the tensor-core route or
        the CUDA-core batched decode kernel, to compare the two where the
        router picks one), or "auto" (chain for M = 1, else calls)."""
        self.lq, self.w, self.dev = lq, w, dev
        W, A = synthetic.draw_workload(w)
        packed = lq.pack(w.fmt, W).reshape(-1).view(np.uint8)
        self.wbytes = packed.nbytes
        R = copies or max(1, math.ceil(2 * L2_BYTES / (self.wbytes + 4 * w.M * (w.K + w.N))))
        R = max(1, min(R, max_bytes // max(self.wbytes, 1)))
        self.R = R
        base = torch.from_numpy(packed).to(dev)
        self.Wd = [base] + [base.clone() for _ in range(R - 1)]
        self.A_host = A.unsqueeze(0).expand(R, -1, -1).contiguous().pin_memory()
        self.Ad = self.A_host.to(dev)
        self.Cd = torch.empty((R, w.M, w.N), dtype=torch.float32, device=dev)
        self.C_host = torch.empty((R, w.M, w.N), dtype=torch.float32).pin_memory()
        self.fn = getattr(lq, f"lq_matmul_{w.fmt}")
        self.bytes_per_launch = algorithmic_bytes(w.fmt, w.M, w.N, w.K)
        self.flops_per_launch = flops(w.M, w.N, w.K)
        self.graph = None
        if mode == "auto":
            mode = "chain" if w.M == 1 else "calls"
        self.problems = None
        if mode.startswith("chain") and w.M == 1:
            # one chain call per 64 problems (the call's limit)
            after = 1 if mode == "chain-dependent" else 0
            self.problems = [
                lq.gemv_problems([(self.Ad[r], self.Wd[r], self.Cd[r], w.N, w.K, after if r > r0 else 0)
                                  for r in range(r0, min(R, r0 + 64))])
                for r0 in range(0, R, 64)]
            if any(lq.lq_gemv_chain(w.fmt, arr) != lq.LQ_OK for arr in self.problems):
                self.problems = None  # outside the chain's path: separate calls
            torch.cuda.synchronize(dev)
        self.mode = mode if self.problems is not None else "calls"
        self.route = None
        self.res = None
        if mode.startswith("argmax") and w.M == 1:
            self.mode = mode
            self.res = torch.zeros((R, 3), dtype=torch.int64, device=dev)
        if mode == "topk" and w.M == 1:
            self.mode = mode
            self.topk = [lq.topk_buffers(w.N, 50, dev) for _ in range(R)]
        if mode in ("tc", "batch") and w.M > 1:
            self.mode = mode
        # kernels of ours per step
        if self.problems is not None:
            self.kernels_per_step = len(self.problems)
        elif self.mode == "topk":
            self.kernels_per_step = 3 * R
        elif self.mode == "argmax-unfused" or w.M >= 2:
            self.kernels_per_step = 2 * R
        else:
            self.kernels_per_step = R

    def step(self, stream=None):
        w = self.w
        if self.problems is not None:
            for arr in self.problems:
                self.lq.lq_gemv_chain(w.fmt, arr, stream)
            return
        if self.mode == "argmax":
            for r in range(self.R):
                self.lq.lq_gemv_argmax(w.fmt, self.Ad[r], self.Wd[r], None, w.N, w.K, self.res[r], stream)
            return
        if self.mode == "topk":
            for r in range(self.R):
                v, i, wk = self.topk[r]
                self.lq.lq_gemv_topk(w.fmt, self.Ad[r], self.Wd[r], self.Cd[r], w.N, w.K, 50, v, i, wk, stream)
            return
        if self.mode in ("tc", "batch"):
            self.lq.force_route(self.lq.ROUTE_TENSOR_CORE if self.mode == "tc" else self.lq.ROUTE_STREAM)
        try:
            for r in range(self.R):
                self.fn(self.Ad[r], self.Wd[r], self.Cd[r], w.M, w.N, w.K, stream)
                if self.mode == "argmax-unfused":
                    self.lq.lq_argmax_f32(self.Cd[r], w.N, self.res[r], stream)
        finally:
            if self.mode in ("tc", "batch"):
                self.lq.force_route(0)

    def capture(self):
        s = torch.cuda.Stream(device=self.dev)
        s.wait_stream(torch.cuda.current_stream(self.dev))
        self.lq.reset_counts()
        with torch.cuda.stream(s):
            self.step()          # eager warm-up (sets kernel attributes)
        torch.cuda.current_stream(self.dev).wait_stream(s)
        torch.cuda.synchronize(self.dev)
        if self.w.M >= 2:
            # launches a step, counted on the eager step: one a matmul, plus
            # the tcgen05 route's A pre-pass where it runs
            lq = self.lq
            self.kernels_per_step = sum(lq.route_count(r) for r in (1, 2, lq.ROUTE_WARP_MMA, lq.COUNT_PREPASS))
            if lq.route_count(1) >= self.R:
                self.route = "batch"        # the CUDA-core batched decode kernel
            elif lq.route_count(lq.ROUTE_WARP_MMA) >= self.R:
                self.route = "warp-mma"     # M = 5..16: warp-level MMAs
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.step()
        torch.cuda.synchronize(self.dev)
        self.graph = g
        # GRAPH_STEPS steps back to back in one graph, as a decode loop issues
        # them: each step's kernels may start streaming their weights while
        # the previous step finishes (programmatic dependent launch works
        # within a graph, not across two graph launches)
        gn = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gn):
            for _ in range(GRAPH_STEPS):
                self.step()
        torch.cuda.synchronize(self.dev)
        self.graph_n = gn
        st = self.lq.last_device_error()
        if st != self.lq.LQ_OK:
            raise RuntimeError(f"device status after warm-up: {self.lq.status_string(st)}")

    def replay(self, steps: int):
        """Exactly `steps` steps: whole GRAPH_STEPS-step graphs, then
        single-step ones."""
        full, rest = divmod(steps, GRAPH_STEPS)
        for _ in range(full):
            self.graph_n.replay()
        for _ in range(rest):
            self.graph.replay()

    def time_graph(self, steps: int, warmup: int, barrier=None):
        """Device time in seconds of `steps` steps replayed from the graphs
        (CUDA events on the replay stream), after `warmup` steps."""
        stream = torch.cuda.current_stream(self.dev)
        self.replay(warmup)
        torch.cuda.synchronize(self.dev)
        if barrier:
            barrier()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        self.replay(steps)
        t1.record(stream)
        torch.cuda.synchronize(self.dev)
        if barrier:
            barrier()
        return t0.elapsed_time(t1) / 1e3

    def replay_spread(self, n: int):
        """p10 / p50 / p90 of the device time of single graph replays, per
        matmul, in µs (each replay bracketed by its own CUDA events)."""
        stream = torch.cuda.current_stream(self.dev)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for a, b in ev:
            a.record(stream)
            self.graph.replay()
            b.record(stream)
        torch.cuda.synchronize(self.dev)
        us = sorted(a.elapsed_time(b) * 1e3 / self.R for a, b in ev)
        q = lambda f: us[min(len(us) - 1, int(f * len(us)))]
        return {"unit": "us_per_matmul", "p10": q(0.1), "p50": q(0.5), "p90": q(0.9), "replays": n}

    def time_e2e(self, steps: int):
        """Through the public API with host buffers: per step the pinned A
        goes to the device, the router runs on every copy, C comes back to
        the host and is read."""
        stream = torch.cuda.current_stream(self.dev)
        torch.cuda.synchronize(self.dev)
        t0 = time.perf_counter()
        checksum = 0.0
        for _ in range(steps):
            self.Ad.copy_(self.A_host, non_blocking=True)
            self.step()
            self.C_host.copy_(self.Cd, non_blocking=True)
            stream.synchronize()
            checksum += float(self.C_host[0, 0, 0])
        dt = time.perf_counter() - t0
        return dt, self.A_host.numel() * 4, self.C_host.numel() * 4, checksum

    def free(self):
        self.graph = self.graph_n = None
        self.Wd = self.Ad = self.Cd = None
        torch.cuda.empty_cache()


def rate(wb: Workbench, seconds_per_launch: float):
    """(value, unit, roofline bound) of one launch of this workload."""
    if wb.w.M >= 128:
        return wb.flops_per_launch / seconds_per_launch / 1e12, "TFLOP/s", "tensor"
    return wb.bytes_per_launch / seconds_per_launch / 1e9, "GB/s", "hbm"


# ---------------------------------------------------------------- CPU oracle
def oracle_rate(w: synthetic.Workload, seconds: float, rows=None):
    """Time the CPU oracle (dequantise + float64 matmul, as it stands) on the
    workload's inputs, restricted to `rows` weight rows, for about `seconds`;
    the oracle's quantisation of those rows is timed on its own. Returns
    (bytes/s of algorithmic traffic, sample description, calls, seconds,
    quantisation seconds)."""
    import oracle as O
    W, A = synthetic.draw_workload(w)
    Wn, An = W.numpy(), A.numpy()
    n = w.N if rows is None else min(rows, w.N)
    tq = time.perf_counter()
    packed = O.pack(w.fmt, Wn[:n])
    quant_s = time.perf_counter() - tq
    calls, t0 = 0, time.perf_counter()
    while True:
        O.reference(w.fmt, An, packed, n, w.K, tensor_core=w.M >= 128)
        calls += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    b = algorithmic_bytes(w.fmt, w.M, n, w.K)
    return (b * calls / dt, f"{calls} oracle call(s) of M={w.M}, N={n} of {w.N}, K={w.K} ({w.fmt})",
            calls, dt, quant_s)


def oracle_subprocess(workload: str, seconds: float, threads):
    """oracle_rate in a fresh interpreter whose BLAS and OpenMP pools have
    `threads` threads (None: the library default, every core), so that the
    thread count is fixed before numpy loads. Returns the parsed dict or an
    {"error": ...} dict."""
    env = dict(os.environ)
    env["CUDA_VISIBLE_DEVICES"] = ""  # the oracle never touches the GPU
    if threads:
        for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            env[k] = str(threads)
    cmd = [sys.executable, os.path.abspath(__file__), "--oracle-sample", workload,
           "--oracle-seconds", str(seconds)]
    try:
        r = subprocess.run(cmd, env=env, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True,
                           timeout=seconds * 6 + 120)
        for line in r.stdout.splitlines()[::-1]:
            if line.startswith("{"):
                return json.loads(line)
        return {"error": (r.stderr or r.stdout).strip().splitlines()[-1:] or ["no output"]}
    except (subprocess.TimeoutExpired, OSError, ValueError) as e:
        return {"error": str(e)}


def workload_config(w: synthetic.Workload) -> dict:
    """The `config` of both arms' lines: the workload itself."""
    return {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "format": w.fmt,
            "l2": "inputs larger than L2 (device arm: rotating weight copies, together "
                  "more than twice the L2)"}


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


# ---------------------------------------------------------------- main
def max_over_ranks(x: float, world: int, device) -> float:
    """The largest of the ranks' values (the job is as slow as its slowest
    rank); the value itself with one rank."""
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def init_dist(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() and args.impl != "reference" else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def run_reference(args, world, rank):
    """The oracle on the headline workload's config, as it stands, on the
    host cores: each step is one oracle call on a row sample sized so that
    the whole run takes about a minute."""
    if rank != 0:
        return
    import oracle as O
    w = synthetic.WORKLOADS[args.workload]
    steps, warmup = args.steps or 20, args.warmup
    _, _, _, dt1, _ = oracle_rate(w, 0.0, rows=64)
    per_row = dt1 / 64
    rows = int(max(8, min(w.N, args.ref_seconds / max(steps + warmup, 1) / max(per_row, 1e-9))))
    W, A = synthetic.draw_workload(w)
    packed = O.pack(w.fmt, W.numpy()[:rows])
    An = A.numpy()
    for _ in range(warmup):
        O.reference(w.fmt, An, packed, rows, w.K, tensor_core=w.M >= 128)
    t0 = time.perf_counter()
    for _ in range(steps):
        O.reference(w.fmt, An, packed, rows, w.K, tensor_core=w.M >= 128)
    dt = time.perf_counter() - t0
    b = algorithmic_bytes(w.fmt, w.M, rows, w.K)
    val = b * steps / dt / 1e9
    sample = f"each step: oracle on M={w.M}, N={rows} of {w.N} rows, K={w.K} ({w.fmt})"
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": "GB/s", "n_gpus": world,
        "steps": steps, "warmup": warmup, "ms_per_step": dt / steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(w),
        "cpu_baseline": {"value": val, "unit": "GB/s", "cores": cpu_cores(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


EXTRA = ["gemv_f16_256x512", "gemv_q4_0_11008x4096_outliers", "gemv_f16_lmhead_151936x2048",
         "gemm_f16_512x6144x2048", "gemm_q8_0_512x6144x2048", "gemm_q4_0_512x6144x2048"] + \
        [f"gemm_{f}_m{m}_6144x2048" for m in (2, 4, 8, 16, 32, 64) for f in ("f16", "q8_0", "q4_0")]


def workload_rank(key: str) -> tuple:
    """Order of the "workloads" entries in the JSON line: the tensor-core
    and batched alternatives of the small-M GEMMs first, then the router's
    small-M GEMMs, the decode GEMVs, the LM head's selections, and the
    prefill GEMMs (M = 512) last, so that a reader keeping only the end of
    the line still has the metric's prefill half and the decode families."""
    if "512x" in key:
        group = 4
    elif "lmhead" in key:
        group = 3
    elif key.startswith("gemv_"):
        group = 2
    elif "[tc]" in key or "[batch]" in key:
        group = 0
    else:
        group = 1
    return (group, key)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: enough for about 1.5 s of device time)")
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(synthetic.WORKLOADS))
    ap.add_argument("--extras", default="all",
                    help="comma-separated extra workloads to time, 'all' or 'none'")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-seconds", type=float, default=60.0,
                    help="--impl reference: seconds of oracle work the whole run aims at")
    ap.add_argument("--mode", default="auto",
                    choices=["auto", "calls", "chain", "chain-dependent", "argmax", "argmax-unfused", "topk",
                             "tc", "batch"],
                    help="how the headline step runs its matmuls (auto: chain for M = 1; argmax modes: "
                         "M = 1, the GEMV with its argmax)")
    ap.add_argument("--oracle-sample", default=None, help=argparse.SUPPRESS)
    ap.add_argument("--oracle-seconds", type=float, default=10.0, help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.oracle_sample:
        w = synthetic.WORKLOADS[args.oracle_sample]
        bps, sample, calls, cdt, quant_s = oracle_rate(w, args.oracle_seconds)
        print(json.dumps({"bps": bps, "sample": sample, "calls": calls, "seconds": cdt,
                          "quantise_s": quant_s}), flush=True)
        return
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world, rank, local = init_dist(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
        return

    import gemm_gemv_f16w_gb300 as lq
    from gemm_gemv_f16w_gb300 import build as lqbuild
    if rank == 0 or not os.path.exists(lq.LIB_PATH):
        lqbuild.build()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    lq.lib()
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    hbm_peak, tc_peak, _, peak_src = peaks()

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    def ranks_max(x: float) -> float:
        return max_over_ranks(x, world, dev)

    # ---- headline workload
    w = synthetic.WORKLOADS[args.workload]
    wb = Workbench(lq, w, dev, mode=args.mode)
    wb.capture()
    probe = wb.time_graph(3, 1)
    steps = args.steps or max(20, int(1.5 / max(probe / 3, 1e-7)))
    lq.reset_counts()
    with ClockSampler(local) as clk:
        dt = wb.time_graph(steps, args.warmup, barrier)
    dt = ranks_max(dt)
    clocks = clk.summary()
    spread = wb.replay_spread(100)  # outside the timed region
    if w.M == 1:
        kernel = KERNEL_OF_MODE[wb.mode]
    else:
        kernel = {"batch": "gemv_batch_kernel", "warp-mma": "gemm_small_kernel"}.get(wb.route, "gemm_tma_kernel")
    launches_per_step = wb.kernels_per_step
    per_gemv = dt / (steps * wb.R)          # one matmul of the workload
    val1, unit, bound = rate(wb, per_gemv)
    value = val1 * world  # every rank runs the same per-GPU work (weak scaling)
    peak = hbm_peak if bound == "hbm" else tc_peak
    # the dominant kernel's launches: the step's work divided evenly
    per_launch = dt / (steps * launches_per_step)
    work_per_launch = (wb.bytes_per_launch if bound == "hbm" else wb.flops_per_launch) * wb.R / launches_per_step
    roofline = {"bound": bound, "achieved": val1, "peak": peak, "unit": unit,
                "frac": val1 / peak, "traffic": ncu_traffic(w.name, kernel),
                "peak_source": f"{peak_src} ({'hbm_gbs' if bound == 'hbm' else 'bf16_tflops'})",
                "kernel": kernel, "algorithmic_per_launch": work_per_launch,
                "us_per_launch": per_launch * 1e6}
    e2e_dt, h2d, d2h, _ = wb.time_e2e(steps)
    e2e_dt = ranks_max(e2e_dt)
    e2e_val = wb.bytes_per_launch * wb.R * steps / e2e_dt / 1e9 * world
    wb.free()

    # ---- the other workload families (same method, shorter runs)
    extras = {}
    names = EXTRA if args.extras == "all" else ([] if args.extras == "none" else args.extras.split(","))
    runs = []
    for name in names:
        if name == w.name:
            continue
        runs.append((name, "auto"))
        if synthetic.WORKLOADS[name].M == 1:
            runs.append((name, "calls"))  # the decode GEMVs both as a chain and as separate calls
        m = synthetic.WORKLOADS[name].M
        if 1 < m <= 32:
            # the router's kernel (warp-MMA) against the tcgen05 kernel and,
            # up to eight rows, the batched decode kernel
            runs.append((name, "tc"))
            if m <= 8:
                runs.append((name, "batch"))
    if w.M == 1 and args.extras != "none":
        runs = [(w.name, "calls"), (w.name, "chain-dependent")] + runs
    lmhead = "gemv_f16_lmhead_151936x2048"
    if lmhead in names or (w.name == lmhead and args.extras != "none"):
        runs += [(lmhead, "argmax"), (lmhead, "argmax-unfused"), (lmhead, "topk")]
    for name, mode in runs:
        x = synthetic.WORKLOADS[name]
        xb = Workbench(lq, x, dev, mode=mode)
        xb.capture()
        p = xb.time_graph(2, 1)
        n = max(5, int(0.25 / max(p / 2, 1e-7)))
        d = ranks_max(xb.time_graph(n, 3, barrier))
        pl = d / (n * xb.R)
        v, u, b = rate(xb, pl)
        pk = hbm_peak if b == "hbm" else tc_peak
        key = f"{name} [{xb.mode}]"
        extras[key] = [round(v, 1), u, round(v / pk, 4), round(pl * 1e6, 3)]
        xb.free()
    extras = dict(sorted(extras.items(), key=lambda kv: workload_rank(kv[0])))

    # ---- CPU oracle baseline (rank 0 at N=1 only): all threads and one
    # thread, each in its own interpreter, quantisation timed separately
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        full = oracle_subprocess(w.name, 10.0, None)
        one = oracle_subprocess(w.name, 10.0, 1)
        if "bps" in full:
            cpu = {"value": full["bps"] / 1e9, "unit": "GB/s", "cores": cpu_cores(), "kind": "oracle",
                   "sample": f"{full['sample']}; {full['seconds']:.1f} s; numpy float64 "
                             f"(dequantise + BLAS matmul, every core)",
                   "value_1_thread": one["bps"] / 1e9 if "bps" in one else None,
                   "quantise_s": {"all_threads": full["quantise_s"],
                                  "1_thread": one.get("quantise_s")},
                   "quantise_sample": f"oracle pack of the same {w.N} x {w.K} weights ({w.fmt})"}
        else:
            cpu = {"value": None, "unit": "GB/s", "cores": cpu_cores(), "kind": "oracle",
                   "sample": f"oracle run failed: {full.get('error')}"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": unit, "n_gpus": world, "steps": steps,
            "warmup": args.warmup, "ms_per_step": dt / steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded torch.randn, recipe in synthetic.py)",
            "config": workload_config(w),
            "step": {"mode": wb.mode, "matmuls": wb.R, "launches": launches_per_step,
                     "weight_copies_mib": round(wb.R * wb.wbytes / 2**20), "l2_mib": L2_BYTES // 2**20,
                     "how": f"one pass over the weight-copy stack; K steps back to back on one stream, "
                            f"replayed from CUDA graphs of {GRAPH_STEPS} steps (and of 1 for the remainder)",
                     "parallelism": f"replicas x{world}"},
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_val, "unit": unit, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            "gpu_launches": steps * launches_per_step,
            "clocks": clocks,
            "spread": spread,
            "workloads_fields": ["value", "unit", "frac", "us"],
            "workloads": extras,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
