#!/usr/bin/env python3
"""Benchmark of the fused split-KV Flash Decode on GB300.

Prints ONE JSON line on rank 0.  A step is one fused decode (all of the hot
path: KV streaming, scores, online softmax, P.V, partial write, arrival and the
last-arriver combine) over one batch of synthetic input.  The default workload is
the largest decode case: B=64 sequences of 8192 tokens, GQA 32/8, d=128, bf16,
W=16 segments each (2.15 GB of K/V per decode).

  value     KV-read GB/s over exactly --steps steps replayed from a CUDA graph,
            inputs resident in HBM, launched back to back; K/V rotate over
            enough copies that every step reads from HBM (copies x bytes >= 4 x L2).
  latency   per-launch device time (CUDA events around every launch).
  isolated  one decode alone: an L2 flush (a read of a 2 x L2 buffer, an unrelated
            kernel) runs before every decode, and events bracket the decode only.
  roofline  KV bytes per launch / mean launch time vs the measured HBM peak.
  extra_cases  the 32K and 128K single-sequence cases, step and isolated figures.
  e2e       the same metric through fd_decode with pinned HOST buffers: every
            step copies q, K, V in and out, lse back.
  cpu_baseline  the fp64 oracle on all host cores (a process per core, split over
            (sequence, query head)) and on 1 core, bounded sample.

``--impl reference`` times the fp64 oracle instead (rank 0 only).
Multi-GPU: N independent replicas (the decode has no cross-GPU exchange).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "batch64_gqa4_d128_L8k_bf16"
DEFAULT_W = 16
# Reported beside the headline: the 32K and 128K single-sequence decode cases.
EXTRA_CASES = ("gqa4_d128_L32k_W8", "gqa8_d128_L128k_W8_spiky")
METRIC = "decode latency (µs) and achieved KV-read HBM GB/s (% of GB300 peak), 1 GPU"
FALLBACK_HBM_GBS = 6800.0


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["fd", "reference"], default="fd")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--W", type=int, default=DEFAULT_W, help="segments for the batch64 W-sweep workload")
    ap.add_argument("--B", type=int, default=64,
                    help="sequences of the batch64 workload (fewer: a smaller case of the same kernel)")
    ap.add_argument("--chunks", type=int, default=0, help="chunks per segment (0 = planner)")
    ap.add_argument("--two-launch", action="store_true", help="split + combine as two kernels")
    ap.add_argument("--ffma", action="store_true", help="CUDA-core consumers even when G >= 4")
    ap.add_argument("--tcgen05", action="store_true", help="tcgen05 tensor cores (d = 128, G >= 4)")
    ap.add_argument("--mma-sync", action="store_true",
                    help="mma.sync tensor cores where tcgen05 is the default (G = 16)")
    ap.add_argument("--cluster-combine", action="store_true",
                    help="combine each (sequence, KV head) pair inside one thread-block cluster")
    ap.add_argument("--combiners", type=int, choices=[1, 2, 4, 8, 16], default=0,
                    help="cap on the CTAs that share one pair's combine (0 = planner)")
    ap.add_argument("--deep-ring", action="store_true",
                    help="two CTAs per SM with 96 KB rings even for many short CTAs")
    ap.add_argument("--no-pdl", action="store_true", help="launch without programmatic dependent launch")
    ap.add_argument("--no-cluster", action="store_true",
                    help="one partial record per chunk (no in-cluster segment merge)")
    ap.add_argument("--cluster", action="store_true",
                    help="always merge chunk partials per segment inside a cluster")
    ap.add_argument("--kv", choices=["native", "e4m3"], default="native",
                    help="K/V storage: the case's 16-bit type, or FP8 E4M3 (q stays 16-bit)")
    ap.add_argument("--paged", type=int, default=0, metavar="P",
                    help="K/V in a shuffled page pool with P tokens per page (block tables)")
    ap.add_argument("--waits", action="store_true",
                    help="fine-grained waits: slot 0 combines partials as their flags arrive")
    ap.add_argument("--soak-s", type=float, default=1.5, help="untimed load before timing (clocks)")
    ap.add_argument("--e2e-steps", type=int, default=30)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-budget-s", type=float, default=120.0)
    ap.add_argument("--no-graph", action="store_true", help="launch each step from Python")
    ap.add_argument("--no-extra", action="store_true", help="skip the 32K / 128K extra cases")
    ap.add_argument("--no-read-floor", action="store_true",
                    help="skip timing a plain read of the same bytes")
    ap.add_argument("--extra-steps", type=int, default=500)
    ap.add_argument("--cpu-baseline-only", action="store_true", help=argparse.SUPPRESS)
    return ap.parse_args(argv)


def make_problem(args):
    import workloads
    if args.workload.startswith("batch64"):
        prob = workloads.batch64_gqa4_d128_L8k_bf16(W=args.W, B=getattr(args, "B", 64))
    elif args.workload in workloads.EXTRA:
        prob = workloads.EXTRA[args.workload]()
    else:
        prob = workloads.CASES[args.workload]()
    if getattr(args, "kv", "native") == "e4m3":
        prob = workloads.with_e4m3_kv(prob)
    return prob


# ---------------------------------------------------------------------------
# Multi-rank plumbing (replicas only).
# ---------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def dist_init(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Largest `value` over all ranks (every rank gets it)."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_throughput(units_per_rank: float, elapsed_s: float, world: int, device=None) -> dict:
    """Whole-job throughput: the units all ranks processed / the slowest rank's time."""
    slowest = max_over_ranks(elapsed_s, world, device)
    return {"elapsed_s": slowest, "units": units_per_rank * world,
            "throughput": units_per_rank * world / slowest if slowest > 0 else float("nan")}


# ---------------------------------------------------------------------------
# Clock sampling during the measured window.
# ---------------------------------------------------------------------------

_REASON_BITS = {
    0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
    0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
    0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown", 0x100: "display_clock_setting",
}


class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active")

    def __init__(self, gpu_id: str, period_ms: int = 100):
        self.gpu_id, self.period_ms = gpu_id, period_ms
        self.lines, self.proc, self.thread = [], None, None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", f"-lms={self.period_ms}"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return self

        def pump():
            for line in self.proc.stdout:
                self.lines.append((time.time(), line.strip()))
        self.thread = threading.Thread(target=pump, daemon=True)
        self.thread.start()
        return self

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float) -> dict:
        sm, mx, pw, reasons = [], [], [], set()
        for ts, line in self.lines:
            if not (t0 <= ts <= t1):
                continue
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 5:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
                pw.append(float(parts[3]))
                bits = int(parts[4], 16)
            except ValueError:
                continue
            for bit, name in _REASON_BITS.items():
                if bits & bit and name != "gpu_idle":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(pw)}


# ---------------------------------------------------------------------------
# CPU side: the fp64 oracle (cpu_baseline and the reference arm).
# ---------------------------------------------------------------------------

def _kv_elem_bytes(problem):
    return 1 if problem.kv_type == "e4m3" else 2


def _oracle_sample(problem, n_tokens):
    """The first n_tokens of every sequence (all heads) as a standalone problem."""
    import numpy as np
    cu = problem.cu_seqlens
    lens = np.minimum(problem.seqlens.astype(np.int64), n_tokens)
    ks = [problem.k[cu[b]:cu[b] + lens[b]] for b in range(problem.B)]
    vs = [problem.v[cu[b]:cu[b] + lens[b]] for b in range(problem.B)]
    k = np.concatenate(ks) if ks else problem.k[:0]
    v = np.concatenate(vs) if vs else problem.v[:0]
    nbytes = int(lens.sum()) * problem.Hkv * problem.d * 2 * _kv_elem_bytes(problem)
    return lens, k, v, nbytes


def time_oracle_step(problem, n_tokens):
    import oracle
    lens, k, v, nbytes = _oracle_sample(problem, n_tokens)
    t = time.perf_counter()
    oracle.decode_reference(problem.q, k, v, lens, problem.dtype, kv_dtype=problem.kv_dtype or None)
    return time.perf_counter() - t, nbytes


# The sample the worker processes decode: set before the pool forks, so that every
# worker inherits it (this process never touches the GPU, so forking is safe).
_SAMPLE = None


def _oracle_heads(heads):
    import oracle
    q, k, v, lens, dtype, kv_dtype = _SAMPLE
    oracle.decode_reference(q, k, v, lens, dtype, heads=heads, kv_dtype=kv_dtype)
    return len(heads)


class ParallelOracle:
    """The fp64 oracle on every host core: one process per core, each decoding a
    contiguous share of the (sequence, query head) pairs of the same sample."""

    def __init__(self, problem, n_tokens, cores=None):
        import multiprocessing as mp
        global _SAMPLE
        lens, k, v, self.nbytes = _oracle_sample(problem, n_tokens)
        _SAMPLE = (problem.q, k, v, lens, problem.dtype, problem.kv_dtype or None)
        self.cores = int(cores or os.cpu_count() or 1)
        pairs = [(b, h) for b in range(problem.B) for h in range(problem.Hq)]
        n = min(self.cores, len(pairs))
        self.shares = [pairs[i * len(pairs) // n:(i + 1) * len(pairs) // n] for i in range(n)]
        self.pool = mp.get_context("fork").Pool(self.cores)

    def step(self):
        t = time.perf_counter()
        self.pool.map(_oracle_heads, self.shares, chunksize=1)
        return time.perf_counter() - t, self.nbytes

    def close(self):
        self.pool.close()
        self.pool.join()


def _choose_sample(prob, budget_s):
    """Tokens per sequence such that one 1-thread oracle decode takes about budget_s."""
    n = int(prob.seqlens.max())
    dt, nb = time_oracle_step(prob, min(n, 2048))
    per_byte = dt / max(nb, 1)
    full = prob.kv_bytes
    return n if per_byte * full <= budget_s else max(256, int(n * budget_s / (per_byte * full)))


def cpu_baseline_only(args):
    """Runs in a subprocess that never touches the GPU: the oracle on a bounded sample,
    about cpu_seconds on all cores, then about cpu_seconds on one core."""
    prob = make_problem(args)
    n = int(prob.seqlens.max())
    n_tok = _choose_sample(prob, args.cpu_seconds / 3.0)
    frac = "all" if n_tok >= n else f"first {n_tok}"
    what = f"fp64 oracle decode of {prob.name} ({frac} tokens of every sequence, all heads)"

    par = ParallelOracle(prob, n_tok)
    par.step()                                         # warm the workers
    pt, pb, pcalls = 0.0, 0, 0
    while pt < args.cpu_seconds and pcalls < 1000:
        dt, nb = par.step()
        pt, pb, pcalls = pt + dt, pb + nb, pcalls + 1
    par.close()

    st, sb, scalls = 0.0, 0, 0
    while st < args.cpu_seconds and scalls < 1000:
        dt, nb = time_oracle_step(prob, n_tok)
        st, sb, scalls = st + dt, sb + nb, scalls + 1
    return {"value": pb / pt / 1e9, "unit": "GB/s", "cores": par.cores, "kind": "oracle",
            "sample": f"{pcalls} x {what}, {pt:.1f} s wall on {par.cores} processes (one per "
                      f"host core, split over (sequence, query head)), 1 BLAS thread each",
            "single_core": {"value": sb / st / 1e9, "unit": "GB/s", "cores": 1,
                            "sample": f"{scalls} x the same decode, {st:.1f} s, 1 thread"}}


def run_cpu_baseline_subprocess(args):
    env = dict(os.environ, **_ONE_THREAD)
    cmd = [sys.executable, os.path.abspath(__file__), "--cpu-baseline-only", "--workload",
           args.workload, "--W", str(args.W), "--B", str(args.B), "--cpu-seconds", str(args.cpu_seconds),
           "--kv", args.kv]
    res = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=900)
    if res.returncode != 0:
        return {"value": None, "unit": "GB/s", "cores": 1, "kind": "oracle",
                "sample": "failed: " + res.stderr.strip().splitlines()[-1] if res.stderr else "failed"}
    return json.loads(res.stdout.strip().splitlines()[-1])


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    prob = make_problem(args)
    n = int(prob.seqlens.max())
    steps, warm = max(1, args.steps), max(0, args.warmup)
    cores = os.cpu_count() or 1
    # Budget per step on all cores; the calibration runs on one.
    n_tok = _choose_sample(prob, cores * args.ref_budget_s / (steps + warm))
    par = ParallelOracle(prob, n_tok, cores)
    for _ in range(warm):
        par.step()
    total_t, total_b = 0.0, 0
    for _ in range(steps):
        dt, nb = par.step()
        total_t += dt
        total_b += nb
    par.close()
    value = total_b / total_t / 1e9
    frac = "all" if n_tok >= n else f"first {n_tok}"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
        "n_gpus": args.gpus, "steps": steps, "warmup": warm,
        "ms_per_step": total_t / steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded N(0,1))",
        "config": {"workload": prob.name, **prob.describe()},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": par.cores, "kind": "oracle",
                         "sample": f"each step: fp64 oracle decode of {prob.name} ({frac} tokens "
                                   f"of every sequence, all heads), {par.cores} processes"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# GPU arm.
# ---------------------------------------------------------------------------

KERNEL_SOURCES = ("split_kv_flash_decode_gb300/csrc/fd_kernel.cuh",
                  "split_kv_flash_decode_gb300/csrc/fd_common.h",
                  "split_kv_flash_decode_gb300/csrc/fd_tcgen05.cuh")


def kernel_source_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def load_traffic(workload: str, kernel: str):
    """DRAM bytes (read + write) per launch from a committed ncu capture of this
    kernel on this workload; None when there is none or the kernel changed since."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            entry = json.load(f).get(workload, {}).get(kernel)
    except (OSError, ValueError):
        return None
    if not entry or entry.get("kernel_source_sha256_16") != kernel_source_hash():
        return None
    return int(entry["dram__bytes_read.sum"]) + int(entry["dram__bytes_write.sum"])


def load_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def to_device(x, dtype, device):
    import numpy as np
    import torch
    if dtype == "f16" or x.dtype == np.uint8:
        t = torch.from_numpy(np.ascontiguousarray(x))
    else:
        t = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16)
    return t.to(device)


def plan_flags(fd, args, prob):
    return (fd.FD_PLAN_LITERAL_W if prob.literal_w else 0) | (
        fd.FD_PLAN_TWO_LAUNCH if args.two_launch else 0) | (fd.FD_PLAN_FFMA if args.ffma else 0) | (
        fd.FD_PLAN_NO_PDL if args.no_pdl else 0) | (fd.FD_PLAN_WAITS if args.waits else 0) | (
        fd.FD_PLAN_NO_CLUSTER if args.no_cluster else 0) | (fd.FD_PLAN_CLUSTER if args.cluster else 0) | (
        fd.FD_PLAN_TCGEN05 if args.tcgen05 else 0) | (
        fd.FD_PLAN_CLUSTER_COMBINE if args.cluster_combine else 0) | (
        fd.FD_PLAN_MMA_SYNC if args.mma_sync else 0) | (
        fd.FD_PLAN_COMBINERS[args.combiners] if args.combiners else 0) | (
        fd.FD_PLAN_DEEP_RING if args.deep_ring else 0)


class CaseRun:
    """One workload on the device: plan, rotated K/V copies, and three CUDA graphs
    over the same K steps: back to back (the timed region), one event pair around
    every launch, and every launch alone after an L2 flush."""

    def __init__(self, fd, args, prob, device, stream, steps):
        import torch
        self.fd, self.args, self.prob, self.stream, self.K = fd, args, prob, stream, steps
        props = torch.cuda.get_device_properties(device)
        self.l2 = int(getattr(props, "L2_cache_size", 126 * 1024 * 1024))
        kv_bytes = prob.kv_bytes
        # Rotate K/V copies so consecutive steps never find their K/V in L2.
        copies = 1 if kv_bytes == 0 else max(1, math.ceil(4 * self.l2 / kv_bytes))
        self.copies = min(copies, max(1, int(40e9 // max(kv_bytes, 1))))
        plan_dtype = "f16_e4m3kv" if prob.kv_type == "e4m3" else prob.dtype
        self.dec = fd.Decoder(prob.Hq, prob.Hkv, prob.d, prob.seqlens, prob.W, plan_dtype,
                              flags=plan_flags(fd, args, prob), chunks=args.chunks, device=device,
                              page_size=args.paged)
        self.q = to_device(prob.q, prob.dtype, device)
        if args.paged:
            import workloads
            kp, vp, table = workloads.to_paged(prob, args.paged)
            k0, v0 = to_device(kp, prob.dtype, device), to_device(vp, prob.dtype, device)
            self.bt = torch.from_numpy(table).to(device)
            self.num_pages = kp.shape[0]
        else:
            k0 = to_device(prob.k, prob.dtype, device)
            v0 = to_device(prob.v, prob.dtype, device)
        self.k0, self.v0 = k0, v0
        self.ks = [k0] + [k0.clone() for _ in range(self.copies - 1)]
        self.vs = [v0] + [v0.clone() for _ in range(self.copies - 1)]
        self.out = torch.empty_like(self.q)
        self.lse = torch.empty((prob.B, prob.Hq), dtype=torch.float32, device=device)
        # An unrelated kernel between isolated decodes: a read of twice the L2 size
        # (a read leaves clean lines, as a weight-streaming GEMM before attention
        # would; a write would leave dirty lines for the decode to write back).
        self.flush = torch.ones(2 * self.l2 // 4, dtype=torch.float32, device=device)
        self.launches_per_step = 2 if args.two_launch else 1
        with torch.cuda.stream(stream):
            for i in range(max(3, args.warmup)):
                self.step(i)
        stream.synchronize()
        self.use_graph = not args.no_graph
        try:
            torch.cuda.Event(enable_timing=True, external=True)
        except TypeError:
            self.use_graph = False
        K = self.K
        self.ev = [(self._event(), self._event()) for _ in range(K)]
        self.ev_iso = [(self._event(), self._event()) for _ in range(K)]
        self.ev_all = (self._event(), self._event())
        self.graphs = {}
        if self.use_graph:
            for name, fn in (("a", self._record_a), ("b", self._record_b), ("c", self._record_c)):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    fn()
                self.graphs[name] = g
            stream.synchronize()

    def _event(self):
        import torch
        # Inside a CUDA graph the events must be "external" to become timing records.
        if self.use_graph:
            return torch.cuda.Event(enable_timing=True, external=True)
        return torch.cuda.Event(enable_timing=True)

    def step(self, i):
        fd, a = self.fd, self.args
        c = i % self.copies
        if a.paged:
            fd.fd_decode_paged(self.dec.plan, self.q, self.ks[c], self.vs[c], self.num_pages, self.bt,
                               self.bt.shape[1], self.out, self.lse, self.dec.workspace, self.stream)
        else:
            fd.fd_decode(self.dec.plan, self.q, self.ks[c], self.vs[c], self.out, self.lse,
                         self.dec.workspace, self.stream)

    def _record_a(self):
        self.ev_all[0].record(self.stream)
        for i in range(self.K):
            self.step(i)
        self.ev_all[1].record(self.stream)

    def _record_b(self):
        for i in range(self.K):
            self.ev[i][0].record(self.stream)
            self.step(i)
            self.ev[i][1].record(self.stream)

    def _record_c(self):
        for i in range(self.K):
            self.flush_sum = self.flush.sum()
            self.ev_iso[i][0].record(self.stream)
            self.step(i)
            self.ev_iso[i][1].record(self.stream)

    def run(self, name):
        import torch
        # A graph replays on torch's current stream: make that the decode stream.
        with torch.cuda.stream(self.stream):
            if self.use_graph:
                self.graphs[name].replay()
            else:
                {"a": self._record_a, "b": self._record_b, "c": self._record_c}[name]()

    def timed_ms(self):
        return self.ev_all[0].elapsed_time(self.ev_all[1])

    def per_launch_us(self, which):
        evs = self.ev if which == "b" else self.ev_iso
        return [x.elapsed_time(y) * 1e3 for x, y in evs]


class ReadFloor:
    """A plain read of the same number of bytes by a library kernel (torch's sum over
    float32 words), timed like the decode: back to back, one event pair around each
    launch, and alone after the same 2 x L2 flush.  It puts the single-decode figures
    next to what any kernel reading those bytes achieves under the same events."""

    def __init__(self, nbytes, l2, device, stream, steps):
        import torch
        self.stream, self.K = stream, steps
        words = max(1, nbytes // 4)
        copies = max(1, math.ceil(4 * l2 / max(nbytes, 1)))
        copies = min(copies, max(1, int(20e9 // max(nbytes, 1))))
        self.bufs = [torch.ones(words, dtype=torch.float32, device=device) for _ in range(copies)]
        self.flush = torch.ones(2 * l2 // 4, dtype=torch.float32, device=device)
        self.res = torch.empty((), dtype=torch.float32, device=device)
        ev = lambda: torch.cuda.Event(enable_timing=True, external=True)  # noqa: E731
        self.ev_all = (ev(), ev())
        self.ev_b = [(ev(), ev()) for _ in range(steps)]
        self.ev_c = [(ev(), ev()) for _ in range(steps)]
        with torch.cuda.stream(stream):
            for i in range(3):
                torch.sum(self.bufs[i % len(self.bufs)], dim=0, out=self.res)
        stream.synchronize()
        self.graphs = {}
        for name in ("a", "b", "c"):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                self._record(name)
            self.graphs[name] = g
        stream.synchronize()

    def _record(self, name):
        import torch
        if name == "a":
            self.ev_all[0].record(self.stream)
        for i in range(self.K):
            if name == "c":
                self.flush_sum = self.flush.sum()
            if name != "a":
                (self.ev_b if name == "b" else self.ev_c)[i][0].record(self.stream)
            torch.sum(self.bufs[i % len(self.bufs)], dim=0, out=self.res)
            if name != "a":
                (self.ev_b if name == "b" else self.ev_c)[i][1].record(self.stream)
        if name == "a":
            self.ev_all[1].record(self.stream)

    def measure(self):
        import torch
        out = {}
        with torch.cuda.stream(self.stream):
            for name in ("a", "a", "b", "c"):
                self.graphs[name].replay()
                self.stream.synchronize()
        out["step_us"] = self.ev_all[0].elapsed_time(self.ev_all[1]) * 1e3 / self.K
        out["latency_us"] = statistics.median(x.elapsed_time(y) * 1e3 for x, y in self.ev_b)
        out["isolated_us"] = statistics.median(x.elapsed_time(y) * 1e3 for x, y in self.ev_c)
        out["what"] = ("torch.sum over the same number of bytes (float32), same three "
                       "graphs and events as the decode; medians")
        return out


def read_floor(nbytes, l2, device, stream, steps):
    """ReadFloor figures, or None where CUDA-graph timing events are unavailable."""
    import torch
    try:
        torch.cuda.Event(enable_timing=True, external=True)
    except TypeError:
        return None
    rf = ReadFloor(nbytes, l2, device, stream, steps)
    out = rf.measure()
    del rf
    torch.cuda.empty_cache()
    return out


def stats_us(xs):
    qs = sorted(xs)

    def pct(p):
        return qs[min(len(qs) - 1, max(0, int(round(p / 100 * (len(qs) - 1)))))]
    return {"mean": statistics.fmean(qs), "median": statistics.median(qs), "p10": pct(10),
            "p90": pct(90), "min": qs[0], "max": qs[-1]}


def extra_case(fd, args, name, device, stream, peak):
    """Step (back to back) and isolated (after an L2 flush) figures of one more case."""
    import copy
    import workloads
    a = copy.copy(args)
    a.workload = name
    prob = make_problem(a)
    run = CaseRun(fd, a, prob, device, stream, max(1, args.extra_steps))
    run.run("a")
    stream.synchronize()
    run.run("a")
    stream.synchronize()
    step_us = run.timed_ms() * 1e3 / run.K
    run.run("b")
    stream.synchronize()
    lat = stats_us(run.per_launch_us("b"))
    run.run("c")
    stream.synchronize()
    iso = stats_us(run.per_launch_us("c"))
    if run.dec.status() != fd.FD_OK:
        raise RuntimeError(f"device status word reported an error on {name}")
    kv = prob.kv_bytes
    l2 = run.l2
    out = {"workload": prob.name, "kv_bytes_per_step": kv, "steps": run.K,
           "ctas": run.dec.info["ctas"], "chunks_per_segment": run.dec.info["chunks"],
           "step_us": step_us, "step_gbs": kv / (step_us * 1e-6) / 1e9,
           "frac_step": kv / (step_us * 1e-6) / 1e9 / peak,
           "latency_us": lat,
           "frac_latency": kv / (lat["median"] * 1e-6) / 1e9 / peak,
           "isolated_us": iso,
           "isolated_gbs": kv / (iso["median"] * 1e-6) / 1e9,
           "frac_isolated": kv / (iso["median"] * 1e-6) / 1e9 / peak}
    del run
    import torch
    torch.cuda.empty_cache()
    if not args.no_read_floor:
        out["plain_read"] = read_floor(kv, l2, device, stream, min(max(1, args.extra_steps), 200))
    return out


def run_fd(args):
    import torch

    import split_kv_flash_decode_gb300 as fd
    from split_kv_flash_decode_gb300 import build

    rank, world, local = dist_env()
    if world > 1:
        torch.cuda.set_device(local)
        dist_init(world, "nccl")
    device = torch.device("cuda", torch.cuda.current_device())
    build.build()
    prob = make_problem(args)
    props = torch.cuda.get_device_properties(device)
    stream = torch.cuda.Stream(device)
    K = max(1, args.steps)
    run = CaseRun(fd, args, prob, device, stream, K)
    dec, kv_bytes, copies, l2 = run.dec, prob.kv_bytes, run.copies, run.l2

    gpu_id = getattr(props, "uuid", None)
    gpu_id = f"GPU-{gpu_id}" if gpu_id is not None and not str(gpu_id).startswith("GPU-") else str(gpu_id or local)
    sampler = ClockSampler(gpu_id).start()
    t_soak = time.time()
    # Soak: the same replay, untimed, so clocks settle and the sampler sees the load.
    while time.time() - t_soak < args.soak_s:
        run.run("a")
        stream.synchronize()
    barrier(world)
    torch.cuda.synchronize(device)
    run.run("a")                  # the timed region: exactly K steps
    stream.synchronize()
    torch.cuda.synchronize(device)
    t_end = time.time()
    barrier(world)
    total_ms = run.timed_ms()
    run.run("b")                  # per-launch latency of the same K steps
    stream.synchronize()
    run.run("c")                  # each decode alone, after an L2 flush
    stream.synchronize()
    sampler.stop()
    clocks = sampler.summary(t_soak, t_end)
    if dec.status() != fd.FD_OK:
        raise RuntimeError("device status word reported an error during the timed region")

    agg = aggregate_throughput(kv_bytes * K / 1e9, total_ms / 1e3, world, device)
    value = agg["throughput"]  # GB/s, whole job
    step_us = total_ms * 1e3 / K
    lat = stats_us(run.per_launch_us("b"))
    iso = stats_us(run.per_launch_us("c"))

    peak, peak_kind = load_peak()
    # Average device time per launch over the timed region (back-to-back launches).
    achieved = kv_bytes / (step_us * 1e-6) / 1e9
    achieved_iso = kv_bytes / (iso["median"] * 1e-6) / 1e9

    # e2e through the public API with pinned host buffers.
    if args.paged:
        e2e = e2e_res = None  # the host-buffer path is measured on the contiguous layout
    else:
        e2e = e2e_measure(fd, dec, prob, device, args.e2e_steps, stream, kv_resident=False)
        e2e_res = e2e_measure(fd, dec, prob, device, max(args.e2e_steps, 200), stream,
                              kv_resident=True, dev_kv=(run.k0, run.v0))
    info = dec.info
    del run
    torch.cuda.empty_cache()
    floor = None if args.no_read_floor else read_floor(kv_bytes, l2, device, stream, min(K, 200))

    extras = {}
    if not args.no_extra and world == 1 and not args.paged:
        for name in EXTRA_CASES:
            if name != prob.name:
                extras[name] = extra_case(fd, args, name, device, stream, peak)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = run_cpu_baseline_subprocess(args)

    kernel_label = ("fd_split_kernel+fd_combine_kernel" if args.two_launch else "fd_split_kernel") + (
        {0: "/ffma", 1: "/mma", 2: "/mma-fp8", 3: "/tcgen05"}[info["path"]]) + ("/waits" if args.waits else "")
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K,
            "warmup": max(3, args.warmup), "ms_per_step": agg["elapsed_s"] * 1e3 / K,
            "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": prob.dtype,
            "data": "synthetic (seeded N(0,1) per tensor)",
            "config": {
                "workload": prob.name, **prob.describe(), "accumulate": "f32",
                "chunks_per_segment": info["chunks"], "ctas": info["ctas"],
                "records_per_segment": info["records_per_segment"],
                "combiners": info["combiners"], "ctas_per_sm": info["ctas_per_sm"],
                "partials_per_sequence_max": info["max_partials"],
                "kv_bytes_per_step": kv_bytes, "two_launch": bool(args.two_launch),
                "kv_storage": prob.kv_type,
                "pdl": not args.no_pdl and not args.waits,
                "kv_layout": f"paged ({args.paged} tokens per page, shuffled pool)" if args.paged
                             else "contiguous [N, Hkv, d]",
                "combine": "fine-grained waits (slot 0 combines as flags arrive)" if args.waits
                           else ("separate combine kernel" if args.two_launch
                                 else (f"in a cluster of {info['combine_cluster']} CTAs per (sequence,"
                                       " KV head), distributed shared memory"
                                       if info["combine_cluster"] else
                                       ("last arriver (atomic counter)" if info["combiners"] == 1 else
                                        f"the last {info['combiners']} arrivers (atomic counter),"
                                        " split by query heads"))),
                "consumer": {0: "FFMA (CUDA cores)", 1: "mma.sync m16n8k16 (tensor cores)",
                             2: "mma.sync m16n8k16 over E4M3 K/V widened in registers",
                             3: "tcgen05.mma (accumulators in tensor memory)"}[info["path"]],
                "l2_policy": f"K/V rotated over {copies} device copies ({copies * kv_bytes / 1e6:.0f} MB"
                             f" >= 4 x L2 {l2 / 1e6:.0f} MB)" if copies > 1 else
                             f"inputs larger than L2: K/V {kv_bytes / 1e6:.0f} MB per step >= 4 x L2"
                             f" {l2 / 1e6:.0f} MB",
                "launch": "CUDA graph replay of the K steps" if run_graph_ok(args) else "eager",
                "parallelism": f"replicas x{world}",
            },
            "latency_us": {**lat, "what": "one decode, CUDA events around each launch, "
                                         "launched back to back (second replay)"},
            "isolated_us": {**iso, "what": "one decode alone: a sum over a 2 x L2 buffer (an "
                                          "unrelated kernel) before each, events around the "
                                          "decode only (third replay)"},
            "step_us": step_us,
            "plain_read": floor,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak,
                         "traffic": load_traffic(prob.name, kernel_label),
                         "traffic_unit": "bytes per launch (ncu dram read + write)",
                         "algorithmic_bytes": kv_bytes,
                         "achieved_from": "KV bytes per launch / (timed-region time / K)",
                         "achieved_isolated": achieved_iso,
                         "frac_isolated": achieved_iso / peak,
                         "peak_kind": f"{peak_kind} (hbm_gbs copy, burst)",
                         "kernel": kernel_label},
            "extra_cases": extras,
            "e2e": e2e, "e2e_resident_kv": e2e_res,
            "gpu_launches": K * (2 if args.two_launch else 1),
            "kv_tokens_per_s": prob.n_tokens * K * world / agg["elapsed_s"],
            "clocks": clocks, "cpu_baseline": cpu,
            "gpu": props.name,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def run_graph_ok(args):
    import torch
    if args.no_graph:
        return False
    try:
        torch.cuda.Event(enable_timing=True, external=True)
    except TypeError:
        return False
    return True


def e2e_measure(fd, dec, prob, device, steps, stream, kv_resident, dev_kv=None):
    """KV GB/s through fd_decode with pinned host inputs copied in and results copied out."""
    import numpy as np
    import torch
    def pinned(x):
        if prob.dtype == "f16" or x.dtype == np.uint8:
            t = torch.from_numpy(np.ascontiguousarray(x))
        else:
            t = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16)
        return t.pin_memory()
    hq = pinned(prob.q)
    dq = torch.empty(hq.shape, dtype=hq.dtype, device=device)
    if kv_resident:
        dk, dv = dev_kv
    else:
        hk, hv = pinned(prob.k), pinned(prob.v)
        dk = torch.empty(hk.shape, dtype=hk.dtype, device=device)
        dv = torch.empty(hv.shape, dtype=hv.dtype, device=device)
    dout = torch.empty_like(dq)
    dlse = torch.empty((prob.B, prob.Hq), dtype=torch.float32, device=device)
    hout = torch.empty(dout.shape, dtype=dout.dtype).pin_memory()
    hlse = torch.empty(dlse.shape, dtype=dlse.dtype).pin_memory()
    h2d = hq.numel() * 2 + (0 if kv_resident else 2 * prob.k.nbytes)
    d2h = hout.numel() * 2 + hlse.numel() * 4

    def one():
        dq.copy_(hq, non_blocking=True)
        if not kv_resident:
            dk.copy_(hk, non_blocking=True)
            dv.copy_(hv, non_blocking=True)
        fd.fd_decode(dec.plan, dq, dk, dv, dout, dlse, dec.workspace, stream)
        hout.copy_(dout, non_blocking=True)
        hlse.copy_(dlse, non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(3):
            one()
        stream.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            one()
        e1.record(stream)
        stream.synchronize()
    ms = e0.elapsed_time(e1) / steps
    return {"value": prob.kv_bytes / (ms * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": ms,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": steps,
            "what": ("q copied in, K/V resident in HBM" if kv_resident else
                     "q, K, V copied in from pinned host memory") + ", out + lse copied back"}


_ONE_THREAD = {"OPENBLAS_NUM_THREADS": "1", "OMP_NUM_THREADS": "1", "MKL_NUM_THREADS": "1",
               "NUMEXPR_NUM_THREADS": "1"}


def main(argv=None):
    args = parse_args(argv)
    if args.cpu_baseline_only or args.impl == "reference":
        # The oracle legs report cores = 1: pin BLAS to one thread before numpy loads.
        os.environ.update(_ONE_THREAD)
    if args.cpu_baseline_only:
        print(json.dumps(cpu_baseline_only(args)), flush=True)
        return 0
    if args.impl == "reference":
        return run_reference(args)
    return run_fd(args)


if __name__ == "__main__":
    sys.exit(main())
