"""Benchmark: attention forward TFLOP/s (bf16, d=128) and fraction of the GB300 dense bf16 peak.

python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step is one call of the library's attention forward over one batch of the
workload (inputs already resident in HBM): the scheduler, TMA loads, both
tcgen05 MMAs, the softmax with delayed rescaling, the correction and the
epilogue all run inside that call. The default workload is the causal
B=4, H=16, N=4096, d=128 problem (Q, K, V iid N(0,1) in bf16, scale 1/sqrt(128)).
FLOPs per step follow the usual convention 4*B*H*N^2*d, halved for causal.

With N > 1 (torchrun), every rank runs its own replica of the workload on its
own GPU (independent problems, no collective on the data path; weak scaling);
a barrier brackets the timed region and the slowest rank's time is used.

``--impl reference`` times the fp64 CPU oracle (the test oracle under
oracle/, as it stands) on a bounded sample of the same workload and prints the
same JSON line with "impl": "reference".
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import fa_inputs  # noqa: E402

METRIC = "attention fwd TFLOPS (bf16, d=128) and % of GB300 dense BF16 tensor peak"
METRIC_BWD = "attention bwd TFLOPS (bf16, d=128) and % of GB300 dense BF16 tensor peak"
DEFAULT_WORKLOAD = "c3_b4h16n4096d128_causal"
FALLBACK_PEAK_TFLOPS = 1900.0
FLOP_PER_CLK_PER_SM = 8192  # dense bf16 tcgen05 rate per SM per clock


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(fa_inputs.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--pass", dest="which", default="fwd", choices=["fwd", "bwd"],
                    help="bwd: time the backward pass instead of the forward")
    a = ap.parse_args()
    if a.warmup < 3:
        ap.error("--warmup must be >= 3")
    return a


# --------------------------------------------------------------------------- distributed plumbing
class Dist:
    def __init__(self, n):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            backend = "nccl" if os.environ.get("FA_BENCH_BACKEND", "nccl") == "nccl" else "gloo"
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        import torch
        dev = "cuda" if self.pg.get_backend() == "nccl" else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


# --------------------------------------------------------------------------- helpers
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            j = json.load(f)
        return float(j["bf16_tflops"]), float(j.get("bf16_tflops_sustained", j["bf16_tflops"])), \
            float(j.get("hbm_gbs", 0.0)), "measured"
    except Exception:
        return FALLBACK_PEAK_TFLOPS, 1700.0, 6800.0, "fallback"


# The sources each pass's kernels are compiled from (a DRAM record stays valid while
# these are unchanged).
KERNEL_SOURCES = {
    "fwd": ("fa_api.cu", "fa_fwd.cuh", "fa_host.cuh", "ptx.cuh"),
    "bwd": ("fa_bwd_api.cu", "fa_bwd.cuh", "fa_fwd.cuh", "fa_host.cuh", "ptx.cuh"),
}


def _code_only(text: str) -> str:
    """C++ source without comments and blank lines (a comment edit is not a kernel change)."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = (re.sub(r"//.*$", "", line).rstrip() for line in text.splitlines())
    return "\n".join(line for line in lines if line)


def kernel_source_hash(which: str = "fwd") -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "attention_forward_tma_gb300", "csrc")
    for name in sorted(KERNEL_SOURCES[which]):
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(name.encode() + _code_only(f.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str, which: str = "fwd"):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on this kernel source."""
    path = os.path.join(ROOT, "profiles", f"fa_{which}_{workload}_dram.txt")
    try:
        kv = {}
        with open(path) as f:
            for line in f:
                if ":" in line and not line.startswith("#"):
                    k, v = line.split(":", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("kernel_source_sha256_16") != kernel_source_hash(which):
            return None
        return float(kv["dram_bytes_per_launch"])
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 20 ms while the benchmark runs;
    each sample carries the host time it was read, so that a time window can be summarised."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
    PERIOD_S = 0.02

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.samples = []   # (host time, sm MHz, max sm MHz, power W, reasons)

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(int(self.PERIOD_S * 1000))], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            t_end = time.perf_counter() + 10.0      # wait (bounded) for the first sample
            while not self.samples and time.perf_counter() < t_end and self.proc.poll() is None:
                time.sleep(0.01)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm, smax = float(parts[0]), float(parts[1])
            except ValueError:
                continue
            try:
                power = float(parts[2])
            except ValueError:
                power = None
            reasons = {n for n, v in zip(self.NAMES, parts[3:7]) if v.lower() == "active"}
            self.samples.append((time.perf_counter(), sm, smax, power, reasons))

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self, t0: float, t1: float):
        """Samples read in [t0 - period, t1 + period] (a short region still gets the samples around it)."""
        win = [x for x in self.samples if t0 - self.PERIOD_S <= x[0] <= t1 + self.PERIOD_S]
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "window_s": round(t1 - t0, 4)}
        reasons = set().union(*(x[4] for x in win))
        powers = [x[3] for x in win if x[3] is not None]
        return {"sm_mhz": statistics.median(x[1] for x in win), "sm_max_mhz": max(x[2] for x in win),
                "reasons": sorted(reasons), "samples": len(win), "window_s": round(t1 - t0, 4),
                "power_w_max": max(powers) if powers else None}


def workload_flops(w, x=None):
    if w.varlen:
        return fa_inputs.varlen_flops(x["lengths"], w.H, w.d, w.causal)
    return fa_inputs.attention_flops(w.B, w.H, w.N, w.d, w.causal, Nk=w.Nk)


def workload_bytes(w, x=None):
    """Compulsory HBM bytes of one step: read Q, K, V once, write O and LSE once."""
    if w.varlen:
        T = int(x["cu_seqlens"][-1])
        rows_q, rows_k = T, T
    else:
        rows_q, rows_k = w.B * w.N, w.B * w.Nk
    return 2.0 * w.d * (2 * rows_q * w.H + 2 * rows_k * w.Hkv) + 4.0 * rows_q * w.H


def oracle_sample(w, x, budget_rows: int, seed: int):
    """A bounded row sample of the workload for the CPU oracle, with its exact FLOPs."""
    rng = np.random.default_rng(seed)
    if w.varlen:
        cu = x["cu_seqlens"]
        T = int(cu[-1])
        toks = rng.integers(0, T, budget_rows)
        heads = rng.integers(0, w.H, budget_rows)
        rows = np.stack([heads, toks], 1).astype(np.int64)
        seq = np.searchsorted(cu, toks, side="right") - 1
        pos = toks - cu[seq]
        L = cu[seq + 1] - cu[seq]
        nkeys = np.minimum(pos + 1, L) if w.causal else L
    else:
        b = rng.integers(0, w.B, budget_rows)
        h = rng.integers(0, w.H, budget_rows)
        i = rng.integers(0, w.N, budget_rows)
        rows = np.stack([b, h, i], 1).astype(np.int64)
        nkeys = np.clip(i + (w.Nk - w.N) + 1, 0, w.Nk) if w.causal else np.full(budget_rows, w.Nk)
    flops = float((4.0 * w.d * nkeys).sum())
    return rows, flops


def run_oracle_rows(w, x, rows, threads):
    import oracle
    if w.varlen:
        return oracle.attention_rows_varlen(x["q"], x["k"], x["v"], x["cu_seqlens"], rows, w.scale, w.causal,
                                            threads=threads, dtype=w.dtype)
    return oracle.attention_rows(x["q"], x["k"], x["v"], rows, w.scale, w.causal, threads=threads, dtype=w.dtype)


def cpu_baseline(w, x, target_s: float = 10.0):
    """The oracle (as it stands) on a bounded row sample; TFLOP/s of the work it did."""
    import oracle
    threads = oracle.default_threads()
    rows, flops = oracle_sample(w, x, 256, seed=1)
    t0 = time.perf_counter()
    run_oracle_rows(w, x, rows, threads)
    dt = max(time.perf_counter() - t0, 1e-6)
    n = int(min(max(256, 256 * target_s / dt), 1 << 20))
    rows, flops = oracle_sample(w, x, n, seed=2)
    t0 = time.perf_counter()
    run_oracle_rows(w, x, rows, threads)
    dt = time.perf_counter() - t0
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"{n} random query rows of {w.name} (fp64 two-pass softmax per row, "
                      f"{flops / 1e9:.1f} GFLOP by the 4*d*keys count), {dt:.1f} s"}


def cpu_baseline_bwd(w, x):
    """The backward oracle (fp64 NumPy, as it stands) on one (sequence, K/V head group) of the workload."""
    import oracle
    Gq = w.H // w.Hkv
    if w.varlen:
        a_, b_ = int(x["cu_seqlens"][0]), int(x["cu_seqlens"][1])
        N, Nk = b_ - a_, b_ - a_
        q, k, v = (x[n][None, a_:b_, :g] for n, g in (("q", Gq), ("k", 1), ("v", 1)))
    else:
        N, Nk = w.N, w.Nk
        q, k, v = x["q"][:1, :, :Gq], x["k"][:1, :, :1], x["v"][:1, :, :1]
    do = fa_inputs.make_qkv(1, N, Gq, w.d, w.seed + 1000, dtype=w.dtype)[0]
    t0 = time.perf_counter()
    oracle.attention_backward(q, k, v, do, w.scale, w.causal, dtype=w.dtype)
    dt = time.perf_counter() - t0
    flops = 2.5 * fa_inputs.attention_flops(1, Gq, N, w.d, w.causal, Nk=Nk)
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count() or 1, "kind": "oracle",
            "sample": f"backward of {'sequence' if w.varlen else 'batch'} 0, K/V head 0 with its {Gq} query "
                      f"head(s) of {w.name} (fp64 NumPy, full matrices per head), {dt:.1f} s"}


def workload_config(w, x, l2_bytes: int, bwd: bool = False):
    """The JSON line's "config", the same for both arms: the workload, its sizes, input
    recipe (scale, seed), FLOPs per step and how the timing treats L2."""
    if w.varlen:
        T = int(x["cu_seqlens"][-1])
        in_bytes = 2 * (2 * T * w.H + 2 * T * w.Hkv) * w.d
    else:
        in_bytes = 2 * (2 * w.B * w.N * w.H + 2 * w.B * w.Nk * w.Hkv) * w.d
    flops = workload_flops(w, x) * (2.5 if bwd else 1.0)
    cfg = {"workload": w.name, "B": w.B, "H": w.H, "H_kv": w.Hkv, "N": w.N, "d": w.d, "causal": w.causal,
           "inputs": w.dtype, "scale": w.scale, "seed": w.seed,
           "l2": ("inputs larger than L2 (Q+K+V+O = %.0f MiB), no flush" % (in_bytes / 2 ** 20))
           if in_bytes > l2_bytes else
           ("inputs smaller than L2 (Q+K+V+O = %.1f MiB): 256 MiB written between steps, value from the "
            "per-step events" % (in_bytes / 2 ** 20)),
           "flops_per_step": flops}
    if bwd:
        cfg["pass"] = "backward (FLOPs = 2.5 x the forward count)"
    if w.Nk != w.N:
        cfg["N_kv"] = w.Nk
    if w.varlen:
        cfg["lengths"] = [int(L) for L in x["lengths"]]
    return cfg, in_bytes


def l2_size_bytes(index: int = 0) -> int:
    """The GPU's L2 size (a property query, no work on the GPU); GB300's if no GPU is visible."""
    try:
        import torch
        if torch.cuda.is_available():
            return int(torch.cuda.get_device_properties(index).L2_cache_size)
    except Exception:
        pass
    return 126 << 20


# --------------------------------------------------------------------------- the reference arm
def run_reference(a, dist):
    w = fa_inputs.WORKLOADS[a.workload]
    if dist.rank != 0:
        return
    import oracle
    x = fa_inputs.make_workload(w)
    threads = oracle.default_threads()
    # size one step so that warmup + steps take about a minute in total
    rows, flops = oracle_sample(w, x, 64, seed=0)
    t0 = time.perf_counter()
    run_oracle_rows(w, x, rows, threads)
    per_row = max(time.perf_counter() - t0, 1e-6) / 64
    total_steps = a.steps + a.warmup
    n_rows = int(max(1, min(4096, 60.0 / total_steps / per_row)))
    samples = [oracle_sample(w, x, n_rows, seed=100 + i) for i in range(total_steps)]
    for i in range(a.warmup):
        run_oracle_rows(w, x, samples[i][0], threads)
    flops = sum(s[1] for s in samples[a.warmup:])
    t0 = time.perf_counter()
    for i in range(a.warmup, total_steps):
        run_oracle_rows(w, x, samples[i][0], threads)
    dt = time.perf_counter() - t0
    value = flops / dt / 1e12
    cfg, _ = workload_config(w, x, l2_size_bytes(dist.local))
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "impl": "reference", "n_gpus": a.gpus,
            "steps": a.steps, "warmup": a.warmup, "ms_per_step": dt / a.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": cfg,
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                             "sample": f"{n_rows} random query rows of {w.name} per step"},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- our arm
def run_ours(a, dist):
    import torch
    import attention_forward_tma_gb300 as fa

    torch.cuda.set_device(dist.local)
    dev = torch.device("cuda", dist.local)
    w = fa_inputs.WORKLOADS[a.workload]
    x = fa_inputs.make_workload(w)
    flops = workload_flops(w, x)

    tdt = torch.float16 if w.dtype == "f16" else torch.bfloat16

    def to_dev(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(tdt).to(dev)

    q, k, v = to_dev(x["q"]), to_dev(x["k"]), to_dev(x["v"])
    o = torch.empty_like(q)
    bwd = a.which == "bwd"
    if w.varlen:
        cu = torch.from_numpy(x["cu_seqlens"]).to(dev)
        maxL = int(x["lengths"].max())
    if bwd:
        # dO drawn like Q from its own seed; O and LSE from one untimed forward
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        flops = 2.5 * flops   # five products against the forward's two
        if w.varlen:
            dout = to_dev(fa_inputs.make_qkv(1, q.shape[0], w.H, w.d, w.seed + 1000, dtype=w.dtype)[0][0])
            lse = torch.empty((w.H, q.shape[0]), dtype=torch.float32, device=dev)
            fa.fa_fwd_varlen(q, k, v, cu, maxL, scale=w.scale, causal=w.causal, out=o, lse=lse)

            def step(s=None):
                fa.fa_bwd_varlen(q, k, v, o, dout, lse, cu, maxL, scale=w.scale, causal=w.causal, dq=dq, dk=dk,
                                 dv=dv, stream=s)
        else:
            dout = to_dev(fa_inputs.make_qkv(w.B, w.N, w.H, w.d, w.seed + 1000, dtype=w.dtype)[0])
            lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
            fa.fa_fwd(q, k, v, scale=w.scale, causal=w.causal, out=o, lse=lse)

            def step(s=None):
                fa.fa_bwd(q, k, v, o, dout, lse, scale=w.scale, causal=w.causal, dq=dq, dk=dk, dv=dv, stream=s)
        splits = 1
        launches_per_step = 3   # preprocessing, backward, dQ conversion
    elif w.varlen:
        lse = torch.empty((w.H, q.shape[0]), dtype=torch.float32, device=dev)

        def step(s=None):
            fa.fa_fwd_varlen(q, k, v, cu, maxL, scale=w.scale, causal=w.causal, out=o, lse=lse,
                             num_splits=w.splits, stream=s)
        splits = fa.num_splits_varlen(len(x["lengths"]), q.shape[0], maxL, w.H, w.Hkv, w.splits)
        launches_per_step = 2 + (1 if splits > 1 else 0)   # schedule, attention (, merge)
    else:
        lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)

        def step(s=None):
            fa.fa_fwd(q, k, v, scale=w.scale, causal=w.causal, out=o, lse=lse, num_splits=w.splits, stream=s)
        splits = fa.num_splits(w.B, w.H, w.Hkv, w.N, w.Nk, w.splits, causal=w.causal, d=w.d)
        launches_per_step = 1 + (1 if splits > 1 else 0)   # attention (, merge)

    stream = torch.cuda.current_stream(dev)
    clocks = ClockSampler(dist.local).__enter__()
    for _ in range(a.warmup):
        step(stream)
    torch.cuda.synchronize(dev)
    st, word = fa.last_device_status(stream)
    if st != fa.FA_OK:
        raise RuntimeError(f"device status {st} ({word:#x}) after warm-up")

    # Inputs that fit in L2 would be served from L2 on repeated steps: then a
    # 256 MiB buffer is written between steps (outside the per-step events) and
    # the value comes from the per-step events alone.
    l2_bytes = torch.cuda.get_device_properties(dev).L2_cache_size
    cfg, in_bytes = workload_config(w, x, l2_bytes, bwd)
    flush_buf = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    flush = flush_buf if in_bytes <= l2_bytes else None

    def eager_steps():
        """K eager steps with CUDA events around each step on the launching stream."""
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(a.steps)]
        dist.barrier()
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        for i in range(a.steps):
            if flush is not None:
                flush.fill_(i & 0xff)
            ev[i][0].record(stream)
            step(stream)
            ev[i][1].record(stream)
        torch.cuda.synchronize(dev)
        t1 = time.perf_counter()
        dist.barrier()
        st, word = fa.last_device_status(stream)
        if st != fa.FA_OK:
            raise RuntimeError(f"device status {st} ({word:#x}) in the timed region")
        per_ms = [e0.elapsed_time(e1) for e0, e1 in ev]
        reg_ms = ev[0][0].elapsed_time(ev[-1][1]) if flush is None else sum(per_ms)
        return per_ms, reg_ms, t0, t1

    graph = None
    if flush is None:
        # timed region: the K steps captured once in a CUDA graph (each call captures
        # after one eager call per shape) and replayed, bracketed by events on the
        # launching stream; the same K steps launched eagerly are reported beside it.
        # Should capture fail, the eager region is the value (stated in `timing`).
        try:
            side = torch.cuda.Stream(dev)
            side.wait_stream(stream)
            with torch.cuda.stream(side):
                step(side)
            stream.wait_stream(side)
            torch.cuda.synchronize(dev)
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                cap = torch.cuda.current_stream(dev)
                for _ in range(a.steps):
                    step(cap)
            graph.replay()
            torch.cuda.synchronize(dev)
        except RuntimeError as e:
            print(f"bench: CUDA graph capture failed ({e}); timing eager launches", file=sys.stderr)
            graph = None
            torch.cuda.synchronize(dev)
        # every rank takes the same path (the paths differ in their barriers)
        if dist.max(0.0 if graph is not None else 1.0) != 0.0:
            graph = None
    if graph is not None:
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        dist.barrier()
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        g0.record(stream)
        graph.replay()
        g1.record(stream)
        torch.cuda.synchronize(dev)
        t1 = time.perf_counter()
        dist.barrier()
        st, word = fa.last_device_status(stream)
        if st != fa.FA_OK:
            raise RuntimeError(f"device status {st} ({word:#x}) in the timed region")
        region_ms = g0.elapsed_time(g1)
        timing = "CUDA graph of the K steps, one replay bracketed by events"
        per_launch_ms, eager_region_ms, _, _ = eager_steps()
        eager = {"ms_per_step": eager_region_ms / a.steps, "avg_launch_ms": sum(per_launch_ms) / a.steps,
                 "min_launch_ms": min(per_launch_ms),
                 "value": dist.world * flops * a.steps / dist.max(eager_region_ms / 1e3) / 1e12,
                 "timing": "K eager launches, events around each step"}
        avg_launch_s = region_ms / a.steps / 1e3
    else:
        per_launch_ms, region_ms, t0, t1 = eager_steps()
        timing = ("K eager launches, 256 MiB written between steps outside the per-step events"
                  if flush is not None else "K eager launches, events around each step (graph capture failed)")
        eager = None
        avg_launch_s = sum(per_launch_ms) / len(per_launch_ms) / 1e3
    wall = t1 - t0
    region_s = dist.max(region_ms / 1e3)
    value = dist.world * flops * a.steps / region_s / 1e12
    clk = clocks.summary(t0, t1)

    # sustained: at least 50 launches over at least 0.5 s, median per-launch time, with L2
    # left warm (back to back) and with 256 MiB written between launches (L2 flushed);
    # each with the clocks sampled over its own window
    n_sus = int(min(max(50, math.ceil(0.5 / max(avg_launch_s, 1e-6))), 20000))

    def sustained(flushed: bool):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_sus)]
        torch.cuda.synchronize(dev)
        s0 = time.perf_counter()
        for i in range(n_sus):
            if flushed:
                flush_buf.fill_(i & 0xff)
            evs[i][0].record(stream)
            step(stream)
            evs[i][1].record(stream)
        torch.cuda.synchronize(dev)
        s1 = time.perf_counter()
        ms = sorted(e0.elapsed_time(e1) for e0, e1 in evs)
        med = statistics.median(ms)
        return {"value": flops / (med / 1e3) / 1e12, "unit": "TFLOP/s", "median_launch_ms": med,
                "p10_launch_ms": ms[len(ms) // 10], "p90_launch_ms": ms[(9 * len(ms)) // 10], "launches": n_sus,
                "seconds": round(s1 - s0, 3), "clocks": clocks.summary(s0, s1)}

    sus = {"warm_l2": sustained(False), "flushed_l2": sustained(True)}
    st, word = fa.last_device_status(stream)
    if st != fa.FA_OK:
        raise RuntimeError(f"device status {st} ({word:#x}) in the sustained runs")
    clocks.__exit__(None, None, None)

    # end to end through the public API with host buffers (pinned), copies inside the region
    n_e2e = max(1, min(a.e2e_steps, a.steps))
    if bwd:
        ins = [q, k, v, o, dout, lse]
        outs = [dq, dk, dv]
    else:
        ins = [q, k, v]
        outs = [o, lse]
    h_in = [t.to("cpu").pin_memory() for t in ins]
    h_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs]
    # Steps are pipelined over three streams with two sets of device buffers: step i+1's
    # host->device copies overlap step i's kernels and step i-1's device->host copies.
    # Every step still copies its own inputs in and its own results out.
    d_in = [[torch.empty_like(t) for t in ins] for _ in range(2)]
    d_out = [[torch.empty_like(t) for t in outs] for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def call(di, do, st):
        if bwd and w.varlen:
            fa.fa_bwd_varlen(*di, cu, maxL, scale=w.scale, causal=w.causal, dq=do[0], dk=do[1], dv=do[2], stream=st)
        elif bwd:
            fa.fa_bwd(*di, scale=w.scale, causal=w.causal, dq=do[0], dk=do[1], dv=do[2], stream=st)
        elif w.varlen:
            fa.fa_fwd_varlen(*di, cu, maxL, scale=w.scale, causal=w.causal, out=do[0], lse=do[1],
                             num_splits=w.splits, stream=st)
        else:
            fa.fa_fwd(*di, scale=w.scale, causal=w.causal, out=do[0], lse=do[1], num_splits=w.splits, stream=st)

    def e2e_steps(n):
        for i in range(n):
            b = i % 2
            if i >= 2:
                s_in.wait_event(ev_comp[b])            # step i-2's kernels have read these inputs
            with torch.cuda.stream(s_in):
                for d_, h_ in zip(d_in[b], h_in):
                    d_.copy_(h_, non_blocking=True)
                ev_in[b].record(s_in)
            stream.wait_event(ev_in[b])
            if i >= 2:
                stream.wait_event(ev_out[b])           # step i-2's results have been copied out
            call(d_in[b], d_out[b], stream)
            ev_comp[b].record(stream)
            s_out.wait_event(ev_comp[b])
            with torch.cuda.stream(s_out):
                for h_, d_ in zip(h_out, d_out[b]):
                    h_.copy_(d_, non_blocking=True)
                ev_out[b].record(s_out)

    e2e_steps(2)
    torch.cuda.synchronize(dev)
    dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    e2e_steps(n_e2e)
    e1.record(s_out)
    torch.cuda.synchronize(dev)
    e2e_s = dist.max(e0.elapsed_time(e1) / 1e3)
    h2d = sum(t.numel() * t.element_size() for t in ins)
    d2h = sum(t.numel() * t.element_size() for t in outs)

    if dist.rank != 0:
        return
    peak, peak_sust, hbm, peak_src = measured_peaks()
    props = torch.cuda.get_device_properties(dev)
    max_mhz = clk["sm_max_mhz"] or sus["warm_l2"]["clocks"]["sm_max_mhz"] or 2070.0
    theoretical = props.multi_processor_count * FLOP_PER_CLK_PER_SM * max_mhz * 1e6 / 1e12
    traffic = profiled_traffic(w.name, a.which)
    # the bound follows the arithmetic intensity: below the ridge of the measured
    # peaks (FLOP per byte) the step is an HBM stream, above it a contraction
    nbytes = workload_bytes(w, x) * (2.0 if bwd else 1.0)   # bwd: Q, K, V, O, dO read; dQ, dK, dV written
    if flops / nbytes < peak * 1e12 / (hbm * 1e9):
        roof = {"bound": "hbm", "achieved": nbytes / avg_launch_s / 1e9, "peak": hbm, "unit": "GB/s",
                "frac": nbytes / avg_launch_s / 1e9 / hbm, "traffic": traffic,
                "peak_source": f"{peak_src} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)",
                "bytes_per_step": nbytes}
    else:
        achieved = flops / avg_launch_s / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "traffic": traffic,
                "peak_source": f"{peak_src} bf16 burst (MEASURED_PEAKS.json)" if peak_src == "measured"
                else "fallback 1.9 PFLOP/s bf16 burst"}
    roof.update({"kernel": ("fa_bwd_kernel (+ preprocessing, dQ conversion)" if bwd else
                            "fa_fwd_kernel" + (" + fa_varlen_schedule_kernel" if w.varlen else "")
                            + (" + fa_combine_kernel" if splits > 1 else "")),
                 "avg_launch_ms": avg_launch_s * 1e3, "duration_from": "timed region / steps" if eager
                 else "mean of the per-step events", "wall_s": wall})
    # the sustained roofline: the median launch of the mode that matches the value's L2
    # policy, against the sustained (power-capped) measured peak
    sus_main = sus["warm_l2"] if flush is None else sus["flushed_l2"]
    med_s = sus_main["median_launch_ms"] / 1e3
    if roof["bound"] == "hbm":
        sus["roofline"] = {"bound": "hbm", "achieved": nbytes / med_s / 1e9, "peak": hbm, "unit": "GB/s",
                           "frac": nbytes / med_s / 1e9 / hbm, "mode": "warm_l2" if flush is None else "flushed_l2",
                           "peak_source": f"{peak_src} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"}
    else:
        sus["roofline"] = {"bound": "tensor", "achieved": flops / med_s / 1e12, "peak": peak_sust,
                           "unit": "TFLOP/s", "frac": flops / med_s / 1e12 / peak_sust,
                           "mode": "warm_l2" if flush is None else "flushed_l2",
                           "peak_source": f"{peak_src} bf16 sustained (MEASURED_PEAKS.json bf16_tflops_sustained)"}
    line = {
        "metric": METRIC_BWD if bwd else METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": dist.world, "steps": a.steps,
        "warmup": a.warmup, "ms_per_step": region_s / a.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic", "config": cfg,
        "pct_of_measured_peak": 100.0 * value / dist.world / peak,
        "pct_of_theoretical_peak": 100.0 * value / dist.world / theoretical,
        "theoretical_peak_tflops": theoretical,
        "roofline": roof,
        "e2e": {"value": dist.world * flops * n_e2e / e2e_s / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n_e2e,
                "overlap": "step i+1's copies in | step i's kernels | step i-1's copies out, three streams"},
        "timing": timing,
        "eager": eager,
        "gpu_launches": launches_per_step * a.steps,
        "clocks": clk,
        "key_splits": splits,
        "sustained": sus,
    }
    if not a.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_bwd(w, x) if bwd else cpu_baseline(w, x)
    print(json.dumps(line), flush=True)


def main():
    a = parse()
    dist = Dist(a.gpus)
    try:
        if a.impl == "reference":
            run_reference(a, dist)
        else:
            run_ours(a, dist)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
