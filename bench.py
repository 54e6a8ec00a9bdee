"""Benchmark of the paged decode step: append the new token, then decode.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference] [--no-cpu-baseline]

A step is one pass of the whole path over one batch: the slot-mapped append
of every sequence's new token, then decode attention (split-K + log-sum-exp
combine) over every sequence's paged context.  Inputs are seeded synthetic
data resident in HBM.  The default workload is the largest of the five:
GQA bf16, 256 sequences, 32 query / 8 kv heads, head_dim 128, block_size 32,
contexts uniform in [1024, 8192] (about 4.8 GB of K/V a step, far larger than
the 129 MB L2, so no flush is needed between its steps).

Prints one JSON line (rank 0).  `value` is the effective HBM throughput of the
step in GB/s (algorithmic bytes: K/V in context, q, out, block-table entries,
and the append's reads and writes), summed over ranks; tokens/s is reported
beside it.  Under torchrun each rank runs its own independent batch (weak
scaling, no collective on the data path).
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import platform
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

REPO = os.path.dirname(os.path.abspath(__file__))
if REPO not in sys.path:
    sys.path.insert(0, REPO)

METRIC = "paged decode: effective KV HBM GB/s (% of GB300 peak) and decode tokens/sec"
DEFAULT_WORKLOAD = "gqa_bf16"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0
DTYPE_NAME = {torch.float32: "f32", torch.float16: "f16", torch.bfloat16: "bf16"}


# ---------------------------------------------------------------------------
# helpers


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def reduce_over_ranks(pg, ms, nbytes):
    """Whole-job time and bytes: the slowest rank's time, all ranks' bytes
    (weak scaling: every rank runs its own batch).  pg is torch.distributed
    with an initialised process group, or None for one process."""
    if pg is None:
        return ms, nbytes
    t = torch.tensor([ms, nbytes], dtype=torch.float64)
    tmax, tsum = t.clone(), t.clone()
    pg.all_reduce(tmax, op=pg.ReduceOp.MAX)
    pg.all_reduce(tsum, op=pg.ReduceOp.SUM)
    return float(tmax[0]), float(tsum[1])


def rank_spec(workload, rank, num_seqs=0):
    """The workload spec of one rank: same shapes, a seed of its own."""
    from paged_kv_cache_24_gb300.workloads import CONFIGS, config_spec

    base = config_spec(CONFIGS[workload])
    over = {"num_seqs": num_seqs} if num_seqs > 0 else {}
    return config_spec(CONFIGS[workload], seed=base.seed + 1000 * rank, **over)


def hbm_peak():
    path = os.path.join(REPO, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def step_bytes(w):
    """Algorithmic bytes of one step of workload `w` at each of its steps."""
    spec = w.spec
    e = torch.tensor([], dtype=spec.dtype).element_size()   # q / out / new tokens
    q8 = spec.kv_fp8 or spec.kv_int8
    row = d_row = spec.head_dim * (1 if q8 else e) + (4 if q8 else 0)
    B, hq, hkv, d, bs = (spec.num_seqs, spec.num_q_heads, spec.num_kv_heads, spec.head_dim,
                         spec.block_size)
    out = []
    tables = w.block_tables.cpu().numpy().astype(np.int64)
    for s in range(w.steps):
        L = w.lens_steps[s].cpu().numpy().astype(np.int64)
        lo = np.maximum(L - spec.window, 0) if spec.window > 0 else np.zeros_like(L)
        ctx = int((L - lo).sum())
        # distinct pool rows the step attends (sequences that share prefix
        # blocks read those rows once from DRAM at best)
        t = np.concatenate([np.arange(a, b) for a, b in zip(lo, L)] or [np.zeros(0, np.int64)])
        seq = np.repeat(np.arange(B), L - lo)
        rows = tables[seq, t // bs] * bs + t % bs
        kv_unique = int(np.unique(rows).size) * 2 * hkv * row
        pages = int((((L - 1) // bs) - (lo // bs) + 1).clip(min=0).sum())
        kv = ctx * 2 * hkv * row            # one K row and one V row per (token, kv head)
        qo = 2 * B * hq * d * e
        meta = pages * 4 + B * 4
        append = B * hkv * (d * e + d_row) * 2 + B * 8  # new rows read, pool rows written
        out.append({"kv": kv, "decode": kv + qo + meta, "append": append,
                    "step": kv + qo + meta + append, "tokens_kvhead": ctx * hkv,
                    "step_unique": kv_unique + qo + meta + append})
    return out


class ClockSampler:
    """Samples SM clock and clock-event reasons through NVML while running."""
    REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
               0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
               0x100: "display_clock_setting"}

    def __init__(self, index, period=0.01):
        self.samples, self.reasons, self.max_mhz = [], 0, None
        self.period, self._stop = period, threading.Event()
        self.ok = False
        try:
            self.nvml = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nvml.nvmlInit_v2() != 0:
                return
            self.h = ctypes.c_void_p()
            if self.nvml.nvmlDeviceGetHandleByIndex_v2(index, ctypes.byref(self.h)) != 0:
                return
            mx = ctypes.c_uint()
            if self.nvml.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = mx.value
            self.ok = True
        except OSError:
            pass

    def _poll(self):
        clk, rsn = ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop.is_set():
            if self.nvml.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(clk)) == 0:
                self.samples.append(clk.value)
            if self.nvml.nvmlDeviceGetCurrentClocksEventReasons(self.h, ctypes.byref(rsn)) == 0:
                self.reasons |= rsn.value
            time.sleep(self.period)

    def __enter__(self):
        if self.ok:
            self._t = threading.Thread(target=self._poll, daemon=True)
            self._t.start()
        return self

    def __exit__(self, *a):
        if self.ok:
            self._stop.set()
            self._t.join()

    def summary(self):
        if not self.ok:
            return None
        names = [n for bit, n in self.REASONS.items() if self.reasons & bit and n != "gpu_idle"]
        return {"sm_mhz": statistics.median(self.samples) if self.samples else None,
                "sm_max_mhz": self.max_mhz, "reasons": names, "samples": len(self.samples)}


def kernel_source_digest(kind="decode"):
    """Digest of the sources of the decode kernels or of the prefill kernels."""
    h = hashlib.sha256()
    csrc = os.path.join(REPO, "paged_kv_cache_24_gb300", "csrc")
    own = ("pkv_decode",) if kind == "decode" else ("pkv_prefill", "pkv_tcgen05")
    for name in sorted(os.listdir(csrc)):
        if name.startswith(own) or name in ("pkv_device.cuh", "pkv_internal.h"):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload, kind="decode"):
    """DRAM bytes per launch of the dominant kernel from a committed ncu
    summary, if it still describes the current kernel source (else None)."""
    path = os.path.join(REPO, "profiles", f"{kind}_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except Exception:
        return None
    ent = rec.get(workload)
    if not ent or ent.get("kernel_digest") != kernel_source_digest(kind):
        return None
    return ent.get("dram_bytes_per_launch")


# ---------------------------------------------------------------------------
# CPU legs: the float64 oracle as it stands


class OracleSampler:
    """Times the float64 oracle, as it stands, on random (sequence, query head)
    pairs of a workload, on the host cores.  Rates are K/V bytes per second,
    counting each pair's share (1/G) of its kv head's context."""

    def __init__(self, w):
        import oracle

        self.oracle = oracle
        self.w = w
        spec = w.spec
        self.e = torch.tensor([], dtype=spec.dtype).element_size()
        self.kc, self.vc = w.k_cache.cpu(), w.v_cache.cpu()
        self.ks = w.k_scale.cpu() if w.k_scale is not None else None
        self.vs = w.v_scale.cpu() if w.v_scale is not None else None
        self.bt = w.block_tables.cpu().numpy()
        self.lens = w.lens_steps[0].cpu().numpy()
        self.q = w.q_steps[0].cpu()
        self.threads = oracle.max_threads()

    def run(self, n_pairs, seed=0, threads=None):
        spec = self.w.spec
        threads = self.threads if threads is None else threads
        rng = np.random.default_rng(seed)
        total = spec.num_seqs * spec.num_q_heads
        flat = rng.choice(total, size=min(n_pairs, total), replace=False)
        pairs = np.stack([flat // spec.num_q_heads, flat % spec.num_q_heads], 1).astype(np.int32)
        t0 = time.perf_counter()
        if spec.kv_fp8 or spec.kv_int8:
            decode = self.oracle.decode_fp8 if spec.kv_fp8 else self.oracle.decode_int8
            decode(self.q, self.kc, self.vc, self.ks, self.vs, self.bt, self.lens, spec.window,
                   self.w.scale, pairs=pairs, threads=threads)
        else:
            self.oracle.decode(self.q, self.kc, self.vc, self.bt, self.lens, spec.window,
                               self.w.scale, pairs=pairs, threads=threads)
        dt = time.perf_counter() - t0
        L = self.lens[pairs[:, 0]].astype(np.int64)
        lo = np.maximum(L - spec.window, 0) if spec.window > 0 else 0
        G = spec.num_q_heads // spec.num_kv_heads
        row = spec.head_dim + 4 if (spec.kv_fp8 or spec.kv_int8) else spec.head_dim * self.e
        kvb = float(((L - lo) * 2 * row).sum()) / G
        return kvb / dt, dt, len(pairs)

    def one_thread(self, pairs_per_s_all, target_s=3.0):
        """The same float64 decode on one host thread, sized to about target_s
        seconds if the threads scaled perfectly: (rate, seconds, pairs)."""
        n = max(4, int(pairs_per_s_all * target_s / max(1, self.threads)))
        return self.run(n, seed=1, threads=1)

    def rate_for(self, target_s):
        """Grow the sample until it takes about target_s seconds; when even the
        whole step is quicker than that, repeat it (fresh pair orders)."""
        n = max(1, self.threads)
        total = self.w.spec.num_seqs * self.w.spec.num_q_heads
        while True:
            rate, dt, got = self.run(n)
            if dt >= 0.5 * target_s:
                return rate, dt, got
            if got >= total:
                break
            n = int(min(total, max(n + 1, n * target_s / max(dt, 1e-3))))
        reps, t_all, b_all = 0, 0.0, 0.0
        while t_all < target_s and reps < 1000:
            rate, dt, got = self.run(total, seed=reps)
            t_all += dt
            b_all += rate * dt
            reps += 1
        return b_all / t_all, t_all, got * reps


def run_reference(args, workload):
    """The oracle as the reference arm, on the host cores (rank 0 only)."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    from paged_kv_cache_24_gb300.workloads import CONFIGS, config_spec, make_workload

    spec = config_spec(CONFIGS[workload])
    w = make_workload(spec, device="cpu", poison=True)
    sampler = OracleSampler(w)
    # calibrate, then size each step so that all warm-up and timed steps take
    # about --reference-seconds (two minutes by default)
    _, dt, got = sampler.run(max(1, sampler.threads))
    per_pair = dt / got
    per_step = args.reference_seconds / max(1, args.steps + args.warmup)
    pairs = int(max(1, min(spec.num_seqs * spec.num_q_heads, per_step / max(per_pair, 1e-6))))
    for i in range(args.warmup):
        sampler.run(pairs, seed=1000 + i)
    rates, times = [], []
    for i in range(args.steps):
        r, dt, _ = sampler.run(pairs, seed=i)
        rates.append(r)
        times.append(dt)
    gbs = statistics.median(rates) / 1e9
    desc = f"{pairs} random (sequence, query head) pairs per step"
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * statistics.median(times), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload, "sample": desc},
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": sampler.threads,
                         "kind": "oracle", "sample": desc, "cpu_model": host_cpu_model()},
        "step_ms_percentiles": percentiles_ms([1e3 * t for t in times]),
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# chunked prefill (a separate workload: tensor-core bound, reported in TFLOP/s)

PREFILL = {
    # batch of sequences with a cached prefix and a 1024-token chunk each
    "prefill_bf16": dict(dtype=torch.bfloat16, num_seqs=4, num_q_heads=32, num_kv_heads=8,
                         head_dim=128, block_size=16, chunk=1024, prefix_lo=2048,
                         prefix_hi=6144, seed=11),
    "prefill_fp16": dict(dtype=torch.float16, num_seqs=4, num_q_heads=32, num_kv_heads=8,
                         head_dim=128, block_size=16, chunk=1024, prefix_lo=2048,
                         prefix_hi=6144, seed=11),
}


def host_cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo), for the baseline line."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.machine()


def percentiles_ms(times_ms):
    """p10 / p50 / p90 of per-step times (ms)."""
    a = np.asarray(times_ms, dtype=np.float64)
    return {f"p{q}": float(np.percentile(a, q)) for q in (10, 50, 90)}


def prefill_inputs(workload):
    """The seeded inputs of a prefill workload on the device: the workload
    (pools holding every sequence's cached prefix), the packed chunk's q, k
    and v, the chunk offsets cu, the lengths L after the chunk, the chunk
    length and the prefixes."""
    from paged_kv_cache_24_gb300.workloads import config_spec, make_workload

    c = PREFILL[workload]
    rng = np.random.default_rng(c["seed"])
    B, chunk = c["num_seqs"], c["chunk"]
    prefix = rng.integers(c["prefix_lo"], c["prefix_hi"] + 1, B)
    lens = (prefix + chunk).tolist()
    spec = config_spec(0, dtype=c["dtype"], num_seqs=B, num_q_heads=c["num_q_heads"],
                       num_kv_heads=c["num_kv_heads"], head_dim=c["head_dim"],
                       block_size=c["block_size"], lens=lens, explicit_pool=None,
                       lens_are_pre_append=False, seed=c["seed"])
    w = make_workload(spec, device="cuda", poison=False)
    g = torch.Generator(device="cuda").manual_seed(c["seed"])
    T, hq, hkv, d = B * chunk, spec.num_q_heads, spec.num_kv_heads, spec.head_dim
    q = torch.randn(T, hq, d, generator=g, device="cuda").to(spec.dtype)
    k = torch.randn(T, hkv, d, generator=g, device="cuda").to(spec.dtype)
    v = torch.randn(T, hkv, d, generator=g, device="cuda").to(spec.dtype)
    cu = torch.arange(0, T + 1, chunk, dtype=torch.int32, device="cuda")
    L = torch.tensor(lens, dtype=torch.int32, device="cuda")
    return w, q, k, v, cu, L, chunk, prefix


def measure_prefill(pkv, workload, steps, warmup):
    """Time `pkv_prefill` on a prefill workload; returns the JSON line's dict."""
    w, q, k, v, cu, L, chunk, prefix = prefill_inputs(workload)
    spec = w.spec
    B, T = spec.num_seqs, q.shape[0]
    hq, hkv, d = spec.num_q_heads, spec.num_kv_heads, spec.head_dim
    out = torch.empty_like(q)
    # algorithmic flops: every (query row, attended key) pair costs 2 D (QK) + 2 D (PV)
    flops = float(sum(int(chunk) * int(p) + chunk * (chunk + 1) // 2 for p in prefix)) * hq * 4 * d

    def step():
        pkv.pkv_prefill(q, k, v, cu, w.k_cache, w.v_cache, w.block_tables, L, 0, w.scale,
                        max_chunk=chunk, out=out)

    # The K/V the step reads (tens of MB) fits in L2: L2 is flushed before
    # every timed step (outside its events), as for the decode lines.
    flush_buf = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device="cuda")
    clean_buf = torch.zeros(2 * L2_BYTES // 4, dtype=torch.int32, device="cuda")
    # warm-up on the capture stream (the stream's workspace then exists), then
    # the timed steps replay a CUDA graph of the same C-ABI call
    gstream = torch.cuda.Stream()
    gstream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(gstream):
        for _ in range(warmup):
            step()
    gstream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=gstream):
        step()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    with ClockSampler(0) as clocks, torch.cuda.stream(gstream):
        for s in range(steps):
            flush_buf.add_(1)
            clean_buf.amax()
            ev[s][0].record(gstream)
            graph.replay()
            ev[s][1].record(gstream)
        torch.cuda.synchronize()
    times = [a.elapsed_time(b) for a, b in ev]
    ms = sum(times) / steps
    tflops = flops / (ms * 1e-3) / 1e12
    peak = None
    try:
        with open(os.path.join(REPO, "MEASURED_PEAKS.json")) as f:
            peak = float(json.load(f)["bf16_tflops"])
        peak_kind = "measured"
    except Exception:
        peak, peak_kind = 1900.0, "fallback"
    # launches a step: the chunk append, the attention (bf16: and its exact
    # second launch)
    per_step = 3 if spec.dtype == torch.bfloat16 else 2
    return {
        "metric": "paged chunked prefill: attention TFLOP/s", "value": tflops,
        "unit": "TFLOP/s", "n_gpus": 1, "steps": steps, "warmup": warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": DTYPE_NAME[spec.dtype], "data": "synthetic",
        "config": {"workload": workload, "num_seqs": B, "chunk": chunk,
                   "mean_prefix": float(prefix.mean()), "num_q_heads": hq, "num_kv_heads": hkv,
                   "head_dim": d, "block_size": spec.block_size,
                   "l2": "flushed between steps (2x L2 written, then 2x L2 read)"},
        "tokens_per_s": T / (ms * 1e-3),
        "step_ms_percentiles": percentiles_ms(times),
        "roofline": {"bound": "tensor", "kernel": "prefill (chunk append + attention)",
                     "achieved": tflops, "peak": peak, "unit": "TFLOP/s", "frac": tflops / peak,
                     "peak_kind": peak_kind,
                     "traffic": recorded_traffic(workload, "prefill")},
        "gpu_launches": per_step * steps, "clocks": clocks.summary()}


def run_prefill(args, pkv):
    print(json.dumps(measure_prefill(pkv, args.workload, args.steps, args.warmup)), flush=True)
    return 0


# ---------------------------------------------------------------------------
# the GPU arm


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--path", default="fused", choices=["fused", "separate"],
                    help="fused: pkv_append_decode (one launch); separate: pkv_append + pkv_decode")
    ap.add_argument("--reference-seconds", type=float, default=120.0,
                    help="--impl reference: host time of all warm-up and timed steps")
    ap.add_argument("--num-seqs", type=int, default=0,
                    help="profiling only: shrink the workload's batch (not a bench line)")
    ap.add_argument("--no-extra-workloads", dest="extra_workloads", action="store_false",
                    help="time only the chosen workload (by default the line also carries "
                         "every other workload's value, roofline and clocks)")
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 3)

    if args.impl == "reference":
        return run_reference(args, args.workload)

    import paged_kv_cache_24_gb300 as pkv
    rank, world, local_rank = dist_env()
    torch.cuda.set_device(local_rank)
    if args.workload in PREFILL:
        return run_prefill(args, pkv)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
        pg = dist

    over = {"num_seqs": args.num_seqs} if args.num_seqs > 0 else {}
    spec = rank_spec(args.workload, rank, args.num_seqs)
    m = measure_decode(pkv, spec, args.steps, args.warmup, args.path, pg, world, local_rank,
                       traffic_key=None if over else args.workload)
    w, sbytes, S = m["w"], m["sbytes"], m["w"].steps
    total_ms_all, bytes_all = m["total_ms"], m["bytes"]
    ms_per_step = total_ms_all / args.steps
    value = bytes_all / (total_ms_all * 1e-3) / 1e9
    tokens_per_s = world * spec.num_seqs * args.steps / (total_ms_all * 1e-3)
    peak, peak_kind = hbm_peak()

    # ---- end to end through the public API, host buffers ----
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(pkv, w, spec, args, sbytes, pg, world)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        sampler = OracleSampler(w)
        rate, dt, got = sampler.rate_for(10.0)
        rate1, dt1, got1 = sampler.one_thread(got / dt)
        cpu = {"value": rate / 1e9, "unit": "GB/s", "cores": sampler.threads, "kind": "oracle",
               "sample": f"{got} random (sequence, query head) pairs of step 0; {dt:.1f} s of "
                         f"float64 decode on the host cores; K/V bytes of the sample / time",
               "cpu_model": host_cpu_model(),
               "one_thread": {"value": rate1 / 1e9, "unit": "GB/s",
                              "sample": f"{got1} pairs, {dt1:.1f} s on one thread"}}

    line = None
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": ("e4m3+f16" if spec.kv_fp8 else "i8+f16" if spec.kv_int8
                      else DTYPE_NAME[spec.dtype]), "data": "synthetic",
            "config": {
                "workload": args.workload + ("" if not over else "-reduced"),
                "num_seqs": spec.num_seqs,
                "num_q_heads": spec.num_q_heads, "num_kv_heads": spec.num_kv_heads,
                "head_dim": spec.head_dim, "block_size": spec.block_size,
                "window": spec.window, "steps_in_workload": S,
                "mean_context": float(w.lens_steps.float().mean()),
                "num_blocks": w.num_blocks,
                "tokens_per_split": m["plan"][0], "num_splits": m["plan"][1],
                "l2": m["l2"],
                "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            },
            "tokens_per_s": tokens_per_s,
            "step_ms_percentiles": percentiles_ms(m["step_ms"]),
            # the same step counted on distinct pool rows (shared prefix blocks once)
            # (every rank's workload has the same shape: rank 0's count x ranks)
            "unique_rows": {"value": world * m["unique"] / (total_ms_all * 1e-3) / 1e9,
                            "unit": "GB/s", "bytes_per_step": m["unique"] / args.steps,
                            "pct_of_hbm_peak": 100.0 * m["unique"] / (total_ms_all * 1e-3) / 1e9
                            / peak},
            "pct_of_hbm_peak": 100.0 * value / (world * peak),
            "path": m["path"],
            "roofline": m["roofline"],
            "gpu_launches": m["gpu_launches"],
            "clocks": m["clocks"],
            "e2e": e2e,
            "cpu_baseline": cpu,
        }
    del m, w
    torch.cuda.empty_cache()
    if rank == 0 and world == 1 and args.extra_workloads and not over:
        line["workloads"] = measure_other_workloads(pkv, args)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()
    return 0


def measure_decode(pkv, spec, steps, warmup, path, pg=None, world=1, local_rank=0,
                   traffic_key=None):
    """Time `steps` decode steps (append + decode) of workload `spec`: CUDA
    graphs of the C-ABI calls replayed on one stream, CUDA events around each
    step and (separate path) around its decode launch.  Returns the measured times, bytes and
    the roofline record (its `traffic` from the committed record for
    `traffic_key`); `w` is the workload (for the end-to-end and CPU legs)."""
    from paged_kv_cache_24_gb300.workloads import make_workload

    w = make_workload(spec, device="cuda", poison=True)
    S = w.steps
    bs = spec.block_size
    sbytes = step_bytes(w)

    slots = [pkv.pkv_slot_mapping(w.block_tables, w.pos_steps[s].contiguous(), bs)
             for s in range(S)]
    lens = [w.lens_steps[s].contiguous() for s in range(S)]
    out = torch.empty_like(w.q_steps[0])
    plan = pkv.pkv_decode_plan(spec.num_seqs, spec.num_q_heads, pkv.cache_layout(w.k_cache),
                               w.max_blocks, spec.window)
    # FP8 pools append through the quantising kernel (no fused form)
    q8 = spec.kv_fp8 or spec.kv_int8
    fused = path == "fused" and not q8
    launches_per_step = (1 if fused else 2) + (1 if plan[1] > 1 else 0)

    def do_append(i):
        if fused:
            return
        if q8:
            append = pkv.pkv_append_fp8 if spec.kv_fp8 else pkv.pkv_append_int8
            append(w.k_steps[i], w.v_steps[i], slots[i], w.k_cache, w.v_cache, w.k_scale,
                   w.v_scale)
        else:
            pkv.pkv_append(w.k_steps[i], w.v_steps[i], slots[i], w.k_cache, w.v_cache)

    def do_decode(i):
        if fused:
            pkv.pkv_append_decode(w.q_steps[i], w.k_steps[i], w.v_steps[i], w.k_cache,
                                  w.v_cache, w.block_tables, lens[i], spec.window, w.scale,
                                  out=out)
        else:
            pkv.pkv_decode(w.q_steps[i], w.k_cache, w.v_cache, w.block_tables, lens[i],
                           spec.window, w.scale, out=out, k_scale=w.k_scale, v_scale=w.v_scale)

    def step(s):
        do_append(s % S)
        do_decode(s % S)

    kv_per_step = statistics.mean(b["kv"] for b in sbytes)
    need_flush = kv_per_step < 4 * L2_BYTES
    flush_buf = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device="cuda") if need_flush else None
    # read after the write so L2 holds clean lines: the next step's reads then
    # pay no write-back of the flush's dirty data
    clean_buf = (torch.zeros(2 * L2_BYTES // 4, dtype=torch.int32, device="cuda")
                 if need_flush else None)

    # The timed steps replay CUDA graphs of these same C-ABI calls (one graph
    # per distinct step input; append and decode captured apart so the
    # decode launch keeps its own events): host-side launch work then never
    # leaves the GPU idle inside a step.  Warm-up runs on the capture stream
    # first, so the library's per-stream workspace exists before capture.
    gstream = torch.cuda.Stream()
    gstream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(gstream):
        for s in range(warmup):
            step(s)
    gstream.synchronize()
    g_app, g_dec = [], []
    for i in range(S):
        if not fused:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=gstream):
                do_append(i)
            g_app.append(g)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=gstream):
            do_decode(i)
        g_dec.append(g)
    torch.cuda.synchronize()
    stream = gstream

    # ---- timed region: exactly `steps` steps ----
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as clocks, torch.cuda.stream(gstream):
        t_start.record(stream)
        for s in range(steps):
            if need_flush:
                flush_buf.add_(1)  # evict the previous step's working set from L2
                clean_buf.amax()
            i = s % S
            ev[s][0].record(stream)
            if not fused:
                # the decode launch's own start (with the fused call the step
                # is that launch: a second event here would only add its own
                # cost, ~2 us of GPU time, to every step)
                g_app[i].replay()
                ev[s][1].record(stream)
            g_dec[i].replay()
            ev[s][2].record(stream)
        t_end.record(stream)
        torch.cuda.synchronize()
    if pg:
        pg.barrier()
    step_ms = [ev[s][0].elapsed_time(ev[s][2]) for s in range(steps)]
    dec_ms = step_ms if fused else [ev[s][1].elapsed_time(ev[s][2]) for s in range(steps)]
    loop_ms = t_start.elapsed_time(t_end)
    # the step time: whole loop / K when nothing else ran in it, else the sum of steps
    total_ms = sum(step_ms) if need_flush else loop_ms
    my_bytes = sum(sbytes[s % S]["step"] for s in range(steps))
    my_unique = sum(sbytes[s % S]["step_unique"] for s in range(steps))
    dec_key = "step" if fused else "decode"  # the fused launch also does the append
    my_dec_bytes = sum(sbytes[s % S][dec_key] for s in range(steps))
    total_ms_all, bytes_all = reduce_over_ranks(pg, total_ms, my_bytes)

    peak, peak_kind = hbm_peak()
    dec_avg_ms = sum(dec_ms) / steps
    achieved = (my_dec_bytes / steps) / (dec_avg_ms * 1e-3) / 1e9
    return {
        "w": w, "sbytes": sbytes, "plan": plan, "total_ms": total_ms_all, "bytes": bytes_all,
        "unique": my_unique, "step_ms": step_ms, "path": "fused" if fused else "separate",
        "l2": ("flushed between steps (2x L2 written, then 2x L2 read)" if need_flush else
               f"inputs larger than L2 ({kv_per_step / 1e9:.2f} GB of K/V per step)"),
        "roofline": {"bound": "hbm",
                     "kernel": ("fused append + decode (split-K) + LSE combine" if fused
                                else "decode (split-K decode + LSE combine)"),
                     "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind,
                     "traffic": recorded_traffic(traffic_key) if traffic_key else None,
                     "algorithmic_bytes_per_launch": my_dec_bytes / steps,
                     "launch_ms": dec_avg_ms},
        "gpu_launches": launches_per_step * steps,
        "clocks": clocks.summary(),
    }


# the other workloads, timed after the headline in the same run
OTHER_WORKLOADS = ["tiny_fp32", "mha_fp16", "sliding_bf16", "serving_fp16", "mha_fp8",
                   "gqa_fp8", "mha_int8", "gqa_int8", "prefill_bf16", "prefill_fp16"]


def measure_other_workloads(pkv, args):
    """Each other workload's line (its value, roofline and clocks), timed in
    this run after the headline: at most 200 steps (serving: its 32) after
    `args.warmup` warm-up steps each."""
    from paged_kv_cache_24_gb300.workloads import CONFIGS, config_spec

    res = {}
    for name in OTHER_WORKLOADS:
        if name == args.workload:
            continue
        steps = min(args.steps, 200)
        if name in PREFILL:
            d = measure_prefill(pkv, name, min(args.steps, 20), args.warmup)
            res[name] = {"metric": d["metric"], "value": d["value"], "unit": d["unit"],
                         "steps": d["steps"], "ms_per_step": d["ms_per_step"],
                         "dtype": d["dtype"], "roofline": d["roofline"], "clocks": d["clocks"],
                         "config": d["config"]}
        else:
            spec = config_spec(CONFIGS[name])
            if spec.steps > 1:
                steps = max(steps, spec.steps)
            m = measure_decode(pkv, spec, steps, args.warmup, args.path, traffic_key=name)
            value = m["bytes"] / (m["total_ms"] * 1e-3) / 1e9
            res[name] = {"metric": METRIC, "value": value, "unit": "GB/s", "steps": steps,
                         "ms_per_step": m["total_ms"] / steps,
                         "tokens_per_s": spec.num_seqs * steps / (m["total_ms"] * 1e-3),
                         "dtype": ("e4m3+f16" if spec.kv_fp8 else "i8+f16" if spec.kv_int8
                                   else DTYPE_NAME[spec.dtype]),
                         "path": m["path"], "roofline": m["roofline"], "clocks": m["clocks"],
                         "unique_rows_gbs": m["unique"] / (m["total_ms"] * 1e-3) / 1e9,
                         "config": {"num_seqs": spec.num_seqs, "window": spec.window,
                                    "tokens_per_split": m["plan"][0],
                                    "num_splits": m["plan"][1], "l2": m["l2"]}}
            del m
        torch.cuda.empty_cache()
    return res


def run_e2e(pkv, w, spec, args, sbytes, pg, world):
    """Same step through the public API (DecodeStep) with host buffers: every
    step copies its staged inputs -- q, the new K/V, positions, lengths and the
    block tables -- from pinned host memory to the device, replays slot
    mapping + append + decode as one CUDA graph, copies the attention output
    back, and the host waits for it."""
    S = w.steps
    step = pkv.DecodeStep(w.k_cache, w.v_cache, spec.num_seqs, spec.num_q_heads, w.max_blocks,
                          spec.window, w.scale, copy_block_tables=True, num_buffers=S,
                          fused=args.path == "fused" and not (spec.kv_fp8 or spec.kv_int8),
                          k_scale=w.k_scale, v_scale=w.v_scale)
    for s in range(S):
        h = step.host[s]
        h["q"].copy_(w.q_steps[s])
        h["k"].copy_(w.k_steps[s])
        h["v"].copy_(w.v_steps[s])
        h["positions"].copy_(w.pos_steps[s])
        h["context_lens"].copy_(w.lens_steps[s])
        h["block_tables"].copy_(w.block_tables)
    for s in range(args.warmup):
        step.run(s % S)
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for s in range(args.steps):
        step.run(s % S)
    ms = (time.perf_counter() - t0) * 1e3
    my_bytes = sum(sbytes[s % S]["step"] for s in range(args.steps))
    ms, my_bytes = reduce_over_ranks(pg, ms, my_bytes)
    return {"value": my_bytes / (ms * 1e-3) / 1e9, "unit": "GB/s",
            "tokens_per_s": world * spec.num_seqs * args.steps / (ms * 1e-3),
            "ms_per_step": ms / args.steps,
            "h2d_bytes_per_step": step.h2d_bytes, "d2h_bytes_per_step": step.d2h_bytes,
            "api": "DecodeStep (one CUDA graph per step, host waits each step)"}


if __name__ == "__main__":
    sys.exit(main())
