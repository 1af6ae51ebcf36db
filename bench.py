#!/usr/bin/env python3
"""Latency / throughput of the CTA-pipelined GEMM chain on one GB300 (or N replicas).

One step = one pass of the whole chain (every GEMM, the scoreboard / work-queue hand-off, all
epilogues) over one batch of seeded synthetic inputs, launched as one CUDA graph replay.  The
L2 cache is flushed (a write of twice its size) between timed steps, outside the timed events.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Rank 0 prints one JSON line.  Under torchrun every rank runs its own replica of the workload
(weak scaling, no collective on the data path); timing is the max over ranks.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import seeded_inputs as si  # noqa: E402

METRIC = "single-batch 2-layer GEMM latency (µs) and TFLOP/s vs roofline on 1 GB300"
DEFAULT_WORKLOAD = "prefill_m2048_d8192"
# tile widths per GEMM measured best on GB300 (0: the library cost model chooses)
TUNED_TILES = {
    "tiny_m64_d256": [64, 64],
    "decode_m128_d4096": [0, 0],
    "prefill_m2048_d8192": [256, 256],
    "llama_m256_4096_14336": [0, 0],
    "gelu4_m512_d8192": [0, 0, 0, 0],
}
TUNED_SPLIT = {}
# every source that shapes the measured launch: the kernel and the host code that picks its tiles,
# raster and scoreboard groups
KERNEL_SOURCES = ["mlp_latency_gb300/csrc/chain_kernel.cuh", "mlp_latency_gb300/csrc/ptx.cuh",
                  "mlp_latency_gb300/csrc/protocol.h", "mlp_latency_gb300/csrc/dep_groups.h",
                  "mlp_latency_gb300/csrc/mlp_chain.cu", "mlp_latency_gb300/csrc/host_protocol.cpp"]
PROFILE_DIR = os.path.join(ROOT, "profiles")


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def recorded_traffic(workload: str):
    """dram bytes per launch from the committed ncu summary, if it was taken on this kernel source."""
    path = os.path.join(PROFILE_DIR, f"chain_kernel_{workload}.md")
    if not os.path.exists(path):
        return None
    vals = {}
    with open(path) as f:
        for line in f:
            if ":" in line and line.strip().startswith("- "):
                k, v = line.strip()[2:].split(":", 1)
                vals[k.strip()] = v.strip().strip("`")
    if vals.get("kernel_source_sha256") != kernel_source_hash():
        return None
    try:
        return float(vals["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# ------------------------------------------------------------------------------ clocks --
class ClockSampler:
    """Samples SM clock and clock-event reasons through NVML (read-only) on a thread."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, uuid: str, period_s: float = 0.0005):
        self.period = period_s
        self.samples = []
        self.max_mhz = None
        self.ok = False
        try:
            self.nvml = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nvml.nvmlInit_v2() != 0:
                return
            self.h = ctypes.c_void_p()
            if self.nvml.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.h)) != 0:
                return
            m = ctypes.c_uint()
            if self.nvml.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(m)) == 0:
                self.max_mhz = m.value
            self._reasons_fn = getattr(self.nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(self.nvml, "nvmlDeviceGetCurrentClocksThrottleReasons")
            self.ok = True
        except OSError:
            self.ok = False

    def _sample(self):
        c = ctypes.c_uint()
        r = ctypes.c_ulonglong()
        if self.nvml.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(c)) == 0 and \
                self._reasons_fn(self.h, ctypes.byref(r)) == 0:
            self.samples.append((c.value, r.value))

    def start(self):
        self.samples = []
        self._stop = threading.Event()

        def loop():
            while not self._stop.is_set():
                self._sample()
                time.sleep(self.period)
        if self.ok:
            self._t = threading.Thread(target=loop, daemon=True)
            self._t.start()

    def stop(self):
        if self.ok:
            self._stop.set()
            self._t.join()
            self._sample()

    def summary(self):
        if not self.ok or not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0,
                    "source": "nvml unavailable"}
        mhz = [s[0] for s in self.samples]
        bits = 0
        for _, r in self.samples:
            bits |= r
        reasons = [name for b, name in self.REASONS.items() if bits & b]
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": self.max_mhz, "reasons": reasons,
                "samples": len(mhz), "source": "nvml"}

    @staticmethod
    def rejected(summary) -> bool:
        bad = {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"}
        if bad & set(summary["reasons"]):
            return True
        if summary["sm_mhz"] and summary["sm_max_mhz"] and summary["sm_mhz"] < 0.6 * summary["sm_max_mhz"] \
                and not summary["reasons"]:
            return True
        return False


# --------------------------------------------------------------------------- distributed --
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value: float, world: int, device=None) -> float:
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------------ phase breakdown --
def phase_breakdown(events: np.ndarray, deps, ctas: np.ndarray = None) -> dict:
    """Per-stage phase times (µs, medians over tiles) of one pipelined run, from its event log:
    the single-GPU analogues of the pages' per-phase overheads (CTA-Pipelining, section III-C,
    Fig. 2b).
      mainloop          tile start (its item taken and, for a consumer, its queue entry and group
                        counter acquired) -> accumulator complete;
      epilogue (T1)     accumulator complete -> release: split-K exchange, bf16 stores, the fence
                        and the scoreboard release, i.e. the producer epilogue with its fence;
      handoff (T3)      for consumer tiles: the last release of its producers -> its start, i.e.
                        the queue push, the consumer's poll and acquire, and the TMA warp's pickup;
      span              first start -> last release of the stage.
    The scheduler's broadcast (T4) happens before a tile's start and is not timed separately.
    `deps[b]` is the dependency CSR (prod_off, prod_tgt) of boundary b.  With the per-CTA records
    (`ctas`: entry, set-up done, exit) it adds the kernel's own span, the CTAs' entry spread, their
    set-up (barriers, TMEM, cluster sync) and the teardown after the last tile's release."""
    out = {}
    t0 = int(events["t_start"].min())
    if ctas is not None and len(ctas):
        entry, setup, exit_ = (ctas[k].astype(np.int64) for k in ("t_start", "t_acc", "t_end"))
        out["kernel"] = {"ctas": int(len(ctas)),
                         "span_us": float(exit_.max() - entry.min()) / 1e3,
                         "entry_spread_us": float(entry.max() - entry.min()) / 1e3,
                         "setup_us": float(np.median(setup - entry)) / 1e3,
                         "first_tile_after_entry_us": float(t0 - entry.min()) / 1e3,
                         "teardown_us": float(exit_.max() - int(events["t_end"].max())) / 1e3}
    for s in sorted(set(int(v) for v in events["stage"])):
        e = events[events["stage"] == s]
        st = {"tiles": int(len(e)),
              "first_start_us": (int(e["t_start"].min()) - t0) / 1e3,
              "span_us": (int(e["t_end"].max()) - int(e["t_start"].min())) / 1e3,
              "mainloop_us": float(np.median((e["t_acc"].astype(np.int64) - e["t_start"].astype(np.int64)))) / 1e3,
              "epilogue_T1_us": float(np.median((e["t_end"].astype(np.int64) - e["t_acc"].astype(np.int64)))) / 1e3}
        if s > 0:
            prev = events[events["stage"] == s - 1]
            t_end_p = dict(zip(prev["tile"].tolist(), prev["t_end"].astype(np.int64).tolist()))
            off, tgt = deps[s - 1]
            last = {}
            for p in range(len(off) - 1):
                for c in tgt[off[p]:off[p + 1]]:
                    last[int(c)] = max(last.get(int(c), 0), t_end_p[p])
            h = [int(r["t_start"]) - last[int(r["tile"])] for r in e]
            st["handoff_T3_us"] = float(np.median(h)) / 1e3
            st["handoff_T3_min_us"] = float(np.min(h)) / 1e3
        out[f"stage{s}"] = st
    return out


# ----------------------------------------------------------------------------- timing --
def time_steps(step_fn, flush_fn, steps: int, stream):
    """Per-step device time (ms) with CUDA events on `stream`; L2 flushed between steps."""
    import torch
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        flush_fn()
        starts[i].record(stream)
        step_fn()
        ends[i].record(stream)
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in zip(starts, ends)]


def pct(xs, q):
    xs = sorted(xs)
    return xs[min(len(xs) - 1, max(0, int(round(q * (len(xs) - 1)))))]


# ------------------------------------------------------------------------- cpu baseline --
def cpu_oracle_baseline(w, X, Ws, budget_s: float, Y_gpu=None):
    """Time the CPU oracle (as it stands) on a bounded row sample of the workload."""
    import oracle  # the one place the bench runs the oracle (plus the reference arm)
    threads = oracle.default_threads()
    per_row_flops = w.flops / w.M
    xb, wb = si.bits(X), [si.bits(t) for t in Ws]
    # pick a row count that takes about budget_s / 3 per call, then repeat within the budget
    rows = si.sample_rows(w.M, min(w.M, 8), seed=3)
    t0 = time.perf_counter()
    oracle.chain(xb, wb, gelu=w.gelu, residual=w.residual, gated=w.gated, rows=rows, threads=threads)
    per_row = (time.perf_counter() - t0) / len(rows)
    n = int(max(1, min(w.M, (budget_s / 3) / max(per_row, 1e-9))))
    rows = np.arange(w.M, dtype=np.int64) if n >= w.M else si.sample_rows(w.M, n, seed=4)
    total_rows, total_t, calls = 0, 0.0, 0
    parity = None
    while total_t < budget_s or calls == 0:
        t0 = time.perf_counter()
        Yo = oracle.chain(xb, wb, gelu=w.gelu, residual=w.residual, gated=w.gated, rows=rows, threads=threads)
        total_t += time.perf_counter() - t0
        total_rows += len(rows)
        calls += 1
        if calls == 1 and Y_gpu is not None:
            ref = oracle.bf16_to_f32(Yo)
            got = Y_gpu[rows].astype(np.float32)
            parity = bool(np.all(np.abs(got - ref) <= 1e-2 * (np.abs(ref) + 1)))
        if calls >= 50:
            break
    value = per_row_flops * total_rows / total_t / 1e12
    sample = (f"{len(rows)} of {w.M} rows of {w.name} per call (rows are independent), "
              f"{calls} calls, {total_t:.1f} s wall")
    return {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": sample,
            "cpu": cpu_model()}, parity, total_t / calls, len(rows)


def cpu_model() -> str:
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part", "hardware")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.machine()


# ----------------------------------------------------------------------------- reference --
def run_reference(args, w):
    """The oracle on the host cores, as the reference arm: same workload, metric and unit."""
    import torch
    world, rank, _ = dist_env()
    if rank != 0:
        return
    X, Ws = si.draw(w, seed=0)
    # each step is a row sample sized so that the whole run stays near two minutes of CPU time
    budget = min(20.0, 120.0 / max(1, args.steps + args.warmup))
    import oracle
    xb, wb = si.bits(X), [si.bits(t) for t in Ws]
    threads = oracle.default_threads()
    rows = si.sample_rows(w.M, min(w.M, 4), seed=3)
    t0 = time.perf_counter()
    oracle.chain(xb, wb, gelu=w.gelu, residual=w.residual, gated=w.gated, rows=rows, threads=threads)
    per_row = (time.perf_counter() - t0) / len(rows)
    n = int(max(1, min(w.M, budget / max(per_row, 1e-9))))
    rows = np.arange(w.M, dtype=np.int64) if n >= w.M else si.sample_rows(w.M, n, seed=4)
    for _ in range(args.warmup):
        oracle.chain(xb, wb, gelu=w.gelu, residual=w.residual, gated=w.gated, rows=rows, threads=threads)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.chain(xb, wb, gelu=w.gelu, residual=w.residual, gated=w.gated, rows=rows, threads=threads)
        times.append(time.perf_counter() - t0)
    step_s = statistics.mean(times)
    flops = w.flops / w.M * len(rows)
    value = flops / step_s / 1e12
    sample = f"{len(rows)} of {w.M} rows of {w.name} per step (rows are independent)"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "M": w.M, "dims": list(w.dims), "gelu": w.gelu,
                   "residual": w.residual, "what": "CPU oracle, plain C, fp32 accumulate"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": sample, "cpu": cpu_model()},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------- sequence-length sweep --
def run_sweep(args):
    """Latency of the 2-GEMM chain against the row count M (the input sequence length) with
    fixed d x d weights, per launch mode, with the micro-batch chunk size swept at every M: the
    single-GPU analogue of the paper's sequence-length study (section IV, Fig. 5).  One JSON
    line per M; Y is checked bit-identical across the modes."""
    import torch
    import mlp_latency_gb300 as mc

    world, rank, local = dist_env()
    if rank != 0:
        return
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    mc.load()
    d = args.sweep_d
    ms_list = [int(v) for v in args.sweep_m.split(",")]
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 128 << 20) or (128 << 20)
    flush_buf = torch.empty(2 * l2, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)
    for M in ms_list:
        w = si.make_workload(f"sweep_m{M}_d{d}", M, (d, d, d))
        X, Ws = si.draw(w, seed=0)
        Xd, Wd = X.to(dev), [t.to(dev) for t in Ws]
        Y = torch.empty(M, d, dtype=torch.bfloat16, device=dev)
        ref = None
        tiles = None     # the first handle's tile widths and splits, kept by every later handle
        line = {"sweep": "sequence length", "M": M, "dims": [d, d, d], "flops": w.flops,
                "l2": "flushed between steps", "graph": "one CUDA graph replay per step"}

        def timed(mode, rows=0, cta_pair=0):
            nonlocal ref, tiles
            # every handle after the first keeps its tile widths and splits, so that all modes add the
            # same k-slices and the bit-identity check holds (the K-granular mode has no CTA pairs)
            kw = dict(tile_n=tiles[0], k_split=tiles[1]) if tiles else {}
            if rows % 128:
                kw["tile_m"] = 64
            if cta_pair:
                kw["cta_pair"] = cta_pair
            with mc.Chain(M, w.dims, mode=mode, microbatch_rows=rows, device=local, **kw) as ch:
                if tiles is None:
                    tiles = (ch.info()["tile_n"], ch.info()["k_split"])
                    line["cta_pair"] = ch.info()["cta_pair"]   # the library's choice for this M
                ws = torch.empty(max(ch.workspace_size(), 256), dtype=torch.uint8, device=dev)
                g = torch.cuda.CUDAGraph()
                with torch.cuda.stream(stream):
                    ch.run(Xd, Wd, Y, ws, stream=stream)
                    torch.cuda.synchronize()
                    if ch.check(stream) != 0:
                        raise RuntimeError(f"device status set ({mode}, M={M})")
                    with torch.cuda.graph(g, stream=stream):
                        ch.run(Xd, Wd, Y, ws, stream=stream)
                    torch.cuda.synchronize()
                    for _ in range(args.warmup):
                        flush_buf.zero_()
                        g.replay()
                    t_est = max(1e-6, w.flops / 1.0e15)          # rough time per step, for the step count
                    steps = int(max(10, min(args.steps, 0.3 / t_est)))
                    med = statistics.median(time_steps(g.replay, flush_buf.zero_, steps, stream)) * 1e3
                    if ch.check(stream) != 0:
                        raise RuntimeError(f"device status set ({mode}, M={M})")
                y = Y.view(torch.int16).clone()
                if ref is None:
                    ref = y
                elif not torch.equal(ref, y):
                    raise RuntimeError(f"{mode} (rows {rows}) differs from the first mode at M={M}")
                return med

        for mode in ("sequential", "sequential_pdl", "pipelined", "pipelined_kwait"):
            line[f"{mode}_us"] = timed(mode)
        best = None
        rows = 64
        while rows <= M // 2:
            for cp in ([0, 2] if rows % 256 == 0 and line["cta_pair"] == 2 else [0]):
                t = timed("microbatch", rows, cp)
                line[f"microbatch_{rows}{'_pair' if cp else ''}_us"] = t
                if best is None or t < best[1]:
                    best = (rows, t)
            rows *= 2
        line["microbatch_best_us"] = best[1] if best else None
        line["microbatch_best_rows"] = best[0] if best else None
        line["bit_identical_across_modes"] = True
        print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------------- main --
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(si.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--tile-n", default=None, help="comma-separated tile widths per GEMM (0 = library choice)")
    ap.add_argument("--k-split", default=None, help="comma-separated split-K factors per GEMM (0 = library choice)")
    ap.add_argument("--mode", default="pipelined", choices=["pipelined", "pipelined_kwait", "pipelined_lamport", "sequential", "sequential_pdl", "microbatch"])
    ap.add_argument("--microbatch-rows", type=int, default=0)
    ap.add_argument("--raster-group", type=int, default=0)
    ap.add_argument("--pipe-stages", type=int, default=0)
    ap.add_argument("--acc-split", type=int, default=0)
    ap.add_argument("--tile-k", type=int, default=0, choices=[0, 64, 128],
                    help="k depth of one ring fill (0 = library choice; 128 = two 64-deep blocks per fill)")
    ap.add_argument("--cta-pair", type=int, default=0, choices=[0, 1, 2],
                    help="0: library choice, 1: one CTA per tile, 2: CTA pairs (256-row tiles, tcgen05 cta_group::2)")
    ap.add_argument("--splitk-exchange", default="global", choices=["global", "dsmem"],
                    help="how split-K siblings add partial sums: through L2, or the owners' shared memory")
    ap.add_argument("--weight-layout", default="kn", choices=["kn", "nk"],
                    help="nk: weights stored transposed (nn.Linear layout)")
    ap.add_argument("--no-baselines", action="store_true", help="skip sequential/micro-batch/cuBLAS lines")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--profile-steps", type=int, default=0,
                    help="only run this many graph replays after warm-up (for ncu); prints nothing")
    ap.add_argument("--sweep-m", default=None,
                    help="comma-separated row counts: time the 2-GEMM chain with d x d weights at each "
                         "(one JSON line per M) instead of the bench step")
    ap.add_argument("--sweep-d", type=int, default=8192)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    w = si.WORKLOADS[args.workload]
    if args.sweep_m:
        run_sweep(args)
        return

    if args.impl == "reference":
        run_reference(args, w)
        return

    import torch
    import mlp_latency_gb300 as mc

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    mc.load()  # raises if the CUDA library was not built: no fallback

    tiles = [int(t) for t in args.tile_n.split(",")][: w.num_gemms] if args.tile_n else TUNED_TILES.get(w.name)
    ksplit = [int(t) for t in args.k_split.split(",")][: w.num_gemms] if args.k_split else TUNED_SPLIT.get(w.name)
    X, Ws = si.draw(w, seed=0)
    Xd = X.to(dev)
    # the library reads W_s as stored; "nk" stores each weight transposed (same values)
    Wd = [(t.t().contiguous() if args.weight_layout == "nk" else t).to(dev) for t in Ws]
    Y = torch.empty(w.M, w.dims[-1], dtype=torch.bfloat16, device=dev)
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 128 << 20) or (128 << 20)
    flush_buf = torch.empty(2 * l2, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def make(mode, rows=0, **kw):
        cta_pair = kw.pop("cta_pair", args.cta_pair)
        # two-block ring fills run with one CTA per tile, outside the K-granular and Lamport modes
        tile_k = 0 if mode in ("pipelined_kwait", "pipelined_lamport") or cta_pair == 2 else args.tile_k
        return mc.Chain(w.M, w.dims, tile_n=tiles, gelu=w.gelu, residual=w.residual, mode=mode,
                        microbatch_rows=rows, device=local, raster_group=args.raster_group,
                        pipe_stages=args.pipe_stages, acc_split=args.acc_split,
                        weight_layout=args.weight_layout, k_split=ksplit, gated=w.gated,
                        cta_pair=cta_pair, splitk_exchange=args.splitk_exchange, tile_k=tile_k, **kw)

    chain = make(args.mode, args.microbatch_rows)
    info = chain.info()
    ws = torch.empty(max(chain.workspace_size(), 256), dtype=torch.uint8, device=dev)

    def capture(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            fn()  # eager once (also encodes the TMA descriptors)
            torch.cuda.synchronize()
            with torch.cuda.graph(g, stream=stream):
                fn()
        torch.cuda.synchronize()
        return g

    with torch.cuda.stream(stream):
        g_main = capture(lambda: chain.run(Xd, Wd, Y, ws, stream=stream))
        status = chain.check(stream)
        if status != 0:
            raise RuntimeError(f"device status {status} after the first run")

        def flush():
            flush_buf.zero_()

        for _ in range(args.warmup):
            flush()
            g_main.replay()
        torch.cuda.synchronize()
        if args.profile_steps:
            for _ in range(args.profile_steps):
                flush()
                g_main.replay()
            torch.cuda.synchronize()
            return

        uuid = "GPU-" + str(getattr(props, "uuid", "")) if getattr(props, "uuid", None) else ""
        sampler = ClockSampler(uuid)
        remeasured = False
        for attempt in range(2):
            barrier(world)
            torch.cuda.synchronize()
            sampler.start()
            ms = time_steps(g_main.replay, flush, args.steps, stream)
            sampler.stop()
            torch.cuda.synchronize()
            barrier(world)
            clocks = sampler.summary()
            if not ClockSampler.rejected(clocks) or attempt == 1:
                break
            remeasured = True
        if chain.check(stream) != 0:
            raise RuntimeError("device status set during the timed region")

        mean_ms = statistics.mean(ms)
        mean_ms_all = max_over_ranks(mean_ms, world, dev)
        value = world * w.flops / (mean_ms_all * 1e-3) / 1e12
        lat_us = statistics.median(ms) * 1e3

        # ---- baselines on this GPU: sequential launches, micro-batching sweep, cuBLAS --------
        baselines = {}
        k_base = min(args.steps, 300)
        if not args.no_baselines:
            for mode in ("sequential", "sequential_pdl", "pipelined", "pipelined_kwait", "pipelined_lamport"):
                if mode == args.mode:
                    continue
                ch = make(mode)
                g = capture(lambda ch=ch: ch.run(Xd, Wd, Y, ws, stream=stream))
                for _ in range(args.warmup):
                    flush(); g.replay()
                baselines[f"{mode}_us"] = statistics.median(time_steps(g.replay, flush, k_base, stream)) * 1e3
                ch.close()
            # Best-tuned micro-batching: every chunk size from 64 rows (64-row tiles below 128), each
            # on one-CTA tiles and, where the chunk holds whole 256-row tiles, on CTA pairs too.
            best = None
            rows = 64
            while rows <= w.M // 2:
                kinds = [1, 2] if rows % 256 == 0 else [1]
                for cp in kinds:
                    try:
                        ch = make("microbatch", rows, tile_m=64 if rows % 128 else 0, cta_pair=cp)
                    except mc.MlpChainError:   # a shape pairs cannot run (gating, split-K)
                        continue
                    g = capture(lambda ch=ch: ch.run(Xd, Wd, Y, ws, stream=stream))
                    for _ in range(args.warmup):
                        flush(); g.replay()
                    t = statistics.median(time_steps(g.replay, flush, k_base, stream)) * 1e3
                    baselines[f"microbatch_{rows}{'_pair' if cp == 2 else ''}_us"] = t
                    if best is None or t < best[1]:
                        best = (rows, t, cp)
                    ch.close()
                rows *= 2
            baselines["microbatch_best_us"] = best[1] if best else None
            baselines["microbatch_best_rows"] = best[0] if best else None
            baselines["microbatch_best_cta_pair"] = best[2] if best else None
            if not w.gelu and not w.residual:
                Wd_kn = [t.t() for t in Wd] if args.weight_layout == "nk" else Wd

                def torch_chain():
                    h = Xd
                    rest = Wd_kn
                    if w.gated:   # SwiGLU block in torch: silu(X Wg) * (X Wu), then the rest
                        h = torch.nn.functional.silu(torch.matmul(h, Wd_kn[0])) * torch.matmul(h, Wd_kn[1])
                        rest = Wd_kn[2:]
                    for t in rest:
                        h = torch.matmul(h, t)
                    Y.copy_(h)
                g = capture(torch_chain)
                for _ in range(args.warmup):
                    flush(); g.replay()
                baselines["torch_matmul_us"] = statistics.median(time_steps(g.replay, flush, k_base, stream)) * 1e3

        # ---- per-phase times of one pipelined run, from the event log (untimed build) ---------
        phases = None
        if args.mode == "pipelined" and w.num_gemms > 1:
            with make("pipelined", event_log=True) as ch:
                for _ in range(3):
                    flush()
                    ch.run(Xd, Wd, Y, ws, stream=stream)
                if ch.check(stream) != 0:
                    raise RuntimeError("device status set in the event-log run")
                phases = phase_breakdown(ch.event_log(), [ch.deps(b)[:2] for b in range(w.num_gemms - 1)],
                                         ch.cta_log())

        # ---- end to end through the host-buffer C-ABI call ------------------------------------
        Xh = X.pin_memory()
        Yh = torch.empty(w.M, w.dims[-1], dtype=torch.bfloat16).pin_memory()
        Xs = torch.empty_like(Xd)
        for _ in range(args.warmup):
            chain.run_host(Xh, Wd, Yh, Xs, Y, ws, stream=stream)
        torch.cuda.synchronize()
        e2e_ms = time_steps(lambda: chain.run_host(Xh, Wd, Yh, Xs, Y, ws, stream=stream), flush,
                            args.steps, stream)
        e2e_mean = max_over_ranks(statistics.mean(e2e_ms), world, dev)
        e2e_value = world * w.flops / (e2e_mean * 1e-3) / 1e12
        if chain.check(stream) != 0:
            raise RuntimeError("device status set during the e2e loop")
        Y_host = Y.float().cpu().numpy()

    # ---- roofline of the dominant kernel (the one chain kernel of the pipelined step) ----------
    peaks = load_peaks()
    t_hbm = w.algorithmic_bytes / (peaks["hbm_gbs"] * 1e9)
    t_tc = w.flops / (peaks["bf16_tflops"] * 1e12)
    launches = info["launches_per_run"]
    launch_s = mean_ms * 1e-3 / launches
    if t_hbm >= t_tc:
        roof = {"bound": "hbm", "achieved": w.algorithmic_bytes / launches / launch_s / 1e9,
                "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    else:
        roof = {"bound": "tensor", "achieved": w.flops / launches / launch_s / 1e12,
                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = recorded_traffic(w.name) if args.mode == "pipelined" and tiles == TUNED_TILES.get(w.name) else None
    roof["peak_source"] = f"{peaks['source']} (MEASURED_PEAKS.json)" if peaks["source"] == "measured" else "fallback"
    roof["t_roof_us"] = max(t_hbm, t_tc) * 1e6
    roof["latency_frac_of_roof"] = max(t_hbm, t_tc) * 1e6 / (mean_ms * 1e3)
    roof["algorithmic_bytes"] = w.algorithmic_bytes
    roof["flops"] = w.flops

    cpu = None
    parity = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu, parity, _, _ = cpu_oracle_baseline(w, X, Ws, args.cpu_budget, Y_host)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": mean_ms_all, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name, "M": w.M, "dims": list(w.dims), "gelu": w.gelu,
                       "residual": w.residual, "gated": w.gated, "mode": args.mode, "tile_m": info["tile_m"], "tile_n": info["tile_n"],
                       "k_split": info["k_split"], "cluster_size": info["cluster_size"], "cta_pair": info["cta_pair"], "splitk_exchange": args.splitk_exchange,
                       "raster_group": info["raster_group"],
                       "tile_k": info["tile_k"], "fill_k": info["fill_k"], "split_across": info["split_across"],
                       "queue_free": info["queue_free"], "grid_ctas": info["grid_ctas"], "pipe_stages": info["pipe_stages"],
                       "graph": "one CUDA graph replay per step",
                       "l2": f"flushed between steps (write of {2 * l2 >> 20} MiB, outside the timed events)",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "latency_us": {"median": lat_us, "mean": mean_ms * 1e3, "p10": pct(ms, 0.1) * 1e3,
                           "p90": pct(ms, 0.9) * 1e3},
            "baselines": baselines,
            "phases": phases,
            "roofline": roof,
            "cpu_baseline": cpu,
            "parity_vs_oracle_sample": parity,
            "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": X.numel() * 2,
                    "d2h_bytes_per_step": Y.numel() * 2, "latency_us": statistics.median(e2e_ms) * 1e3,
                    "what": "mlp_chain_run_host: pinned X -> device, chain whose last GEMM stores into pinned Y on the host, per step"},
            "gpu_launches": args.steps * launches,
            "clocks": {**clocks, "remeasured": remeasured},
            "kernel_source_sha256": kernel_source_hash(),
        }
        print(json.dumps(line), flush=True)
    chain.close()
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
