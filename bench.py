#!/usr/bin/env python3
"""Benchmark: paged MLA decode, nh128 b64 ctx8192 (bf16 cache, page_size 1).

One step = one decode call (mla_decode_fwd + mla_decode_combine when the plan
splits) over the whole batch, with every input already resident in HBM.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                  [--workload dense|ragged_bf16|ragged_fp8|fp8_long|mtp]

With --gpus N > 1 outside torchrun the script starts the N ranks itself
(torch.distributed.run, 127.0.0.1); under torchrun WORLD_SIZE must equal N.

Prints ONE JSON line (rank 0).  ``value`` is the whole-job KV-cache read rate
in TB/s (KV bytes of all ranks / max-over-ranks time); the per-call latency is
in ``us_per_call``.  Under torchrun (N > 1) every rank runs an independent
replica of the workload: the op has no exchange step, so there is no
collective on the data path (scaling: weak).

``--impl reference`` times the fp64 CPU oracle, as it stands, on a bounded
sample of the same workload on this host's cores (there is no reference
library to install: the pages hold no code).
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
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import mla_synth as syn  # noqa: E402

METRIC = "MLA decode µs/call & KV-cache TB/s (frac of roofline), nh128 b64 ctx8192"
UNIT = "TB/s"
HBM_FALLBACK_GBS = 6800.0
BF16_FALLBACK_TFLOPS = 1900.0
MI355X_HK_US = {"dense": 132.878}  # the pages' HK m16x8 time for this workload (other hardware)


# ------------------------------------------------------------------ workload ---

def make_workload(name: str, seed: int = 0, batch: int = 0, ctx: int = 0, heads: int = 0,
                  sq: int = 0, page_size: int = 0) -> syn.Problem:
    if name == "dense":
        return syn.dense(batch or 64, ctx or 8192, seed=seed)
    if name == "ragged_bf16":
        return syn.ragged(syn.KV_BF16, seed=seed)
    if name == "ragged_fp8":
        return syn.ragged(syn.KV_FP8_E4M3, seed=seed)
    if name == "fp8_long":
        return syn.fp8_long(ctx or 109440, seed=seed)
    if name == "mtp":
        return syn.mtp(heads or 64, sq or 2, page_size or 1, seed=seed)
    raise ValueError(name)


def visible_keys(p: syn.Problem) -> np.ndarray:
    """[B, Sq] keys each query token attends to."""
    lens = p.seq_lens.astype(np.int64)[:, None]
    i = np.arange(p.sq)[None, :]
    n = lens - p.sq + i + 1 if p.causal else np.broadcast_to(lens, (p.batch, p.sq))
    return np.clip(n, 0, lens)


def algorithmic(p: syn.Problem):
    """Bytes and FLOPs one decode call must move / do (no padding, no partials)."""
    row_bytes = 1152 if p.kv_dtype == syn.KV_BF16 else 576
    kv = int(p.seq_lens.astype(np.int64).sum()) * row_bytes
    rows = p.batch * p.sq * p.heads
    q_b = rows * 576 * 2
    out_b = rows * 512 * 2 + rows * 4
    bt_b = int(sum(-(-int(c) // p.page_size) for c in p.seq_lens)) * 4
    flops = 2 * int(visible_keys(p).sum()) * p.heads * (576 + 512)
    return dict(kv_bytes=kv, bytes=kv + q_b + out_b + bt_b + p.batch * 4, flops=flops)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d["bf16_tflops_sustained"]), "measured"
    except Exception:
        return HBM_FALLBACK_GBS, BF16_FALLBACK_TFLOPS, 1700.0, "fallback"


# ------------------------------------------------------------------- clocks ---

class NvmlClockSampler:
    """SM clock and clock-event reasons read through NVML (libnvidia-ml, read-only
    queries) every 0.5 ms while the timed region runs: a region of a few
    milliseconds still gets several samples.  Raises OSError when NVML is not
    there; the caller then falls back to nvidia-smi."""

    REASONS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
               "hw_thermal_slowdown": 0x40}

    def __init__(self, gpu_index: int, period_s: float = 0.0005):
        import ctypes
        self.nv = ctypes.CDLL("libnvidia-ml.so.1")
        if self.nv.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        if self.nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(gpu_index), ctypes.byref(self.h)) != 0:
            raise OSError("no NVML handle")
        self.period = period_s
        self.samples = []
        self.stop_flag = False
        self.t = None
        self.max_mhz = self._max_clock()

    def _clock(self):
        import ctypes
        v = ctypes.c_uint(0)  # NVML_CLOCK_SM = 1
        return v.value if self.nv.nvmlDeviceGetClockInfo(self.h, ctypes.c_int(1), ctypes.byref(v)) == 0 else None

    def _max_clock(self):
        import ctypes
        v = ctypes.c_uint(0)
        ok = self.nv.nvmlDeviceGetMaxClockInfo(self.h, ctypes.c_int(1), ctypes.byref(v)) == 0
        return v.value if ok else None

    def _reasons(self):
        import ctypes
        v = ctypes.c_ulonglong(0)
        fn = getattr(self.nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(self.nv, "nvmlDeviceGetCurrentClocksThrottleReasons")
        return v.value if fn(self.h, ctypes.byref(v)) == 0 else 0

    def _run(self):
        while not self.stop_flag:
            self.samples.append((self._clock(), self._reasons()))
            time.sleep(self.period)

    def start(self):
        self.t = threading.Thread(target=self._run, daemon=True)
        self.t.start()
        time.sleep(0.01)

    def stop(self):
        self.stop_flag = True
        self.t.join(timeout=2)
        sm = [c for c, _ in self.samples if c]
        reasons = sorted(n for n, bit in self.REASONS.items()
                         if any(r & bit for _, r in self.samples))
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": self.max_mhz,
                "samples": len(sm), "reasons": reasons, "source": "nvml, 0.5 ms"}


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.gpu)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, mx, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(power) if power else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# --------------------------------------------------------------- distributed ---

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(value: float, device=None) -> float:
    """Max over ranks (identity when not distributed)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_rate(units_per_rank: float, world: int, seconds_max: float) -> float:
    """Whole-job rate: every rank processed the same units; time is the max."""
    return units_per_rank * world / seconds_max


# ---------------------------------------------------------------- CPU oracle ---

def oracle_sample_rate(p: syn.Problem, target_s: float = 12.0):
    """Time the oracle on whole (sequence, all heads, all tokens) slices of the
    workload, growing the sample until it takes ~target_s; returns (KV bytes
    per second of the full workload extrapolated from the sample, description)."""
    import oracle
    oracle.build()
    row_bytes = 1152 if p.kv_dtype == syn.KV_BF16 else 576
    nb = 1
    while True:
        t0 = time.perf_counter()
        oracle.decode(p.q_bits, p.cache, p.kv_dtype, p.kv_scale, p.page_size, p.block_table,
                      p.seq_lens, p.softmax_scale, p.causal, b_range=(0, nb))
        dt = time.perf_counter() - t0
        if dt >= target_s / 3 or nb >= p.batch:
            break
        nb = min(p.batch, max(nb + 1, int(nb * target_s / max(dt, 1e-3) / 2)))
    sample_keys = int(p.seq_lens[:nb].astype(np.int64).sum())
    full_keys = int(p.seq_lens.astype(np.int64).sum())
    t_full = dt * full_keys / max(sample_keys, 1)
    kv_rate = full_keys * row_bytes / t_full
    desc = (f"first {nb} of {p.batch} sequences (all {p.heads} heads x {p.sq} tokens, "
            f"{sample_keys} keys) in {dt:.2f} s; full-batch time extrapolated by keys: "
            f"{t_full:.1f} s")
    return kv_rate, dt, nb, t_full, desc


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    p = make_workload(args.workload, batch=args.batch, ctx=args.ctx, heads=args.heads, sq=args.sq,
                      page_size=args.page_size)
    import oracle
    oracle.build()
    per_step = []
    nb = None
    for _ in range(args.warmup + args.steps):
        rate, dt, nb, t_full, desc = oracle_sample_rate(p, target_s=max(2.0, 30.0 / max(1, args.steps + args.warmup)))
        per_step.append((rate, t_full, desc))
    timed = per_step[args.warmup:]
    rate = statistics.median(r for r, _, _ in timed)
    t_full = statistics.median(t for _, t, _ in timed)
    value = rate / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_full * 1e3,
        "us_per_call": t_full * 1e6, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded N(0,1))",
        "config": config_of(p, args.workload),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": timed[-1][2]},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line))
    return 0


def config_of(p: syn.Problem, workload: str):
    lens = p.seq_lens.astype(np.int64)
    return {"workload": p.name, "workload_key": workload, "batch": p.batch, "heads": p.heads,
            "sq": p.sq, "ctx": int(lens.max()) if len(set(lens.tolist())) == 1 else "ragged",
            "sum_ctx": int(lens.sum()), "page_size": p.page_size,
            "kv_dtype": "bf16" if p.kv_dtype == syn.KV_BF16 else "fp8_e4m3",
            "causal": p.causal, "softmax_scale": p.softmax_scale,
            "l2": "inputs larger than L2 (KV cache %.0f MB vs 129 MB L2), no flush"
                  % (p.cache.nbytes / 1e6),
            "parallelism": "replicas"}


# ------------------------------------------------------------------- GPU arm ---

def run_gpu(args):
    import torch
    import paged_mla_decode_latent_gb300 as mla
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from parity import to_device

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    mla.build()
    p = make_workload(args.workload, seed=rank, batch=args.batch, ctx=args.ctx, heads=args.heads,
                      sq=args.sq, page_size=args.page_size)
    alg = algorithmic(p)
    t = to_device(p, dev)
    out = torch.empty((p.batch, p.sq, p.heads, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((p.batch, p.sq, p.heads), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    if args.dplan:
        # device-planned: the partition is computed on the GPU every step
        plan = mla.dplan_info(p.batch, p.heads, p.sq, p.page_size, p.kv_dtype, p.causal,
                              int(t["bt"].shape[1]) * p.page_size)
        ws = torch.empty(int(plan.workspace_bytes), dtype=torch.uint8, device=dev)
        launches_per_step = 3

        def pre(s):
            mla.plan_device(plan, t["lens"], ws, stream=s)

        def fwd_call(s):
            mla.fwd_dplan(plan, t["q"], t["cache"], t["scale"], t["bt"], p.softmax_scale, out, lse,
                          ws, stream=s)

        def post(s):
            mla.combine_dplan(plan, out, lse, ws, stream=s)

        def status():
            return mla.dplan_check(plan, ws)
    else:
        plan = mla.plan(p.seq_lens, p.heads, p.sq, p.page_size, p.kv_dtype, p.causal)
        ws = mla.workspace_for(plan, dev)
        launches_per_step = 1 + (1 if plan.num_splits > 1 else 0)

        def pre(s):
            pass

        def fwd_call(s):
            mla.fwd(plan, t["q"], t["cache"], t["scale"], t["bt"], t["lens"], p.softmax_scale,
                    out, lse, ws, s)

        def post(s):
            mla.combine(plan, t["lens"], out, lse, ws, s)

        def status():
            return mla.check(plan, ws)

    def step():
        pre(stream)
        fwd_call(stream)
        post(stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    st = status()
    if st != 0:
        raise RuntimeError(f"device status {st:#x} after warm-up")

    # choose K so the timed region lasts long enough for clock samples
    steps = args.steps
    if steps <= 0:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(5):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        per = e0.elapsed_time(e1) / 5 / 1e3
        steps = int(min(20000, max(20, math.ceil(2.5 / max(per, 1e-6)))))

    n_ev = steps
    ev_s = [torch.cuda.Event(enable_timing=True) for _ in range(n_ev)]
    ev_f = [torch.cuda.Event(enable_timing=True) for _ in range(n_ev)]
    ev_e = [torch.cuda.Event(enable_timing=True) for _ in range(n_ev)]
    gpu_index = dev.index if world == 1 else int(os.environ.get("LOCAL_RANK", 0))
    try:  # NVML numbers the GPUs of the machine, CUDA the visible ones
        nvml_index = torch.cuda._get_nvml_device_index(dev)
    except Exception:
        nvml_index = gpu_index
    try:
        clocks = NvmlClockSampler(nvml_index)
    except (OSError, AttributeError):
        clocks = ClockSampler(gpu_index)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for k in range(steps):
        pre(stream)
        ev_s[k].record(stream)
        fwd_call(stream)
        ev_f[k].record(stream)
        post(stream)
        ev_e[k].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    clk = clocks.stop()
    total_s = t_start.elapsed_time(t_end) / 1e3
    fwd_ms = [ev_s[k].elapsed_time(ev_f[k]) for k in range(steps)]
    step_ms = [ev_s[k].elapsed_time(ev_e[k]) for k in range(steps)]
    st = status()
    if st != 0:
        raise RuntimeError(f"device status {st:#x} after the timed steps")

    total_max = reduce_max(total_s, dev)
    ms_per_step = total_max / steps * 1e3
    fwd_mean_ms = statistics.mean(fwd_ms)
    kv_rate = aggregate_rate(alg["kv_bytes"] * steps, world, total_max)

    hbm, tc, tc_sus, peak_src = load_peaks()
    t_hbm = alg["bytes"] / (hbm * 1e9)
    t_tc = alg["flops"] / (tc * 1e12)
    bound = "hbm" if t_hbm >= t_tc else "tensor"
    if bound == "hbm":
        achieved = alg["bytes"] / (fwd_mean_ms / 1e3) / 1e9
        peak, unit = hbm, "GB/s"
    else:
        achieved = alg["flops"] / (fwd_mean_ms / 1e3) / 1e12
        peak, unit = tc, "TFLOP/s"
    roof = {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
            "frac": achieved / peak, "traffic": None, "peak_source": peak_src,
            "kernel": "mla_decode_fwd", "roofline_us": max(t_hbm, t_tc) * 1e6,
            "alg_bytes_per_launch": alg["bytes"], "alg_flops_per_launch": alg["flops"],
            "fwd_us_mean": fwd_mean_ms * 1e3, "fwd_us_median": statistics.median(fwd_ms) * 1e3}
    if bound == "tensor":  # the same against the tensor rate sustained over seconds
        roof["peak_sustained"] = tc_sus
        roof["frac_sustained"] = achieved / tc_sus
    prof = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(prof) and not args.dplan:
        try:
            tr = json.load(open(prof)).get(args.workload)
            if (tr and tr.get("kernel_rev") == kernel_revision(tr.get("sources"))
                    and tr.get("alg_bytes_per_launch") == alg["bytes"]):
                roof["traffic"] = tr["dram_bytes_per_launch"]
        except Exception:
            pass

    # the same step captured once as a CUDA graph (fwd + combine) and replayed
    graph = None
    if args.graph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            cap = torch.cuda.current_stream()
            pre(cap)
            fwd_call(cap)
            post(cap)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for _ in range(steps):
            g.replay()
        g1.record(stream)
        torch.cuda.synchronize()
        gsec = reduce_max(g0.elapsed_time(g1) / 1e3, dev)
        graph = {"us_per_call": gsec / steps * 1e6,
                 "value": aggregate_rate(alg["kv_bytes"] * steps, world, gsec) / 1e12,
                 "unit": UNIT, "steps": steps}
        st = status()
        if st != 0:
            raise RuntimeError(f"device status {st:#x} after the graph replays")

    # end to end through the public API with host buffers: H2D of q, block
    # table and lengths from pinned memory, decode, D2H of out and lse
    e2e = None if (args.no_e2e or args.dplan) else e2e_measure(mla, p, t, plan, ws, stream, dev,
                                                                max(10, min(steps, 400)), world)

    line = {
        "metric": METRIC, "value": kv_rate / 1e12, "unit": UNIT, "n_gpus": world,
        "steps": steps, "warmup": max(3, args.warmup), "ms_per_step": ms_per_step,
        "us_per_call": ms_per_step * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if p.kv_dtype == syn.KV_BF16 else "fp8_e4m3->bf16",
        "data": "synthetic (seeded N(0,1), numpy Philox)",
        "config": dict(config_of(p, args.workload), **(
            {"planner": "device", "unit_capacity": plan.max_units, "num_sms": plan.num_sms}
            if args.dplan else
            {"splits": plan.num_splits, "chunk_len": plan.chunk_len, "num_sms": plan.num_sms})),
        "roofline": roof, "clocks": clk, "e2e": e2e,
        **({"cuda_graph": graph} if graph is not None else {}),
        "gpu_launches": steps * launches_per_step,
        "context": {"mi355x_hk_m16x8_us": MI355X_HK_US.get(args.workload),
                    "note": "the pages' MI355X time for this shape (fp8 kernels, other hardware)"},
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, dt, nb, t_full, desc = oracle_sample_rate(p)
        import oracle
        line["cpu_baseline"] = {"value": rate / 1e12, "unit": UNIT, "cores": oracle.num_threads(),
                                "kind": "oracle", "sample": desc}
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def e2e_measure(mla, p, t, plan, ws, stream, dev, steps, world):
    """The decode through the public C-ABI calls with inputs and results in
    pinned host memory: every step copies its q, block table and lengths in
    and its out and lse back inside the timed region.

    Steps are pipelined as a serving loop runs them: two slots of device
    buffers, step i's inputs copied in (one copy stream) and step i-1's
    results copied out (another) while step i-1 / i computes on ``stream``.
    ``us_per_call`` is the pipelined time per step; ``serial_us_per_call``
    the time of one step at a time (copy in, compute, copy out, no overlap).
    """
    import torch
    q_h = t["q"].cpu().pin_memory()
    bt_h = t["bt"].cpu().pin_memory()
    lens_h = t["lens"].cpu().pin_memory()
    oshape, lshape = (p.batch, p.sq, p.heads, 512), (p.batch, p.sq, p.heads)
    out_h = [torch.empty(oshape, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    lse_h = [torch.empty(lshape, dtype=torch.float32).pin_memory() for _ in range(2)]
    q_d = [torch.empty_like(t["q"]) for _ in range(2)]
    bt_d = [torch.empty_like(t["bt"]) for _ in range(2)]
    lens_d = [torch.empty_like(t["lens"]) for _ in range(2)]
    out_d = [torch.empty(oshape, dtype=torch.bfloat16, device=dev) for _ in range(2)]
    lse_d = [torch.empty(lshape, dtype=torch.float32, device=dev) for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev = lambda: torch.cuda.Event()  # noqa: E731
    in_ready = [ev() for _ in range(2)]
    computed = [ev() for _ in range(2)]
    read_back = [ev() for _ in range(2)]
    used = [False, False]

    def step(i):
        k = i % 2
        with torch.cuda.stream(s_in):
            if used[k]:
                s_in.wait_event(computed[k])  # the slot's inputs are free again
            q_d[k].copy_(q_h, non_blocking=True)
            bt_d[k].copy_(bt_h, non_blocking=True)
            lens_d[k].copy_(lens_h, non_blocking=True)
            in_ready[k].record(s_in)
        stream.wait_event(in_ready[k])
        if used[k]:
            stream.wait_event(read_back[k])  # the slot's results were copied out
        mla.fwd(plan, q_d[k], t["cache"], t["scale"], bt_d[k], lens_d[k], p.softmax_scale,
                out_d[k], lse_d[k], ws, stream)
        mla.combine(plan, lens_d[k], out_d[k], lse_d[k], ws, stream)
        computed[k].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(computed[k])
            out_h[k].copy_(out_d[k], non_blocking=True)
            lse_h[k].copy_(lse_d[k], non_blocking=True)
            read_back[k].record(s_out)
        used[k] = True

    def timed(n, pipelined):
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        s_in.wait_event(e0)
        for i in range(n):
            step(i)
            if not pipelined:  # the next step's copies and compute start after this one is back
                s_in.wait_event(read_back[i % 2])
                stream.wait_event(read_back[i % 2])
        for k in range(2):
            if used[k]:
                stream.wait_event(read_back[k])  # every result is on the host
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / 1e3

    for _ in range(3):
        step(0)
    timed(3, True)
    sec = reduce_max(timed(steps, True), dev)
    serial = reduce_max(timed(max(3, steps // 4), False), dev) / max(3, steps // 4)
    kv = algorithmic(p)["kv_bytes"]
    h2d = q_h.numel() * 2 + bt_h.numel() * 4 + lens_h.numel() * 4
    d2h = out_h[0].numel() * 2 + lse_h[0].numel() * 4
    return {"value": aggregate_rate(kv * steps, world, sec) / 1e12, "unit": UNIT,
            "us_per_call": sec / steps * 1e6, "steps": steps,
            "serial_us_per_call": serial * 1e6, "pipelined": "2 steps in flight",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)}


def run_epilogue_bench(args):
    """The decode epilogue alone (q-concat + latent-row insert, one token per
    sequence at decode, H query rows + one cache row per token): µs per call
    and GB/s moved, CUDA events over back-to-back calls, inputs resident."""
    import torch
    import paged_mla_decode_latent_gb300 as mla
    torch.cuda.set_device(0)
    mla.build()
    T, H = args.tokens or 1, args.heads or 8
    fp8 = args.kv == "fp8"
    ps, pages = 64, max(4, (4 * T) // 64 + 4)  # noqa: E501
    g = np.random.default_rng(0)
    mk = lambda *sh: torch.randn(*sh, dtype=torch.float32, device="cuda").to(torch.bfloat16)  # noqa: E731
    ql, qp, kc, kp = mk(T, H, 512), mk(T, H, 64), mk(T, 512), mk(T, 64)
    slots = torch.from_numpy(g.choice(pages * ps, size=T, replace=False).astype(np.int64)).cuda()
    q = torch.empty((T, H, 576), dtype=torch.bfloat16, device="cuda")
    cache = (torch.zeros((pages, ps, 576), dtype=torch.uint8, device="cuda") if fp8 else
             torch.zeros((pages, ps, 576), dtype=torch.bfloat16, device="cuda"))
    scale = torch.tensor([0.0123], dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    call = lambda s: mla.epilogue(ql, qp, kc, kp, slots, q, cache, scale, stream=s)  # noqa: E731
    for _ in range(max(3, args.warmup)):
        call(stream)
    # Host-side launch cost (the ctypes call) exceeds this kernel's time, so
    # the calls are captured once as a CUDA graph and replayed: the device
    # time per call is what is measured.
    per_graph = 100
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cap = torch.cuda.current_stream()
        for _ in range(per_graph):
            call(cap)
    g.replay()
    reps = max(1, (args.steps if args.steps > 0 else 2000) // per_graph)
    steps = reps * per_graph
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(reps):
        g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) / steps * 1e3
    moved = T * H * 1152 * 2 + T * 1152 + T * (576 if fp8 else 1152) + T * 8
    hbm, _, _, src = load_peaks()
    gbs = moved / (us * 1e-6) / 1e9
    print(json.dumps({
        "metric": "MLA decode epilogue µs/call (q-concat + latent cache insert)", "value": us,
        "unit": "us", "higher_is_better": False, "steps": steps, "n_gpus": 1,
        "dtype": "bf16" if not fp8 else "bf16->fp8_e4m3",
        "config": {"workload": f"epilogue_t{T}_h{H}_{'fp8' if fp8 else 'bf16'}", "tokens": T,
                   "heads": H, "page_size": ps, "timing": "CUDA graph of 100 calls, replayed",
                   "l2": "working set %.1f MB: L2-resident (decode-size call)" % (moved / 1e6)},
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s",
                     "frac": gbs / hbm, "bytes_per_call": moved, "peak_source": src},
        "context": {"b300_page_kernel_us": 2.06,
                    "note": "the page's fused epilogue on B300, Kimi-K3 TP8 decode at concurrency 1"},
        "gpu_launches": steps}))
    return 0


def run_gather_kvb_bench(args):
    """The cached-prefix expansion alone (gather_kv_b_proj): the pages' shape,
    12 TP8-local heads, fp8 cache at page size 1, one sequence of --ctx cached
    tokens (default 32000); µs per call, TB/s moved and TFLOP/s against the
    measured peaks.  Synthetic kv_b_proj weights ~ N(0, 1/512)."""
    import torch
    import paged_mla_decode_latent_gb300 as mla
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from parity import to_device
    torch.cuda.set_device(0)
    mla.build()
    H = args.heads or 12
    batch = args.batch or 1
    ctx = args.ctx or 32000
    fp8 = args.kv != "bf16"
    p = syn.make_problem(batch, 1, 4, [ctx] * batch, 1, syn.KV_FP8_E4M3 if fp8 else syn.KV_BF16,
                         False, seed=0, name=f"gather_kvb_h{H}_b{batch}_ctx{ctx}")
    t = to_device(p)
    w = (torch.randn((H, 256, 512), device="cuda") / math.sqrt(512.0)).to(torch.bfloat16)
    cu = torch.arange(batch + 1, dtype=torch.int32, device="cuda") * ctx
    T = batch * ctx
    k = torch.empty((T, H, 192), dtype=torch.bfloat16, device="cuda")
    v = torch.empty((T, H, 128), dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    call = lambda: mla.gather_kv_b_proj(t["cache"], t["scale"], t["bt"], t["lens"], cu, ctx, w, k,  # noqa: E731
                                        v, status, stream)
    for _ in range(max(3, args.warmup)):
        call()
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"status {int(status.item()):#x}")
    steps = args.steps if args.steps > 0 else 50
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        call()
    e1.record(stream)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) / steps * 1e3
    row = 576 if fp8 else 1152
    moved = T * row + T * H * (192 + 128) * 2 + H * 256 * 512 * 2 + batch * 8
    flops = 2.0 * T * H * 256 * 512
    hbm, tc, _, src = load_peaks()
    t_hbm, t_tc = moved / (hbm * 1e9), flops / (tc * 1e12)
    bound = "tensor" if t_tc >= t_hbm else "hbm"
    achieved = flops / (us * 1e-6) / 1e12 if bound == "tensor" else moved / (us * 1e-6) / 1e9
    peak = tc if bound == "tensor" else hbm
    print(json.dumps({
        "metric": "gather_kv_b_proj µs/call (cached-prefix K/V expansion)", "value": us,
        "unit": "us", "higher_is_better": False, "steps": steps, "n_gpus": 1,
        "dtype": "fp8_e4m3->bf16" if fp8 else "bf16",
        "config": {"workload": p.name, "heads": H, "batch": batch, "ctx": ctx, "page_size": 1},
        "tb_per_s": moved / (us * 1e-6) / 1e12,
        "roofline": {"bound": bound, "achieved": achieved, "peak": peak,
                     "unit": "TFLOP/s" if bound == "tensor" else "GB/s", "frac": achieved / peak,
                     "roofline_us": max(t_hbm, t_tc) * 1e6, "bytes_per_call": moved,
                     "flops_per_call": flops, "peak_source": src},
        "context": {"mi355x_page_ms": {"4096": 0.038, "32000": 0.227, "65536": 0.442,
                                       "109440": 0.711},
                    "note": "the page's Triton kernel on MI355X (Kimi-K3 TP8, 12 heads, fp8, ps 1)"},
        "gpu_launches": steps}))
    return 0


def kernel_revision(sources=None) -> str:
    """Hash of the sources that define a kernel (default: all of csrc/): a
    recorded traffic figure is void once any of them changes."""
    import hashlib
    h = hashlib.sha1()
    csrc = os.path.join(ROOT, "paged_mla_decode_latent_gb300", "csrc")
    for f in sorted(sources or os.listdir(csrc)):
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:12]


def _free_port() -> int:
    import socket
    with socket.socket() as so:
        so.bind(("127.0.0.1", 0))
        return so.getsockname()[1]


def launch_replicas(n: int, argv) -> int:
    """Start one rank per GPU (torch.distributed.run on 127.0.0.1) running
    this script with the same arguments; returns the launcher's exit code."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           f"--nproc-per-node={n}", "--master-addr", "127.0.0.1",
           "--master-port", str(_free_port()), os.path.abspath(__file__), *argv]
    return subprocess.call(cmd)


def run_launch_check(args):
    """The replica launch and the cross-rank reduction alone, on CPU ranks
    (gloo): no decode runs.  Rank 0 prints what every rank saw."""
    import torch.distributed as dist
    world, rank, _ = dist_env()
    dist.init_process_group("gloo")
    t = reduce_max(1.0 + 0.5 * rank)
    seen = [None] * world
    dist.all_gather_object(seen, {"rank": rank, "world": world, "max_s": t,
                                  "rate": aggregate_rate(1000.0, world, t)})
    if rank == 0:
        print(json.dumps({"launch_check": {"gpus": args.gpus, "world": world, "ranks": seen}}))
    dist.destroy_process_group()
    return 0


def main(argv=None):
    argv = list(sys.argv[1:] if argv is None else argv)
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1,
                    help="replicas, one per GPU; started here through torch.distributed.run "
                         "unless already launched that way with WORLD_SIZE == N")
    ap.add_argument("--launch-check", action="store_true",
                    help="only start the ranks and check the cross-rank reduction (CPU, gloo)")
    ap.add_argument("--steps", type=int, default=0, help="0 = enough for ~2.5 s of timed work")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="dense",
                    choices=["dense", "ragged_bf16", "ragged_fp8", "fp8_long", "mtp", "epilogue",
                             "gather_kvb"])
    ap.add_argument("--tokens", type=int, default=0, help="epilogue workload: tokens (default 1)")
    ap.add_argument("--heads", type=int, default=0,
                    help="epilogue (default 8), gather_kvb (12) or mtp (64) workload: heads")
    ap.add_argument("--sq", type=int, default=0, help="mtp workload: query tokens (default 2)")
    ap.add_argument("--page-size", type=int, default=0, help="mtp workload: page size (default 1)")
    ap.add_argument("--kv", default="", choices=["", "bf16", "fp8"],
                    help="epilogue (default bf16) / gather_kvb (default fp8) workload: cache")
    ap.add_argument("--batch", type=int, default=0, help="dense workload: batch (default 64)")
    ap.add_argument("--ctx", type=int, default=0,
                    help="dense (default 8192) or fp8_long (default 109440) workload: context")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--dplan", action="store_true",
                    help="device-planned path: the partition computed on the GPU each step")
    ap.add_argument("--graph", action="store_true",
                    help="also time the step captured as one CUDA graph and replayed")
    args = ap.parse_args(argv)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.gpus > 1 and "RANK" not in os.environ:
        return launch_replicas(args.gpus, argv)
    if args.gpus != world:
        raise SystemExit(f"bench.py: --gpus {args.gpus} but WORLD_SIZE={world}: launch one rank "
                         "per GPU with --nproc-per-node equal to --gpus")
    if args.launch_check:
        return run_launch_check(args)
    if args.workload == "epilogue":
        return run_epilogue_bench(args)
    if args.workload == "gather_kvb":
        return run_gather_kvb_bench(args)
    if args.impl == "reference":
        if args.steps <= 0:
            args.steps = 3
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
