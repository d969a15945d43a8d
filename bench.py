#!/usr/bin/env python
"""Throughput of one MLA decode step (weight-absorbed, latent cache) on GB300.

A step is the whole hot path for one batch through the C-ABI call
mla_decode_step: absorb_q -> decode split -> LSE combine -> out_proj (for
bf16 the combine and out_proj run as one fused kernel).  The default workload is
DeepSeek-V2-Lite decode in bf16: B=8 sequences of S=4096 cached rows, H=16.
Each step reads one "layer": the bench keeps L copies of cache + weights
(L chosen so that their total exceeds 3x the L2 size) and step k uses layer
k mod L, so no step finds its cache in L2.

Prints one JSON line.  `value` is latent-cache GB/s of the whole step
(algorithmic cache bytes B*S*576*2 per step over the device time of the
timed steps); `tokens_per_s` is B*steps/time.  `roofline` covers the split
kernel (the dominant kernel), timed with CUDA events around each of its
launches inside the timed region.

`--impl reference` times the fp64 CPU oracle instead (the reference arm).
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

METRIC = "MLA decode latent-cache GB/s (vs ~8 TB/s HBM) and decode tokens/s"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0
# DRAM bytes per split launch measured by ncu: a list of records, each naming the
# kernel, the workload and the sources (with their sha256) it was measured on.
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "split_traffic.json")
SPLIT_KERNEL = {"bf16": "split_tc_kernel", "fp8": "split_fp8_kernel", "f32": "split_f32_kernel"}
DTYPE_NAME = {"bf16": "bf16", "fp8": "fp8_e4m3 cache, bf16 weights", "f32": "f32"}


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="v2lite_bf16_b8_s4096")
    ap.add_argument("--splits", type=int, default=0, help="KV chunks per sequence (0 = auto)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--op", default="step",
                    choices=["step", "cache_append", "wo_proj", "kq_proj", "ov_proj", "absorb_q",
                             "combine", "out_proj"],
                    help="step: the decode step (default); cache_append / wo_proj: the steps "
                         "around it, timed alone on the workload's sizes")
    return ap.parse_args(argv)


# ----------------------------------------------------------------------------- peaks, traffic
def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def sources_sha(sources):
    h = hashlib.sha256()
    for rel in sources:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def recorded_traffic(kernel, workload):
    """The recorded DRAM bytes per launch of `kernel` on `workload`, or None when
    there is no record or its sources have changed since it was taken."""
    try:
        with open(TRAFFIC_FILE) as f:
            records = json.load(f)
    except Exception:
        return None
    for d in records:
        if d.get("kernel") != kernel or d.get("workload") != workload:
            continue
        try:
            if d.get("source_sha256") == sources_sha(d.get("sources", [])):
                return d.get("dram_bytes_per_launch")
        except OSError:
            return None
    return None


# ----------------------------------------------------------------------------- clocks (NVML)
class ClockSampler:
    """Samples SM clock and clock-event reasons through NVML while running."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
               0x2: "applications_clocks_setting", 0x10: "sync_boost"}

    def __init__(self, bus_id: str | None, period_s: float = 0.002):
        self.ok = False
        self.samples = []
        self.reasons = 0
        self.period = period_s
        try:
            self.nvml = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nvml.nvmlInit_v2() != 0:
                return
            self.h = ctypes.c_void_p()
            if bus_id is not None:
                r = self.nvml.nvmlDeviceGetHandleByPciBusId_v2(bus_id.encode(), ctypes.byref(self.h))
            else:
                r = self.nvml.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(self.h))
            if r != 0:
                return
            mx = ctypes.c_uint()
            self.nvml.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx))
            self.max_mhz = mx.value
            self.ok = True
        except OSError:
            pass

    def _poll(self):
        clk = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        fn = getattr(self.nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.nvml.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self._stop.is_set():
            if self.nvml.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(clk)) == 0:
                self.samples.append(clk.value)
            if fn(self.h, ctypes.byref(rs)) == 0:
                self.reasons |= rs.value
            time.sleep(self.period)

    def __enter__(self):
        if self.ok:
            self._stop = threading.Event()
            self._t = threading.Thread(target=self._poll, daemon=True)
            self._t.start()
        return self

    def __exit__(self, *a):
        if self.ok:
            self._stop.set()
            self._t.join()

    def summary(self):
        if not self.ok or not self.samples:
            return None
        names = [n for bit, n in self.REASONS.items() if self.reasons & bit]
        return {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": names, "samples": len(self.samples), "source": "nvml"}


def bus_id_of(device_index: int):
    try:
        rt = ctypes.CDLL("libcudart.so.13")
        buf = ctypes.create_string_buffer(64)
        if rt.cudaDeviceGetPCIBusId(buf, 64, device_index) == 0:
            return buf.value.decode()
    except OSError:
        pass
    return None


# ----------------------------------------------------------------------------- CPU oracle leg
def oracle_throughput(cfg, budget_s: float, max_steps: int | None = None, warmup: int = 0,
                      rows_per_step: int | None = None):
    """Time the fp64 oracle's absorbed path on sequences of `cfg` (inputs converted
    to fp64 beforehand, outside the timing).  Returns (GB/s, tokens/s, steps, rows, cores)."""
    import numpy as np
    from oracle import mla_oracle as O
    from workloads import make_inputs
    inp = make_inputs(cfg, seed=0)
    seqs = [inp.as_float64_numpy(b) for b in range(cfg.batch)]
    for a in seqs:
        if a["cache"] is None:   # FP8 cache: the oracle decodes the E4M3 codes
            a["cache"] = O.e4m3_to_float64(a["cache_e4m3"])
    rows = cfg.s_max if rows_per_step is None else max(1, min(cfg.s_max, rows_per_step))

    def one(i):
        a = seqs[i % cfg.batch]
        n = rows
        O.decode_absorbed(a["q_nope"], a["q_rope"], a["w_uk"], a["w_uv"], a["cache"][:, :n],
                          np.array([n]), np.array([n - 1]), cfg.softmax_scale, cfg.rope_base)

    for i in range(warmup):
        one(i)
    t0 = time.perf_counter()
    steps = 0
    while True:
        one(steps)
        steps += 1
        el = time.perf_counter() - t0
        if max_steps is not None and steps >= max_steps:
            break
        if max_steps is None and el >= budget_s:
            break
    el = time.perf_counter() - t0
    byts = steps * rows * cfg.row * cfg.elt_bytes
    return byts / el / 1e9, steps / el, steps, rows, el


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


# ----------------------------------------------------------------------------- reference arm
def run_reference(args, cfg, rank, world):
    if rank != 0:
        return 0
    # Size each step so that warm-up + steps stay within about two minutes.
    import numpy as np  # noqa: F401
    probe_gbs, _, _, _, probe_el = oracle_throughput(cfg, 0.0, max_steps=1, rows_per_step=cfg.s_max)
    per_full = probe_el
    budget = 120.0
    rows = cfg.s_max
    if per_full * (args.steps + args.warmup) > budget:
        rows = max(32, int(cfg.s_max * budget / (per_full * (args.steps + args.warmup))))
    gbs, tps, steps, rows, el = oracle_throughput(cfg, 0.0, max_steps=args.steps,
                                                  warmup=args.warmup, rows_per_step=rows)
    sample = (f"each step: fp64 NumPy oracle (absorbed form, exact softmax) on one sequence's "
              f"first {rows} of {cfg.s_max} rows, H={cfg.heads}, cycling over the {cfg.batch} "
              f"sequences of the workload")
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": steps, "warmup": args.warmup, "ms_per_step": el / steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "tokens_per_s": tps,
        "config": workload_config(cfg, None, None),
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": cpu_cores(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(cfg, layers, splits):
    c = {"workload": cfg.name, "batch": cfg.batch, "heads": cfg.heads, "seq_len": cfg.s_max,
         "d_c": cfg.d_c, "d_rope": cfg.d_rope, "d_nope": cfg.d_nope, "d_v": cfg.d_v,
         "cache_dtype": cfg.dtype, "parallelism": "replicas (one batch per GPU, no collective)"}
    if layers is not None:
        c["l2"] = (f"inputs larger than L2: {layers} layer copies of cache + W_UK + W_UV rotated, "
                   f"step k reads layer k mod {layers}")
    if splits is not None:
        c["kv_splits"] = splits
    if cfg.q_len > 1:
        c["q_len"] = cfg.q_len
    return c


# ----------------------------------------------------------------------------- ranks
def max_over_ranks(x: float, device, world: int) -> float:
    """The slowest rank's time: every rank contributes its own, all receive the max."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank_step: float, steps: int, world: int, seconds: float) -> float:
    """Units all ranks processed (each rank runs its own replica of the workload) per
    second of the slowest rank."""
    return units_per_rank_step * steps * world / seconds


# ----------------------------------------------------------------------------- around the step
def run_op(args, cfg, rank):
    """Time mla_cache_append, mla_wo_proj, or the materialised projections
    (mla_absorb_q_materialized: x . W^KQ and RoPE; mla_ov_proj: W^OV on o_c) alone
    on the workload's sizes: K launches
    in one CUDA graph over L rotating weight copies (more than 3x L2), CUDA events
    around the replay.  The dominant bytes are the weight's; the line reports them
    per second against the measured HBM peak."""
    import torch
    import head_latent_attention_absorbed_gb300 as mla
    from workloads import (cache_storage, make_append_inputs, make_inputs,
                           make_materialized_inputs, make_wo_inputs)
    mla.load()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    dt = cache_storage(cfg)   # the cache's type names the library dtype
    d = mla.dims(cfg.batch, cfg.heads, cfg.s_max, mla.dtype_code(dt))
    l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or 126 * 2 ** 20
    if args.op == "cache_append":
        inp = make_append_inputs(cfg, seed=0)
        wbytes = inp.w_kva.numel() * inp.w_kva.element_size()
        L = max(2, math.ceil(3 * l2 / wbytes))
        ws = [inp.w_kva.to(dev) for _ in range(L)]
        x, pos = inp.x.to(dev), inp.positions.to(dev)
        cache = torch.zeros((cfg.batch, cfg.s_max, cfg.row), dtype=dt, device=dev)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        moved = wbytes + x.numel() * x.element_size() + cfg.batch * cfg.row * cache.element_size()
        launch = lambda k: mla.cache_append(d, x, ws[k % L], pos, cache, cfg.rope_base, status)
        metric = "cache append: kv_a_proj weight + token + row bytes per second"
    elif args.op in ("absorb_q", "out_proj", "combine"):
        # The three kernels of the step around the split, each alone: absorb (a1 + a2,
        # bound by W_UK), combine (a4, the chunk partials), out_proj (a5, bound by W_UV).
        inp = make_inputs(cfg, seed=0)
        B, H = cfg.batch, cfg.heads
        q_abs = torch.empty((B, H, cfg.d_c), dtype=torch.float32, device=dev)
        q_pe = torch.empty((B, H, cfg.d_rope), dtype=torch.float32, device=dev)
        o_c = torch.empty((B, H, cfg.d_c), dtype=torch.float32, device=dev)
        lse = torch.empty((B, H), dtype=torch.float32, device=dev)
        out = torch.empty((B, H, cfg.d_v), dtype=torch.float32, device=dev)
        qn, qr = inp.q_nope.to(dev), inp.q_rope.to(dev)
        pos, lengths = inp.positions.to(dev), inp.lengths.to(dev)
        wbytes = inp.w_uk.numel() * inp.w_uk.element_size()
        L = max(2, math.ceil(3 * l2 / wbytes))
        if args.op == "absorb_q":
            ws = [inp.w_uk.to(dev) for _ in range(L)]
            moved = (wbytes + qn.numel() * qn.element_size() + qr.numel() * qr.element_size() +
                     pos.numel() * 4 + q_abs.numel() * 4 + q_pe.numel() * 4)
            launch = lambda k: mla.absorb_q(d, qn, qr, ws[k % L], pos, q_abs, q_pe, cfg.rope_base)
            metric = "absorb: W_UK + queries + q_abs + q_pe bytes per second"
        elif args.op == "out_proj":
            ws = [inp.w_uv.to(dev) for _ in range(L)]
            o_c.normal_()
            moved = wbytes + o_c.numel() * 4 + out.numel() * 4
            launch = lambda k: mla.out_proj(d, o_c, ws[k % L], out)
            metric = "out_proj: W_UV + o_c + o bytes per second"
        else:
            L = 1
            splits = mla.num_splits(d, args.splits)
            wsp = torch.empty((mla.workspace_bytes(d, args.splits),), dtype=torch.uint8, device=dev)
            status = torch.zeros(1, dtype=torch.int32, device=dev)
            mla.absorb_q(d, qn, qr, inp.w_uk.to(dev), pos, q_abs, q_pe, cfg.rope_base)
            mla.decode_split(d, q_abs, q_pe, inp.cache.to(dev), lengths, wsp, cfg.softmax_scale,
                             args.splits, status)
            torch.cuda.synchronize()
            if int(status.item()) != 0:
                raise RuntimeError("device status after the split that fills the partials")
            chunk = (-(-cfg.s_max // splits) + 7) // 8 * 8
            used = sum(-(-int(n) // chunk) for n in inp.lengths.tolist())   # chunks with rows
            moved = used * H * (cfg.d_c + 1) * 4 + o_c.numel() * 4 + lse.numel() * 4
            launch = lambda k: mla.decode_combine(d, lengths, wsp, o_c, args.splits, lse)
            metric = "combine: chunk partials read + o_c + lse bytes per second (partials in L2)"
    elif args.op in ("kq_proj", "ov_proj"):
        m = make_materialized_inputs(cfg, seed=0)
        wdt = m.w_o.dtype
        H = cfg.heads
        if args.op == "kq_proj":
            w0 = torch.empty((H * cfg.d_c, cfg.hidden), dtype=wdt, device=dev)
            mla.materialize_wkq(d, m.w_q_nope.to(dev), m.base.w_uk.to(dev), w0)
        else:
            w0 = torch.empty((cfg.hidden, H * cfg.d_c), dtype=wdt, device=dev)
            mla.materialize_wov(d, m.w_o.to(dev), m.base.w_uv.to(dev), w0)
        wbytes = w0.numel() * w0.element_size()
        L = max(2, math.ceil(3 * l2 / wbytes))
        ws = [w0.clone() for _ in range(L)]
        x = m.x.to(dev)
        q_rope, pos = m.base.q_rope.to(dev), m.base.positions.to(dev)
        q_abs = torch.empty((cfg.batch, H, cfg.d_c), dtype=torch.float32, device=dev)
        q_pe = torch.empty((cfg.batch, H, cfg.d_rope), dtype=torch.float32, device=dev)
        o_c = torch.randn((cfg.batch, H, cfg.d_c), generator=torch.Generator().manual_seed(0)).to(dev)
        y = torch.empty((cfg.batch, cfg.hidden), dtype=torch.float32, device=dev)
        if args.op == "kq_proj":
            moved = (wbytes + x.numel() * x.element_size() + q_abs.numel() * 4 +
                     q_rope.numel() * q_rope.element_size() + q_pe.numel() * 4)
            launch = lambda k: mla.absorb_q_materialized(d, x, ws[k % L], q_rope, pos, q_abs, q_pe,
                                                         cfg.rope_base)
            metric = "materialised absorb: W^KQ weight + x + q bytes per second"
        else:
            moved = wbytes + o_c.numel() * 4 + y.numel() * 4
            launch = lambda k: mla.ov_proj(d, o_c, ws[k % L], y)
            metric = "materialised output: W^OV weight + o_c + y bytes per second"
    else:
        inp = make_wo_inputs(cfg, seed=0)
        wbytes = inp.w_o.numel() * inp.w_o.element_size()
        L = max(2, math.ceil(3 * l2 / wbytes))
        ws = [inp.w_o.to(dev) for _ in range(L)]
        o = inp.o.to(dev)
        y = torch.empty((cfg.batch, cfg.hidden), dtype=torch.float32, device=dev)
        moved = wbytes + o.numel() * 4 + y.numel() * 4
        launch = lambda k: mla.wo_proj(d, o, ws[k % L], y)
        metric = "W^O projection: weight + input + output bytes per second"
    K, W = args.steps, args.warmup
    for k in range(W):
        launch(k)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream(device=dev)
    with torch.cuda.graph(g, stream=cap, capture_error_mode="thread_local"):
        for k in range(K):
            launch(k)
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    g.replay()
    e1.record()
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / K
    gbs = moved / (us * 1e-6) / 1e9
    peak, peak_kind = measured_peaks()
    line = {"op": args.op, "metric": metric, "value": gbs, "unit": "GB/s", "n_gpus": 1,
            "steps": K, "warmup": W, "us_per_launch": us, "higher_is_better": True,
            "dtype": DTYPE_NAME[cfg.dtype], "data": "synthetic",
            "config": {"workload": cfg.name, "batch": cfg.batch, "heads": cfg.heads,
                       "hidden": cfg.hidden,
                       "l2": (f"{L} rotating weight copies, more than 3x L2" if args.op != "combine"
                              else "the partials, written by the split just before, in L2")},
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s",
                         "frac": gbs / peak, "peak_kind": f"{peak_kind} (copy bandwidth, burst)",
                         "bytes_per_launch": moved}}
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def launches_per_step(cfg) -> int:
    """Library kernels one step launches: absorb, (FP8: the query image), split,
    then the fused combine + W_UV (one token, bf16/FP8, batch x heads <= 256) or
    combine and out_proj."""
    fused = cfg.q_len == 1 and cfg.dtype != "f32" and cfg.batch * cfg.heads <= 256
    return 1 + (1 if cfg.dtype == "fp8" else 0) + 1 + (1 if fused else 2)


# ----------------------------------------------------------------------------- our arm
def main():
    return main_with(parse(), int(os.environ.get("RANK", "0")),
                     int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("LOCAL_RANK", "0")))


def main_with(args, rank: int, world: int, local: int = 0):
    from workloads import BY_NAME
    cfg = BY_NAME[args.workload]

    if args.impl == "reference":
        return run_reference(args, cfg, rank, world)
    if args.op != "step":
        return run_op(args, cfg, rank)

    import torch
    import torch.distributed as dist
    import head_latent_attention_absorbed_gb300 as mla
    from workloads import cache_storage, make_inputs

    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    mla.load()

    dt = cache_storage(cfg)   # the cache's type names the library dtype
    inp = make_inputs(cfg, seed=rank)
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 0) or 126 * 2 ** 20
    per_layer = (inp.cache.numel() * inp.cache.element_size() +
                 (inp.w_uk.numel() + inp.w_uv.numel()) * inp.w_uk.element_size())
    L = max(2, math.ceil(3 * l2 / per_layer))
    caches = [inp.cache.to(dev) for _ in range(L)]
    wuk = [inp.w_uk.to(dev) for _ in range(L)]
    wuv = [inp.w_uv.to(dev) for _ in range(L)]
    qn = [inp.q_nope.to(dev) for _ in range(L)]
    qr = [inp.q_rope.to(dev) for _ in range(L)]
    lengths = inp.lengths.to(dev)
    positions = inp.positions.to(dev)
    step = mla.DecodeStep(cfg.batch, cfg.heads, cfg.s_max, dt, device=dev,
                          num_splits_requested=args.splits, rope_base=cfg.rope_base,
                          softmax_scale=cfg.softmax_scale, q_len=cfg.q_len)
    d = step.dims
    cache_bytes = int(inp.lengths.to(torch.int64).sum()) * cfg.row * inp.cache.element_size()

    def one_step(k):
        # The whole step through the single call mla_decode_step: absorb, split,
        # and (bf16) the fused combine + W_UV kernel.
        l = k % L
        step.run(qn[l], qr[l], caches[l], lengths, positions, wuk[l], wuv[l])

    K, W = args.steps, args.warmup
    for k in range(W):
        one_step(k)
    torch.cuda.synchronize()
    if int(step.status.item()) != 0:
        raise RuntimeError(f"device status {int(step.status.item())} after warm-up")

    # The K timed steps, captured as one CUDA graph (four launches per step).
    cap = torch.cuda.Stream(device=dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=cap, capture_error_mode="thread_local"):
        for k in range(K):
            one_step(k)
    g.replay()                       # one untimed replay (graph upload, warm)
    torch.cuda.synchronize()

    t_begin = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(bus_id_of(dev.index))
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with sampler:
        t_begin.record()
        g.replay()
        t_end.record()
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    elapsed_ms = t_begin.elapsed_time(t_end)
    if int(step.status.item()) != 0:
        raise RuntimeError(f"device status {int(step.status.item())} after the timed steps")

    elapsed_ms = max_over_ranks(elapsed_ms, dev, world)
    sec = elapsed_ms / 1e3
    value = whole_job_rate(cache_bytes, K, world, sec) / 1e9
    tokens = whole_job_rate(cfg.batch * cfg.q_len, K, world, sec)

    # The dominant kernel alone: Ks back-to-back split launches over the same
    # rotating layer copies, one CUDA graph, CUDA events on the replay stream.
    # (Event nodes between the launches of the step graph would themselves add
    # microseconds per launch.)
    Ks = min(K, 400)
    gs = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gs, stream=cap, capture_error_mode="thread_local"):
        for k in range(Ks):
            if cfg.q_len == 1:
                mla.decode_split(d, step.q_abs, step.q_pe, caches[k % L], lengths,
                                 step.workspace, step.scale, args.splits, step.status)
            else:   # the split has no separate multi-token entry: split + combine
                mla.decode_attn_multi(d, cfg.q_len, step.q_abs, step.q_pe, caches[k % L],
                                      lengths, step.o_c, step.workspace, step.scale, args.splits,
                                      step.lse, step.status)
    gs.replay()
    torch.cuda.synchronize()
    s_begin = torch.cuda.Event(enable_timing=True)
    s_end = torch.cuda.Event(enable_timing=True)
    s_begin.record()
    gs.replay()
    s_end.record()
    torch.cuda.synchronize()
    split_avg_s = s_begin.elapsed_time(s_end) / 1e3 / Ks
    if int(step.status.item()) != 0:
        raise RuntimeError(f"device status {int(step.status.item())} after the split-only replay")

    # End-to-end through the public API with host buffers: every step copies the
    # queries, lengths and positions from pinned host memory and reads o back
    # into pinned host memory.  Each layer copy's step is captured once with
    # DecodeStep.capture and replayed.
    e2e = None
    if not args.no_e2e:
        hosts = [step.capture(caches[l], wuk[l], wuv[l]) for l in range(L)]
        for l, hs in enumerate(hosts):          # the host side fills each step's inputs
            hs.q_nope.copy_(inp.q_nope)
            hs.q_rope.copy_(inp.q_rope)
            hs.lengths.copy_(inp.lengths)
            hs.positions.copy_(inp.positions)
        Ke = min(K, 2000)
        for k in range(min(W, 20)):
            hosts[k % L].replay()
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for k in range(Ke):
            hosts[k % L].replay()
        e1.record()
        torch.cuda.synchronize()
        e_ms = e0.elapsed_time(e1)
        if int(step.status.item()) != 0:
            raise RuntimeError(f"device status {int(step.status.item())} after the e2e steps")
        e_ms = max_over_ranks(e_ms, dev, world)
        bi, bo = hosts[0].h2d_bytes, hosts[0].d2h_bytes
        e2e = {"value": whole_job_rate(cache_bytes, Ke, world, e_ms / 1e3) / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo, "steps": Ke,
               "tokens_per_s": whole_job_rate(cfg.batch * cfg.q_len, Ke, world, e_ms / 1e3),
               "path": ("DecodeStep.capture: per step one CUDA-graph replay of mla_decode_step"
                        + ("" if cfg.q_len == 1 else "_multi") + " on pinned host buffers -- its "
                        "kernels read the queries, lengths and positions and write o over the "
                        "host link, no copy nodes")}

    peak, peak_kind = measured_peaks()
    achieved = cache_bytes / split_avg_s / 1e9
    kname = SPLIT_KERNEL[cfg.dtype]
    roofline = {"bound": "hbm",
                "kernel": (f"{kname} (mla_decode_split)" if cfg.q_len == 1 else
                           f"{kname} + combine_kernel (mla_decode_attn_multi)"),
                "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "peak_kind": f"{peak_kind} (copy bandwidth, burst)",
                "frac_of_nominal_8TBs": achieved / NOMINAL_HBM_GBS,
                "traffic": recorded_traffic(kname, cfg.name),
                "bytes_per_launch": cache_bytes,
                "avg_launch_us": split_avg_s * 1e6,
                "launches_timed": Ks,
                "timing": "graph of back-to-back split launches, CUDA events around its replay"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        gbs, tps, nsteps, rows, el = oracle_throughput(cfg, args.cpu_seconds)
        cpu = {"value": gbs, "unit": "GB/s", "cores": cpu_cores(), "kind": "oracle",
               "tokens_per_s": tps,
               "sample": (f"{nsteps} single-sequence decode steps ({rows} rows, H={cfg.heads}) "
                          f"of this workload through the fp64 NumPy oracle, {el:.1f} s; inputs "
                          f"converted to fp64 before timing")}

    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": elapsed_ms / K, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": DTYPE_NAME[cfg.dtype],
        "data": "synthetic (seeded N(0,1) cache and queries, N(0,0.02^2) weights)",
        "tokens_per_s": tokens,
        "config": workload_config(cfg, L, step.splits),
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": launches_per_step(cfg) * K,
        "clocks": sampler.summary(),
        "timing": "one CUDA-graph replay of the timed steps (no event nodes inside), CUDA events "
                  "on the replay stream",
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
