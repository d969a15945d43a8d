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
kernel (the dominant kernel) and, under `decode_attn`, mla_decode_attn
(split + LSE combine), each timed as a CUDA graph of back-to-back plain
launches (each starting after the previous one ended) with the overlapped
figure beside it; `roofline_workloads` gives the same two for the ragged,
128-head and long-context workloads; `steady` replays a long graph of steps
with the SM clock sampled throughout.  The CPU leg (`cpu_baseline`) times the
fp64 oracle on all cores and on one thread, and compares the last timed
step's outputs with the oracle (`check`); the run fails if they disagree.

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
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the split / decode_attn rooflines of the other workloads")
    ap.add_argument("--steady-steps", type=int, default=2000,
                    help="steps per replay of the long steady-state graph (0: skip)")
    ap.add_argument("--cpu-single-thread", action="store_true", help=argparse.SUPPRESS)
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

    def summary(self, bins: bool = False):
        if not self.ok or not self.samples:
            return None
        names = [n for bit, n in self.REASONS.items() if self.reasons & bit]
        out = {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz,
               "reasons": names, "samples": len(self.samples), "source": "nvml"}
        if bins:   # samples per 15 MHz clock step
            hist = {}
            for v in self.samples:
                k = str(int(v // 15 * 15))
                hist[k] = hist.get(k, 0) + 1
            out["sm_mhz_bins"] = dict(sorted(hist.items(), key=lambda kv: -int(kv[0])))
        return out


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


def blas_threads():
    """(library, threads) of NumPy's BLAS, read from the loaded OpenBLAS itself
    (no extra package needed); (None, None) if it cannot be read."""
    import numpy as np
    np.ones(2) @ np.ones(2)               # make sure the BLAS library is loaded
    try:
        paths = sorted({ln.split()[-1] for ln in open("/proc/self/maps")
                        if "openblas" in ln.lower() and ln.strip().endswith(".so") or
                        ("openblas" in ln.lower() and ".so" in ln.split()[-1])})
    except OSError:
        return None, None
    for path in paths:
        try:
            lib = ctypes.CDLL(path)
        except OSError:
            continue
        for name in ("scipy_openblas_get_num_threads64_", "openblas_get_num_threads64_",
                     "openblas_get_num_threads"):
            fn = getattr(lib, name, None)
            if fn is not None:
                fn.restype = ctypes.c_int
                return os.path.basename(path), int(fn())
    return None, None


def single_thread_oracle(cfg, seconds: float):
    """The same oracle leg in a child process whose BLAS and OpenMP pools have
    one thread.  Returns its JSON dict or None."""
    import subprocess
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")
    cmd = [sys.executable, os.path.abspath(__file__), "--cpu-single-thread", "--workload",
           cfg.name, "--cpu-seconds", str(seconds)]
    try:
        r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=seconds + 120)
        return json.loads(r.stdout.strip().splitlines()[-1]) if r.returncode == 0 else None
    except Exception:
        return None


def oracle_check(cfg, gpu_out, seed: int):
    """The last timed step's outputs (o, o_c, lse; every step of the timed graph
    reads identical copies of the same inputs) against the fp64 oracle on up to
    eight sequences of the workload, with the parity tolerances."""
    import numpy as np
    from oracle import mla_oracle as O
    from workloads import (TOL_BF16_MAX_ABS, TOL_BF16_REL_L2, TOL_F32_MAX_ABS, make_inputs)
    inp = make_inputs(cfg, seed=seed)
    nb = min(cfg.batch, 8)
    seqs = sorted({round(i * (cfg.batch - 1) / max(nb - 1, 1)) for i in range(nb)})
    res, ok = {"sequences": seqs, "step": "last timed step"}, True
    refs = {k: [] for k in ("o", "o_c", "lse")}
    rows = []
    for b in seqs:
        for i in range(cfg.q_len):
            rows.append(b * cfg.q_len + i)
        a = inp.as_float64_numpy(b)
        if a["cache"] is None:
            a["cache"] = O.e4m3_to_float64(a["cache_e4m3"])
        if cfg.q_len == 1:
            n = int(a["lengths"][0])
            r = O.decode_absorbed(a["q_nope"], a["q_rope"], a["w_uk"], a["w_uv"],
                                  a["cache"][:, :n], a["lengths"], a["positions"],
                                  cfg.softmax_scale, cfg.rope_base)
            for k in refs:
                refs[k].append(r[k][0])
        else:   # rows b * q_len .. + q_len - 1 are sequence b's tokens
            T = cfg.q_len
            n = int(a["lengths"][0])
            qn = inp.q_nope[b * T:(b + 1) * T].double().numpy()[None]
            qr = inp.q_rope[b * T:(b + 1) * T].double().numpy()[None]
            r = O.decode_multi_token(qn, qr, a["w_uk"], a["w_uv"], a["cache"][:, :n],
                                     np.array([n]), T, cfg.softmax_scale, cfg.rope_base)
            for k in refs:
                refs[k].extend(list(r[k][0]))
    for k in ("o", "o_c", "lse"):
        ref = np.stack(refs[k])
        got = gpu_out[k][rows]
        ma = float(np.max(np.abs(got - ref)))
        rl = float(np.linalg.norm((got - ref).ravel()) / max(np.linalg.norm(ref.ravel()), 1e-300))
        fin = bool(np.all(np.isfinite(got)))
        good = fin and (ma <= TOL_F32_MAX_ABS if cfg.dtype == "f32"
                        else ma <= TOL_BF16_MAX_ABS and rl <= TOL_BF16_REL_L2)
        res[k] = {"max_abs": ma, "rel_l2": rl}
        ok = ok and good
    res["tolerance"] = ({"max_abs": TOL_F32_MAX_ABS} if cfg.dtype == "f32" else
                        {"max_abs": TOL_BF16_MAX_ABS, "rel_l2": TOL_BF16_REL_L2})
    res["ok"] = ok
    return res


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


# ----------------------------------------------------------------------------- timing helpers
def graph_time(mla, stream, launch, n: int, reps: int, overlap: bool = True, bus=None):
    """Capture n calls launch(0..n-1) as one CUDA graph on `stream`, with the
    library's programmatic launches on or off; replay it once untimed, then
    `reps` times with CUDA events around each replay on the replaying stream.
    Returns (microseconds per launch of each replay, clock summary or None);
    the SM clock is sampled only when `bus` is given."""
    import torch
    mla.set_launch_overlap(overlap)
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
            for k in range(n):
                launch(k)
    finally:
        mla.set_launch_overlap(True)
    g.replay()
    torch.cuda.synchronize()
    sampler = ClockSampler(bus) if bus is not None else None
    out = []
    with (sampler if sampler is not None else _Nothing()):
        for _ in range(reps):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            g.replay()
            e1.record()
            torch.cuda.synchronize()
            out.append(e0.elapsed_time(e1) * 1e3 / n)
    del g
    return out, (sampler.summary(bins=True) if sampler is not None else None)


class _Nothing:
    def __enter__(self):
        return self

    def __exit__(self, *a):
        return False


# The other workloads whose split and mla_decode_attn rooflines the default run
# reports beside the bench workload's: the ragged batch, the 128-head batch and
# the long context at its 128 chunks per sequence.
OTHER_WORKLOADS = ("v2lite_bf16_b64_ragged512_8192", "v3heads_bf16_h128_b32_s16384",
                   "v2lite_bf16_b4_s65536_split128")


def workload_rooflines(mla, dev, stream, peak, bus):
    """Split-only and mla_decode_attn rooflines of OTHER_WORKLOADS: plain launches
    (programmatic launch off) over two or more cache copies larger than L2 in all,
    median of three replays; bytes are the valid rows' (ragged tails excluded)."""
    import torch
    from workloads import BY_NAME, cache_storage, make_inputs
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 0) or 126 * 2 ** 20
    res = []
    for name in OTHER_WORKLOADS:
        c = BY_NAME[name]
        inp = make_inputs(c, seed=0)
        per = inp.cache.numel() * inp.cache.element_size()
        L = max(2, math.ceil(3 * l2 / per))
        caches = [inp.cache.to(dev) for _ in range(L)]
        lengths, pos = inp.lengths.to(dev), inp.positions.to(dev)
        d = mla.dims(c.batch, c.heads, c.s_max, mla.dtype_code(cache_storage(c)))
        B, H = c.batch, c.heads
        q_abs = torch.empty((B, H, c.d_c), dtype=torch.float32, device=dev)
        q_pe = torch.empty((B, H, c.d_rope), dtype=torch.float32, device=dev)
        o_c = torch.empty((B, H, c.d_c), dtype=torch.float32, device=dev)
        lse = torch.empty((B, H), dtype=torch.float32, device=dev)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        mla.absorb_q(d, inp.q_nope.to(dev), inp.q_rope.to(dev), inp.w_uk.to(dev), pos, q_abs,
                     q_pe, c.rope_base)
        ws = torch.empty((mla.workspace_bytes(d, c.num_splits),), dtype=torch.uint8, device=dev)
        nbytes = int(inp.lengths.to(torch.int64).sum()) * c.row * c.elt_bytes
        n = max(8, min(200, int(20e-3 / (nbytes / 5e12))))    # about 20 ms per replay
        split = lambda k: mla.decode_split(d, q_abs, q_pe, caches[k % L], lengths, ws,
                                           c.softmax_scale, c.num_splits, status)
        attn = lambda k: mla.decode_attn(d, q_abs, q_pe, caches[k % L], lengths, o_c, ws,
                                         c.softmax_scale, c.num_splits, lse, status)
        sp, clk = graph_time(mla, stream, split, n, 3, overlap=False, bus=bus)
        at, _ = graph_time(mla, stream, attn, n, 3, overlap=False)
        if int(status.item()) != 0:
            raise RuntimeError(f"device status {int(status.item())} on {name}")
        splits, chunk, persistent = mla.plan(d, c.num_splits)
        hpc = mla.heads_per_cta(d)
        entry = {"workload": name, "batch": B, "heads": H, "s_max": c.s_max,
                 "kv_splits": splits, "chunk_rows": chunk, "bytes_per_launch": nbytes,
                 "split_form": ("persistent (one CTA per SM)" if persistent else
                                "one CTA per (head group, chunk, sequence)"),
                 "heads_per_cta": hpc,
                 "operand_parts": "one bf16 part" if hpc == 64 else "bf16 hi + lo",
                 "launches_timed": n, "replays": 3, "clocks": clk}
        for key, us_list in (("split", sp), ("decode_attn", at)):
            us = statistics.median(us_list)
            gbs = nbytes / (us * 1e-6) / 1e9
            entry[key] = {"avg_launch_us": us, "achieved": gbs, "frac": gbs / peak,
                          "spread_us": [min(us_list), max(us_list)]}
        entry["split"]["traffic"] = recorded_traffic(SPLIT_KERNEL[c.dtype], name)
        res.append(entry)
        del caches, ws, inp
        torch.cuda.empty_cache()
    return res


# ----------------------------------------------------------------------------- our arm
def main():
    return main_with(parse(), int(os.environ.get("RANK", "0")),
                     int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("LOCAL_RANK", "0")))


def main_with(args, rank: int, world: int, local: int = 0):
    from workloads import BY_NAME
    cfg = BY_NAME[args.workload]

    if args.cpu_single_thread:   # child of the CPU leg, BLAS limited to one thread
        gbs, tps, nsteps, rows, el = oracle_throughput(cfg, args.cpu_seconds)
        print(json.dumps({"value": gbs, "unit": "GB/s", "cores": 1, "steps": nsteps,
                          "rows": rows, "seconds": el, "tokens_per_s": tps,
                          "env": "OPENBLAS_NUM_THREADS=OMP_NUM_THREADS=MKL_NUM_THREADS=1"}))
        return 0
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
    splits_req = args.splits or cfg.num_splits   # the workload's own chunk count, if any
    bus = bus_id_of(dev.index)
    step = mla.DecodeStep(cfg.batch, cfg.heads, cfg.s_max, dt, device=dev,
                          num_splits_requested=splits_req, rope_base=cfg.rope_base,
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
    sampler = ClockSampler(bus)
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

    # Outputs of the last timed step, kept for the oracle check of the CPU leg
    # before the graphs below overwrite them.
    last_out = {"o": step.out.double().cpu().numpy(), "o_c": step.o_c.double().cpu().numpy(),
                "lse": step.lse.double().cpu().numpy()}

    # The dominant kernel and mla_decode_attn (split + combine) alone: graphs of Ks
    # back-to-back launches over the rotating layer copies, timed with CUDA events
    # around each of `reps` replays (median reported).  "plain": programmatic launch
    # off, so each launch starts after the previous one ended and the average is one
    # launch's whole duration; "overlapped": the library's default launches, where
    # a launch's set-up and first cache boxes overlap the previous launch's tail.
    Ks, reps = 400, 5

    def split_launch(k):
        mla.decode_split(d, step.q_abs, step.q_pe, caches[k % L], lengths, step.workspace,
                         step.scale, splits_req, step.status)

    def attn_launch(k):
        if cfg.q_len == 1:
            mla.decode_attn(d, step.q_abs, step.q_pe, caches[k % L], lengths, step.o_c,
                            step.workspace, step.scale, splits_req, step.lse, step.status)
        else:
            mla.decode_attn_multi(d, cfg.q_len, step.q_abs, step.q_pe, caches[k % L], lengths,
                                  step.o_c, step.workspace, step.scale, splits_req, step.lse,
                                  step.status)

    if cfg.q_len > 1:    # no separate multi-token split entry: split + combine
        split_launch = attn_launch
    split_plain, clk_split = graph_time(mla, cap, split_launch, Ks, reps, overlap=False,
                                        bus=bus)
    split_ovl, _ = graph_time(mla, cap, split_launch, Ks, reps, overlap=True)
    attn_plain, clk_attn = graph_time(mla, cap, attn_launch, Ks, reps, overlap=False, bus=bus)
    attn_ovl, _ = graph_time(mla, cap, attn_launch, Ks, reps, overlap=True)
    if int(step.status.item()) != 0:
        raise RuntimeError(f"device status {int(step.status.item())} after the split-only replay")

    # The same step graph, long: `--steady-steps` steps per replay, five replays,
    # with the SM clock sampled throughout (a timed region long enough for many
    # samples), so that the step time can be read against the clock.
    steady = None
    if args.steady_steps > 0:
        st_us, st_clk = graph_time(mla, cap, one_step, args.steady_steps, 5, overlap=True,
                                   bus=bus)
        if int(step.status.item()) != 0:
            raise RuntimeError(f"device status {int(step.status.item())} after the steady replays")
        med = statistics.median(st_us)
        steady = {"steps_per_replay": args.steady_steps, "replays": len(st_us),
                  "us_per_step": med, "us_per_step_min": min(st_us),
                  "us_per_step_max": max(st_us),
                  "value": cache_bytes / (med * 1e-6) / 1e9, "unit": "GB/s",
                  "tokens_per_s": cfg.batch * cfg.q_len / (med * 1e-6),
                  "clocks": st_clk,
                  "us_x_sm_mhz": med * st_clk["sm_mhz"] if st_clk else None}

    # End-to-end through the public API with host buffers: every step reads the
    # queries, lengths and positions from pinned host memory and writes o into
    # pinned host memory.  Each layer copy's step is set up once with
    # DecodeStep.capture; the headline makes each step one direct
    # mla_decode_step call (HostStep.launch, arguments converted at capture), and
    # the same steps as one CUDA-graph replay each are timed beside it.
    e2e = None
    if not args.no_e2e:
        hosts = [step.capture(caches[l], wuk[l], wuv[l]) for l in range(L)]
        for l, hs in enumerate(hosts):          # the host side fills each step's inputs
            hs.q_nope.copy_(inp.q_nope)
            hs.q_rope.copy_(inp.q_rope)
            hs.lengths.copy_(inp.lengths)
            hs.positions.copy_(inp.positions)
        Ke = min(K, 2000)

        def time_host_steps(how):
            for k in range(min(W, 20)):
                getattr(hosts[k % L], how)()
            torch.cuda.synchronize()
            if world > 1:
                dist.barrier()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            t0 = time.perf_counter()
            e0.record()
            for k in range(Ke):
                getattr(hosts[k % L], how)()
            e1.record()
            torch.cuda.synchronize()
            wall_ms = (time.perf_counter() - t0) * 1e3
            e_ms = e0.elapsed_time(e1)
            if int(step.status.item()) != 0:
                raise RuntimeError(f"device status {int(step.status.item())} after the e2e steps")
            return max_over_ranks(e_ms, dev, world), wall_ms

        l_ms, l_wall = time_host_steps("launch")
        r_ms, r_wall = time_host_steps("replay")
        bi, bo = hosts[0].h2d_bytes, hosts[0].d2h_bytes
        suffix = "" if cfg.q_len == 1 else "_multi"
        e2e = {"value": whole_job_rate(cache_bytes, Ke, world, l_ms / 1e3) / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo, "steps": Ke,
               "us_per_step": l_ms * 1e3 / Ke, "host_wall_us_per_step": l_wall * 1e3 / Ke,
               "tokens_per_s": whole_job_rate(cfg.batch * cfg.q_len, Ke, world, l_ms / 1e3),
               "path": (f"HostStep.launch: per step one mla_decode_step{suffix} call on pinned "
                        "host buffers -- its kernels read the queries, lengths and positions "
                        "and write o over the host link, no copy nodes; consecutive steps "
                        "overlap by programmatic dependent launch"),
               "graph_replay": {
                   "value": whole_job_rate(cache_bytes, Ke, world, r_ms / 1e3) / 1e9,
                   "unit": "GB/s", "us_per_step": r_ms * 1e3 / Ke,
                   "host_wall_us_per_step": r_wall * 1e3 / Ke,
                   "path": "the same steps, each one replay of its captured CUDA graph"}}

    peak, peak_kind = measured_peaks()
    kname = SPLIT_KERNEL[cfg.dtype]

    def rate(us_list):
        us = statistics.median(us_list)
        gbs = cache_bytes / (us * 1e-6) / 1e9
        return {"achieved": gbs, "frac": gbs / peak, "avg_launch_us": us,
                "spread_us": [min(us_list), max(us_list)]}

    sp, so, ap, ao = rate(split_plain), rate(split_ovl), rate(attn_plain), rate(attn_ovl)
    attn_name = "mla_decode_attn" if cfg.q_len == 1 else "mla_decode_attn_multi"
    roofline = {"bound": "hbm",
                "kernel": (f"{kname} (mla_decode_split)" if cfg.q_len == 1 else
                           f"{kname} + combine_kernel ({attn_name})"),
                "achieved": sp["achieved"], "peak": peak, "unit": "GB/s", "frac": sp["frac"],
                "peak_kind": f"{peak_kind} (copy bandwidth, burst)",
                "frac_of_nominal_8TBs": sp["achieved"] / NOMINAL_HBM_GBS,
                "traffic": recorded_traffic(kname, cfg.name),
                "bytes_per_launch": cache_bytes,
                "avg_launch_us": sp["avg_launch_us"], "spread_us": sp["spread_us"],
                "launches_timed": Ks, "replays": reps,
                "timing": (f"plain launches (programmatic launch off): a CUDA graph of {Ks} "
                           f"back-to-back launches over the rotating layer copies, each starting "
                           f"after the previous one ended; CUDA events around each replay, "
                           f"median of {reps} replays"),
                "clocks": clk_split,
                "us_x_sm_mhz": sp["avg_launch_us"] * clk_split["sm_mhz"] if clk_split else None,
                "overlapped": dict(so, timing="the library's default programmatic launches: "
                                   "each launch's set-up and first cache boxes overlap the "
                                   "previous launch's tail (a pipelined throughput)"),
                "decode_attn": dict(ap, call=attn_name, kernels="split + LSE combine",
                                    bytes_per_launch=cache_bytes, target_frac=0.70,
                                    timing="plain launches, as above", clocks=clk_attn,
                                    overlapped=ao)}

    others = None
    if not args.no_workloads and world == 1 and cfg.name == "v2lite_bf16_b8_s4096":
        others = workload_rooflines(mla, dev, cap, peak, bus)

    cpu, check = None, None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        blas_lib, blas_n = blas_threads()
        gbs, tps, nsteps, rows, el = oracle_throughput(cfg, args.cpu_seconds)
        single = single_thread_oracle(cfg, min(args.cpu_seconds, 5.0))
        cpu = {"value": gbs, "unit": "GB/s", "cores": cpu_cores(), "kind": "oracle",
               "tokens_per_s": tps, "blas": blas_lib, "blas_threads": blas_n,
               "sample": (f"{nsteps} single-sequence decode steps ({rows} rows, H={cfg.heads}) "
                          f"of this workload through the fp64 NumPy oracle, {el:.1f} s; inputs "
                          f"converted to fp64 before timing"),
               "single_thread": single}
        # The oracle leg also checks the GPU's last timed step against the oracle.
        check = oracle_check(cfg, last_out, seed=rank)

    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": elapsed_ms / K, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": DTYPE_NAME[cfg.dtype],
        "data": "synthetic (seeded N(0,1) cache and queries, N(0,0.02^2) weights)",
        "tokens_per_s": tokens,
        "config": workload_config(cfg, L, step.splits),
        "roofline": roofline, "roofline_workloads": others, "steady": steady,
        "cpu_baseline": cpu, "check": check, "e2e": e2e,
        "gpu_launches": launches_per_step(cfg) * K,
        "clocks": sampler.summary(),
        "timing": "one CUDA-graph replay of the timed steps (no event nodes inside), CUDA events "
                  "on the replay stream",
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    if check is not None and not check["ok"]:
        print("bench: the last timed step does not match the oracle", file=sys.stderr)
        return 1
    return 0


if __name__ == "__main__":
    sys.exit(main())
