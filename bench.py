#!/usr/bin/env python
"""Benchmark of the GDN recurrence on GB300: decode-step state HBM GB/s and gdn_scan tokens/s.

One bench step is one ``gdn_decode_step`` (one token for every sequence of the batch) on the
Qwen-style decode workload B=64, Hk=16, Hv=32, Dk=Dv=128, bf16 activations, f32 state
(134 MB, updated in place).  The JSON line's value is the algorithmic HBM traffic of a step
(one read and one write of the state plus the step's inputs and output) over the device
time of the step.  Supplementary: the prefill and long-context scans (tokens/s).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

``--impl reference`` times the fp64 CPU oracle (there is no other implementation of this
method to run) on a bounded sample of the same workload.  Under torchrun each rank runs its
own copy of the per-GPU workload (independent batches, no collective on the data path).
"""
from __future__ import annotations

import argparse
import csv
import ctypes
import datetime as _dt
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from linear_attention_recurrence_gdn_gb300.workloads import (  # noqa: E402
    DECODE_B64, DECODE_B256_HM, LONG_B2, PREFILL_B4, Workload, make_inputs)

METRIC = "GDN decode step: state HBM GB/s (% of peak); gdn_scan tokens/sec"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
MMA_SYNC_MAC_PER_CLK_SM = 1024  # measured issue rate of mma.sync bf16 m16n8k16 per SM
FP32_LANES_PER_SM = 128          # FP32 FMA lanes per SM
MAX_SM_MHZ_FALLBACK = 2070.0


# ------------------------------------------------------------------------ roofline model

def decode_bytes(w: Workload) -> int:
    """Algorithmic HBM bytes of one decode step: read + write of the f32 state, q and k per
    key head, v and z per value head, the f32 output, two f32 gates and the f32 norm weight."""
    e = w.elem_bytes
    return (8 * w.B * w.Hv * w.Dv * w.Dk + 2 * w.B * w.Hk * w.Dk * e
            + w.B * w.Hv * (2 * w.Dv * e + 4 * w.Dv + 8) + 4 * w.Dv)


def scan_flops(w: Workload) -> int:
    """6 Dk Dv FLOP per (token, value head): S.k, S.q and the rank-1 update."""
    return 6 * w.Dk * w.Dv * w.B * w.S * w.Hv


def scan_mma_flops(w: Workload) -> int:
    """Tensor-core FLOPs the block form issues per launch for its row MMAs.

    Per warp (16 memory rows) and 16-token block: X and Y (4 KST MMAs per operand term), d and
    O (6 each, hi/lo split operands on both sides), the update (NTILE per term); bf16 inputs are
    exact bf16 operands (2 terms), other types split into hi + lo (3 terms).  Each m16n8k16 MMA
    is 2 * 16 * 8 * 16 FLOP.  The per-chunk KK / QX tables (under 4% more) are not counted.
    """
    terms = 2 if w.act == "bf16" else 3
    kst, ntile = w.Dk // 16, w.Dk // 8       # the update runs over the Dk / 8 n-tiles of a row
    per_warp_block = 4 * kst * terms + 12 + ntile * terms
    warps_per_head = w.Dv // 16
    return (w.B * w.Hv * warps_per_head * per_warp_block * 2 * 16 * 8 * 16 * w.S) // 16


def scan_tmem_mma_flops(w: Workload) -> int:
    """Tensor-core FLOPs the tensor-memory chunked kernel issues per launch (M = 128 MMAs).

    Per head and 32-token chunk c of n: the chunk tables (8 MMAs with N = 32, 16 from the
    second chunk on, when the cross table with the previous chunk's keys is added), [x | y]
    from S' hi / lo (16, N = 64), d = R T (6, N = 32), O (6, N = 32), the update (4, N = 128)
    and the next chunk's correction (6, N = 64, all chunks but the last).  Each M x N x 16 MMA
    is 2 * 128 * N * 16 FLOP; rows the tables compute beyond the 64 real ones are counted too.
    """
    n = (w.S + 31) // 32
    per = 2 * 128 * 16
    tables = (8 + 16 * (n - 1)) * 32
    pre = 16 * n * 64
    d_o = 12 * n * 32
    upd = 4 * n * 128
    corr = 6 * (n - 1) * 64
    return w.B * w.Hv * per * (tables + pre + d_o + upd + corr)


def scan_wy_mma_flops(w: Workload) -> int:
    """Tensor-core FLOPs the chunked (WY) kernel issues per launch (M = 128, K = 16 MMAs).

    Per head and 64-token chunk: the tables [K; Q] K^T (8 MMAs, N = 64), W^T and U^T (8 each,
    N = 64: hi and lo B operands over K = 64), X = U^T - S W^T (24, N = 64: hi.hi, hi.lo, lo.hi
    over K = 128), Y = S Q^T (16, N = 64), the update (8, N = 128) and the intra-chunk output
    (12, N = 64).  Each M x N x 16 MMA is 2 * 128 * N * 16 FLOP.  The mma.sync tiles of the
    triangular inverse (under 1%) are not counted.
    """
    n = (w.S + 63) // 64
    per = 2 * 128 * 16
    return w.B * w.Hv * n * per * ((8 + 8 + 8 + 24 + 16 + 12) * 64 + 8 * 128)


def scan_bytes(w: Workload) -> int:
    e = w.elem_bytes
    s0 = 4 * w.B * w.Hv * w.Dv * w.Dk if w.s0_std is not None else 0
    return (2 * w.B * w.S * w.Hk * w.Dk * e + w.B * w.S * w.Hv * (2 * w.Dv * e + 4 * w.Dv + 8)
            + s0 + 4 * w.B * w.Hv * w.Dv * w.Dk + 4 * w.Dv)


def load_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured",
                "bf16_tflops": float(d.get("bf16_tflops", FALLBACK_BF16_TFLOPS)),
                "sm_max_mhz": float(d.get("sm_max_mhz", MAX_SM_MHZ_FALLBACK))}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": FALLBACK_HBM_GBS, "source": "fallback",
                "bf16_tflops": FALLBACK_BF16_TFLOPS, "sm_max_mhz": MAX_SM_MHZ_FALLBACK}


def code_hash(source: str) -> str:
    """sha256 of C/C++/CUDA source with its comments and all whitespace removed: the hash
    changes with the code, not with its comments or layout."""
    out, i, n = [], 0, len(source)
    while i < n:
        if source.startswith("//", i):
            j = source.find("\n", i)
            i = n if j < 0 else j
        elif source.startswith("/*", i):
            j = source.find("*/", i + 2)
            i = n if j < 0 else j + 2
        elif source[i] == '"':                     # string literal, kept verbatim
            j = i + 1
            while j < n and source[j] != '"':
                j += 2 if source[j] == "\\" else 1
            out.append(source[i:j + 1])
            i = j + 1
        else:
            if not source[i].isspace():
                out.append(source[i])
            i += 1
    return hashlib.sha256("".join(out).encode()).hexdigest()


def profiled_traffic(kernel_file: str, summary: str):
    """DRAM bytes per launch recorded by an ncu capture, if the kernel code is unchanged.

    ``summary`` (under profiles/) holds lines ``code_sha256: <hex>`` (``code_hash`` of the
    kernel source) and ``dram_bytes_per_launch: <int>``; a mismatch means the counters are
    stale -> None.
    """
    try:
        text = open(os.path.join(ROOT, "profiles", summary)).read()
        src = open(os.path.join(ROOT, "linear_attention_recurrence_gdn_gb300", "csrc",
                                kernel_file)).read()
    except OSError:
        return None
    fields = dict(line.split(":", 1) for line in text.splitlines() if ":" in line)
    if fields.get("code_sha256", "").strip() != code_hash(src):
        return None
    try:
        return int(fields["dram_bytes_per_launch"].strip())
    except (KeyError, ValueError):
        return None


# ------------------------------------------------------------------------- distributed

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def dist_init(world: int, backend: str):
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def barrier(world: int):
    if world > 1:
        torch.distributed.barrier()


def allreduce_max(x: float, world: int, device=None) -> float:
    """Max of a scalar over ranks (the slowest rank sets the job time)."""
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def aggregate_rate(units_per_rank: float, world: int, seconds_max: float) -> float:
    """Whole-job throughput: the units every rank processed over the slowest rank's time."""
    return units_per_rank * world / seconds_max


# ------------------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons, kept with host timestamps."""

    FIELDS = ("timestamp,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None, period_ms: int = 50):
        self.uuid = uuid
        self.file = tempfile.NamedTemporaryFile(prefix="gdn_clocks_", suffix=".csv", delete=False)
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(period_ms)], stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        self.file.close()

    def samples(self):
        out = []
        try:
            rows = list(csv.reader(open(self.file.name)))
        except OSError:
            return out
        for r in rows:
            if len(r) < 10:
                continue
            r = [c.strip() for c in r]
            if self.uuid and self.uuid not in r[1]:
                continue
            try:
                ts = _dt.datetime.strptime(r[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                out.append({"t": ts, "sm": float(r[2]), "max": float(r[3]),
                            "reasons": {"hw_slowdown": r[6], "hw_thermal_slowdown": r[7],
                                        "sw_thermal_slowdown": r[8], "sw_power_cap": r[9]}})
            except ValueError:
                continue
        return out

    def summary(self, t0: float, t1: float) -> dict:
        s = self.samples()
        inside = [x for x in s if t0 <= x["t"] <= t1]
        window = "timed region"
        if not inside:   # region shorter than the sampling period: nearest samples
            inside = sorted(s, key=lambda x: min(abs(x["t"] - t0), abs(x["t"] - t1)))[:3]
            window = "nearest samples to a timed region shorter than the sampling period"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi unavailable"}
        reasons = sorted({k for x in inside for k, v in x["reasons"].items()
                          if v.lower() == "active"})
        return {"sm_mhz": statistics.median(x["sm"] for x in inside),
                "sm_max_mhz": max(x["max"] for x in inside), "reasons": reasons,
                "samples": len(inside), "window": window}


def device_uuid(dev) -> str | None:
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return None


# ---------------------------------------------------------------------------- decode

def decode_params(gdn, w: Workload, dev, sets: int):
    """Device buffers and C-ABI parameter blocks for `sets` independent decode problems."""
    bufs, params = [], []
    base = make_inputs(w)
    for i in range(sets):
        inp = base if i == 0 else make_inputs(w, seed=w.seed + 7919 * i)
        d = {k: (None if v is None else v.to(dev)) for k, v in inp.items()}
        state = d["s0"].clone()
        y = torch.empty(d["v"].shape, dtype=torch.float32, device=dev)
        prm = gdn.make_params(d["q"], d["k"], d["v"], d["log_decay"], d["beta"], state, y,
                              z=d["z"], gn=d["gn"], head_major=w.head_major)
        bufs.append((d, state, y))
        params.append(prm)
    return bufs, params


def run_decode_steps(lib, params, stream_handle, n: int, start: int = 0):
    for i in range(start, start + n):
        st = lib.gdn_decode_step(ctypes.byref(params[i % len(params)]), stream_handle)
        if st != 0:
            raise RuntimeError(f"gdn_decode_step failed with status {st}")


def bench_decode(gdn, w: Workload, dev, steps: int, warmup: int, world: int, sampler):
    lib = gdn.library()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    state_bytes = 4 * w.B * w.Hv * w.Dv * w.Dk
    sets = max(2, -(-4 * l2 // state_bytes))          # >= 4x L2 of distinct state
    bufs, params = decode_params(gdn, w, dev, sets)
    stream = torch.cuda.current_stream(dev)
    handle = stream.cuda_stream
    run_decode_steps(lib, params, handle, warmup)
    torch.cuda.synchronize(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(dev)
    t0 = time.time()
    ev0.record(stream)
    run_decode_steps(lib, params, handle, steps, start=warmup)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    t1 = time.time()
    barrier(world)
    ms = allreduce_max(ev0.elapsed_time(ev1), world, dev)
    clocks = sampler.summary(t0, t1) if sampler else None
    return {"ms_total": ms, "ms_per_step": ms / steps, "sets": sets, "clocks": clocks,
            "bufs": bufs, "params": params}


def e2e_decode(gdn, w: Workload, dev, steps: int, world: int):
    """Same metric end to end: every step moves its inputs from pinned host memory to the
    GPU, runs the C-ABI decode step on the resident state, and brings y back to the host.

    Through the binding's HostDecodeStep: the per-step inputs (q, k, v, z, log_decay, beta)
    sit in one pinned host buffer and y in pinned host memory; a step is one C-ABI call with
    GDN_FLAG_HOST_IO, whose kernel reads the inputs from host memory and writes y there over
    the chip-to-chip link, then a wait on an event recorded behind it.
    """
    inp = make_inputs(w)
    names = ["q", "k", "v", "z", "log_decay", "beta"]
    state = inp["s0"].to(dev)
    gn = inp["gn"].to(dev)
    stepper = gdn.HostDecodeStep({k: inp[k] for k in names}, state, gn,
                                 head_major=w.head_major)
    for k in names:
        stepper.host[k].copy_(inp[k])
    for _ in range(5):
        stepper.run()
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(steps):
        stepper.run()
    sec = allreduce_max(time.perf_counter() - t0, world, dev)
    return {"value": aggregate_rate(decode_bytes(w), world, sec / steps) / 1e9, "unit": "GB/s",
            "h2d_bytes_per_step": stepper.h2d_bytes, "d2h_bytes_per_step": stepper.d2h_bytes,
            "steps": steps, "ms_per_step": 1e3 * sec / steps,
            "note": "state resident in HBM; per step one C-ABI call reading the inputs from "
                    "pinned host memory and writing y to pinned host memory "
                    "(GDN_FLAG_HOST_IO), then a wait on an event recorded behind it"}


# ------------------------------------------------------------------------------ scan

def bench_split(gdn, w: Workload, dev, reps: int):
    """gdn_scan against gdn_scan_split at several segment counts on one workload (tokens/s,
    median of `reps` CUDA-event-timed calls each; the workspace allocated once)."""
    inp = make_inputs(w)
    d = {k: (None if v is None else v.to(dev)) for k, v in inp.items()}
    y = torch.empty(d["v"].shape, dtype=torch.float32, device=dev)
    st = torch.empty((w.B, w.Hv, w.Dv, w.Dk), dtype=torch.float32, device=dev)
    args = (d["q"], d["k"], d["v"], d["log_decay"], d["beta"], st, y)
    kw = dict(s0=d["s0"], z=d["z"], gn=d["gn"], head_major=w.head_major)
    stream = torch.cuda.current_stream(dev)

    def timed(fn):
        fn()
        torch.cuda.synchronize(dev)
        ts = []
        for _ in range(max(3, reps)):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            torch.cuda.synchronize(dev)
            ts.append(e0.elapsed_time(e1))
        return statistics.median(ts)

    tokens = w.B * w.S
    out = {"config": w.as_config(), "metric": "tokens/s", "lines": []}
    ms = timed(lambda: gdn.gdn_scan(*args, **kw))
    y_ref, st_ref = y.clone(), st.clone()
    out["lines"].append({"segments": 1, "ms": ms, "value": tokens / (ms * 1e-3)})

    def rel_diff(a, ref):                # max |a - ref| / (1 + |ref|), the scan tolerance's form
        return float(((a - ref).abs() / (1 + ref.abs())).max())

    for nseg in (2, 4, 8):
        prm = gdn.make_params(*args, z=d["z"], gn=d["gn"], s0=d["s0"], head_major=w.head_major)
        wsb = torch.empty(max(16, gdn.gdn_scan_split_workspace(prm, nseg)), dtype=torch.uint8,
                          device=dev)
        ms_s = timed(lambda: gdn.gdn_scan_split(*args, segments=nseg, workspace=wsb, **kw))
        out["lines"].append({"segments": nseg, "ms": ms_s, "value": tokens / (ms_s * 1e-3),
                             "speedup": ms / ms_s,
                             "max_rel_diff_vs_gdn_scan": {"y": rel_diff(y, y_ref),
                                                          "state": rel_diff(st, st_ref)}})
    return out


SCAN_KERNELS = {
    "chunked": "chunked WY on tcgen05 (GDN_FLAG_SCAN_CHUNKED)",
    "block16": "16-token block on mma.sync (GDN_FLAG_SCAN_BLOCK16)",
    "tmem": "tensor-memory 32-token look-ahead (GDN_FLAG_SCAN_TMEM)",
    "general": "general head dims (f32 on CUDA cores)",
}


def _tiled(d: int) -> bool:
    return (16 <= d <= 128 and d % 16 == 0) or d == 256


def bench_scan(gdn, w: Workload, dev, reps: int, sms: int, sm_mhz: float, peaks: dict,
               kernel: str = "default"):
    """gdn_scan on workload `w` with the given kernel ("default": no flag; the line then names
    the kernel the default ran, found by comparing its output bit for bit with each kernel's)."""
    inp = make_inputs(w)
    d = {k: (None if v is None else v.to(dev)) for k, v in inp.items()}
    y = torch.empty(d["v"].shape, dtype=torch.float32, device=dev)
    st = torch.empty((w.B, w.Hv, w.Dv, w.Dk), dtype=torch.float32, device=dev)

    def call(which):
        gdn.gdn_scan(d["q"], d["k"], d["v"], d["log_decay"], d["beta"], st, y, s0=d["s0"],
                     z=d["z"], gn=d["gn"], head_major=w.head_major, tmem=which == "tmem",
                     block16=which == "block16", chunked=which == "chunked")

    ran = kernel
    if kernel == "default":
        # which kernel the default ran: only one applies outside bf16 / f16 heads of 128
        if not (_tiled(w.Dk) and _tiled(w.Dv)):
            ran = "general"
        elif not (w.act in ("bf16", "f16") and w.Dk == w.Dv == 128):
            ran = "block16"
        else:
            call("default")
            ref = y.clone()
            ran = "other"
            for cand in ("chunked", "block16"):
                call(cand)
                if torch.equal(y, ref):
                    ran = cand
                    break

    def run():
        call(kernel)

    run()
    torch.cuda.synchronize(dev)
    stream = torch.cuda.current_stream(dev)
    times = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        run()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        times.append(e0.elapsed_time(e1))
    ms = statistics.median(times)
    secs = ms * 1e-3
    fp32_peak = sms * FP32_LANES_PER_SM * 2 * sm_mhz * 1e6 / 1e12
    fp32_eq = scan_flops(w) / secs / 1e12
    mma = scan_mma_flops(w) / secs / 1e12
    mma_sync_peak = sms * MMA_SYNC_MAC_PER_CLK_SM * 2 * sm_mhz * 1e6 / 1e12
    bf16 = peaks["bf16_tflops"]
    method = scan_flops(w) / secs / 1e12
    roof = {"bound": "tensor", "achieved": method, "peak": bf16, "unit": "TFLOP/s",
            "frac": method / bf16, "traffic": None,
            "work": "6 Dk Dv FLOP per token-head: the method's own products (S.k, S.q and the "
                    "rank-1 update), whatever the kernel issues",
            "peak_note": f"{peaks['source']} cuBLAS bf16 dense"}
    label = SCAN_KERNELS.get(ran, ran)
    cfg = dict(w.as_config(), kernel=("default: " + label) if kernel == "default" else label)
    if ran == "tmem":
        tc = scan_tmem_mma_flops(w) / secs / 1e12
        roof["issued"] = {"achieved": tc, "frac": tc / bf16, "unit": "TFLOP/s",
                          "work": "tcgen05 MMA FLOPs the tensor-memory kernel issues (tables, "
                                  "[x | y], d, O, update, correction; hi/lo terms counted)"}
    elif ran == "chunked":
        tc = scan_wy_mma_flops(w) / secs / 1e12
        roof["issued"] = {"achieved": tc, "frac": tc / bf16, "unit": "TFLOP/s",
                          "work": "tcgen05 MMA FLOPs the chunked kernel issues (tables, W, U, "
                                  "X, Y, update, intra-chunk output; hi/lo terms counted)"}
    else:
        roof["issued"] = {"achieved": mma, "frac": mma / bf16, "unit": "TFLOP/s",
                          "frac_of_mma_sync_ceiling": mma / mma_sync_peak,
                          "work": "mma.sync FLOPs the block form issues for its row MMAs (X, "
                                  "Y, d, O, update; hi/lo operand terms counted)",
                          "ceiling_note": f"mma.sync's own ceiling {MMA_SYNC_MAC_PER_CLK_SM} "
                                          f"MAC/clk/SM = {mma_sync_peak:.0f} TFLOP/s at "
                                          f"{sm_mhz:.0f} MHz"}
    return {"config": cfg, "value": w.B * w.S / secs, "unit": "tokens/s", "ms": ms,
            "reps": reps, "roofline": roof,
            "fp32_equivalent": {"achieved": fp32_eq, "peak": fp32_peak, "unit": "TFLOP/s",
                                "frac": fp32_eq / fp32_peak,
                                "work": "6 Dk Dv FLOP per token-head (the sequential "
                                        "recurrence's own count)",
                                "peak_note": f"{sms} SMs x {FP32_LANES_PER_SM} FP32 lanes x 2 "
                                             f"x {sm_mhz:.0f} MHz: the sequential form's "
                                             f"FP32 roofline"},
            "hbm_bytes": scan_bytes(w)}


def scan_lines(gdn, workloads, dev, reps: int, sms: int, sm_mhz: float, peaks: dict) -> list:
    """Per workload: the default gdn_scan, then the other of the two main kernels; then the
    first workload through the tensor-memory kernel."""
    out = []
    for x in workloads:
        line = bench_scan(gdn, x, dev, reps, sms, sm_mhz, peaks)
        out.append(line)
        other = "block16" if "chunked" in line["config"]["kernel"] else "chunked"
        out.append(bench_scan(gdn, x, dev, reps, sms, sm_mhz, peaks, kernel=other))
    out.append(bench_scan(gdn, workloads[0], dev, reps, sms, sm_mhz, peaks, kernel="tmem"))
    return out


# ------------------------------------------------------------------- oracle baselines

def oracle_decode_sample(w: Workload, batch: int, threads: int, min_seconds: float,
                         max_calls: int | None = None):
    """Time the fp64 oracle on decode steps of the first `batch` sequences of `w`."""
    import oracle   # the CPU-baseline leg is the one place bench.py runs the oracle
    ws = w.replace(B=batch)
    inp = make_inputs(ws)
    oracle.run(inp["q"], inp["k"], inp["v"], inp["log_decay"], inp["beta"], z=inp["z"],
               gn=inp["gn"], s0=inp["s0"], threads=threads)          # warm-up / load
    calls, t0 = 0, time.perf_counter()
    while True:
        oracle.run(inp["q"], inp["k"], inp["v"], inp["log_decay"], inp["beta"], z=inp["z"],
                   gn=inp["gn"], s0=inp["s0"], threads=threads)
        calls += 1
        el = time.perf_counter() - t0
        if (max_calls and calls >= max_calls) or (not max_calls and el >= min_seconds):
            break
    sec = el / calls
    return {"value": decode_bytes(ws) / sec / 1e9, "unit": "GB/s", "cores": threads,
            "kind": "oracle", "seconds_per_call": sec,
            "sample": f"{calls} oracle decode step(s) of {batch} of {w.B} sequences "
                      f"(all {w.Hv} value heads) of {w.name}, fp64, {threads} threads"}


def oracle_scan_sample(w: Workload, threads: int, min_seconds: float, tokens: int = 512):
    """Time the fp64 oracle on the first `tokens` tokens of one sequence of scan workload `w`
    (all its value heads), repeated until `min_seconds` have passed; tokens/s as gdn_scan's
    metric counts them (B * S per call, all heads)."""
    import oracle
    ws = w.replace(B=1, S=min(tokens, w.S))
    inp = make_inputs(ws)
    calls, t0 = 0, time.perf_counter()
    while True:
        oracle.run(inp["q"], inp["k"], inp["v"], inp["log_decay"], inp["beta"], z=inp["z"],
                   gn=inp["gn"], s0=inp["s0"], threads=threads)
        calls += 1
        el = time.perf_counter() - t0
        if el >= min_seconds:
            break
    return {"workload": w.name, "value": ws.S * calls / el, "unit": "tokens/s", "cores": threads,
            "sample": f"{calls} oracle scan(s) of the first {ws.S} tokens of one of {w.B} "
                      f"sequences (all {w.Hv} value heads), fp64, {threads} threads"}


def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.processor() or platform.machine()


def cpu_baselines(w: Workload, scans, seconds: float) -> dict:
    """The oracle as it stands on this host: the decode workload on all cores (the line's
    cpu_baseline value) and on one thread, and tokens/s of the scan workloads (all cores and
    one thread)."""
    cores = os.cpu_count() or 1
    out = oracle_decode_sample(w, w.B, cores, seconds)
    out.pop("seconds_per_call", None)
    one = oracle_decode_sample(w, max(1, w.B // 16), 1, seconds / 4)
    one.pop("seconds_per_call", None)
    out["threads1"] = one
    out["cpu_model"] = cpu_model()
    out["scan"] = [oracle_scan_sample(x, cores, seconds / 4) for x in scans]
    out["scan"] += [oracle_scan_sample(x, 1, seconds / 8, tokens=128) for x in scans]
    return out


def reference_arm(args, w: Workload):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    threads = os.cpu_count() or 1
    # size the per-step sample so that warmup + steps finish in about a minute
    probe = oracle_decode_sample(w, 1, threads, 0.0, max_calls=1)
    per_seq = probe["seconds_per_call"]
    budget = 60.0 / max(1, args.steps + args.warmup)
    batch = max(1, min(w.B, int(budget / max(per_seq, 1e-6))))
    ws = w.replace(B=batch)
    inp = make_inputs(ws)

    def step():
        oracle.run(inp["q"], inp["k"], inp["v"], inp["log_decay"], inp["beta"], z=inp["z"],
                   gn=inp["gn"], s0=inp["s0"], threads=threads)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    sec = (time.perf_counter() - t0) / args.steps
    value = decode_bytes(ws) / sec / 1e9
    sample = (f"each step: one fp64 oracle decode step of {batch} of {w.B} sequences (all "
              f"{w.Hv} value heads) of {w.name} on {threads} host threads")
    line = {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sec,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": dict(w.as_config(), sample_batch=batch),
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------------------ main

def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=2000)
    ap.add_argument("--scan-reps", type=int, default=5)
    ap.add_argument("--no-scan", action="store_true", help="skip the supplementary scans")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--only", choices=["all", "decode", "scan", "rect", "split"], default="all",
                    help="decode: skip the scans; scan: time only the scans (profiling runs); "
                         "rect: time the separate-key/value-head-dim workloads; split: the "
                         "sequence-split scan against the scan on a long sequence with few heads")
    ap.add_argument("--scan-S", type=int, default=0,
                    help="override the scan workloads' sequence length (profiling runs)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    w = DECODE_B64

    if args.impl == "reference":
        return reference_arm(args, w)

    import linear_attention_recurrence_gdn_gb300 as gdn
    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (there is no CPU path)")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dist_init(world, "nccl")
    gdn.library()
    props = torch.cuda.get_device_properties(dev)
    peaks = load_peaks()

    scan_workloads = [PREFILL_B4, LONG_B2]
    if args.scan_S > 0:
        scan_workloads = [x.replace(S=args.scan_S, name=f"{x.name}_S{args.scan_S}")
                          for x in scan_workloads]
    if args.only == "scan":
        out = scan_lines(gdn, scan_workloads, dev, args.scan_reps, props.multi_processor_count,
                         peaks["sm_max_mhz"], peaks)
        if rank == 0:
            print(json.dumps({"scan": out}), flush=True)
        return 0
    if args.only == "split":
        # the long-context workload with a quarter of its value heads (8 heads of one
        # sequence): too few heads to fill the GPU, the case the sequence split is for
        ws = LONG_B2.replace(name="long_f16_b1_s16384_hk2_hv8_d128", B=1, Hk=2, Hv=8)
        if rank == 0:
            print(json.dumps({"split": bench_split(gdn, ws, dev, args.scan_reps)}), flush=True)
        return 0
    if args.only == "rect":
        # the headline workloads with Dk != Dv (same heads, same token counts), and with head
        # dims of 256 (half the heads, so twice the state per token)
        decs = [DECODE_B64.replace(name="decode_bf16_b64_hk16_hv32_dk128_dv64", Dv=64),
                DECODE_B64.replace(name="decode_bf16_b64_hk8_hv16_d256", Hk=8, Hv=16, Dk=256,
                                   Dv=256),
                # head dims that are not multiples of 16: the general kernel
                DECODE_B64.replace(name="decode_bf16_b64_hk16_hv32_dk100_dv72", Dk=100, Dv=72)]
        scans = [PREFILL_B4.replace(name="prefill_bf16_b4_s4096_hk16_hv32_dk64_dv128", Dk=64),
                 PREFILL_B4.replace(name="prefill_bf16_b4_s4096_hk8_hv16_d256", Hk=8, Hv=16,
                                    Dk=256, Dv=256),
                 PREFILL_B4.replace(name="prefill_bf16_b4_s1024_hk16_hv32_dk100_dv72", S=1024,
                                    Dk=100, Dv=72)]
        lines = []
        for rd in decs:
            dec = bench_decode(gdn, rd, dev, args.steps, args.warmup, world, None)
            gbs = decode_bytes(rd) / (dec["ms_per_step"] * 1e-3) / 1e9
            lines.append({"config": rd.as_config(), "metric": "decode state HBM GB/s",
                          "value": gbs, "ms_per_step": dec["ms_per_step"],
                          "frac_of_measured_hbm": gbs / peaks["hbm_gbs"]})
            del dec
            torch.cuda.empty_cache()
        for rs in scans:
            lines.append(bench_scan(gdn, rs, dev, args.scan_reps, props.multi_processor_count,
                                    peaks["sm_max_mhz"], peaks))
        if rank == 0:
            print(json.dumps({"rect": lines}), flush=True)
        return 0

    sampler = ClockSampler(device_uuid(dev)) if rank == 0 else None
    time.sleep(0.5 if sampler else 0.0)
    dec = bench_decode(gdn, w, dev, args.steps, args.warmup, world, sampler)
    del dec["bufs"], dec["params"]
    torch.cuda.empty_cache()
    ms_step = dec["ms_per_step"]
    value = aggregate_rate(decode_bytes(w), world, ms_step * 1e-3) / 1e9
    per_launch = decode_bytes(w) / (ms_step * 1e-3) / 1e9

    # the large-batch decode workload (B = 256, head-major operands): each step moves four
    # times the bytes, so a quarter of the steps
    wl = DECODE_B256_HM
    steps_l = max(args.warmup, args.steps // 4)
    dec_l = bench_decode(gdn, wl, dev, steps_l, args.warmup, world, sampler)
    sets_l = dec_l["sets"]
    del dec_l["bufs"], dec_l["params"]
    torch.cuda.empty_cache()

    def decode_entry(wd: Workload, d: dict, steps: int, sets: int, traffic_file: str) -> dict:
        gbs = decode_bytes(wd) / (d["ms_per_step"] * 1e-3) / 1e9
        return {"config": dict(wd.as_config(), bytes_per_step=decode_bytes(wd),
                               l2=f"rotating {sets} independent state/input sets"),
                "value": aggregate_rate(decode_bytes(wd), world, d["ms_per_step"] * 1e-3) / 1e9,
                "unit": "GB/s", "steps": steps, "ms_per_step": d["ms_per_step"],
                "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"],
                             "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"],
                             "traffic": profiled_traffic("gdn_decode.cuh", traffic_file),
                             "peak_source": peaks["source"], "kernel": "gdn_decode_kernel",
                             "frac_of_nominal_8tbs": gbs / 8000.0},
                "clocks": d["clocks"]}

    decodes = [decode_entry(w, dec, args.steps, dec["sets"], "decode_b64_dram_traffic.txt"),
               decode_entry(wl, dec_l, steps_l, sets_l, "decode_b256_hm_dram_traffic.txt")]

    e2e = e2e_decode(gdn, w, dev, args.e2e_steps, world)
    scan = None
    if not args.no_scan and args.only == "all":
        sm_mhz = peaks["sm_max_mhz"]
        scan = {"metric": "gdn_scan tokens/sec", "note": "supplementary, not the headline",
                "workloads": scan_lines(gdn, scan_workloads, dev, args.scan_reps,
                                        props.multi_processor_count, sm_mhz, peaks)}
    if sampler:
        sampler.stop()

    if rank != 0:
        return 0
    cpu = None
    if not args.no_cpu_baseline:
        cpu = cpu_baselines(w, [PREFILL_B4, LONG_B2], args.cpu_seconds)
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": dict(w.as_config(), l2=f"rotating {dec['sets']} independent state/input sets "
                       f"({dec['sets']} x {4 * w.B * w.Hv * w.Dv * w.Dk / 1e6:.0f} MB state > "
                       f"4 x L2 {props.L2_cache_size / 1e6:.0f} MB)",
                       parallelism=f"replicas x{world}" if world > 1 else "single GPU",
                       bytes_per_step=decode_bytes(w)),
        "roofline": {"bound": "hbm", "achieved": per_launch, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": per_launch / peaks["hbm_gbs"],
                     "traffic": profiled_traffic("gdn_decode.cuh", "decode_b64_dram_traffic.txt"),
                     "peak_source": peaks["source"], "kernel": "gdn_decode_kernel",
                     "frac_of_nominal_8tbs": per_launch / 8000.0},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": args.steps,
        "clocks": dec["clocks"],
        "decode_workloads": decodes,
        "scan": scan,
        "device": props.name,
    }
    print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
