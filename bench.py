"""Benchmark of the MXFP8 training matmul on GB300.

Default workload (one "step"): the dense forward layer M=16384 tokens,
K=7168, N=18432 -- MX-quantize X rowwise (E4M3), MX-quantize W columnwise
(E4M3), block-scaled GEMM with BF16 output, all through the C ABI.  The
line's value is the step's GEMM work (2MNK) over the step time in TFLOP/s.
Inputs are larger than L2 (X 235 MB, W 264 MB, Y 604 MB), so every step
streams from HBM.

The same JSON line carries per-kernel measurements of every hot-path row
(quantize bandwidth sweep, dense forward / dgrad / wgrad GEMMs, the MoE
grouped GEMM), each against its roofline, the end-to-end number with host
buffers, SM clocks sampled during the timed region, and the CPU oracle
timed on a bounded sample as a reported baseline.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
Under torchrun each rank runs its own batch (weak scaling, no collective
on the data path); rank 0 prints the line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("MXFP8 GEMM TFLOP/s and % dense MXFP8 peak; quantize GB/s and % HBM peak (1 GB300)")
UNIT = "TFLOP/s"
FWD = dict(m=16384, n=18432, k=7168)
WORKLOAD = "dense forward layer: quantize X[16384x7168] rowwise + W[7168x18432] colwise " \
           "(MXFP8 E4M3, 32-blocks, E8M0) + block-scaled GEMM, BF16 out"
NOMINAL_FP8_OVER_BF16 = 2.0            # 4.5 / 2.25 PFLOP/s dense, nominal ratio
REF_ROWS, REF_COLS = 32, 256   # per-step sample of the reference (oracle) arm
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------- clocks

CLOCK_FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]


def _sample_time(field: str):
    """Host epoch seconds of an nvidia-smi timestamp ("2026/12/03 05:29:22.123"),
    or None."""
    try:
        day, clock = field.strip().split(" ")
        hms, _, frac = clock.partition(".")
        t = time.mktime(time.strptime(f"{day} {hms}", "%Y/%m/%d %H:%M:%S"))
        return t + (float("0." + frac) if frac else 0.0)
    except ValueError:
        return None


class ClockSampler:
    """nvidia-smi sampling (every `period_ms`) while the timed regions run.
    Every sample carries nvidia-smi's timestamp, so a measurement can take
    the median SM clock of the samples inside its own host-time window."""

    def __init__(self, gpu_index: int, period_ms: int = 100):
        self.gpu = gpu_index
        self.period_ms = period_ms
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={CLOCK_FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.period_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]
        return False

    @staticmethod
    def _parse(line: str):
        """(epoch seconds or None, sm MHz, max MHz, active reasons) or None."""
        parts = [p.strip() for p in line.split(",")]
        t = None
        if parts and "/" in parts[0]:          # leading timestamp field
            t = _sample_time(parts[0])
            parts = parts[1:]
        if len(parts) < 9:
            return None
        try:
            sm, mx_ = float(parts[1]), float(parts[2])
        except ValueError:
            return None
        reasons = {name for name, val in zip(REASONS, parts[5:9])
                   if val.lower() in ("active", "0x1", "1", "yes")}
        return t, sm, mx_, reasons

    def summary(self, t0: float | None = None, t1: float | None = None):
        """Median SM clock under load (samples at >= half the highest one),
        highest max clock and the throttle reasons seen; with t0, t1 (host
        epoch seconds) only the samples inside that window."""
        sm, mx_, reasons = [], [], set()
        for line in self.lines:
            rec = self._parse(line)
            if rec is None:
                continue
            t, s_, m_, r_ = rec
            if t0 is not None and (t is None or t < t0 or t > t1):
                continue
            sm.append(s_)
            mx_.append(m_)
            reasons |= r_
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        busy = [s for s in sm if s >= 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": max(mx_) if mx_ else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- device helpers

def setup_dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value: float, world: int, device) -> float:
    """Largest value over all ranks (the slowest rank sets the step time)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value: float, world: int, device) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


class ForwardLayer:
    """Preallocated buffers and the three C-ABI calls of one forward step."""

    def __init__(self, mx, x, w, stream):
        import torch
        self.mx = mx
        m, k = x.shape
        k2, n = w.shape
        assert k == k2
        self.m, self.n, self.k = m, n, k
        dev = x.device
        self.x, self.w = x, w
        self.qx = torch.empty((m, k), dtype=torch.uint8, device=dev)
        self.sx = torch.empty(mx.mx_scale_bytes(m, k), dtype=torch.uint8, device=dev)
        self.qw = torch.empty((n, k), dtype=torch.uint8, device=dev)
        self.sw = torch.empty(mx.mx_scale_bytes(n, k), dtype=torch.uint8, device=dev)
        self.y = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
        self.stream = stream
        self.h = int(stream.cuda_stream)

    def quantize_x(self):
        mx = self.mx
        st = mx.mx_quantize(self.x.data_ptr(), 0, self.m, self.k, self.k, 0, 1, 0,
                            self.qx.data_ptr(), self.sx.data_ptr(), None, None, self.h)
        assert st == 0, st

    def quantize_w(self):
        mx = self.mx
        st = mx.mx_quantize(self.w.data_ptr(), 0, self.k, self.n, self.n, 0, 2, 0, None, None,
                            self.qw.data_ptr(), self.sw.data_ptr(), self.h)
        assert st == 0, st

    def gemm(self):
        mx = self.mx
        st = mx.mx_gemm(self.m, self.n, self.k, self.qx.data_ptr(), self.sx.data_ptr(), 0,
                        self.qw.data_ptr(), self.sw.data_ptr(), 0, self.y.data_ptr(), 0, self.n,
                        self.h)
        assert st == 0, st

    def step(self):
        self.quantize_x()
        self.quantize_w()
        self.gemm()

    launches_per_step = 3


# Per-row kernel timings: warm-up launches, then the median of timed
# launches; each row's timed region lasts at least ROW_SECONDS so that
# several clock samples fall inside it.
ROW_WARMUP = 10
ROW_REPS = 50
ROW_MAX_REPS = 4000
ROW_SECONDS = 0.25


def _reps_for(one_ms: float, reps: int | None) -> int:
    if reps is not None:
        return reps
    return int(min(ROW_MAX_REPS, max(ROW_REPS, ROW_SECONDS * 1e3 / max(one_ms, 1e-4))))


def _estimate_ms(fn, stream) -> float:
    import torch
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(5):
        fn()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / 5


def timed_launches(fn, stream, reps: int | None = None, warmup: int = ROW_WARMUP, pre=None):
    """Median duration (ms) of fn() over timed launches, each between two
    CUDA events on `stream`, and the host-time window (epoch seconds) of the
    timed region.  `pre` (e.g. an L2 flush) is enqueued before each launch,
    outside its events; nothing synchronizes the host between `pre`, the
    launch and the events, so the host's launch latency is not timed."""
    import torch
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        n = _reps_for(_estimate_ms(fn, stream) + (_estimate_ms(pre, stream) if pre else 0.0),
                      reps)
        events = []
        t0 = time.time()
        for _ in range(n):
            if pre is not None:
                pre()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            events.append((a, b))
        torch.cuda.synchronize()
        t1 = time.time()
    return statistics.median(a.elapsed_time(b) for a, b in events), (t0, t1)


def time_kernel(fn, stream, reps: int | None = ROW_REPS, warmup: int = ROW_WARMUP) -> float:
    """Median duration (ms) of fn() over reps launches, CUDA events on `stream`."""
    return timed_launches(fn, stream, reps, warmup)[0]


BURST_IDLE_S = 0.5
BURST_LAUNCHES = 8


def timed_burst(fn, stream, launches: int = BURST_LAUNCHES, idle_s: float = BURST_IDLE_S) -> float:
    """Median duration (ms) of `launches` back-to-back launches of an
    already warmed-up fn(), started after the GPU has idled for `idle_s`
    seconds: the kernel timed alone, before the power cap lowers the clock
    (the counterpart of the measured burst peak)."""
    import torch
    torch.cuda.synchronize()
    time.sleep(idle_s)
    with torch.cuda.stream(stream):
        events = []
        for _ in range(launches):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            events.append((a, b))
        torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in events)


def timed_graph(call, nbuf: int, stream, launches: int):
    """Steady-state duration (ms) per launch: `launches` calls (call(i) runs
    on `stream` with buffer set i % nbuf) captured in one CUDA graph and
    replayed, timed by CUDA events around the replays.  Consecutive launches
    touch different buffer sets totalling more than four times the L2, so
    every launch reads its input from HBM."""
    import torch
    with torch.cuda.stream(stream):
        for i in range(nbuf):
            call(i)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(launches):
                call(i % nbuf)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        g.replay()
        b.record(stream)
        torch.cuda.synchronize()
        one = a.elapsed_time(b)
        n = int(min(200, max(3, ROW_SECONDS * 1e3 / max(one, 1e-3))))
        t0 = time.time()
        a.record(stream)
        for _ in range(n):
            g.replay()
        b.record(stream)
        torch.cuda.synchronize()
        t1 = time.time()
    del g
    return a.elapsed_time(b) / (n * launches), (t0, t1)


class RowClocks:
    """The host-time window of every row's timed region; once the clock
    sampler has stopped, each row gets the median SM clock of the samples
    in its window.  (No throughput is scaled by it: under the power cap the
    sampled clock reads well below the clock the kernels effectively ran
    at, so GEMM rows carry a burst time instead, see gemm rows.)"""

    def __init__(self):
        self.windows = []

    def mark(self, row: dict, window, key: str):
        self.windows.append((row, window, key))

    def fill(self, sampler):
        for row, (t0, t1), _key in self.windows:
            c = sampler.summary(t0, t1)
            row["sm_mhz_median"] = c["sm_mhz"]
            row["clock_samples"] = c["samples"]


def flush_l2(buf):
    buf.add_(1)


def launch_floor(stream, scrub, clean) -> dict:
    """The timing harness's own floor: the per-launch time (CUDA events
    around one launch, behind the same flushes as the bandwidth rows) of a
    trivial kernel, a one-block fill of 16 floats."""
    import torch
    tiny = torch.zeros(16, device=scrub.device)
    t, _ = timed_launches(lambda: tiny.fill_(1.0), stream, pre=lambda: flush_l2(scrub))
    tc, _ = timed_launches(lambda: tiny.fill_(1.0), stream,
                           pre=lambda: (flush_l2(scrub), clean.sum()))
    return {"flush_ms": round(t, 4), "clean_l2_ms": round(tc, 4),
            "form": "one-block fill of 16 floats between the same CUDA events, behind the "
                    "same flushes"}


def bandwidth_row(fn, stream, scrub, clean, nbytes: float, hbm: float, bpe: float,
                  clocks: RowClocks, steady=None, floor=None) -> dict:
    """A bandwidth row: one launch timed right behind an L2 write flush, and
    behind the write flush plus a read pass (clean L2); with `steady`
    (call(i), buffer sets, launches per graph), also the steady-state time
    per launch of back-to-back launches over rotating buffers; with `floor`
    (launch_floor()), the clean-L2 rate once the harness floor is taken off."""
    t, win = timed_launches(fn, stream, pre=lambda: flush_l2(scrub))
    tc, _ = timed_launches(fn, stream, pre=lambda: (flush_l2(scrub), clean.sum()))
    gbs = nbytes / (t * 1e-3) / 1e9
    gbc = nbytes / (tc * 1e-3) / 1e9
    row = {"ms": round(t, 4), "GB/s": round(gbs, 1), "frac_hbm": round(gbs / hbm, 3),
           "bytes_per_elem": bpe,
           "clean_l2": {"ms": round(tc, 4), "GB/s": round(gbc, 1), "frac_hbm": round(gbc / hbm, 3)}}
    if floor is not None and tc > floor["clean_l2_ms"]:
        gbf = nbytes / ((tc - floor["clean_l2_ms"]) * 1e-3) / 1e9
        row["clean_l2"]["frac_hbm_beyond_floor"] = round(gbf / hbm, 3)
    if steady is not None:
        call, nbuf, launches = steady
        ts, _ = timed_graph(call, nbuf, stream, launches)
        gss = nbytes / (ts * 1e-3) / 1e9
        row["steady"] = {"ms": round(ts, 4), "GB/s": round(gss, 1), "frac_hbm": round(gss / hbm, 3),
                         "form": f"CUDA graph of {launches} launches over {nbuf} buffer sets "
                                 "(> 4x L2), replayed; time per launch"}
    clocks.mark(row, win, "GB/s")
    return row


# ---------------------------------------------------------------- per-row measurements

def moe_roofline(sizes, n: int, k: int, kind: str, flops_peak: float, hbm_gbs: float,
                 w_code_bytes: float = 1.0) -> dict:
    """Roofline of a mixture-of-experts GEMM.  Per expert with t tokens
    (codes 1 byte and scales 1/32 byte per element; the expert weights'
    codes w_code_bytes per element, 0.5 for packed MXFP4):
      forward  y[t, n] = x[t, k] w_g[n, k]^T, BF16 out
      dgrad    dx[t, k] = dy[t, n] w_g[n, k], FP32 out
      wgrad    dw_g[n, k] = dy[t, n]^T x[t, k], FP32 out (written for every
               expert, zeros without tokens)
    time_ms is the lower bound max(sum FLOP / tensor peak, sum bytes / HBM)
    for a kernel that overlaps experts freely; per_expert_ms is the sum over
    experts of max(FLOP_g / peak, bytes_g / HBM), the bound when experts run
    one after another (small experts bound by their weight or output bytes).
    flops_peak in TFLOP/s, hbm_gbs in GB/s."""
    sc = 1.0 + 1.0 / 32.0
    wsc = w_code_bytes + 1.0 / 32.0
    flops_sum = bytes_sum = per_expert = 0.0
    for t in sizes:
        t = int(t)
        flops = 2.0 * t * n * k
        if kind == "forward":
            nbytes = t * k * sc + n * k * wsc + t * n * 2 if t else 0.0
        elif kind == "dgrad":
            nbytes = (t * n + n * k) * sc + t * k * 4 if t else 0.0
        elif kind == "wgrad":
            nbytes = (t * n + t * k) * sc + n * k * 4
        else:
            raise ValueError(kind)
        flops_sum += flops
        bytes_sum += nbytes
        per_expert += max(flops / (flops_peak * 1e12), nbytes / (hbm_gbs * 1e9))
    tc = flops_sum / (flops_peak * 1e12)
    tm = bytes_sum / (hbm_gbs * 1e9)
    return {"bound": "tensor" if tc >= tm else "hbm", "time_ms": round(max(tc, tm) * 1e3, 4),
            "tensor_ms": round(tc * 1e3, 4), "hbm_ms": round(tm * 1e3, 4),
            "bytes": int(bytes_sum), "per_expert_ms": round(per_expert * 1e3, 4)}


def with_roofline(row: dict, roof: dict) -> dict:
    row["roofline"] = dict(roof, frac=round(roof["time_ms"] / row["ms"], 3),
                           per_expert_frac=round(roof["per_expert_ms"] / row["ms"], 3))
    if "burst" in row:
        row["burst"]["roofline_frac"] = round(roof["time_ms"] / row["burst"]["ms"], 3)
    return row


def measure_rows(mx, peaks, dev, stream, local: int = 0):
    """Per-kernel measurements of the other hot-path rows (rank 0, N=1), with
    the SM clock sampled during each row."""
    import torch
    with ClockSampler(local, period_ms=50) as sampler:
        clocks = RowClocks()
        out = _measure_rows(mx, peaks, dev, stream, clocks)
    clocks.fill(sampler)
    return out


def _gemm_row(fl: float, t: float, tb: float, fp8_peak: float, fp8_sustained: float) -> dict:
    """A GEMM row: `t` the median over a >= 0.25 s loop of launches (the
    power cap active, compared with the sustained peak as well), `tb` the
    burst time after an idle pause (compared with the burst peak)."""
    tf = fl / (t * 1e-3) / 1e12
    tfb = fl / (tb * 1e-3) / 1e12
    return {"ms": round(t, 4), "TFLOP/s": round(tf, 1),
            "frac_fp8_peak": round(tf / fp8_peak, 3),
            "frac_fp8_sustained_peak": round(tf / fp8_sustained, 3),
            "burst": {"ms": round(tb, 4), "TFLOP/s": round(tfb, 1),
                      "frac_fp8_peak": round(tfb / fp8_peak, 3),
                      "form": f"median of {BURST_LAUNCHES} back-to-back launches after "
                              f"{BURST_IDLE_S:g} s idle"}}


def _measure_rows(mx, peaks, dev, stream, clocks: RowClocks):
    import torch
    from mxfp8_block_scaled_mx_gb300 import workloads as W
    h = int(stream.cuda_stream)
    out = {}
    hbm = peaks["hbm_gbs"]
    fp8_peak = peaks["bf16_tflops"] * NOMINAL_FP8_OVER_BF16
    fp8_sustained = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]) * NOMINAL_FP8_OVER_BF16
    scrub = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    clean = torch.ones(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    l2_bytes = torch.cuda.get_device_properties(dev).L2_cache_size

    def gemm_row(name, fn, fl, extra=None):
        t, win = timed_launches(fn, stream)
        tb = timed_burst(fn, stream)
        row = _gemm_row(fl, t, tb, fp8_peak, fp8_sustained)
        if extra:
            row.update(extra)
        clocks.mark(row, win, "TFLOP/s")
        out[name] = row
        return row

    # quantize bandwidth sweep: 4096x4096 and 16384x8192.  Each launch is
    # timed alone right behind an L2 write flush (and behind a flush plus a
    # read pass), and back to back over rotating buffer sets in a CUDA graph.
    floor = launch_floor(stream, scrub, clean)
    out["launch_floor"] = floor
    for (r, c), seed in (((4096, 4096), 0), ((16384, 8192), 1)):
        set_bytes = r * c * 2 + r * c + mx.mx_scale_bytes(r, c)
        nbuf = max(2, -(-4 * l2_bytes // set_bytes) + 1)
        xs = [W.quantize_sweep((r, c), seed=seed, device=dev)]
        xs += [xs[0].roll(i, 0) for i in range(1, nbuf)]          # distinct buffers, same data
        x = xs[0]
        qrs = [torch.empty((r, c), dtype=torch.uint8, device=dev) for _ in range(nbuf)]
        srs = [torch.empty(mx.mx_scale_bytes(r, c), dtype=torch.uint8, device=dev) for _ in range(nbuf)]
        qr, sr = qrs[0], srs[0]
        qc = torch.empty((c, r), dtype=torch.uint8, device=dev)
        sc = torch.empty(mx.mx_scale_bytes(c, r), dtype=torch.uint8, device=dev)
        for mode, axis, bpe in (("row", 1, 3.03125), ("col", 2, 3.03125), ("both", 3, 4.0625)):
            def q(axis=axis):
                st = mx.mx_quantize(x.data_ptr(), 0, r, c, c, 0, axis, 0,
                                    qr.data_ptr() if axis & 1 else None,
                                    sr.data_ptr() if axis & 1 else None,
                                    qc.data_ptr() if axis & 2 else None,
                                    sc.data_ptr() if axis & 2 else None, h)
                assert st == 0
            steady = None
            if mode == "row":
                def qi(i):
                    st = mx.mx_quantize(xs[i].data_ptr(), 0, r, c, c, 0, 1, 0, qrs[i].data_ptr(),
                                        srs[i].data_ptr(), None, None, h)
                    assert st == 0
                steady = (qi, nbuf, 4 * nbuf)
            out[f"quantize_{r}x{c}_{mode}"] = bandwidth_row(q, stream, scrub, clean,
                                                            r * c * bpe, hbm, bpe, clocks, steady,
                                                            floor)
        if (r, c) == (16384, 8192):
            # the page's conservative (ceil) scale rule, rowwise E4M3
            def qceil():
                st = mx.mx_quantize(x.data_ptr(), 0, r, c, c, 0, 1, 1, qr.data_ptr(),
                                    sr.data_ptr(), None, None, h)
                assert st == 0
            out[f"quantize_{r}x{c}_row_ceil"] = bandwidth_row(qceil, stream, scrub, clean,
                                                              r * c * 3.03125, hbm, 3.03125, clocks)
            # MXFP4 codes (E2M1, 16-element containers: one byte per element)
            def q4():
                st = mx.mx_quantize(x.data_ptr(), 0, r, c, c, 4, 1, 0, qr.data_ptr(),
                                    sr.data_ptr(), None, None, h)
                assert st == 0
            out[f"quantize_{r}x{c}_row_e2m1"] = bandwidth_row(q4, stream, scrub, clean,
                                                              r * c * 3.03125, hbm, 3.03125, clocks)
            # the same codes in packed storage (two per byte): 2 + 1/2 + 1/32 B per element
            q4p_codes = torch.empty((r, c // 2), dtype=torch.uint8, device=dev)

            def q4p():
                st = mx.mx_quantize(x.data_ptr(), 0, r, c, c, 7, 1, 0, q4p_codes.data_ptr(),
                                    sr.data_ptr(), None, None, h)
                assert st == 0
            out[f"quantize_{r}x{c}_row_e2m1_packed"] = bandwidth_row(
                q4p, stream, scrub, clean, r * c * 2.53125, hbm, 2.53125, clocks)
            del q4p_codes
            # stochastic rounding (E5M2, the gradient format): the 16-bit
            # random draws are an input, +2 bytes per element
            rb = W.random_bits16((r, c), seed=11, device=dev)

            def qsr():
                st = mx.mx_quantize_sr(x.data_ptr(), 0, r, c, c, rb.data_ptr(), c, 1, 1, 0,
                                       qr.data_ptr(), sr.data_ptr(), None, None, h)
                assert st == 0
            out[f"quantize_{r}x{c}_row_sr_e5m2"] = bandwidth_row(qsr, stream, scrub, clean,
                                                                 r * c * 5.03125, hbm, 5.03125,
                                                                 clocks)

            # both orientations with stochastic rounding (gradients feeding the
            # data and the weight gradient): 2 + 2 + 2 x (1 + 1/32) B per element
            def qsr_both():
                st = mx.mx_quantize_sr(x.data_ptr(), 0, r, c, c, rb.data_ptr(), c, 1, 3, 0,
                                       qr.data_ptr(), sr.data_ptr(), qc.data_ptr(), sc.data_ptr(),
                                       h)
                assert st == 0
            out[f"quantize_{r}x{c}_both_sr_e5m2"] = bandwidth_row(
                qsr_both, stream, scrub, clean, r * c * 6.0625, hbm, 6.0625, clocks)
            # stochastic rounding to packed MXFP4 (gradients in E2M1): bf16 and
            # draws read, half a byte of code written per element
            q4s_codes = torch.empty((r, c // 2), dtype=torch.uint8, device=dev)

            def qsr4():
                st = mx.mx_quantize_sr(x.data_ptr(), 0, r, c, c, rb.data_ptr(), c, 7, 1, 0,
                                       q4s_codes.data_ptr(), sr.data_ptr(), None, None, h)
                assert st == 0
            out[f"quantize_{r}x{c}_row_sr_e2m1_packed"] = bandwidth_row(
                qsr4, stream, scrub, clean, r * c * 4.53125, hbm, 4.53125, clocks)
            del rb, q4s_codes
            # FP32 input (the same values): 4 bytes read per element
            xf = x.float()
            for mode, axis, bpe in (("row", 1, 5.03125), ("both", 3, 6.0625)):
                def qf(axis=axis):
                    st = mx.mx_quantize(xf.data_ptr(), 1, r, c, c, 0, axis, 0,
                                        qr.data_ptr() if axis & 1 else None,
                                        sr.data_ptr() if axis & 1 else None,
                                        qc.data_ptr() if axis & 2 else None,
                                        sc.data_ptr() if axis & 2 else None, h)
                    assert st == 0
                out[f"quantize_{r}x{c}_fp32_{mode}"] = bandwidth_row(
                    qf, stream, scrub, clean, r * c * bpe, hbm, bpe, clocks)
            del xf
        del x, xs, qr, sr, qrs, srs, qc, sc

    # backward GEMMs (FP32 out), the fused bias+SiLU forward, MXFP4/6 operands
    x, w = W.dense_forward(device=dev)
    xq = mx.quantize(x, "e4m3", "row", stream=stream)
    wq = mx.quantize(w, "e4m3", "col", stream=stream)
    bias = torch.randn(w.shape[1], device=dev, dtype=torch.float32)
    yf = torch.empty((x.shape[0], w.shape[1]), dtype=torch.bfloat16, device=dev)
    fl = 2 * x.shape[0] * w.shape[1] * x.shape[1]
    gemm_row("forward_16384x18432x7168_bf16",
             lambda: mx.gemm(xq, wq, "bf16", out=yf, stream=stream), fl)
    gemm_row("forward_bias_silu_16384x18432x7168_bf16",
             lambda: mx.gemm(xq, wq, "bf16", out=yf, stream=stream, bias=bias, act="silu"), fl)
    del xq, wq, bias
    for tag, fa, fb in (("mxfp4_weights_e4m3xe2m1", "e4m3", "e2m1"),
                        ("mxfp4_packed_weights_e4m3xe2m1", "e4m3", "e2m1_packed"),
                        ("mxfp6_e3m2xe3m2", "e3m2", "e3m2")):
        xq = mx.quantize(x, fa, "row", stream=stream)
        wq = mx.quantize(w, fb, "col", stream=stream)
        gemm_row(f"forward_{tag}_16384x18432x7168_bf16",
                 lambda: mx.gemm(xq, wq, "bf16", out=yf, stream=stream), fl)
        del xq, wq
    del yf
    dy = W.dense_grad_output(device=dev)
    rq = mx.quantize(dy, "e5m2", "row", stream=stream)
    wq = mx.quantize(w, "e4m3", "row", stream=stream)
    dx = torch.empty((dy.shape[0], w.shape[0]), dtype=torch.float32, device=dev)
    gemm_row("dgrad_16384x7168x18432_e5m2xe4m3_fp32",
             lambda: mx.gemm(rq, wq, "fp32", out=dx, stream=stream),
             2 * dy.shape[0] * w.shape[0] * dy.shape[1])
    del rq, wq, dx
    xq = mx.quantize(x, "e4m3", "col", stream=stream)
    dq = mx.quantize(dy, "e5m2", "col", stream=stream)
    dw = torch.empty((x.shape[1], dy.shape[1]), dtype=torch.float32, device=dev)
    gemm_row("wgrad_7168x18432x16384_e4m3xe5m2_fp32",
             lambda: mx.gemm(xq, dq, "fp32", out=dw, stream=stream),
             2 * x.shape[1] * dy.shape[1] * x.shape[0])
    del xq, dq, dw, x, w, dy

    xm, wm, offsets = W.moe_inputs(device=dev)
    e, n, k = wm.shape
    d_off = torch.from_numpy(offsets).to(dev)
    qa = mx.quantize_grouped(xm, d_off, "e4m3", stream=stream)
    qw = mx.quantize(wm.view(e * n, k), "e4m3", "row", stream=stream)
    qb = mx.MxTensor(qw.codes.view(e, n, k), qw.scales, "e4m3")
    ym = torch.empty((xm.shape[0], n), dtype=torch.bfloat16, device=dev)
    fl = 2 * xm.shape[0] * n * k
    sizes = [int(v) for v in (offsets[1:] - offsets[:-1])]
    row = gemm_row("moe_grouped_64x(2048x7168)_65536tok_bf16",
                   lambda: mx.grouped_gemm(qa, d_off, qb, "bf16", out=ym, stream=stream), fl,
                   {"group_sizes_min_max": [min(sizes), max(sizes)],
                    "empty_groups": sizes.count(0)})
    with_roofline(row, moe_roofline(sizes, n, k, "forward", fp8_peak, hbm))
    # the same with MXFP4 expert weights in packed storage (two codes a byte)
    qw4 = mx.quantize(wm.view(e * n, k), "e2m1_packed", "row", stream=stream)
    qb4 = mx.MxTensor(qw4.codes.view(e, n, k // 2), qw4.scales, "e2m1_packed")
    row = gemm_row("moe_grouped_mxfp4_packed_weights_64x(2048x7168)_65536tok_bf16",
                   lambda: mx.grouped_gemm(qa, d_off, qb4, "bf16", out=ym, stream=stream), fl)
    with_roofline(row, moe_roofline(sizes, n, k, "forward", fp8_peak, hbm, w_code_bytes=0.5))
    del qw4, qb4

    # grouped rowwise quantize into the buffers above (the C call: no
    # allocation inside the timed launches; inputs 940 MB, larger than L2)
    def qrow():
        st = mx.mx_quantize_grouped(xm.data_ptr(), 0, xm.shape[0], k, k, 0, 0, e,
                                    d_off.data_ptr(), qa.codes.data_ptr(), qa.scales.data_ptr(), h)
        assert st == 0
    t, win = timed_launches(qrow, stream)
    gbs = xm.numel() * 3.03125 / (t * 1e-3) / 1e9
    row = {"ms": round(t, 4), "GB/s": round(gbs, 1), "frac_hbm": round(gbs / hbm, 3)}
    clocks.mark(row, win, "GB/s")
    out["moe_quantize_grouped_65536x7168"] = row
    del ym, qa

    # mixture-of-experts backward: dX_g = dY_g W_g^T (experts side by side
    # along K) and dW_g = dY_g^T X_g (grouped along K), FP32 out
    total = xm.shape[0]
    dym = W.moe_grad_output(device=dev)
    qa = mx.quantize_grouped(dym, d_off, "e5m2", stream=stream)
    qb = mx.quantize(wm.view(e * n, k), "e4m3", "col", stream=stream)
    dx = torch.empty((total, k), dtype=torch.float32, device=dev)
    row = gemm_row("moe_dgrad_64x(7168x2048)_65536tok_fp32",
                   lambda: mx.grouped_gemm_bcat(qa, d_off, qb, "fp32", out=dx, stream=stream), fl)
    with_roofline(row, moe_roofline(sizes, n, k, "dgrad", fp8_peak, hbm))
    del qa, qb, dx
    ldq = mx.mx_grouped_cols_capacity(total, e)
    qa = mx.quantize_grouped(dym, d_off, "e5m2", axis="col", ldq=ldq, stream=stream)
    qb = mx.quantize_grouped(xm, d_off, "e4m3", axis="col", ldq=ldq, stream=stream)
    dw = torch.empty((e, n, k), dtype=torch.float32, device=dev)
    row = gemm_row("moe_wgrad_64x(2048x7168)_65536tok_fp32",
                   lambda: mx.grouped_gemm_wgrad(qa, d_off, qb, total, "fp32", out=dw,
                                                 stream=stream), fl)
    with_roofline(row, moe_roofline(sizes, n, k, "wgrad", fp8_peak, hbm))
    del dw

    # grouped columnwise quantize of X (per-expert token blocks), into the
    # buffers above; the codes of the 128-padded segments are written too
    def qcol():
        st = mx.mx_quantize_grouped_ex(xm.data_ptr(), 0, total, k, k, 0, 2, 0, e, d_off.data_ptr(),
                                       None, None, qb.codes.data_ptr(), ldq,
                                       qb.scales.data_ptr(), h)
        assert st == 0
    t, win = timed_launches(qcol, stream)
    gbs = xm.numel() * 3.03125 / (t * 1e-3) / 1e9
    row = {"ms": round(t, 4), "GB/s": round(gbs, 1), "frac_hbm": round(gbs / hbm, 3)}
    clocks.mark(row, win, "GB/s")
    out["moe_quantize_grouped_cols_65536x7168"] = row
    return out


# ---------------------------------------------------------------- CPU oracle baseline

def oracle_sample(rows: int = 4096, cols: int = 4096):
    """The CPU oracle, as it stands, on a bounded sample of the forward
    workload: `rows` token rows of X and `cols` columns of W with the full
    K = 7168, drawn from the workload's distributions; oracle quantize of
    both slices plus the oracle block-scaled GEMM.
    Returns (TFLOP/s, seconds, description)."""
    from mxfp8_block_scaled_mx_gb300 import workloads as W
    from oracle import mx_oracle as O
    k = FWD["k"]
    xs = W.synth_matrix((rows, k), 1.0, 0.005, 50.0, 500.0, seed=404)
    ws = W.synth_matrix((k, cols), 0.02, seed=405)
    t0 = time.perf_counter()
    a = O.quantize(xs.float().double().numpy(), "e4m3", "row")
    b = O.quantize(ws.float().double().numpy(), "e4m3", "col")
    O.gemm(a, b)
    dt = time.perf_counter() - t0
    flops = 2 * rows * cols * k
    return flops / dt / 1e12, dt, (f"oracle quantize of X[{rows}x{k}] rowwise and W[{k}x{cols}] "
                                   f"colwise, then oracle GEMM {rows}x{cols}x{k} "
                                   "(float64 numpy), same distributions as the forward layer")


def cpu_threads():
    return os.cpu_count() or 1


def oracle_parts(gemm_rows: int, quant: bool = True) -> dict:
    """The oracle's pieces timed on the host: quantization of the full
    4096x4096 tensor of the quantize sweep (rowwise and columnwise, GB/s on
    the algorithmic 3.03125 B/element), and the block-scaled GEMM of a
    `gemm_rows`-row slice of the forward layer (full N = 18432, K = 7168)
    with its time extrapolated to all 16384 rows."""
    import numpy as np
    from mxfp8_block_scaled_mx_gb300 import workloads as W
    from oracle import mx_oracle as O
    out = {}
    if quant:
        x = W.quantize_sweep((4096, 4096), seed=0).float().double().numpy()
        for axis in ("row", "col"):
            t0 = time.perf_counter()
            O.quantize(x, "e4m3", axis)
            dt = time.perf_counter() - t0
            out[f"quantize_4096x4096_{axis}_GB/s"] = round(4096 * 4096 * 3.03125 / dt / 1e9, 4)
    m, n, k = FWD["m"], FWD["n"], FWD["k"]
    rng = np.random.default_rng(5)
    # operands of the layer's formats and block structure (E4M3 codes with
    # per-block scales near 2^0); the GEMM's cost does not depend on the values
    fin = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    a = O.MxBlocks(rng.choice(fin, (gemm_rows, k)), rng.integers(120, 134, (gemm_rows, k // 32),
                                                                 dtype=np.uint8), O.FORMATS["e4m3"])
    b = O.MxBlocks(rng.choice(fin, (n, k)), rng.integers(120, 134, (n, k // 32), dtype=np.uint8),
                   O.FORMATS["e4m3"])
    t0 = time.perf_counter()
    O.gemm(a, b)
    dt = time.perf_counter() - t0
    out["gemm_slice"] = f"{gemm_rows}x{n}x{k}"
    out["gemm_slice_s"] = round(dt, 3)
    out["gemm_TFLOP/s"] = round(2 * gemm_rows * n * k / dt / 1e12, 6)
    out["gemm_full_16384_rows_s_extrapolated"] = round(dt * m / gemm_rows, 1)
    return out


def oracle_one_thread() -> dict:
    """oracle_parts in a child process limited to one thread (BLAS and
    OpenMP pools of one), on a smaller GEMM slice."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               NUMEXPR_NUM_THREADS="1")
    res = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-one-thread"],
                         capture_output=True, text=True, env=env, timeout=600)
    if res.returncode != 0:
        return {"error": res.stderr.strip().splitlines()[-1:] or ["failed"]}
    return json.loads(res.stdout.strip().splitlines()[-1])


def cpu_baseline_record() -> dict:
    """The reported CPU baseline: the oracle, as it stands, on bounded
    samples (about half a minute of host work in all)."""
    v, dt, desc = oracle_sample(2048, 4096)
    rec = {"value": v, "unit": UNIT, "cores": cpu_threads(), "kind": "oracle", "sample": desc,
           "seconds": round(dt, 2)}
    rec["all_threads"] = dict(oracle_parts(128), threads=cpu_threads())
    rec["one_thread"] = dict(oracle_one_thread(), threads=1)
    return rec


# ---------------------------------------------------------------- main arms

def run_reference(args):
    world, rank, _ = setup_dist()
    if rank != 0:
        return 0
    # each step: a small bounded sample so K steps end within minutes
    for _ in range(args.warmup):
        oracle_sample(REF_ROWS, REF_COLS)
    vals, secs = [], []
    for _ in range(args.steps):
        v, dt, desc = oracle_sample(REF_ROWS, REF_COLS)
        vals.append(v)
        secs.append(dt)
    value = statistics.median(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": statistics.median(secs) * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "sample": desc},
        "cpu_baseline": {"kind": "oracle", "value": value, "unit": UNIT, "cores": cpu_threads(),
                         "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


PAIR_KERNEL_SOURCES = ("gemm_pair.cu", "epilogue.cuh", "tiles.cuh", "groups.cuh", "ptx.cuh",
                       "kernels.h")


def pair_kernel_sources_sha() -> str:
    """sha256 over the block-pair GEMM's source files, in a fixed order."""
    h = hashlib.sha256()
    for name in PAIR_KERNEL_SOURCES:
        with open(os.path.join(ROOT, "mxfp8_block_scaled_mx_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def gemm_traffic_record():
    """DRAM bytes per launch of the forward GEMM (the block-pair kernel) from
    the committed ncu summary, valid only while the kernel's sources are
    unchanged (the sha256 of their concatenation recorded beside the
    figure)."""
    path = os.path.join(ROOT, "profiles", "mx_gemm_pair_forward_16384x18432x7168_dram.md")
    try:
        text = open(path).read()
        sha = pair_kernel_sources_sha()
    except OSError:
        return None
    rec = {}
    for line in text.splitlines():
        if ":" in line and line.strip().startswith("- "):
            key, val = line.strip()[2:].split(":", 1)
            rec[key.strip()] = val.strip().strip("`")
    if rec.get("pair kernel sources sha256") != sha:
        return None
    try:
        return float(rec["dram bytes per full-size launch"])
    except (KeyError, ValueError):
        return None


def run_gpu(args):
    import torch
    import mxfp8_block_scaled_mx_gb300 as mx
    from mxfp8_block_scaled_mx_gb300 import workloads as W

    world, rank, local = setup_dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    mx.lib()
    peaks, peak_src = read_peaks()
    stream = torch.cuda.Stream(device=dev)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    with torch.cuda.stream(stream):
        x, w = W.dense_forward(seed=rank, device=dev)
        layer = ForwardLayer(mx, x, w, stream)
        torch.cuda.synchronize()
        for _ in range(args.warmup):
            layer.step()
        torch.cuda.synchronize()

        # ---------------- device-resident timed region
        ev = []
        barrier()
        torch.cuda.synchronize()
        with ClockSampler(local) as clocks:
            start = torch.cuda.Event(enable_timing=True)
            stop = torch.cuda.Event(enable_timing=True)
            start.record(stream)
            for _ in range(args.steps):
                layer.quantize_x()
                layer.quantize_w()
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record(stream)
                layer.gemm()
                b.record(stream)
                ev.append((a, b))
            stop.record(stream)
            torch.cuda.synchronize()
        barrier()
        elapsed_ms = start.elapsed_time(stop)
        gemm_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
        elapsed_ms = max_over_ranks(elapsed_ms, world, dev)
        assert mx.mx_device_status(stream) == 0

        flops_step = 2 * layer.m * layer.n * layer.k
        ms_per_step = elapsed_ms / args.steps
        value = world * flops_step / (ms_per_step * 1e-3) / 1e12

        # quantize kernels timed alone (same buffers) for their GB/s
        tq_x = time_kernel(layer.quantize_x, stream, ROW_REPS)
        tq_w = time_kernel(layer.quantize_w, stream, ROW_REPS)

        # ---------------- end to end: host buffers through the C ABI
        hx = torch.empty(x.shape, dtype=x.dtype, pin_memory=True)
        hw = torch.empty(w.shape, dtype=w.dtype, pin_memory=True)
        hx.copy_(x)
        hw.copy_(w)
        hy = torch.empty(layer.y.shape, dtype=layer.y.dtype, pin_memory=True)
        # the device-timed figure's K steps: the streamed form's pipeline fill
        # and drain (one upload, one download) are amortized as in a long run
        e2e_steps = max(3, args.steps)
        for _ in range(2):
            x.copy_(hx, non_blocking=True)
            w.copy_(hw, non_blocking=True)
            layer.step()
            hy.copy_(layer.y, non_blocking=True)
        torch.cuda.synchronize()
        barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(e2e_steps):
            x.copy_(hx, non_blocking=True)
            w.copy_(hw, non_blocking=True)
            layer.step()
            hy.copy_(layer.y, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        barrier()
        serial_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world, dev)
        serial_value = world * flops_step / (serial_ms * 1e-3) / 1e12
        h2d = hx.numel() * hx.element_size() + hw.numel() * hw.element_size()
        d2h = hy.numel() * hy.element_size()

        # Streaming form of the same job: step i's upload, compute and
        # download run on their own streams, so the upload of step i+1 and
        # the download of step i-1 overlap the compute of step i.  Device
        # buffers are double-buffered; every step still copies its inputs
        # from pinned host memory and its result back inside the timed region.
        s_up = torch.cuda.Stream(device=dev)
        s_dn = torch.cuda.Stream(device=dev)
        layers = [layer, ForwardLayer(mx, torch.empty_like(x), torch.empty_like(w), stream)]
        hys = [hy, torch.empty(layer.y.shape, dtype=layer.y.dtype, pin_memory=True)]

        def pipelined(n, start_ev):
            up_ev = [None, None]
            comp_ev = [None, None]
            dn_ev = [None, None]
            s_up.wait_event(start_ev)
            for i in range(n):
                j = i % 2
                L = layers[j]
                with torch.cuda.stream(s_up):
                    if comp_ev[j] is not None:
                        s_up.wait_event(comp_ev[j])      # step i-2 is done with these inputs
                    L.x.copy_(hx, non_blocking=True)
                    L.w.copy_(hw, non_blocking=True)
                    up_ev[j] = torch.cuda.Event()
                    up_ev[j].record(s_up)
                stream.wait_event(up_ev[j])
                if dn_ev[j] is not None:
                    stream.wait_event(dn_ev[j])          # step i-2's result has been read out
                L.step()
                comp_ev[j] = torch.cuda.Event()
                comp_ev[j].record(stream)
                with torch.cuda.stream(s_dn):
                    s_dn.wait_event(comp_ev[j])
                    hys[j].copy_(L.y, non_blocking=True)
                    dn_ev[j] = torch.cuda.Event()
                    dn_ev[j].record(s_dn)
            for ev_ in dn_ev:
                if ev_ is not None:
                    stream.wait_event(ev_)

        w0 = torch.cuda.Event()
        w0.record(stream)
        pipelined(3, w0)                                  # warm-up
        torch.cuda.synchronize()
        barrier()
        p0 = torch.cuda.Event(enable_timing=True)
        p1 = torch.cuda.Event(enable_timing=True)
        p0.record(stream)
        pipelined(e2e_steps, p0)
        p1.record(stream)
        torch.cuda.synchronize()
        barrier()
        e2e_ms = max_over_ranks(p0.elapsed_time(p1) / e2e_steps, world, dev)
        e2e_value = world * flops_step / (e2e_ms * 1e-3) / 1e12
        assert torch.equal(hys[(e2e_steps - 1) % 2], layers[(e2e_steps - 1) % 2].y.cpu())
        del layers[1]

        rows = None
        if rank == 0 and world == 1 and not args.no_rows:
            del hx, hw, hy
            rows = measure_rows(mx, peaks, dev, stream, local)

    if rank != 0:
        return 0

    fp8_peak = peaks["bf16_tflops"] * NOMINAL_FP8_OVER_BF16
    gemm_tflops = flops_step / (gemm_ms * 1e-3) / 1e12
    traffic = gemm_traffic_record()
    hbm = peaks["hbm_gbs"]
    qx_bytes = layer.m * layer.k * 3.03125
    qw_bytes = layer.k * layer.n * 3.03125
    clk = clocks.summary()
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "m": layer.m, "n": layer.n, "k": layer.k,
                   "l2": "inputs larger than L2 (X 235 MB, W 264 MB, Y 604 MB per step)",
                   "per_rank_batch": "one 16384-token batch per GPU",
                   "value_def": "2*M*N*K of the step / step time (quantize X + quantize W + GEMM)"},
        "roofline": {"bound": "tensor", "achieved": round(gemm_tflops, 1),
                     "peak": round(fp8_peak, 1), "unit": "TFLOP/s",
                     "frac": round(gemm_tflops / fp8_peak, 4), "traffic": traffic,
                     "kernel": "mx_gemm_pair_kernel (cta_group::2 block pairs, forward, BF16 out)",
                     "peak_source": f"{peak_src} bf16 burst {peaks['bf16_tflops']} TFLOP/s x "
                                    f"{NOMINAL_FP8_OVER_BF16} (nominal dense fp8/bf16 ratio)",
                     "frac_of_sustained": round(
                         gemm_tflops / (peaks["bf16_tflops_sustained"] * NOMINAL_FP8_OVER_BF16), 4)},
        "step_parts_ms": {"gemm": round(gemm_ms, 4), "quantize_x_alone": round(tq_x, 4),
                          "quantize_w_alone": round(tq_w, 4)},
        "quantize": {"x_rowwise_GB/s": round(qx_bytes / (tq_x * 1e-3) / 1e9, 1),
                     "w_colwise_GB/s": round(qw_bytes / (tq_w * 1e-3) / 1e9, 1),
                     "hbm_peak_GB/s": hbm,
                     "x_frac_hbm": round(qx_bytes / (tq_x * 1e-3) / 1e9 / hbm, 3),
                     "w_frac_hbm": round(qw_bytes / (tq_w * 1e-3) / 1e9 / hbm, 3)},
        "e2e": {"value": round(e2e_value, 2), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "form": "streamed: upload / compute / download of consecutive steps overlap "
                        "on three streams, double-buffered device tensors",
                "serial_value": round(serial_value, 2),
                "serial_form": "one stream: upload, quantize x2, GEMM, download per step"},
        "gpu_launches": layer.launches_per_step * args.steps,
        "clocks": clk,
    }
    if rows is not None:
        line["rows"] = rows
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_record()
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="mx", choices=["mx", "reference"])
    ap.add_argument("--no-rows", action="store_true", help="skip the per-row extra kernels")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--oracle-one-thread", action="store_true", help=argparse.SUPPRESS)
    args = ap.parse_args(argv)
    if args.oracle_one_thread:
        print(json.dumps(oracle_parts(16)), flush=True)
        return 0
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
