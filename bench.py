#!/usr/bin/env python
"""Benchmark of the row-wise LayerNorm / RMSNorm hot path on one GB300.

One step = one pass of the whole path over the bf16 workload with N = 8192
rows and H in {1024, 5120}: for each H, LayerNorm forward + backward, RMSNorm
forward + backward and the fused residual-add + RMSNorm forward (10 calls, 14
kernel launches).  Each call is timed on the device with CUDA events on the
launching stream, with L2 flushed before every call, as in training where
the forward's outputs are long gone from L2 when the backward runs.  The flush
writes a buffer larger than twice the L2 size and then reads another one of
that size, so the dirty lines of the write are back in HBM before the timed
call starts: the call finds L2 cold and clean (the state ncu's cache control
leaves), and is not charged for writing back the flush's own data.

Metric: achieved HBM GB/s = algorithmic bytes of the step / summed device
time of its calls.  Algorithmic bytes per call (e = 2 bytes, bf16):
  LN fwd 2NHe + 2He + 8N,  RMS fwd 2NHe + He + 4N,  fused 4NHe + He + 4N,
  LN bwd 3NHe + 3He + 8N,  RMS bwd 3NHe + 2He + 4N.

The JSON line also carries: per-call microseconds (the backward per shape
included), a roofline object for the call with the largest share of the step,
the SM clocks sampled during the timed region, an end-to-end figure through
the public API with pinned host buffers and the copies inside the timed
region, and the fp64 CPU oracle timed on the host as a reported baseline.

``--impl reference`` times the CPU oracle alone on a bounded row sample of the
same workload (there is no other implementation of this path to run).
Under torchrun (N > 1) every rank runs an independent replica of the step
(rows are independent; nothing is exchanged) and rank 0 prints the aggregate.
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

WORKLOAD = "LN+RMSNorm fwd+bwd and fused add+RMSNorm fwd, bf16, N=8192, H in {1024, 5120}"
SHAPES = [(8192, 1024), (8192, 5120)]
EPS, EPS_FUSED = 1e-5, 1e-6
FALLBACK_HBM_GBS = 6800.0
METRIC = "LN/RMSNorm fwd+bwd achieved HBM GB/s and % of GB300 peak; bwd µs per shape (bf16)"
OPS = ("ln_fwd", "ln_bwd", "rms_fwd", "rms_bwd", "fused_fwd")
# Measured by --sweep / --profile-op, not part of the step: the fused-add
# backward (dx and dres from the stored h, plus the residual-stream gradient).
EXTRA_OPS = ("fused_bwd", "ln_bwd_y", "rms_bwd_y", "fused_fwd_ip")
LAUNCHES = {"ln_fwd": 1, "rms_fwd": 1, "fused_fwd": 1, "ln_bwd": 2, "rms_bwd": 2, "fused_bwd": 2, "ln_bwd_y": 2,
            "rms_bwd_y": 2, "fused_fwd_ip": 1}


def alg_bytes(op: str, N: int, H: int, e: int = 2, ew: int = 2) -> int:
    """Algorithmic HBM bytes of one call (each tensor byte read or written once)."""
    nh = N * H * e
    return {
        "ln_fwd": 2 * nh + 2 * H * ew + 8 * N,
        "rms_fwd": 2 * nh + H * ew + 4 * N,
        "fused_fwd": 4 * nh + H * ew + 4 * N,
        "ln_bwd": 3 * nh + 8 * N + H * ew + 2 * H * ew,
        "rms_bwd": 3 * nh + 4 * N + H * ew + H * ew,
        # reads dy, h, the stream gradient; writes dx and dres
        "fused_bwd": 5 * nh + 4 * N + H * ew + H * ew,
        # the fused add updating the residual stream in place (h_out = x)
        "fused_fwd_ip": 4 * nh + H * ew + 4 * N,
        # from the saved output: reads dy, y, rstd, gamma (and beta)
        "ln_bwd_y": 3 * nh + 4 * N + 2 * H * ew + 2 * H * ew,
        "rms_bwd_y": 3 * nh + 4 * N + H * ew + H * ew,
    }[op]


# ---------------------------------------------------------------------------
# environment
# ---------------------------------------------------------------------------

def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def src_digest():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "rmsnorm_ln_fwd_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(op_key: str):
    """dram read+write bytes per launch of `op_key` from the committed ncu
    summary, or None when absent or taken on other kernel sources."""
    path = os.path.join(ROOT, "profiles", "roofline_traffic.txt")
    try:
        with open(path) as f:
            kv = dict(line.strip().split("=", 1) for line in f if "=" in line and not line.startswith("#"))
    except OSError:
        return None
    if kv.get("src_digest") != src_digest():
        return None
    v = kv.get(op_key)
    return float(v) if v else None


def record_traffic(paths, out_path):
    """Write the per-call DRAM traffic table that roofline.traffic reads.

    Each path is an ncu raw CSV (``--csv --page raw`` with the metrics
    dram__bytes_read.sum and dram__bytes_write.sum) of one call captured with
    ``bench.py --profile-op OP --shape NxH``, named ``traffic_OP_NxH.csv``;
    the call's traffic is the sum over the launches captured (a backward: its
    main kernel and its partial reduction).  The table records the digest of
    the kernel sources it was taken on, computed here, so bench.py stops
    reporting it once a source changes."""
    import csv
    rows = {}
    for path in paths:
        name = os.path.basename(path)
        if not (name.startswith("traffic_") and name.endswith(".csv")):
            raise ValueError(f"{path}: expected traffic_<op>_<N>x<H>.csv")
        key = name[len("traffic_"):-len(".csv")]
        with open(path) as f:
            lines = [r for r in csv.reader(f)]
        head = next(i for i, r in enumerate(lines) if r and r[0] == "ID")
        h, units = lines[head], dict(zip(lines[head], lines[head + 1]))  # the row after the header: units
        scale = {"byte": 1, "kbyte": 1e3, "mbyte": 1e6, "gbyte": 1e9, "tbyte": 1e12,
                 "kibyte": 1024, "mibyte": 1 << 20, "gibyte": 1 << 30}
        total, launches = 0.0, 0
        for r in lines[head + 2:]:
            if len(r) != len(h):
                continue
            d = dict(zip(h, r))
            for m in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
                total += float(d[m].replace(",", "")) * scale[units[m].strip().lower()]
            launches += 1
        if launches == 0:
            raise ValueError(f"{path}: no captured launch")
        rows[key] = (int(total), launches)
    with open(out_path, "w") as f:
        f.write("# DRAM read+write bytes per call (every kernel of the call, ncu dram__bytes_read.sum +\n")
        f.write("# dram__bytes_write.sum, cold caches), written by `python bench.py --record-traffic` from\n")
        f.write("# captures of `ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum --clock-control none\n")
        f.write("# -k regex:'fwd_|bwd_' -s <forward launches> -c <kernels of one call> --csv --page raw\n")
        f.write("# python bench.py --profile-op OP --shape NxH --iters 2`.  Writes still dirty in L2 when a\n")
        f.write("# kernel ends are not counted.  src_digest: the kernel sources the captures ran on.\n")
        f.write(f"src_digest={src_digest()}\n")
        for key in sorted(rows):
            f.write(f"{key}={rows[key][0]}\n")
    return rows


class L2Flush:
    """Evicts L2 between timed calls: a write of a buffer larger than twice the
    L2 size, then a read of a second one of the same size.  The read pushes the
    write's dirty lines back to HBM inside the flush, so the next call starts
    from a cold, clean L2."""

    def __init__(self, dev):
        import torch
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        n = max(2 * l2, 256 << 20) // 4
        self.w = torch.empty(n, dtype=torch.float32, device=dev)
        self.r = torch.zeros(n, dtype=torch.float32, device=dev)
        self.out = torch.empty((), dtype=torch.float32, device=dev)
        self.mib = n * 4 >> 20

    def __call__(self):
        import torch
        self.w.zero_()
        torch.sum(self.r, dim=0, out=self.out)

    def describe(self):
        return (f"flushed before every timed call: a {self.mib} MiB write, then a {self.mib} MiB read that "
                f"writes the dirty lines back before the call starts (cold, clean L2)")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        import tempfile
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:  # no nvidia-smi: no clock record
            self.proc = None
            os.unlink(self.path)
            return
        t0 = time.time()
        while time.time() - t0 < 5.0 and os.path.getsize(self.path) == 0:
            time.sleep(0.02)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) == 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------
# the workload on the GPU
# ---------------------------------------------------------------------------

class Shape:
    """Device tensors of one (N, H) shape and argument tuples for the C ABI."""

    def __init__(self, N, H, dev, seed, lib, extra=False, dtype="bf16", x_offset=0.0, x_scale=1.0):
        import torch
        from rmsnorm_ln_fwd_gb300 import synth, ops
        self.N, self.H, self.lib, self.dev = N, H, lib, dev
        host = synth.norm_inputs(N, H, dtype, seed=seed, with_residual=True, with_dh_stream=extra,
                                 x_offset=x_offset, x_scale=x_scale)
        self.code = {"f32": 0, "bf16": 1, "f16": 2}[dtype]
        self.esize = 4 if dtype == "f32" else 2
        self.host = host
        t = {k: v.to(dev) for k, v in host.items()}
        self.t = t
        e = torch.empty
        bf = synth.DTYPES[dtype]
        self.y = e(N, H, dtype=bf, device=dev)
        self.yr = e(N, H, dtype=bf, device=dev)
        self.yf = e(N, H, dtype=bf, device=dev)
        self.h = e(N, H, dtype=bf, device=dev)
        self.dx = e(N, H, dtype=bf, device=dev)
        self.dxr = e(N, H, dtype=bf, device=dev)
        self.mean = e(N, dtype=torch.float32, device=dev)
        self.rstd = e(N, dtype=torch.float32, device=dev)
        self.rstd_r = e(N, dtype=torch.float32, device=dev)
        self.rstd_f = e(N, dtype=torch.float32, device=dev)
        self.dg = e(H, dtype=bf, device=dev)
        self.db = e(H, dtype=bf, device=dev)
        self.dgr = e(H, dtype=bf, device=dev)
        self.wsb = ops.bwd_workspace_bytes(H, dev)
        self.ws = e((self.wsb + 3) // 4, dtype=torch.float32, device=dev)
        self.bytes = {op: alg_bytes(op, N, H, bf.itemsize, bf.itemsize) for op in OPS}
        if extra:
            self.dxf = e(N, H, dtype=bf, device=dev)
            self.dresf = e(N, H, dtype=bf, device=dev)
            self.dgf = e(H, dtype=bf, device=dev)

    def call(self, op, stream):
        L, t, N, H = self.lib, self.t, self.N, self.H
        BF = self.code
        if op == "ln_fwd":
            st = L.ln_forward(t["x"].data_ptr(), H, t["gamma"].data_ptr(), t["beta"].data_ptr(), self.y.data_ptr(),
                              H, self.mean.data_ptr(), self.rstd.data_ptr(), N, H, EPS, BF, BF, stream)
        elif op == "ln_bwd":
            st = L.ln_backward(t["dy"].data_ptr(), H, t["x"].data_ptr(), H, self.mean.data_ptr(),
                               self.rstd.data_ptr(), t["gamma"].data_ptr(), self.dx.data_ptr(), H,
                               self.dg.data_ptr(), self.db.data_ptr(), self.ws.data_ptr(), self.wsb, N, H, BF, BF,
                               stream)
        elif op == "rms_fwd":
            st = L.rms_forward(t["x"].data_ptr(), H, t["gamma"].data_ptr(), self.yr.data_ptr(), H,
                               self.rstd_r.data_ptr(), N, H, EPS, BF, BF, stream)
        elif op == "rms_bwd":
            st = L.rms_backward(t["dy"].data_ptr(), H, t["x"].data_ptr(), H, self.rstd_r.data_ptr(),
                                t["gamma"].data_ptr(), self.dxr.data_ptr(), H, self.dgr.data_ptr(),
                                self.ws.data_ptr(), self.wsb, N, H, BF, BF, stream)
        elif op == "ln_bwd_y":
            st = L.ln_backward_from_output(t["dy"].data_ptr(), H, self.y.data_ptr(), H, self.rstd.data_ptr(),
                                           t["gamma"].data_ptr(), t["beta"].data_ptr(), self.dxf.data_ptr(), H,
                                           self.dg.data_ptr(), self.db.data_ptr(), self.ws.data_ptr(), self.wsb, N,
                                           H, BF, BF, stream)
        elif op == "rms_bwd_y":
            st = L.rms_backward_from_output(t["dy"].data_ptr(), H, self.yr.data_ptr(), H, self.rstd_r.data_ptr(),
                                            t["gamma"].data_ptr(), self.dxf.data_ptr(), H, self.dgr.data_ptr(),
                                            self.ws.data_ptr(), self.wsb, N, H, BF, BF, stream)
        elif op == "fused_fwd_ip":
            st = L.fused_add_rms_forward(t["x"].data_ptr(), H, t["residual"].data_ptr(), H, t["gamma"].data_ptr(),
                                         self.yf.data_ptr(), H, t["x"].data_ptr(), H, self.rstd_f.data_ptr(), N, H,
                                         EPS_FUSED, BF, BF, stream)
        elif op == "fused_bwd":
            st = L.fused_add_rms_backward(t["dy"].data_ptr(), H, self.h.data_ptr(), H, self.rstd_f.data_ptr(),
                                          t["gamma"].data_ptr(), t["dh_stream"].data_ptr(), H, self.dxf.data_ptr(),
                                          H, self.dresf.data_ptr(), H, self.dgf.data_ptr(), self.ws.data_ptr(),
                                          self.wsb, N, H, BF, BF, stream)
        else:
            st = L.fused_add_rms_forward(t["x"].data_ptr(), H, t["residual"].data_ptr(), H, t["gamma"].data_ptr(),
                                         self.yf.data_ptr(), H, self.h.data_ptr(), H, self.rstd_f.data_ptr(), N, H,
                                         EPS_FUSED, BF, BF, stream)
        if st != 0:
            raise RuntimeError(f"{op} {N}x{H}: status {st}")


# Every configuration of the workload's specification, timed call by call
# after the step (the step itself is the C2 workload): (config, op, N, H,
# row dtype, x offset, x scale).  C2's backwards are listed again so that
# their main-kernel / partial-reduction split is reported too.
CONFIGS = [
    ("C1", "ln_fwd", 64, 256, "f32", 0.0, 1.0),
    ("C1", "ln_bwd", 64, 256, "f32", 0.0, 1.0),
    ("C2", "ln_bwd", 8192, 1024, "bf16", 0.0, 1.0),
    ("C2", "rms_bwd", 8192, 1024, "bf16", 0.0, 1.0),
    ("C2", "ln_bwd", 8192, 5120, "bf16", 0.0, 1.0),
    ("C2", "rms_bwd", 8192, 5120, "bf16", 0.0, 1.0),
    ("C2s", "ln_fwd", 8192, 1024, "f32", 1000.0, 1e-2),
    ("C2s", "ln_bwd", 8192, 1024, "f32", 1000.0, 1e-2),
    ("C2s", "rms_fwd", 8192, 1024, "f32", 1000.0, 1e-2),
    ("C2s", "rms_bwd", 8192, 1024, "f32", 1000.0, 1e-2),
    ("C3", "fused_fwd", 16384, 4096, "bf16", 0.0, 1.0),
    ("C4", "ln_bwd", 32768, 1024, "bf16", 0.0, 1.0),
    ("C4", "rms_bwd", 32768, 1024, "bf16", 0.0, 1.0),
    ("C4", "ln_bwd", 16384, 2048, "bf16", 0.0, 1.0),
    ("C4", "rms_bwd", 16384, 2048, "bf16", 0.0, 1.0),
    ("C5", "ln_fwd", 2048, 16384, "bf16", 0.0, 1.0),
    ("C5", "rms_fwd", 2048, 16384, "bf16", 0.0, 1.0),
    ("C5", "ln_bwd", 2048, 16384, "bf16", 0.0, 1.0),
    ("C5", "rms_bwd", 2048, 16384, "bf16", 0.0, 1.0),
    ("C5", "ln_fwd", 512, 16384, "bf16", 0.0, 1.0),
    ("C5", "rms_fwd", 512, 16384, "bf16", 0.0, 1.0),
    ("C5", "ln_bwd", 512, 16384, "bf16", 0.0, 1.0),
    ("C5", "rms_bwd", 512, 16384, "bf16", 0.0, 1.0),
]


def time_call(s, op, stream, flush, iters, split=False):
    """Per-call device µs of `op` on shape `s`: L2 flushed before each call,
    CUDA events on the launching stream.  With split, the backward's main
    kernel and its partial reduction are timed apart (an event recorded
    between them by the library; the reduction then runs as an ordinary
    launch instead of a programmatic dependent one)."""
    import ctypes
    import torch
    sh = stream.cuda_stream
    if op in FORWARD_OF:
        s.call(FORWARD_OF[op], sh)
    for _ in range(3):
        flush()
        s.call(op, sh)
    ev = []
    for _ in range(iters):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        s.call(op, sh)
        b.record(stream)
        ev.append((a, b))
    torch.cuda.synchronize()
    us = [a.elapsed_time(b) * 1e3 for a, b in ev]
    out = {"us_mean": round(statistics.fmean(us), 2), "us_median": round(statistics.median(us), 2),
           "us_min": round(min(us), 2)}
    if split:
        sp = []
        for _ in range(iters):
            flush()
            a, m, b = (torch.cuda.Event(enable_timing=True) for _ in range(3))
            m.record(stream)  # creates the event's handle; the library records it again
            a.record(stream)
            s.lib.norm_set_bwd_split_event(ctypes.c_void_p(m.cuda_event))
            s.call(op, sh)
            b.record(stream)
            sp.append((a, m, b))
        s.lib.norm_set_bwd_split_event(None)
        torch.cuda.synchronize()
        out["main_us_mean"] = round(statistics.fmean(a.elapsed_time(m) * 1e3 for a, m, _ in sp), 2)
        out["reduce_us_mean"] = round(statistics.fmean(m.elapsed_time(b) * 1e3 for _, m, b in sp), 2)
        out["split_note"] = "main + reduce timed apart, the reduction launched without PDL"
    return out


def run_configs(lib, dev, stream, flush, peak, iters):
    import torch
    out = {}
    cache = {}
    for cfg, op, N, H, dt, off, scale in CONFIGS:
        key = (N, H, dt, off, scale)
        if key not in cache:
            cache.clear()
            torch.cuda.empty_cache()
            cache[key] = Shape(N, H, dev, seed=11, lib=lib, dtype=dt, x_offset=off, x_scale=scale)
        s = cache[key]
        r = time_call(s, op, stream, flush, iters, split="bwd" in op)
        byts = alg_bytes(op, N, H, s.esize, s.esize)
        gbs = byts / (r["us_mean"] * 1e-6) / 1e9
        r.update({"config": cfg, "op": op, "N": N, "H": H, "dtype": dt, "bytes": byts, "gbs": round(gbs, 1),
                  "frac": round(gbs / peak, 3), "launches": LAUNCHES[op]})
        if off:
            r["x"] = f"{off:g} + {scale:g}*N(0,1)"
        out[f"{cfg}_{op}_{dt}_{N}x{H}"] = r
    cache.clear()
    torch.cuda.empty_cache()
    return out


def step_calls(shapes):
    return [(s, op) for s in shapes for op in OPS]


def aggregate(step_ms, step_bytes, world, dist=None, device=None):
    """(max step time over ranks, whole-job GB/s).  Every rank runs an
    independent replica of the same step (rows are independent; nothing is
    exchanged), so the job moves world * step_bytes in the slowest rank's time."""
    import torch
    t = torch.tensor([float(step_ms)], dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    ms = float(t.item())
    return ms, world * step_bytes / (ms * 1e-3) / 1e9


def run_ours(args):
    import torch
    import torch.distributed as dist

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    from rmsnorm_ln_fwd_gb300 import _build
    _build.build()
    import rmsnorm_ln_fwd_gb300 as nl
    lib = nl.load_library()
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    shapes = [Shape(N, H, dev, seed=rank * 100 + i, lib=lib) for i, (N, H) in enumerate(SHAPES)]
    calls = step_calls(shapes)
    flush = L2Flush(dev)

    for _ in range(args.warmup):
        for s, op in calls:
            flush()
            s.call(op, sh)
    torch.cuda.synchronize()

    n = len(calls)
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
          for _ in range(args.steps)]
    sampler = ClockSampler(dev.index)
    sampler.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    for k in range(args.steps):
        for i, (s, op) in enumerate(calls):
            flush()
            ev[k][i][0].record(stream)
            s.call(op, sh)
            ev[k][i][1].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t_wall
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()

    per_call = [[ev[k][i][0].elapsed_time(ev[k][i][1]) for k in range(args.steps)] for i in range(n)]
    step_ms = sum(sum(c) for c in per_call) / args.steps
    step_bytes = sum(s.bytes[op] for s, op in calls)
    step_ms_max, value = aggregate(step_ms, step_bytes, world, dist, dev)

    peak, peak_kind = measured_peak()
    breakdown = {}
    for i, (s, op) in enumerate(calls):
        us = statistics.median(per_call[i]) * 1e3
        mean_us = statistics.fmean(per_call[i]) * 1e3
        gbs = s.bytes[op] / (mean_us * 1e-6) / 1e9
        breakdown[f"{op}_{s.N}x{s.H}"] = {"us_median": round(us, 2), "us_mean": round(mean_us, 2),
                                          "us_min": round(min(per_call[i]) * 1e3, 2),
                                          "gbs": round(gbs, 1), "frac": round(gbs / peak, 3),
                                          "bytes": s.bytes[op], "launches": LAUNCHES[op]}
    # the call with the largest share of the step
    dom_i = max(range(n), key=lambda i: sum(per_call[i]))
    ds, dop = calls[dom_i]
    dkey = f"{dop}_{ds.N}x{ds.H}"
    d_us = statistics.fmean(per_call[dom_i]) * 1e3
    achieved = ds.bytes[dop] / (d_us * 1e-6) / 1e9
    traffic = recorded_traffic(dkey)

    e2e = run_e2e(args, shapes, stream, dev, world, dist)
    configs = run_configs(lib, dev, stream, flush, peak, args.config_iters) if args.config_iters > 0 else None
    out = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(step_ms_max, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "rows": 8192, "widths": [1024, 5120],
                   "calls_per_step": [op for op in OPS],
                   "l2": flush.describe(),
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "frac_of_peak": round(value / world / peak, 3),
        "peak_gbs": peak,
        "peak_kind": peak_kind,
        "bwd_us": bwd_us(breakdown, configs),
        "breakdown": breakdown,
        "roofline": {"bound": "hbm", "kernel": dkey + (" (main + partial-reduce kernels)" if "bwd" in dop else ""),
                     "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 3), "traffic": traffic,
                     "algorithmic_bytes": ds.bytes[dop], "peak_kind": f"{peak_kind} (hbm_gbs copy)"},
        "configs": configs,
        "clocks": clocks,
        "e2e": e2e,
        "gpu_launches": args.steps * sum(LAUNCHES[op] for _, op in calls),
        "wall_s_timed_region": round(wall, 3),
    }
    if rank == 0:
        out["cpu_baseline"] = cpu_baseline(args)
        print(json.dumps(out), flush=True)
    if world > 1:
        dist.destroy_process_group()


def bwd_us(breakdown, configs):
    """Backward µs (mean) per bf16 shape: the step's calls, then every bf16
    backward of the configurations, with the main/reduce split where timed."""
    out = {k.replace("_bwd", ""): {"us": v["us_mean"]} for k, v in breakdown.items() if "_bwd_" in k}
    for k, v in (configs or {}).items():
        if v["dtype"] == "bf16" and "_bwd" in v["op"]:
            e = out.setdefault(f"{v['op'].replace('_bwd', '')}_{v['N']}x{v['H']}", {"us": v["us_mean"]})
            e["main_us"], e["reduce_us"] = v["main_us_mean"], v["reduce_us_mean"]
    return out


OUT_NAMES = ("y", "mean", "rstd", "dx", "dg", "db", "yr", "rstd_r", "dxr", "dgr", "yf", "h", "rstd_f")


def run_e2e(args, shapes, stream, dev, world, dist):
    """The same step through the C ABI with host buffers: every step copies its
    inputs from pinned host memory to the device, runs the ten calls and copies
    every output back to pinned host memory, all inside the timed region (no L2
    flush: the copies are the traffic).  Copies overlap compute the way a
    caller would arrange it: inputs stream in on one copy stream, outputs
    stream out on another, and each width has two device buffer sets so step
    k+1's uploads and step k's downloads run while the other set computes."""
    import torch
    lib = shapes[0].lib
    slots = [[s, Shape(s.N, s.H, dev, seed=0, lib=lib)] for s in shapes]
    hin = [{k: v.pin_memory() for k, v in pair[0].host.items()} for pair in slots]
    hout = [{n: torch.empty(getattr(pair[0], n).shape, dtype=getattr(pair[0], n).dtype, pin_memory=True)
             for n in OUT_NAMES} for pair in slots]
    h2d = sum(v.numel() * v.element_size() for d in hin for v in d.values())
    d2h = sum(v.numel() * v.element_size() for d in hout for v in d.values())
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()  # noqa: E731
    # per width and buffer set: inputs landed, compute done, downloads done
    landed = [[ev(), ev()] for _ in slots]
    computed = [[ev(), ev()] for _ in slots]
    drained = [[None, None] for _ in slots]
    freed = [[None, None] for _ in slots]

    def one_step(k):
        b = k % 2
        for i, pair in enumerate(slots):
            s = pair[b]
            with torch.cuda.stream(s_in):
                if freed[i][b] is not None:
                    s_in.wait_event(freed[i][b])  # the calls that read this set are done
                for name, src in hin[i].items():
                    s.t[name].copy_(src, non_blocking=True)
                landed[i][b].record(s_in)
            stream.wait_event(landed[i][b])
            if drained[i][b] is not None:
                stream.wait_event(drained[i][b])  # the last downloads from this set are done
            for op in OPS:
                s.call(op, stream.cuda_stream)
            computed[i][b].record(stream)
            freed[i][b] = computed[i][b]
            with torch.cuda.stream(s_out):
                s_out.wait_event(computed[i][b])
                for name in OUT_NAMES:
                    hout[i][name].copy_(getattr(s, name), non_blocking=True)
                e = ev()
                e.record(s_out)
                drained[i][b] = e

    for k in range(max(1, args.warmup)):
        one_step(k)
    torch.cuda.synchronize()
    e2e_steps = max(1, min(args.steps, args.e2e_steps))
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    s_in.wait_event(a)
    s_out.wait_event(a)
    for k in range(e2e_steps):
        one_step(k)
    stream.wait_stream(s_in)
    stream.wait_stream(s_out)
    z.record(stream)
    torch.cuda.synchronize()
    step_bytes = sum(s.bytes[op] for s in shapes for op in OPS)
    ms, gbs = aggregate(a.elapsed_time(z) / e2e_steps, step_bytes, world, dist, dev)
    return {"value": round(gbs, 1), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(ms, 4),
            "steps": e2e_steps, "how": "C ABI calls; pinned host buffers; uploads, compute and downloads on three "
                                      "streams, two device buffer sets per width"}


# ---------------------------------------------------------------------------
# the CPU oracle: baseline and reference arm
# ---------------------------------------------------------------------------

def oracle_step(samples):
    import oracle as O
    for x, dy, res, g, b in samples:
        O.layer_norm_forward(x, g, b, EPS)
        O.layer_norm_backward(dy, x, g, EPS)
        O.rms_norm_forward(x, g, EPS)
        O.rms_norm_backward(dy, x, g, EPS)
        O.fused_add_rms_norm_forward(x, res, g, EPS_FUSED, "bfloat16")


def oracle_samples(rows, seed=0):
    from rmsnorm_ln_fwd_gb300 import synth
    out = []
    for i, (N, H) in enumerate(SHAPES):
        c = synth.norm_inputs(rows, H, "bf16", seed=seed * len(SHAPES) + i, with_residual=True)
        f = {k: v.double().numpy() for k, v in c.items()}
        out.append((f["x"], f["dy"], f["residual"], f["gamma"], f["beta"]))
    return out


def sample_bytes(rows):
    return sum(alg_bytes(op, rows, H) for _, H in SHAPES for op in OPS)


def _cpu_worker(rows, target_s, seed):
    """Repeat the oracle over one row sample for target_s seconds -> (reps, s)."""
    samples = oracle_samples(rows, seed)
    t0 = time.perf_counter()
    reps = 0
    while True:
        oracle_step(samples)
        reps += 1
        if time.perf_counter() - t0 >= target_s:
            break
    return reps, time.perf_counter() - t0


def cpu_baseline(args, target_s=None):
    """The oracle as it stands, on one core and then on every host core (one
    process per core, each on its own row sample; spawned, never forked after
    CUDA is up).  The JSON value is the all-core figure."""
    import multiprocessing as mp
    target_s = args.cpu_seconds if target_s is None else target_s
    rows = args.cpu_rows
    reps, dt = _cpu_worker(rows, target_s, 0)
    single = reps * sample_bytes(rows) / dt / 1e9
    cores = os.cpu_count() or 1
    with mp.get_context("spawn").Pool(cores) as pool:
        res = pool.starmap(_cpu_worker, [(rows, target_s, i) for i in range(cores)])
    multi = sum(r / t for r, t in res) * sample_bytes(rows) / 1e9
    return {"value": round(multi, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{rows} of 8192 rows per width, all 10 calls, repeated for {target_s:.0f} s in each of "
                      f"{cores} processes (one per core, own sample each); numpy fp64",
            "single_core": {"value": round(single, 4), "unit": "GB/s", "cores": 1,
                            "sample": f"the same loop in one process: {reps} repetitions in {dt:.1f} s"}}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    rows = args.ref_rows
    samples = oracle_samples(rows)
    for _ in range(args.warmup):
        oracle_step(samples)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(samples)
    dt = time.perf_counter() - t0
    step_ms = dt / args.steps * 1e3
    gbs = sample_bytes(rows) / (step_ms * 1e-3) / 1e9
    sample = f"{rows} of 8192 rows per width per step, all 10 calls, numpy fp64 single-threaded"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_ms, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "rows_per_step": rows, "widths": [1024, 5120]},
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


# ---------------------------------------------------------------------------
# extra modes: per-config sweep and a single-call loop for profilers
# ---------------------------------------------------------------------------

SWEEP = [("ln_fwd", 8192, 1024), ("rms_fwd", 8192, 1024), ("ln_bwd", 8192, 1024), ("rms_bwd", 8192, 1024),
         ("ln_fwd", 8192, 5120), ("rms_fwd", 8192, 5120), ("ln_bwd", 8192, 5120), ("rms_bwd", 8192, 5120),
         ("fused_fwd", 16384, 4096), ("ln_bwd", 32768, 1024), ("rms_bwd", 32768, 1024), ("ln_bwd", 16384, 2048),
         ("rms_bwd", 16384, 2048), ("ln_fwd", 2048, 16384), ("rms_fwd", 2048, 16384), ("ln_bwd", 2048, 16384),
         ("rms_bwd", 2048, 16384), ("ln_fwd", 512, 16384), ("rms_fwd", 512, 16384), ("ln_bwd", 512, 16384),
         ("rms_bwd", 512, 16384), ("fused_bwd", 8192, 1024), ("fused_bwd", 8192, 5120), ("fused_bwd", 16384, 4096),
         ("ln_bwd_y", 8192, 1024), ("ln_bwd_y", 8192, 5120), ("rms_bwd_y", 8192, 1024), ("rms_bwd_y", 8192, 5120),
         # the backward shapes "Rewrite Triton normalization backward kernel_1 (#499)" times (Results table)
         ("ln_bwd", 1024, 8192), ("ln_bwd", 2048, 4096), ("ln_bwd", 16384, 1024), ("ln_bwd", 4096, 4096),
         ("ln_bwd", 8192, 4096), ("rms_bwd", 4096, 4096), ("rms_bwd", 2048, 4096), ("rms_bwd", 16384, 1024),
         # in place over x (last: it rewrites the shape's x on every call)
         ("fused_fwd_ip", 16384, 4096)]

FORWARD_OF = {"ln_bwd": "ln_fwd", "rms_bwd": "rms_fwd", "fused_bwd": "fused_fwd", "ln_bwd_y": "ln_fwd",
              "rms_bwd_y": "rms_fwd"}


def run_sweep(args):
    import torch
    from rmsnorm_ln_fwd_gb300 import _build
    _build.build()
    import rmsnorm_ln_fwd_gb300 as nl
    lib = nl.load_library()
    nl._lib.set_kernel_path(args.path)
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    peak, kind = measured_peak()
    flush = L2Flush(dev)
    cache = {}
    for op, N, H in SWEEP:
        if (N, H) not in cache:
            cache.clear()
            torch.cuda.empty_cache()
            cache[(N, H)] = Shape(N, H, dev, seed=7, lib=lib, extra=True, dtype=args.dtype)
        s = cache[(N, H)]
        if op in FORWARD_OF:
            s.call(FORWARD_OF[op], stream.cuda_stream)
        for _ in range(5):
            flush()
            s.call(op, stream.cuda_stream)
        ts = []
        for _ in range(args.sweep_iters):
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            s.call(op, stream.cuda_stream)
            b.record(stream)
            ts.append((a, b))
        torch.cuda.synchronize()
        us = [a.elapsed_time(b) * 1e3 for a, b in ts]
        byts = s.bytes.get(op) or alg_bytes(op, N, H, s.esize, s.esize)
        med = statistics.median(us)
        print(json.dumps({"op": op, "N": N, "H": H, "dtype": args.dtype, "path": args.path, "us_median": round(med, 2),
                          "us_min": round(min(us), 2),
                          "gbs": round(byts / (med * 1e-6) / 1e9, 1), "frac": round(byts / (med * 1e-6) / 1e9 / peak, 3),
                          "bytes": byts, "peak": peak, "peak_kind": kind}), flush=True)


def run_profile_loop(args):
    """Run one call `--iters` times (after one untimed forward for a backward):
    a small, self-terminating target for ncu captures."""
    import torch
    from rmsnorm_ln_fwd_gb300 import _build
    _build.build()
    import rmsnorm_ln_fwd_gb300 as nl
    lib = nl.load_library()
    nl._lib.set_kernel_path(args.path)
    N, H = (int(v) for v in args.shape.split("x"))
    dev = torch.device("cuda", 0)
    s = Shape(N, H, dev, seed=3, lib=lib, extra=True, dtype=args.dtype)
    sh = torch.cuda.current_stream(dev).cuda_stream
    op = args.profile_op
    if op in FORWARD_OF:
        s.call(FORWARD_OF[op], sh)
    for _ in range(args.iters):
        s.call(op, sh)
    torch.cuda.synchronize()
    print(json.dumps({"profiled": op, "N": N, "H": H, "iters": args.iters}))


def run_calibrate(args):
    """Reference points for the per-call numbers, under the same flush and
    events: an almost empty kernel (the floor of an event-timed call), plain
    device copies moving the bytes of the step's calls, back-to-back copies
    over rotating buffers, and the host link (pinned host memory)."""
    import torch
    from rmsnorm_ln_fwd_gb300 import _build
    _build.build()
    import rmsnorm_ln_fwd_gb300 as nl
    lib = nl.load_library()
    dev = torch.device("cuda", 0)
    st = torch.cuda.current_stream(dev)
    flush = L2Flush(dev)
    peak, kind = measured_peak()

    def timed(fn, iters=60, do_flush=True):
        for _ in range(5):
            if do_flush:
                flush()
            fn()
        ev = []
        for _ in range(iters):
            if do_flush:
                flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(st)
            fn()
            b.record(st)
            ev.append((a, b))
        torch.cuda.synchronize()
        us = [a.elapsed_time(b) * 1e3 for a, b in ev]
        return round(statistics.fmean(us), 2), round(min(us), 2)

    def emit(**kw):
        print(json.dumps(kw), flush=True)

    tiny = torch.zeros(1, device=dev)
    m, mn = timed(lambda: tiny.add_(1))
    emit(what="torch add on one element (the floor of an event-timed call)", us_mean=m, us_min=mn)
    one = Shape(1, 256, dev, seed=0, lib=lib)
    m, mn = timed(lambda: one.call("rms_fwd", st.cuda_stream))
    emit(what="rms_forward on one row of 256 (one CTA)", us_mean=m, us_min=mn)
    del one
    for mib in (8, 16, 32, 40, 64, 80, 128, 256):
        n = mib * (1 << 20) // 2
        src = torch.ones(n, dtype=torch.bfloat16, device=dev)
        dst = torch.empty_like(src)
        m, mn = timed(lambda: dst.copy_(src))
        byts = 4 * n
        emit(what=f"device copy {mib} MiB -> {mib} MiB", bytes=byts, us_mean=m, us_min=mn,
             gbs=round(byts / (m * 1e-6) / 1e9, 1), frac=round(byts / (m * 1e-6) / 1e9 / peak, 3))
        del src, dst
    n = 16 * (1 << 20) // 2
    bufs = [(torch.ones(n, dtype=torch.bfloat16, device=dev), torch.empty(n, dtype=torch.bfloat16, device=dev))
            for _ in range(16)]  # 512 MiB in all: every copy reads buffers L2 no longer holds
    reps = 4
    for _ in range(2):
        for a_, b_ in bufs:
            b_.copy_(a_)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    flush()
    a.record(st)
    for _ in range(reps):
        for a_, b_ in bufs:
            b_.copy_(a_)
    b.record(st)
    torch.cuda.synchronize()
    per = a.elapsed_time(b) * 1e3 / (reps * len(bufs))
    emit(what="device copy 16 MiB -> 16 MiB, 64 copies back to back over 16 buffer pairs", us_per_copy=round(per, 2),
         frac=round(4 * n / (per * 1e-6) / 1e9 / peak, 3))
    del bufs
    n = 1 << 30
    h = torch.empty(n, dtype=torch.uint8, pin_memory=True)
    h2 = torch.empty(n, dtype=torch.uint8, pin_memory=True)
    d = torch.empty(n, dtype=torch.uint8, device=dev)
    d2 = torch.empty(n, dtype=torch.uint8, device=dev)
    m, _ = timed(lambda: d.copy_(h, non_blocking=True), iters=5, do_flush=False)
    emit(what="host -> device, 1 GiB from pinned memory", gbs=round(n / (m * 1e-6) / 1e9, 1), us_mean=m)
    m, _ = timed(lambda: h.copy_(d, non_blocking=True), iters=5, do_flush=False)
    emit(what="device -> host, 1 GiB to pinned memory", gbs=round(n / (m * 1e-6) / 1e9, 1), us_mean=m)
    s2 = torch.cuda.Stream(dev)

    def both():
        ev0 = torch.cuda.Event()
        ev0.record(st)
        s2.wait_event(ev0)
        d.copy_(h, non_blocking=True)
        with torch.cuda.stream(s2):
            h2.copy_(d2, non_blocking=True)
        st.wait_stream(s2)
    m, _ = timed(both, iters=5, do_flush=False)
    emit(what="both directions at once, 1 GiB each", gbs_each=round(n / (m * 1e-6) / 1e9, 1), us_mean=m)
    emit(what="peak", hbm_gbs=peak, kind=kind)


def main():
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=300)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--e2e-steps", type=int, default=50)
    p.add_argument("--config-iters", type=int, default=50,
                   help="timed calls per configuration call after the step (0: skip the configs object)")
    p.add_argument("--cpu-rows", type=int, default=512)
    p.add_argument("--cpu-seconds", type=float, default=10.0)
    p.add_argument("--ref-rows", type=int, default=64)
    p.add_argument("--sweep", action="store_true", help="per-call timings over every configured shape")
    p.add_argument("--record-traffic", nargs="+", default=None, metavar="CSV",
                   help="write the per-call DRAM traffic table from ncu captures named traffic_<op>_<N>x<H>.csv")
    p.add_argument("--traffic-out", default=os.path.join(ROOT, "profiles", "roofline_traffic.txt"))
    p.add_argument("--calibrate", action="store_true",
                   help="reference points: event floor, plain device copies, host link")
    p.add_argument("--sweep-iters", type=int, default=50)
    p.add_argument("--dtype", choices=["bf16", "f16", "f32"], default="bf16",
                   help="row dtype of --sweep / --profile-op (the step itself is bf16)")
    p.add_argument("--path", type=int, default=0, help="kernel-family policy: 0 auto, 1 register rows, 2 loop, 3 bulk-copy pipeline")
    p.add_argument("--profile-op", choices=list(OPS + EXTRA_OPS), default=None)
    p.add_argument("--shape", default="8192x1024")
    p.add_argument("--iters", type=int, default=3)
    args = p.parse_args()
    if args.impl == "ours" and not (args.sweep or args.profile_op):
        args.warmup = max(args.warmup, 3)  # at least three untimed warm-up steps
    if args.record_traffic:
        print(json.dumps(record_traffic(args.record_traffic, args.traffic_out)))
    elif args.impl == "reference":
        run_reference(args)
    elif args.sweep:
        run_sweep(args)
    elif args.calibrate:
        run_calibrate(args)
    elif args.profile_op:
        run_profile_loop(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
