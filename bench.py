#!/usr/bin/env python3
"""Benchmark: dense GEMM throughput (TFLOP/s = 2MNK / t) on one GB300.

One step is one pass of the whole hot path: an fp32 product at n = 3072 on the
SIMT kernel (gemm_f32) and a bf16-input / fp32-accumulate product at
8192^3 on the tcgen05 kernel (gemm_bf16_f32acc), on seeded synthetic inputs
already resident in HBM. `value` = total FLOPs of the K timed steps / their
device time (CUDA events on the launching stream). Each kernel's own time is
taken with events around it and reported in `parts` with its roofline.

Inputs rotate over several copies whose total size exceeds the 129 MB L2, so
no timed launch finds its operands in L2 from the previous step.

`e2e` is the same metric through the public tensor API with HOST tensors: the
host->device copy of A and B and the device->host copy of C are inside the
timed region.

    python bench.py [--gpus N --steps K --warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs the same step on its own GPU
(replicas); value = FLOPs of all ranks / max time over ranks.
`--impl reference` times the CPU oracle on the host cores on a bounded sample
of the same workload.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GEMM TFLOP/s (2MNK/t) fp32 n=3072 and bf16 8192³; % of GB300 peak"
UNIT = "TFLOP/s"
L2_BYTES = 129 * 1024 * 1024
WORKLOAD_NAME = "fp32 3072^3 (gemm_f32) + bf16->fp32 8192^3 (gemm_bf16_f32acc), one of each per step"

# (workload name, kernel, roofline bound, C-ABI entry name, kernel source file).
# The entry points are the workspace (stream-K) variants; a workspace is
# allocated once, outside the timed region, where the product uses one.
PARTS = [
    ("f32_3072", "sgemm_simt_kernel", "alu", "gemm_f32_ws", "sgemm_simt.cu"),
    ("bf16_8192", "hgemm_tc2_kernel", "tensor", "gemm_bf16_f32acc_ws", "hgemm_tc2.cu"),
]


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sustained-s", type=float, default=1.5,
                    help="seconds of the sustained leg (back-to-back steps with their own "
                         "clock record; 0: skip)")
    ap.add_argument("--cpu-1t-seconds", type=float, default=3.0,
                    help="target single-thread oracle seconds per fp32 config (1-3) "
                         "in cpu_baseline (0: skip)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target oracle seconds per part for cpu_baseline")
    ap.add_argument("--only", choices=[p[0] for p in PARTS], default=None,
                    help="time one part only (for profiling; not a bench line)")
    ap.add_argument("--table", action="store_true",
                    help="time every named workload alone and print one JSON line per workload "
                         "(the parity workloads' speeds; not the bench line)")
    ap.add_argument("--table-tf32", action="store_true",
                    help="time fp32 inputs in every arithmetic (FFMA, TF32, 3xTF32) at 3072^3 "
                         "and 8192^3, one JSON line each")
    ap.add_argument("--table-only", default=None, metavar="WORKLOAD",
                    help="with --table: one named workload (for profiling)")
    ap.add_argument("--tf32-only", default=None, metavar="SHAPE:MODE",
                    help="with --table-tf32: one shape (f32_3072 or f32_8192) and one mode "
                         "(fp32, tf32 or 3xtf32), e.g. f32_3072:3xtf32 (for profiling)")
    ap.add_argument("--tf32-plain", action="store_true",
                    help="with --table-tf32: call without a workspace (the plain entry "
                         "points: the fp32 kernel's own loader, the tf32 converter kernel)")
    ap.add_argument("--fma-ceiling", action="store_true",
                    help="measure the FFMA throughput a register-only loop reaches "
                         "(packed and scalar), one JSON line each (not the bench line)")
    ap.add_argument("--table-ex", action="store_true",
                    help="time the extended call (stored transposes, alpha/beta) on the fp32 "
                         "3072^3 and 16-bit 8192^3 workloads, one JSON line per variant")
    ap.add_argument("--table-soft", action="store_true",
                    help="time bf16 products whose operands TMA cannot read (odd pitches, "
                         "2-byte offsets) through the plain call, against the same kernel "
                         "on 16-byte pitches, one JSON line per shape")
    ap.add_argument("--soft-only", default=None, metavar="SHAPE",
                    help="with --table-soft: one shape, unaligned call only (for profiling)")
    return ap.parse_args()


# ------------------------------------------------------------------ distributed plumbing

class Dist:
    def __init__(self, n_gpus: int):
        import torch
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.n_gpus = n_gpus
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            backend = "nccl" if torch.cuda.is_available() else "gloo"
            if backend == "nccl":
                torch.cuda.set_device(self.local_rank)
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        import torch
        dev = "cuda" if torch.cuda.is_available() else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """SM clock, power and clock-event reasons of one GPU, sampled in a thread
    every `period_s` while a timed region runs (start() just before its first
    launch, stop() just after its last event), read through NVML (the driver's
    libnvidia-ml, read-only queries). Where NVML cannot be loaded, nvidia-smi
    is sampled at its fastest period instead."""

    # clock-event reason bits of NVML's public header
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}
    SMI_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                  "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                  "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int, period_s: float = 0.002):
        self.dev = device_index
        self.period = period_s
        self.samples = []  # (sm_mhz, power_w, reason bits)
        self.sm_max = None
        self.source = None
        self._nvml = None
        self._handle = None
        self._thread = None
        self._stop = None
        self._proc = None
        self._open_nvml()

    def _open_nvml(self):
        import ctypes
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                return
            h = ctypes.c_void_p()
            uuid = None
            try:
                import torch
                uuid = str(torch.cuda.get_device_properties(self.dev).uuid)
            except Exception:
                uuid = None
            ok = False
            if uuid:
                ok = nv.nvmlDeviceGetHandleByUUID(f"GPU-{uuid}".encode(), ctypes.byref(h)) == 0
            if not ok and nv.nvmlDeviceGetHandleByIndex_v2(self.dev, ctypes.byref(h)) != 0:
                return
            mx = ctypes.c_uint(0)
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:  # 1: SM clock
                self.sm_max = float(mx.value)
            # the reasons query under its current name, else its older one
            self._reasons_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(nv, "nvmlDeviceGetCurrentClocksThrottleReasons")
            self._nvml, self._handle = nv, h
            self.source = "nvml"
        except (OSError, AttributeError):
            self._nvml = None

    def _sample_nvml(self):
        import ctypes
        nv, h = self._nvml, self._handle
        mhz, mw, why = ctypes.c_uint(0), ctypes.c_uint(0), ctypes.c_ulonglong(0)
        while not self._stop.is_set():
            if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(mhz)) == 0:
                nv.nvmlDeviceGetPowerUsage(h, ctypes.byref(mw))
                self._reasons_fn(h, ctypes.byref(why))
                self.samples.append((float(mhz.value), mw.value / 1e3, int(why.value)))
            self._stop.wait(self.period)

    def start(self):
        import threading
        self.samples = []
        if self._nvml is not None:
            self._stop = threading.Event()
            self._thread = threading.Thread(target=self._sample_nvml, daemon=True)
            self._thread.start()
            return
        try:
            self._out = open(self._path(), "w")
            self._proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.SMI_FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "10", "-i", str(self.dev)], stdout=self._out, stderr=subprocess.DEVNULL)
            self.source = "nvidia-smi"
        except (OSError, FileNotFoundError):
            self._proc = None

    def _path(self):
        import tempfile
        return os.path.join(tempfile.gettempdir(), f"gemm14_clocks_{os.getpid()}_{self.dev}.csv")

    def stop(self) -> dict:
        if self._thread is not None:
            self._stop.set()
            self._thread.join()
            self._thread = None
        elif self._proc is not None:
            self._proc.terminate()
            try:
                self._proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self._proc.kill()
            self._out.close()
            self._proc = None
            names = {5: 0x8, 6: 0x40, 7: 0x20, 8: 0x4}
            with open(self._path()) as f:
                for line in f:
                    cols = [c.strip() for c in line.split(",")]
                    if len(cols) < 9:
                        continue
                    try:
                        sm, smax = float(cols[1]), float(cols[2])
                        pw = float(cols[3]) if cols[3].replace(".", "", 1).isdigit() else 0.0
                    except ValueError:
                        continue
                    bits = sum(b for i, b in names.items() if cols[i].lower().startswith("active"))
                    self.samples.append((sm, pw, bits))
                    self.sm_max = max(self.sm_max or 0.0, smax)
        return self.summary()

    def summary(self) -> dict:
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.sm_max, "reasons": ["no samples"],
                    "samples": 0, "source": self.source}
        sm = [x[0] for x in self.samples]
        counts = {name: sum(1 for x in self.samples if x[2] & bit)
                  for bit, name in self.REASONS.items()}
        return {"sm_mhz": statistics.median(sm), "sm_min_mhz": min(sm), "sm_max_mhz": self.sm_max,
                "reasons": sorted(n for n, c in counts.items() if c),
                "reason_samples": {n: c for n, c in counts.items() if c},
                "power_w_max": max(x[1] for x in self.samples),
                "samples": len(sm), "period_ms": self.period * 1e3, "source": self.source}


# ------------------------------------------------------------------ helpers

def source_sha(fname: str) -> str:
    h = hashlib.sha256()
    for f in (fname, "ptx.cuh", "kernels.h"):
        with open(os.path.join(ROOT, "dense_gemm_14_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_for(kernel: str, src: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, only if it was taken
    on the current source of the kernel (else null)."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    e = d.get(kernel)
    if not e or e.get("source_sha") != source_sha(src) or e.get("workload") != workload:
        return None
    return e.get("dram_bytes_per_launch")


def workload_info(name):
    from dense_gemm_14_gb300 import inputs, roofline
    w = inputs.WORKLOADS[name]
    in_b = 4 if w.dtype == "f32" else 2
    return w, roofline.flops(w.M, w.N, w.K), roofline.ideal_bytes(w.M, w.N, w.K, in_b, 4)


# ------------------------------------------------------------------ CPU oracle timing

def time_oracle_sample(name: str, target_s: float, A=None, B=None, want_rows=False,
                       threads: int = 0):
    """Times the oracle on the first R rows of the named product, R sized so
    the call takes about target_s seconds, on `threads` threads (0: all the
    host's). Returns (flops, seconds, rows, threads), and with want_rows also
    the oracle's R x N rows (float64)."""
    import oracle
    from dense_gemm_14_gb300 import inputs, roofline
    w = inputs.WORKLOADS[name]
    if A is None:
        A, B = inputs.make_workload(name)
    Ah, Bh = inputs.host_view(A), inputs.host_view(B)
    M, (K, N) = Ah.shape[0], Bh.shape
    # two probes: 32 rows (whose time is mostly start-up), then about half a
    # second's worth, from which the sample's rows are sized
    rows = min(M, 32)
    for probe_s in (0.5, target_s):
        t0 = time.perf_counter()
        oracle.gemm(Ah[:rows], Bh, w.dtype, threads=threads, with_abs=False)
        probe = time.perf_counter() - t0
        rows = int(max(1, min(M, rows * min(probe_s, target_s) / max(probe, 1e-6))))
    t0 = time.perf_counter()
    ref, _ = oracle.gemm(Ah[:rows], Bh, w.dtype, threads=threads, with_abs=False)
    dt = time.perf_counter() - t0
    out = (roofline.flops(rows, N, K), dt, rows, threads or oracle.max_threads())
    return out + (ref,) if want_rows else out


# The element-wise bounds the parity tests hold the products to:
# |C - C_ref| <= bound * (|A| |B|) element by element.
ELEMENT_BOUND = {"f32": 1e-5, "bf16": 4e-3}


def accuracy_of(name, A, B, C_dev, ref_rows, abs_rows=16):
    """The GPU product's first rows against the oracle: relative RMSE
    ||C - C_ref||_2 / ||C_ref||_2 over the rows the oracle timing computed,
    and the largest |C - C_ref| / (|A| |B|) over the first abs_rows rows
    (its bound beside it)."""
    import numpy as np

    import oracle
    from dense_gemm_14_gb300 import inputs
    w = inputs.WORKLOADS[name]
    r = ref_rows.shape[0]
    got = C_dev[:r].double().cpu().numpy()
    rmse = float(np.linalg.norm(got - ref_rows) / max(np.linalg.norm(ref_rows), 1e-300))
    ra = min(abs_rows, r)
    Ah, Bh = inputs.host_view(A), inputs.host_view(B)
    ref, refabs = oracle.gemm(np.ascontiguousarray(Ah[:ra]), Bh, w.dtype, with_abs=True)
    ok, worst = oracle.within_bound(got[:ra], ref, refabs, ELEMENT_BOUND[w.dtype])
    return {"workload": name, "rows_rmse": r, "rel_rmse": rmse, "rows_bound": ra,
            "max_err_over_abs": worst, "bound": ELEMENT_BOUND[w.dtype], "within": ok}


def run_reference(args, dist: Dist, data=None):
    """The oracle arm: the CPU oracle on host cores, a bounded sample per step.
    Under torchrun only rank 0 works and prints; `data` overrides the inputs."""
    if dist.rank != 0:
        return None
    import oracle
    from dense_gemm_14_gb300 import inputs
    oracle.build()
    if data is None:
        data = {name: inputs.make_workload(name) for name, *_ in PARTS}
    per_step_s = max(0.5, 120.0 / max(1, args.steps + args.warmup)) / len(PARTS)
    # calibrate rows per part once
    rows = {}
    for name, *_ in PARTS:
        _, dt, r, _ = time_oracle_sample(name, per_step_s, *data[name])
        rows[name] = r
    tot_f, tot_t = 0.0, 0.0
    for step in range(args.warmup + args.steps):
        for name, *_ in PARTS:
            w = inputs.WORKLOADS[name]
            A, B = data[name]
            r = rows[name]
            t0 = time.perf_counter()
            oracle.gemm(inputs.host_view(A)[:r], inputs.host_view(B), w.dtype, with_abs=False)
            dt = time.perf_counter() - t0
            if step >= args.warmup:
                tot_f += 2.0 * r * B.shape[1] * B.shape[0]
                tot_t += dt
    value = tot_f / tot_t / 1e12
    sample = ", ".join(f"first {rows[n]} rows of {n}" for n, *_ in PARTS) + " per step"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": tot_t / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD_NAME, "sample": sample},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.max_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return line


# ------------------------------------------------------------------ GPU arm

def run_ours(args, dist: Dist):
    import torch

    import dense_gemm_14_gb300 as g14
    from dense_gemm_14_gb300 import inputs, roofline

    g14.load()
    dev = torch.device("cuda", dist.local_rank if dist.world > 1 else 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    peaks = roofline.measured_peaks()

    entries = {"gemm_f32_ws": g14.gemm_f32_ws, "gemm_bf16_f32acc_ws": g14.gemm_bf16_f32acc_ws}
    codes = {"f32": g14.GEMM14_DTYPE_F32, "bf16": g14.GEMM14_DTYPE_BF16}
    parts = []
    host = {}
    for name, kernel, bound, entry, src in PARTS:
        if args.only and name != args.only:
            continue
        w, fl, ib = workload_info(name)
        A, B = inputs.make_workload(name)
        host[name] = (A, B)
        per_set = A.numel() * A.element_size() + B.numel() * B.element_size() + w.M * w.N * 4
        nsets = max(2, -(-2 * L2_BYTES // per_set))
        a0, b0 = A.to(dev), B.to(dev)
        sets = [(a0, b0, torch.empty(w.M, w.N, device=dev))]
        for _ in range(nsets - 1):
            sets.append((a0.clone(), b0.clone(), torch.empty(w.M, w.N, device=dev)))
        # the workspace the call asks for with these operands (stream-K region,
        # and copies of operands in a storage its kernel reads faster)
        a0, b0, c0 = sets[0]
        ws_bytes = g14.workspace_bytes_ex(codes[w.dtype], 0, 0, w.M, w.N, w.K, a0.data_ptr(), w.K,
                                          b0.data_ptr(), w.N, c0.data_ptr(), w.N)
        ws = torch.zeros(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
        # kernels one call launches: the product, and one copy kernel when the
        # workspace holds copies (asked for beyond the stream-K region)
        launches = 2 if ws_bytes > g14.workspace_bytes(codes[w.dtype], w.M, w.N, w.K, 0) else 1
        parts.append(dict(name=name, kernel=kernel, bound=bound, fn=entries[entry], src=src,
                          launches=launches,
                          w=w, flops=fl, ideal_bytes=ib, sets=sets, ws=ws, ws_bytes=ws_bytes,
                          entry=entry))

    def launch(p, step):
        a, b, c = p["sets"][step % len(p["sets"])]
        w = p["w"]
        p["fn"](w.M, w.N, w.K, a.data_ptr(), w.K, b.data_ptr(), w.N, c.data_ptr(), w.N,
                p["ws"].data_ptr(), p["ws_bytes"], stream.cuda_stream)

    # warm-up (also configures the kernels' shared-memory attributes)
    for step in range(args.warmup):
        for p in parts:
            launch(p, step)
    st = g14.check_device_error(stream.cuda_stream)
    if st:
        raise RuntimeError(f"device error during warm-up: {g14.status_string(st)}")

    K = args.steps
    ev = {p["name"]: ([torch.cuda.Event(enable_timing=True) for _ in range(K)],
                      [torch.cuda.Event(enable_timing=True) for _ in range(K)]) for p in parts}
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(dev.index)
    dist.barrier()
    torch.cuda.synchronize()
    # The value: K steps back to back between one pair of events, nothing in
    # between the kernels, so that each launch overlaps the end of the one
    # before it (the kernels wait for their predecessor on the device). The
    # clocks are sampled from just before the first launch to just after the
    # last event (every 2 ms).
    clocks.start()
    start.record(stream)
    for step in range(K):
        for p in parts:
            launch(p, step)
    end.record(stream)
    end.synchronize()
    clk = clocks.stop()
    # Each kernel's own duration (the roofline): the same K steps again with an
    # event pair around every kernel (which keeps consecutive kernels apart),
    # with a clock record of its own.
    clocks_parts = ClockSampler(dev.index)
    clocks_parts.start()
    for step in range(K):
        for p in parts:
            s_ev, e_ev = ev[p["name"]]
            s_ev[step].record(stream)
            launch(p, step)
            e_ev[step].record(stream)
    torch.cuda.synchronize()
    clk_parts = clocks_parts.stop()
    dist.barrier()
    st = g14.check_device_error(stream.cuda_stream)
    if st:
        raise RuntimeError(f"device error in the timed region: {g14.status_string(st)}")
    elapsed_s = start.elapsed_time(end) / 1e3
    elapsed_max = dist.max(elapsed_s)
    flops_step = sum(p["flops"] for p in parts)
    value = flops_step * K * dist.world / elapsed_max / 1e12

    # The SM clock the tensor-core part actually runs at. NVML reports the
    # clock the GPU targets, which under a dense tensor load can sit above
    # the one the SMs run at. A one-thread kernel that spins for a fixed
    # number of SM cycles (torch.cuda._sleep) is started on a second stream
    # together with each product; it shares an SM with the product's CTAs
    # (they leave room for it), so cycles / event time is the clock while the
    # product runs. Kept only when the spin ended before the product did.
    effective = {}
    for p in parts:
        if p["bound"] != "tensor":
            continue
        side = torch.cuda.Stream(dev)
        cycles = 200_000
        mhz = []
        for step in range(10):
            pre = torch.cuda.Event()
            pre.record(stream)
            g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            g0.record(stream)
            launch(p, step)
            g1.record(stream)
            side.wait_event(pre)
            with torch.cuda.stream(side):
                s0.record(side)
                torch.cuda._sleep(cycles)
                s1.record(side)
            torch.cuda.synchronize()
            spin_ms = s0.elapsed_time(s1)
            # the spin lies inside the product's run: it started after the
            # product's start event and ended before its end event
            if g0.elapsed_time(s0) >= 0 and s1.elapsed_time(g1) >= 0 and spin_ms > 0:
                mhz.append(cycles / (spin_ms * 1e3))
        effective[p["name"]] = {"sm_mhz_median": statistics.median(mhz) if mhz else None,
                                "samples": len(mhz), "method": "spin of 200000 SM cycles on a "
                                "second stream inside the product's run, 10 tries"}

    # A sustained leg: the same step back to back for about args.sustained_s
    # seconds (the clock settles under the power cap), one event pair, its own
    # clock record. Reported beside the value, not in it.
    sustained = None
    if args.sustained_s > 0:
        n_sus = max(1, int(args.sustained_s / max(elapsed_s / K, 1e-6)))
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        clocks_sus = ClockSampler(dev.index, period_s=0.005)
        torch.cuda.synchronize()
        clocks_sus.start()
        s0.record(stream)
        for step in range(n_sus):
            for p in parts:
                launch(p, step)
        s1.record(stream)
        s1.synchronize()
        clk_sus = clocks_sus.stop()
        st = g14.check_device_error(stream.cuda_stream)
        if st:
            raise RuntimeError(f"device error in the sustained leg: {g14.status_string(st)}")
        sus_s = dist.max(s0.elapsed_time(s1) / 1e3)
        sustained = {"steps": n_sus, "seconds": sus_s, "ms_per_step": sus_s / n_sus * 1e3,
                     "value": flops_step * n_sus * dist.world / sus_s / 1e12, "unit": UNIT,
                     "clocks": clk_sus}

    part_out = []
    for p in parts:
        s_ev, e_ev = ev[p["name"]]
        ms = [s_ev[i].elapsed_time(e_ev[i]) for i in range(K)]
        avg_s = statistics.mean(ms) / 1e3
        tflops = p["flops"] / avg_s / 1e12
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        mhz = clk_parts.get("sm_mhz")
        if p["bound"] == "tensor":
            # a short back-to-back region runs at burst clocks; seconds of
            # load settle at the power-capped sustained rate
            if elapsed_s >= 1.0:
                peak = peaks["bf16_tflops_sustained"]
                peak_note = f"bf16 dense, sustained ({peaks['source']}; timed region >= 1 s)"
            else:
                peak = peaks["bf16_tflops"]
                peak_note = f"bf16 dense, burst ({peaks['source']}; timed region < 1 s)"
            # dense bf16: 8192 FLOP (4096 multiply-adds) per SM per clock, at
            # the clock sampled while the parts ran
            per_clock = 8192
        else:
            peak = roofline.fp32_alu_peak_tflops()
            peak_note = "FFMA: 152 SMs x 128 lanes x 2 FLOP x 2070 MHz (unit counts)"
            per_clock = 256
        at_clock = None
        if mhz:
            pk = sms * per_clock * mhz * 1e6 / 1e12
            at_clock = {"sm_mhz_median": mhz, "peak_tflops": pk, "frac": tflops / pk,
                        "note": f"{sms} SMs x {per_clock} FLOP/clock x the median SM clock "
                                "NVML reported while the parts were timed"}
        eff = effective.get(p["name"])
        if eff and eff["sm_mhz_median"]:
            pk = sms * per_clock * eff["sm_mhz_median"] * 1e6 / 1e12
            eff = dict(eff, peak_tflops=pk, frac=tflops / pk)
        part_out.append({
            "workload": p["name"], "kernel": p["kernel"], "entry": p["entry"],
            "launches_per_call": p["launches"],
            "schedule": "stream-K" if p["ws_bytes"] else "data-parallel",
            "workspace_bytes": p["ws_bytes"], "M": p["w"].M, "N": p["w"].N,
            "K": p["w"].K, "ms_mean": statistics.mean(ms), "ms_median": statistics.median(ms),
            "ms_min": min(ms), "tflops": tflops, "at_sampled_clock": at_clock,
            "at_effective_clock": eff,
            "roofline": {"bound": p["bound"], "achieved": tflops, "peak": peak, "unit": UNIT,
                         "frac": tflops / peak, "peak_kind": peak_note,
                         "traffic": traffic_for(p["kernel"], p["src"], p["name"]),
                         "ideal_bytes": p["ideal_bytes"],
                         "hbm_floor_ms": p["ideal_bytes"] / (peaks["hbm_gbs"] * 1e9) * 1e3},
        })
    dominant = max(part_out, key=lambda x: x["ms_mean"])

    # ---- end to end through the public API with host tensors
    e2e = None
    if not args.no_e2e:
        # inputs and the result buffers in pinned host memory, allocated once
        # (as a caller reusing its buffers would); every step sends A and B to
        # the GPU and brings C back inside the timed region
        pinned = {n: (a.pin_memory(), b.pin_memory()) for n, (a, b) in host.items()}
        outs = {p["name"]: torch.empty((p["w"].M, p["w"].N), dtype=torch.float32,
                                       pin_memory=True) for p in parts}
        h2d = sum(a.numel() * a.element_size() + b.numel() * b.element_size()
                  for a, b in pinned.values())
        d2h = sum(p["w"].M * p["w"].N * 4 for p in parts)
        e2e_steps = max(1, min(K, 10))

        def issue_all():
            hs = []
            for _ in range(e2e_steps):
                for n, (a, b) in pinned.items():
                    hs.append(g14.gemm_async(a, b, out=outs[n]))
            return hs

        # warm-up in the timed pattern, so that the caching allocator holds
        # the device buffers of every product in flight (a steady state)
        for h in issue_all():
            h.wait()
        dist.barrier()
        torch.cuda.synchronize()
        # every product of every step issued through gemm_async (the next
        # one's operands go in while the one before computes and its result
        # comes out), all results waited for inside the timed region
        t0 = time.perf_counter()
        for h in issue_all():
            h.wait()
        torch.cuda.synchronize()
        t_e2e = dist.max(time.perf_counter() - t0)
        e2e = {"value": flops_step * e2e_steps * dist.world / t_e2e / 1e12, "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
               "ms_per_step": t_e2e / e2e_steps * 1e3,
               "issue": "gemm_async per product (C ABI gemm14_gemm_host on pinned host "
                        "buffers), results waited for at the end"}

    # ---- CPU oracle baseline (rank 0, one GPU only)
    cpu = None
    accuracy = None
    if dist.world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        tf, tt, desc, threads = 0.0, 0.0, [], 1
        accuracy = []
        for p in parts:
            f, t, r, threads, ref_rows = time_oracle_sample(p["name"], args.cpu_seconds,
                                                            *host[p["name"]], want_rows=True)
            tf += f
            tt += t
            desc.append(f"first {r} rows of {p['name']}")
            # the rows the oracle computed, against the GPU's C (every operand
            # set holds the same A and B, so set 0's C is the product's)
            accuracy.append(accuracy_of(p["name"], *host[p["name"]], p["sets"][0][2], ref_rows))
        cpu = {"value": tf / tt / 1e12, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": "; ".join(desc) + " (fp64 oracle, product only)", "seconds": tt}
        # the oracle on one thread, on the three fp32 configs (a bounded
        # sample of rows each, the whole product when it fits the time)
        if args.cpu_1t_seconds > 0:
            one = []
            for name in ("f32_256", "f32_3072", "f32_ragged"):
                f1, t1, r1, _ = time_oracle_sample(name, args.cpu_1t_seconds, threads=1)
                w1 = inputs.WORKLOADS[name]
                one.append({"workload": name, "rows": r1, "of_rows": w1.M, "seconds": t1,
                            "gflops": f1 / t1 / 1e9})
            cpu["one_thread"] = one

    if dist.rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": dist.world,
            "steps": K, "warmup": args.warmup, "ms_per_step": elapsed_max / K * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32 (FFMA) + bf16xbf16->f32 (tcgen05)", "data": "synthetic",
            "config": {"workload": WORKLOAD_NAME,
                       "l2": "inputs rotate over copies totalling > 2x L2 (no flush)",
                       "parallelism": f"replicas x{dist.world}"},
            "roofline": {k: dominant["roofline"][k] for k in
                         ("bound", "achieved", "peak", "unit", "frac", "traffic")},
            "dominant_kernel": dominant["kernel"],
            "parts": part_out,
            "gpu_launches": sum(p["launches"] for p in parts) * K,
            "timing": {"value": "K steps back to back between one event pair",
                       "parts": "the same K steps again, an event pair around each kernel",
                       "launches_timed_in_total": 2 * sum(p["launches"] for p in parts) * K},
            "clocks": clk,
            "clocks_parts": clk_parts,
            "sustained": sustained,
            "e2e": e2e,
            "cpu_baseline": cpu,
            "accuracy": accuracy,
        }
        print(json.dumps(line), flush=True)


def run_table(args):
    """Every named workload timed alone (CUDA events per launch, operand copies
    rotating over > 2x L2), with its roofline fraction. One JSON line each."""
    import torch

    import dense_gemm_14_gb300 as g14
    from dense_gemm_14_gb300 import inputs, roofline

    g14.load()
    peaks = roofline.measured_peaks()
    entry = {"f32": g14.gemm_f32, "bf16": g14.gemm_bf16_f32acc, "f16": g14.gemm_f16_f32acc}
    entry_ws = {"f32": g14.gemm_f32_ws, "bf16": g14.gemm_bf16_f32acc_ws,
                "f16": g14.gemm_f16_f32acc_ws}
    code = {"f32": g14.GEMM14_DTYPE_F32, "bf16": g14.GEMM14_DTYPE_BF16,
            "f16": g14.GEMM14_DTYPE_F16}
    stream = torch.cuda.current_stream()
    if not args.table_only:
        # the floor of a launch timed this way: a one-thread kernel that spins for
        # 100 SM cycles, timed alone and back to back like the products below
        for i in range(5):
            torch.cuda._sleep(100)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(50)]
        for e0, e1 in evs:
            e0.record(stream)
            torch.cuda._sleep(100)
            e1.record(stream)
        b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        b0.record(stream)
        for _ in range(50):
            torch.cuda._sleep(100)
        b1.record(stream)
        torch.cuda.synchronize()
        alone = statistics.median(e0.elapsed_time(e1) for e0, e1 in evs)
        print(json.dumps({"launch_floor": {"kernel": "one thread, 100 SM cycles",
                                           "us_alone_median": alone * 1e3,
                                           "us_back_to_back": b0.elapsed_time(b1) / 50 * 1e3}}),
              flush=True)
    for name, w in inputs.WORKLOADS.items():
        if args.table_only and name != args.table_only:
            continue
        _, fl, ib = workload_info(name)
        A, B = inputs.make_workload(name)
        per_set = A.numel() * A.element_size() + B.numel() * B.element_size() + w.M * w.N * 4
        nsets = max(2, -(-2 * L2_BYTES // per_set))
        sets = [(A.cuda(), B.cuda(), torch.empty(w.M, w.N, device="cuda")) for _ in range(nsets)]
        # the workspace for these operands: the stream-K region, and room to
        # re-pitch operands TMA cannot read (same alignment in every set)
        a0, b0, c0 = sets[0]
        ws_bytes = g14.workspace_bytes_ex(code[w.dtype], 0, 0, w.M, w.N, w.K, a0.data_ptr(), w.K,
                                          b0.data_ptr(), w.N, c0.data_ptr(), w.N)
        ws = torch.zeros(max(ws_bytes, 256), dtype=torch.uint8, device="cuda")
        for schedule in ("data-parallel", "stream-K"):
            if schedule == "stream-K" and ws_bytes == 0:
                continue
            time_one(args, name, w, fl, ib, sets, nsets, stream, peaks, roofline, g14, schedule,
                     entry[w.dtype], entry_ws[w.dtype], ws, ws_bytes)
        del sets
        torch.cuda.empty_cache()


def time_one(args, name, w, fl, ib, sets, nsets, stream, peaks, roofline, g14, schedule, fn,
             fn_ws, ws, ws_bytes):
    """One --table line: `schedule` selects the plain or the workspace entry point."""
    import torch
    def launch(i):
        a, b, c = sets[i % nsets]
        if schedule == "stream-K":
            fn_ws(w.M, w.N, w.K, a.data_ptr(), w.K, b.data_ptr(), w.N, c.data_ptr(), w.N,
                  ws.data_ptr(), ws_bytes, stream.cuda_stream)
        else:
            fn(w.M, w.N, w.K, a.data_ptr(), w.K, b.data_ptr(), w.N, c.data_ptr(), w.N,
               stream.cuda_stream)

    for i in range(args.warmup):
        launch(i)
    reps = max(args.steps, 5)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(reps)]
    clocks = ClockSampler(torch.cuda.current_device(), period_s=0.001)
    torch.cuda.synchronize()
    clocks.start()
    for i, (e0, e1) in enumerate(evs):
        e0.record(stream)
        launch(i)
        e1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if g14.check_device_error(stream.cuda_stream):
        raise RuntimeError(f"device error in {name}")
    ms = [e0.elapsed_time(e1) for e0, e1 in evs]
    # the same launches back to back between one event pair: consecutive
    # products overlap launch and set-up with the end of the one before
    b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    b0.record(stream)
    for i in range(reps):
        launch(i)
    b1.record(stream)
    torch.cuda.synchronize()
    if g14.check_device_error(stream.cuda_stream):
        raise RuntimeError(f"device error in {name}")
    ms_b2b = b0.elapsed_time(b1) / reps
    mean = statistics.mean(ms)
    tf = fl / (mean / 1e3) / 1e12
    if w.dtype == "f32":
        peak, kind = roofline.fp32_alu_peak_tflops(), "alu"
    else:
        peak, kind = peaks["bf16_tflops"], "tensor"  # each workload is timed alone: burst
    gbs = ib / (mean / 1e3) / 1e9
    print(json.dumps({"workload": name, "schedule": schedule, "M": w.M, "N": w.N, "K": w.K,
                      "dtype": w.dtype, "ms_mean": mean, "ms_median": statistics.median(ms), "ms_min": min(ms), "tflops": tf,
                      "bound": kind, "peak_tflops": peak, "frac_compute": tf / peak,
                      "algorithmic_bytes": ib, "gbs": gbs,
                      "frac_hbm": gbs / peaks["hbm_gbs"],
                      "workspace_bytes": ws_bytes if schedule == "stream-K" else 0,
                      "clocks": clk,
                      "back_to_back": {"ms": ms_b2b, "tflops": fl / (ms_b2b / 1e3) / 1e12,
                                       "gbs": ib / (ms_b2b / 1e3) / 1e9,
                                       "frac_hbm": ib / (ms_b2b / 1e3) / 1e9 / peaks["hbm_gbs"]}}),
          flush=True)


# (transa, transb, alpha, beta) variants of the extended call
EX_VARIANTS = [(0, 0, 1.0, 0.0), (1, 0, 1.0, 0.0), (0, 1, 1.0, 0.0), (1, 1, 1.0, 0.0),
               (0, 0, -1.5, 0.0), (0, 0, -1.5, 0.5)]


def run_table_ex(args):
    """gemm14_gemm_ex timed alone per variant: the operands stored as the
    variant says (transposed copies made before timing), C read too when
    beta != 0 (its bytes added to the algorithmic traffic). Operand copies
    rotate over > 2x L2; the workspace entry (stream-K where it applies)."""
    import torch

    import dense_gemm_14_gb300 as g14
    from dense_gemm_14_gb300 import inputs, roofline

    g14.load()
    peaks = roofline.measured_peaks()
    code = {"f32": g14.GEMM14_DTYPE_F32, "bf16": g14.GEMM14_DTYPE_BF16,
            "f16": g14.GEMM14_DTYPE_F16}
    stream = torch.cuda.current_stream()
    for name in ("f32_3072", "bf16_8192", "f16_8192"):
        w, fl, ib = workload_info(name)
        A, B = inputs.make_workload(name)
        for ta, tb, alpha, beta in EX_VARIANTS:
            As = (A.t().contiguous() if ta else A).cuda()
            Bs = (B.t().contiguous() if tb else B).cuda()
            per_set = As.numel() * As.element_size() + Bs.numel() * Bs.element_size() + w.M * w.N * 4
            nsets = max(2, -(-2 * L2_BYTES // per_set))
            sets = [(As.clone(), Bs.clone(), torch.zeros(w.M, w.N, device="cuda"))
                    for _ in range(nsets)]
            lda, ldb = As.shape[1], Bs.shape[1]
            # the workspace this call asks for (stream-K region, and copies of
            # operands in a storage its kernel reads slowly)
            ws_bytes = g14.workspace_bytes_ex(code[w.dtype], ta, tb, w.M, w.N, w.K,
                                              sets[0][0].data_ptr(), lda, sets[0][1].data_ptr(),
                                              ldb, sets[0][2].data_ptr(), w.N)
            ws = torch.zeros(max(ws_bytes, 256), dtype=torch.uint8, device="cuda")

            def launch(i):
                a, b, c = sets[i % nsets]
                g14.gemm_ex(code[w.dtype], ta, tb, w.M, w.N, w.K, alpha, a.data_ptr(), lda,
                            b.data_ptr(), ldb, beta, c.data_ptr(), w.N, ws.data_ptr(), ws_bytes,
                            stream.cuda_stream)

            for i in range(args.warmup):
                launch(i)
            reps = max(args.steps, 5)
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(reps)]
            for i, (e0, e1) in enumerate(evs):
                e0.record(stream)
                launch(i)
                e1.record(stream)
            torch.cuda.synchronize()
            if g14.check_device_error(stream.cuda_stream):
                raise RuntimeError(f"device error in {name}")
            ms = [e0.elapsed_time(e1) for e0, e1 in evs]
            mean = statistics.mean(ms)
            tf = fl / (mean / 1e3) / 1e12
            if w.dtype == "f32":
                peak, kind = roofline.fp32_alu_peak_tflops(), "alu"
            else:
                peak, kind = peaks["bf16_tflops"], "tensor"
            nbytes = ib + (w.M * w.N * 4 if beta != 0.0 else 0)
            gbs = nbytes / (mean / 1e3) / 1e9
            print(json.dumps({"workload": name, "transa": ta, "transb": tb, "alpha": alpha,
                              "beta": beta, "ms_mean": mean, "ms_median": statistics.median(ms), "ms_min": min(ms), "tflops": tf,
                              "bound": kind, "peak_tflops": peak, "frac_compute": tf / peak,
                              "algorithmic_bytes": nbytes, "gbs": gbs,
                              "frac_hbm": gbs / peaks["hbm_gbs"]}), flush=True)
            del sets, As, Bs
            torch.cuda.empty_cache()


# bf16 products with operands TMA cannot read: (name, M, N, K, transa, transb,
# extra pitch of A, extra pitch of B, element offset of A and B), the stored
# rows' pitches being their lengths plus the extra.
SOFT_SHAPES = [
    ("8192x8192x8191_lda_odd", 8192, 8192, 8191, 0, 0, 0, 0, 0),
    ("4096_nn_odd", 4096, 4096, 4096, 0, 0, 1, 1, 0),
    ("4096_tt_odd", 4096, 4096, 4096, 1, 1, 1, 1, 0),
    ("4096_nn_pitch+2_offset1", 4096, 4096, 4096, 0, 0, 2, 2, 1),
    ("1000x777x1000_ldb_odd", 1000, 777, 1000, 0, 0, 0, 1, 0),
    ("16384x64x4096_odd", 16384, 64, 4096, 0, 0, 1, 1, 0),
]


def run_table_soft(args):
    """The 16-bit software loader: bf16 products through the plain call (no
    workspace, so no re-pitching) with operands that TMA cannot read, against
    the same one-SM kernel on copies with 16-byte pitches (CTA pairs off for
    both). Operand copies rotate over > 2x L2; the two results must agree bit
    for bit."""
    import torch

    import dense_gemm_14_gb300 as g14
    from dense_gemm_14_gb300 import roofline

    g14.load()
    peaks = roofline.measured_peaks()
    stream = torch.cuda.current_stream()
    prev = g14.set_pair_kernel(False)
    try:
        for name, M, N, K, ta, tb, xa, xb, off in SOFT_SHAPES:
            if args.soft_only and name != args.soft_only:
                continue
            ar, ac = (K, M) if ta else (M, K)
            br, bc = (N, K) if tb else (K, N)
            g = torch.Generator(device="cuda").manual_seed(14100)
            variants = {"unaligned": (ac + xa, bc + xb, off)}
            if not args.soft_only:
                variants["tma"] = (-(-ac // 8) * 8, -(-bc // 8) * 8, 0)
            res, outs = {}, {}
            for v, (lda, ldb, o) in variants.items():
                per_set = (ar * lda + br * ldb) * 2 + M * N * 4
                nsets = max(2, -(-2 * L2_BYTES // per_set))
                sets = []
                for _ in range(nsets):
                    a = torch.zeros(o + ar * lda, dtype=torch.bfloat16, device="cuda")
                    b = torch.zeros(o + br * ldb, dtype=torch.bfloat16, device="cuda")
                    a[o:].view(ar, lda)[:, :ac] = (torch.randn(ar, ac, device="cuda", generator=g)
                                                    * 0.05).to(torch.bfloat16)
                    b[o:].view(br, ldb)[:, :bc] = (torch.randn(br, bc, device="cuda", generator=g)
                                                    * 0.05).to(torch.bfloat16)
                    sets.append((a, b, torch.zeros(M, N, device="cuda")))
                if v == "tma":  # the same operand values as the unaligned sets
                    for (a, b, _), (ua, ub, _) in zip(sets, outs["sets"]):
                        ula, ulb, uo = variants["unaligned"]
                        a.view(ar, lda)[:, :ac] = ua[uo:].view(ar, ula)[:, :ac]
                        b.view(br, ldb)[:, :bc] = ub[uo:].view(br, ulb)[:, :bc]

                def launch(i):
                    a, b, c = sets[i % nsets]
                    g14.gemm_ex(g14.GEMM14_DTYPE_BF16, ta, tb, M, N, K, 1.0,
                                a.data_ptr() + 2 * o, lda, b.data_ptr() + 2 * o, ldb, 0.0,
                                c.data_ptr(), N, None, 0, stream.cuda_stream)

                for i in range(args.warmup):
                    launch(i)
                reps = max(args.steps, 5)
                evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                       for _ in range(reps)]
                for i, (e0, e1) in enumerate(evs):
                    e0.record(stream)
                    launch(i)
                    e1.record(stream)
                torch.cuda.synchronize()
                if g14.check_device_error(stream.cuda_stream):
                    raise RuntimeError(f"device error in {name} ({v})")
                ms = [e0.elapsed_time(e1) for e0, e1 in evs]
                res[v] = {"lda": lda, "ldb": ldb, "offset": o, "ms_median": statistics.median(ms),
                          "ms_min": min(ms)}
                launch(0)
                torch.cuda.synchronize()
                outs[v] = sets[0][2].clone()
                if v == "unaligned":
                    outs["sets"] = sets
                else:
                    del sets
            fl = roofline.flops(M, N, K)
            line = {"shape": name, "M": M, "N": N, "K": K, "transa": ta, "transb": tb}
            for v, r in res.items():
                tf = fl / (r["ms_median"] / 1e3) / 1e12
                line[v] = dict(r, tflops=tf, frac_of_bf16_peak=tf / peaks["bf16_tflops"])
            if "tma" in outs:
                line["bit_identical"] = bool(torch.equal(outs["unaligned"], outs["tma"]))
                line["unaligned_over_tma"] = res["unaligned"]["ms_median"] / res["tma"]["ms_median"]
            print(json.dumps(line), flush=True)
            outs.clear()
            torch.cuda.empty_cache()
    finally:
        g14.set_pair_kernel(prev)


def run_table_tf32(args):
    """fp32 inputs timed alone in each arithmetic: gemm_f32 (FFMA), gemm_tf32_f32acc
    and gemm_f32_3xtf32 (tensor cores), at the 3072^3 workload and at an 8192^3
    product of the same distribution (U[-1,1), seed 14007), each with the
    workspace it asks for (with --tf32-plain: none). Operand copies rotate over
    > 2x L2."""
    import torch

    import dense_gemm_14_gb300 as g14
    from dense_gemm_14_gb300 import inputs, roofline

    g14.load()
    peaks = roofline.measured_peaks()
    stream = torch.cuda.current_stream()
    shapes = [("f32_3072", None), ("f32_8192", (8192, 8192, 8192, 14007))]
    modes = [("fp32 FFMA", g14.GEMM14_DTYPE_F32), ("tf32", g14.GEMM14_DTYPE_TF32),
             ("3xtf32", g14.GEMM14_DTYPE_F32_3XTF32)]
    if args.tf32_only:
        only_shape, only_mode = args.tf32_only.split(":")
        shapes = [sh for sh in shapes if sh[0] == only_shape]
        modes = [m for m in modes if m[0].split()[0] == only_mode]
    for name, spec in shapes:
        if spec is None:
            w = inputs.WORKLOADS[name]
            M, N, K = w.M, w.N, w.K
            A, B = inputs.make_workload(name)
        else:
            M, N, K, seed = spec
            A, B = inputs.make(M, N, K, "f32", "uniform", 1.0, seed=seed)
        fl = roofline.flops(M, N, K)
        ib = roofline.ideal_bytes(M, N, K, 4, 4)
        per_set = (M * K + K * N + M * N) * 4
        nsets = max(2, -(-2 * L2_BYTES // per_set))
        sets = [(A.cuda(), B.cuda(), torch.empty(M, N, device="cuda")) for _ in range(nsets)]
        for mode, code in modes:
            # the workspace each mode asks for with these operands (TF32 on
            # row-major B: room for its K-major copy)
            a0, b0, c0 = sets[0]
            ws_bytes = 0 if args.tf32_plain else g14.workspace_bytes_ex(
                code, 0, 0, M, N, K, a0.data_ptr(), K, b0.data_ptr(), N, c0.data_ptr(), N)
            ws = (None if args.tf32_plain else
                  torch.zeros(max(ws_bytes, 256), dtype=torch.uint8, device="cuda"))

            def launch(i):
                a, b, c = sets[i % nsets]
                g14.gemm_ex(code, 0, 0, M, N, K, 1.0, a.data_ptr(), K, b.data_ptr(), N, 0.0,
                            c.data_ptr(), N, ws.data_ptr() if ws is not None else None,
                            ws_bytes, stream.cuda_stream)

            for i in range(args.warmup):
                launch(i)
            reps = max(args.steps, 5)
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(reps)]
            for i, (e0, e1) in enumerate(evs):
                e0.record(stream)
                launch(i)
                e1.record(stream)
            torch.cuda.synchronize()
            if g14.check_device_error(stream.cuda_stream):
                raise RuntimeError(f"device error in {name} {mode}")
            ms = [e0.elapsed_time(e1) for e0, e1 in evs]
            mean = statistics.mean(ms)
            tf = fl / (mean / 1e3) / 1e12
            mma_flops = fl * (3 if code == g14.GEMM14_DTYPE_F32_3XTF32 else 1)
            if code == g14.GEMM14_DTYPE_F32:
                peak, kind = roofline.fp32_alu_peak_tflops(), "alu"
            else:
                # tf32 dense peak: the measured bf16 burst figure x the nominal
                # tf32 / bf16 ratio (1.1 / 2.25 PFLOP/s)
                peak, kind = peaks["bf16_tflops"] * 1.1 / 2.25, "tensor (tf32)"
            print(json.dumps({"workload": name, "mode": mode, "M": M, "N": N, "K": K,
                              "workspace_bytes": ws_bytes, "ms_mean": mean, "ms_median": statistics.median(ms), "ms_min": min(ms), "tflops": tf,
                              "mma_tflops": mma_flops / (mean / 1e3) / 1e12, "bound": kind,
                              "peak_tflops": peak,
                              "frac_compute": mma_flops / (mean / 1e3) / 1e12 / peak,
                              "vs_ffma_peak": tf / roofline.fp32_alu_peak_tflops(),
                              "gbs": ib / (mean / 1e3) / 1e9}), flush=True)
        del sets
        torch.cuda.empty_cache()


FMA_CEILING_SRC = r"""
#include <cstdint>
// Each thread runs 32 independent accumulator chains of fused multiply-adds
// on register operands only: packed fma.rn.f32x2 (MODE 0) or scalar
// fma.rn.f32 (MODE 1). No memory traffic but one store per thread at the end.
template <int MODE>
__global__ void fma_loop(float* out, int iters, float a0, float b0) {
  constexpr int NCH = 32;
  uint64_t acc2[NCH], a2, b2;
  float acc1[NCH];
  asm("mov.b64 %0, {%1, %2};" : "=l"(a2) : "f"(a0), "f"(a0 + 1.0f));
  asm("mov.b64 %0, {%1, %2};" : "=l"(b2) : "f"(b0), "f"(b0 - 1.0f));
#pragma unroll
  for (int i = 0; i < NCH; ++i) {
    asm("mov.b64 %0, {%1, %2};" : "=l"(acc2[i]) : "f"((float)i), "f"((float)(i + threadIdx.x)));
    acc1[i] = (float)(3 * i + threadIdx.x);
  }
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int i = 0; i < NCH; ++i) {
      if (MODE == 0) asm volatile("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc2[i]) : "l"(a2), "l"(b2));
      else asm volatile("fma.rn.f32 %0, %1, %2, %0;" : "+f"(acc1[i]) : "f"(a0), "f"(b0));
    }
  }
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < NCH; ++i) {
    float x, y;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(x), "=f"(y) : "l"(acc2[i]));
    s += x + y + acc1[i];
  }
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}
// out: blocks x threads floats on the device; launches on the default stream.
extern "C" int fma_ceiling_run(float* out, int mode, int blocks, int threads, int iters) {
  if (mode == 0) fma_loop<0><<<blocks, threads>>>(out, iters, 1.0001f, 0.9999f);
  else fma_loop<1><<<blocks, threads>>>(out, iters, 1.0001f, 0.9999f);
  return (int)cudaGetLastError();
}
"""


def run_fma_ceiling(args):
    """The FFMA throughput register-only loops reach on this GPU against the
    unit-count peak (SMs x 128 lanes x 2 FLOP x clock): 32 independent chains
    a thread, packed (fma.rn.f32x2, what the fp32 kernel issues) and scalar,
    at 16 warps per SM and at the fp32 kernel's 8. Compiled here with nvcc
    into a scratch folder; one JSON line per case."""
    import ctypes
    import tempfile

    import torch

    from dense_gemm_14_gb300 import build, roofline
    tmp = tempfile.mkdtemp(prefix="fma_ceiling_")
    src, lib = os.path.join(tmp, "fma.cu"), os.path.join(tmp, "libfma.so")
    with open(src, "w") as f:
        f.write(FMA_CEILING_SRC)
    subprocess.run([build.nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-O3",
                    "-Xcompiler", "-fPIC", "-shared", "-o", lib, src], check=True)
    so = ctypes.CDLL(lib)
    so.fma_ceiling_run.argtypes = [ctypes.c_void_p] + [ctypes.c_int] * 4
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    threads = 256
    cases = ((0, "packed fma.rn.f32x2", 2, 20000, 32), (1, "scalar fma.rn.f32", 2, 20000, 32),
             (0, "packed fma.rn.f32x2", 1, 20000, 32), (1, "scalar fma.rn.f32", 1, 20000, 32))
    for mode, name, per_sm, iters, fma_per_iter in cases:
        blocks = per_sm * sms
        out = torch.empty(blocks * threads, device="cuda")
        torch.cuda.synchronize()
        assert so.fma_ceiling_run(out.data_ptr(), mode, blocks, threads, 100) == 0
        clocks = ClockSampler(torch.cuda.current_device(), period_s=0.001)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        clocks.start()
        e0.record(torch.cuda.default_stream())
        so.fma_ceiling_run(out.data_ptr(), mode, blocks, threads, iters)
        e1.record(torch.cuda.default_stream())
        torch.cuda.synchronize()
        clk = clocks.stop()
        ms = e0.elapsed_time(e1)
        fmas = float(iters) * fma_per_iter * (1 if mode == 1 else 2) * blocks * threads
        tflops = 2 * fmas / (ms * 1e-3) / 1e12
        peak = roofline.fp32_alu_peak_tflops()
        print(json.dumps({"fma_ceiling": name, "ms": ms, "tflops": tflops,
                          "unit_count_peak_tflops": peak, "frac_of_unit_count_peak": tflops / peak,
                          "fma_per_clock_per_sm_at_2070": fmas / (ms * 1e-3) / sms / 2.07e9,
                          "grid": f"{blocks} x {threads} threads ({8 * per_sm} warps per SM), "
                                  f"{fma_per_iter} chains each",
                          "clocks": clk}), flush=True)


def main():
    args = parse_args()
    if args.fma_ceiling:
        run_fma_ceiling(args)
        return
    if args.table_tf32:
        run_table_tf32(args)
        return
    if args.table:
        run_table(args)
        return
    if args.table_ex:
        run_table_ex(args)
        return
    if args.table_soft:
        run_table_soft(args)
        return
    dist = Dist(args.gpus)
    try:
        if args.impl == "reference":
            run_reference(args, dist)
        else:
            run_ours(args, dist)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
