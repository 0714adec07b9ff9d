"""Benchmark: device-wide scan throughput at n = 1e8 on one GB300.

One step = four single-pass scans of 1e8 elements each: int32 exclusive and
inclusive (uniform integers in [-1000, 1000], seed 2) and fp32 exclusive and
inclusive (uniform [0, 1), seed 1), inputs resident in HBM.  `value` is
elements scanned per second (G-elem/s) over all ranks; the roofline line
converts the scan kernel's average launch time to GB/s on its algorithmic
bytes, 2 * n * 4 bytes per launch (read once, write once).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the sequential CPU oracle on the same metric (a
bounded sample of the same inputs per step).  Under torchrun each rank runs
its own replica on its own GPU (independent problems, no collective on the
data path); rank 0 prints one JSON line.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np

METRIC = "scan G-elem/s & HBM GB/s vs 2n·sizeof(T) roofline, int32/fp32 at n=1e8"
UNIT = "G-elem/s"
N = 100_000_000
BYTES_PER_ELEM = 8  # one 4-byte read + one 4-byte write
L2_BYTES = 129 * 1024 * 1024
# fp64 scan roofline: GB300's nominal FP64 rate is 1.25 TFLOP/s counting an FMA as two
# operations, i.e. 625e9 FP64 adds per second; the lane-blocked fp64 kernel makes about 2.3
# adds per element (15 in-lane adds per 16 elements, ~4 warp-scan adds per lane, and one
# add per output).
FP64_DADD_PER_S = 625e9
FP64_ADDS_PER_ELEM = 2.3
FALLBACK_HBM_GBS = 6800.0
VARIANTS = [("i32", False), ("i32", True), ("f32", False), ("f32", True)]
DATA = "synthetic, seeded SplitMix64: int32 U[-1000,1000] (seed 2), fp32 U[0,1) (seed 1)"
WORKLOAD = "scan n=1e8; step = int32 excl+incl, fp32 excl+incl (4 launches)"
KERNEL_SOURCES = ["stream_compaction_pass_gb300/csrc/scan_pipe.cu", "stream_compaction_pass_gb300/csrc/scan.cu",
                  "stream_compaction_pass_gb300/csrc/scan_body.cuh", "stream_compaction_pass_gb300/csrc/tile.cuh",
                  "stream_compaction_pass_gb300/csrc/lookback.cuh", "stream_compaction_pass_gb300/csrc/bulk.cuh"]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "k_scan_lookback_pipe_sb_n1e8.md")


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def max_over_ranks(elapsed_ms: float, device=None) -> float:
    """Largest elapsed time over all ranks (every rank gets it)."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(elapsed_ms)
    t = torch.tensor([elapsed_ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(elems_per_rank: int, world: int, max_elapsed_ms: float) -> float:
    """Elements all ranks processed, per second, in G-elem/s."""
    return elems_per_rank * world / (max_elapsed_ms * 1e-3) / 1e9


def emit(obj) -> None:
    print(json.dumps(obj, separators=(",", ":")), flush=True)


# --------------------------------------------------------------------------
# measurement helpers

def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured (MEASURED_PEAKS.json hbm_gbs)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback (6.8 TB/s, one earlier GB300 copy measurement)"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic():
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources; else None."""
    try:
        text = open(TRAFFIC_FILE).read()
    except OSError:
        return None
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9]+)", text)
    h = re.search(r"kernel_source_hash:\s*([0-9a-f]+)", text)
    if not m or not h or h.group(1) != kernel_source_hash():
        return None
    return int(m.group(1))


class ClockSampler:
    """SM clock and clock-event (throttle) reasons, sampled every ~1 ms by a
    thread while the timed region runs.  Reads NVML directly (read-only
    queries; the timed region is a few ms, shorter than nvidia-smi's first
    sample); falls back to nvidia-smi at 100 ms if NVML cannot be loaded."""

    # NVML clock-event reason bits (nvmlClocksEventReason*)
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        import threading
        self.proc = None
        self.nvml = None
        self.samples = []  # (sm_mhz, reasons bitmask)
        self.max_mhz = None
        if gpu_id is None:
            return
        try:
            import ctypes
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                raise OSError("nvmlInit failed")
            h = ctypes.c_void_p()
            if nv.nvmlDeviceGetHandleByUUID(gpu_id.encode(), ctypes.byref(h)) != 0:
                raise OSError("no NVML handle for this GPU")
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:  # NVML_CLOCK_SM
                self.max_mhz = float(mx.value)
            self.nvml, self.handle = nv, h
            self.stop_flag = threading.Event()
            self.thread = threading.Thread(target=self._run_nvml, daemon=True)
            self.thread.start()
            return
        except Exception:
            self.nvml = None
        try:
            import tempfile
            fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
            self.fh = os.fdopen(fd, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", gpu_id, "-lms", "100"], stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def _run_nvml(self):
        import ctypes
        clk, rsn = ctypes.c_uint(), ctypes.c_ulonglong()
        get_reasons = getattr(self.nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.nvml.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self.stop_flag.is_set():
            if self.nvml.nvmlDeviceGetClockInfo(self.handle, 1, ctypes.byref(clk)) == 0 and \
                    get_reasons(self.handle, ctypes.byref(rsn)) == 0:
                self.samples.append((float(clk.value), int(rsn.value)))
            time.sleep(0.001)

    def stop(self):
        if self.nvml is not None:
            self.stop_flag.set()
            self.thread.join(timeout=5)
            reasons = set()
            for _mhz, bits in self.samples:
                for bit, name in self.REASONS.items():
                    if bits & bit:
                        reasons.add(name)
            sm = [m for m, _b in self.samples]
            return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": self.max_mhz,
                    "reasons": sorted(reasons), "samples": len(sm), "source": "nvml"}
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        self.raw = open(self.path).read()
        os.unlink(self.path)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.raw.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm), "source": "nvidia-smi"}


def gpu_uuid(torch, dev) -> str | None:
    try:
        u = torch.cuda.get_device_properties(dev).uuid
        s = str(u)
        return s if s.startswith("GPU-") else "GPU-" + s
    except Exception:
        return None


# --------------------------------------------------------------------------
# CPU side: the oracle as a baseline / reference arm

def oracle_step(orc, xs, xf, m: int) -> None:
    orc.scan_i32(xs[:m], False)
    orc.scan_i32(xs[:m], True)
    orc.scan_f32(xf[:m], False)
    orc.scan_f32(xf[:m], True)


def cpu_baseline(xs, xf, budget_s: float = 10.0):
    import oracle as orc
    orc.load()
    m = N
    t0 = time.perf_counter()
    reps = 0
    while True:
        oracle_step(orc, xs, xf, m)
        reps += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return {"value": _sig(4 * m * reps / dt / 1e9), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{reps} full steps (4 scans of 1e8) in {dt:.1f} s, one core"}


def run_reference(args) -> None:
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import seeded_inputs as si
    import oracle as orc
    orc.load()
    budget_elems = 2.0e10  # ~20-40 s of oracle work over the whole run
    m = int(min(N, max(100_000, budget_elems / (4 * (args.steps + args.warmup)))))
    xs = si.workload_int_pm1000(m, seed=2)
    xf = si.workload_f32_unit(m, seed=1)
    for _ in range(args.warmup):
        oracle_step(orc, xs, xf, m)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(orc, xs, xf, m)
    dt = time.perf_counter() - t0
    value = 4 * m * args.steps / dt / 1e9
    sample = f"first {m} elements of the 1e8-element inputs per scan, 4 scans per step"
    emit({"metric": METRIC, "value": value, "unit": UNIT, "impl": "reference", "n_gpus": world,
          "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
          "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int32/fp32",
          "data": DATA, "config": {"workload": WORKLOAD, "n": N, "sample_elems_per_scan": m},
          "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
          "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}})


# --------------------------------------------------------------------------
# GPU side

def time_region(torch, stream, fn, reps: int, warmup: int = 3) -> float:
    """Mean ms per call of fn() on `stream`, CUDA events, after warm-up."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(reps):
        fn()
    b.record(stream)
    b.synchronize()
    return a.elapsed_time(b) / reps


def time_flushed(torch, stream, fn, scratch, reps: int) -> float:
    """Mean ms of fn() on `stream` with L2 flushed before each call: the
    scratch buffer (larger than L2) is written between calls, and only fn()
    is inside the CUDA events."""
    fn()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    with torch.cuda.stream(stream):
        for a, b in ev:
            scratch.zero_()
            a.record(stream)
            fn()
            b.record(stream)
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in ev) / reps


def _sig(v: float, digits: int = 4) -> float:
    """v rounded to `digits` significant digits (keeps the JSON line short)."""
    if v == 0 or not np.isfinite(v):
        return float(v)
    return float(f"{v:.{digits}g}")


def sweep_sizes():
    """The int32 size sweep: 2^10 .. 2^30, 2^k - 1 and 2^k + 1 around the
    tile-sized and large powers, and 10^3 .. 10^9."""
    sizes = {1 << k for k in range(10, 31)}
    for k in (10, 12, 13, 16, 20, 24, 27, 30):
        sizes |= {(1 << k) - 1, (1 << k) + 1}
    sizes |= {10 ** k for k in range(3, 10)}
    return sorted(sizes)


def size_label(n: int) -> str:
    for k in range(10, 31):
        for d, tag in ((0, ""), (-1, "-1"), (1, "+1")):
            if n == (1 << k) + d:
                return f"2^{k}{tag}"
    for k in range(3, 10):
        if n == 10 ** k:
            return f"1e{k}"
    return str(n)


def row_rates(torch, ss, stream, dev, xs_d, xf_d, out_d, launch_ms_by_variant):
    """Secondary rows, one short entry each: [ms per call, fraction of the
    measured HBM peak on the row's algorithmic bytes] (CUDA events, mean of
    20 after 3 warm-ups; L2 flushed before every call where the data would
    fit in L2)."""
    import seeded_inputs as si
    rows = {}
    peak, _ = measured_hbm_peak()
    sh = stream.cuda_stream
    scratch = torch.empty(80_000_000, dtype=torch.int32, device=dev)  # 320 MB, over twice the L2

    def entry(bytes_, ms):
        return [_sig(ms), round(bytes_ / (ms * 1e-3) / 1e9 / peak, 3)]

    def timed(fn, nbytes, reps=20):
        # inputs that fit in L2 twice over get a flush before every call
        if nbytes < 2 * L2_BYTES:
            return time_flushed(torch, stream, fn, scratch, reps)
        return time_region(torch, stream, fn, reps)

    # C2 at n = 1e8 and the headline variants, from the step's own per-launch events
    for (kind, incl), ms in launch_ms_by_variant.items():
        rows[f"{kind}{'i' if incl else 'x'}_1e8"] = entry(8 * N, ms)
    # C2: fp32 inclusive and exclusive at 1e6 and 1e7: [ms and fraction with L2 flushed,
    # ms warm (back to back, the arrays L2-resident)]
    for nf in (1_000_000, 10_000_000):
        xf_s = torch.from_numpy(si.workload_f32_unit(nf, seed=1)).to(dev)
        of_s = torch.empty_like(xf_s)
        for incl in (True, False):
            fn = (lambda: ss.scan_inclusive_f32(xf_s, of_s, stream=sh)) if incl else \
                 (lambda: ss.scan_exclusive_f32(xf_s, of_s, stream=sh))
            rows[f"f32{'i' if incl else 'x'}_{nf:.0e}".replace("+0", "")] = (
                entry(8 * nf, timed(fn, 8 * nf)) + [_sig(time_region(torch, stream, fn, 20), 3)])
        del xf_s, of_s
    # C1: int32 n = 4096, an inclusive and an exclusive scan per step, per call from
    # Python and per replay of a captured graph (launch latency, not bandwidth): [us, us]
    x_small = torch.from_numpy(si.workload_int_0_100(4096, seed=0)).to(dev)
    o_small = torch.empty_like(x_small)

    def small_step():
        ss.scan_inclusive_i32(x_small, o_small, stream=sh)
        ss.scan_exclusive_i32(x_small, o_small, stream=sh)
    ms = time_region(torch, stream, small_step, 200)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        small_step()
    ms_g = time_region(torch, stream, graph.replay, 200)
    rows["c1_4096_us"] = [_sig(ms * 1e3, 3), _sig(ms_g * 1e3, 3)]
    del graph, x_small, o_small
    # C3: int32 exclusive over the whole size sweep, us per call (the fraction is
    # 8n bytes / time / peak); prefixes of one seeded input in [-1000, 1000]
    top = sweep_sizes()[-1]
    gen = torch.Generator(device=dev)
    gen.manual_seed(2)
    xi = torch.randint(-1000, 1001, (top,), dtype=torch.int32, device=dev, generator=gen)
    oi = torch.empty_like(xi)
    sweep = {}
    for ns in sweep_sizes():
        a, o = xi[:ns], oi[:ns]
        ms = timed(lambda: ss.scan_exclusive_i32(a, o, stream=sh), 8 * ns, 20 if ns < (1 << 29) else 5)
        sweep[size_label(ns)] = _sig(ms * 1e3, 3)
    # 2^k - 1 and 2^k + 1 sit beside 2^k: "2^k": [us(2^k), us(2^k - 1), us(2^k + 1)]
    for lbl in [k for k in sweep if k.startswith("2^") and k[-2:] not in ("-1", "+1")]:
        if lbl + "-1" in sweep:
            sweep[lbl] = [sweep[lbl], sweep.pop(lbl + "-1"), sweep.pop(lbl + "+1")]
    rows["i32x_sweep_us"] = sweep
    del xi, oi
    # copy probe with the scan's loader: the practical roofline of this access pattern
    ms = time_region(torch, stream, lambda: ss.ss_copy_u32(xs_d, out_d, N, stream=sh), 20)
    rows["copy_1e8"] = entry(8 * N, ms)
    # ablations (reduce-then-scan, three kernels) at the same int32 workload, on 2n bytes
    for name, algo in (("rts", ss.SS_ALGO_REDUCE_THEN_SCAN), ("rts_bl", ss.SS_ALGO_RTS_BLELLOCH),
                       ("rts_bl32", ss.SS_ALGO_RTS_BLELLOCH_PAD32), ("rts_bl2", ss.SS_ALGO_RTS_BLELLOCH_PAD2)):
        ms = time_region(torch, stream, lambda a=algo: ss.ss_scan(ss.SS_I32, False, a, xs_d, out_d, stream=sh), 20)
        rows[f"{name}_1e8"] = entry(8 * N, ms)
    # C5: uint32 Poisson(8) counts, n = 2^27, out of place and in place
    nc = 1 << 27
    cnt = torch.from_numpy(si.workload_poisson_counts(nc, seed=4).view(np.int32)).to(dev)
    cnt_out = torch.empty_like(cnt)
    rows["pois"] = entry(8 * nc, time_region(torch, stream, lambda: ss.scan_exclusive_u32(cnt, cnt_out, stream=sh), 20))
    rows["pois_inpl"] = entry(8 * nc, time_region(
        torch, stream, lambda: ss.scan_exclusive_u32(cnt_out, cnt_out, stream=sh), 20))
    del cnt, cnt_out
    # C4: flag compaction, n = 2^28, p in {0.01, 0.5, 0.99}, on 5n + 4k bytes; and the
    # unordered (warp-aggregated atomics) ablation on the same inputs, ms only
    nk = 1 << 28
    keys = torch.from_numpy(si.uniform_u32(nk, 6).view(np.int32)).to(dev)
    kout = torch.empty_like(keys)
    dcount = torch.zeros(1, dtype=torch.int64, device=dev)
    unord = []
    for p in (0.01, 0.5, 0.99):
        flags_np = si.bernoulli_flags(nk, p, 7)
        flags = torch.from_numpy(flags_np).to(dev)
        kept = int(flags_np.sum(dtype=np.int64))
        ms = time_region(torch, stream, lambda: ss.compact_u32(keys, flags, kout, dcount, stream=sh), 20)
        rows[f"cmp_p{p}"] = entry(nk * 5 + 4 * kept + 8, ms)
        unord.append(_sig(time_region(torch, stream, lambda: ss.ss_compact_u32_unordered(
            keys, flags, kout, dcount, stream=sh), 20)))
        del flags
    rows["cmp_unord_ms"] = unord
    del keys
    # predicate compaction (keep v > 0, fp32, no flag array), on 4n + 4k bytes; unordered ms
    unord = []
    for p in (0.01, 0.5, 0.99):
        xp = torch.from_numpy(si.workload_positive_f32(nk, p, seed=5)).to(dev)
        pout = kout.view(torch.float32)
        ss.compact_positive_f32(xp, pout, dcount, stream=sh)
        stream.synchronize()
        kept = int(dcount.item())
        ms = time_region(torch, stream, lambda: ss.compact_positive_f32(xp, pout, dcount, stream=sh), 20)
        rows[f"pos_p{p}"] = entry(nk * 4 + 4 * kept + 8, ms)
        unord.append(_sig(time_region(torch, stream, lambda: ss.ss_compact_positive_unordered(
            ss.SS_F32, xp, pout, dcount, stream=sh), 20)))
        del xp
    rows["pos_unord_ms"] = unord
    del kout
    # MoE counts and 64-aligned offsets, 256 experts, top-8: [us per call, us per graph replay]
    for tokens in (4096, 65536, 1 << 20):
        ids = torch.from_numpy(si.topk_ids(tokens, 8, 256, seed=6)).to(dev)
        cnt_e = torch.empty(256, dtype=torch.int32, device=dev)
        off_e = torch.empty(257, dtype=torch.int32, device=dev)
        ms = time_region(torch, stream, lambda: ss.ss_moe_counts_offsets(ids, 256, 64, cnt_e, off_e, stream=sh), 100)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            ss.ss_moe_counts_offsets(ids, 256, 64, cnt_e, off_e, stream=sh)
        ms_g = time_region(torch, stream, graph.replay, 100)
        rows[f"moe_t{tokens}_us"] = [_sig(ms * 1e3, 3), _sig(ms_g * 1e3, 3)]
        del graph, ids
    # scans with 64-bit sums at n = 1e8: uint32 -> uint64 (12 B per element), int64 and fp64 (16 B)
    w_in = torch.from_numpy(si.uniform_u32(N, seed=60).view(np.int32)).to(dev)
    w_64 = torch.from_numpy(si.uniform_f32(N, seed=64).astype(np.float64)).to(dev)
    w_out = torch.empty(N, dtype=torch.float64, device=dev)
    for name, fn, per in (
            ("u32_u64", lambda: ss.ss_scan_wide(ss.SS_WIDE_U32_U64, True, w_in, w_out, stream=sh), 12),
            ("i64", lambda: ss.ss_scan_wide(ss.SS_WIDE_I64, True, w_64.view(torch.int64), w_out, stream=sh), 16),
            ("f64", lambda: ss.ss_scan_wide(ss.SS_WIDE_F64, True, w_64, w_out, stream=sh), 16)):
        ms = time_region(torch, stream, fn, 20)
        rows[f"{name}_1e8"] = entry(per * N, ms)
    # fp64 is bound by FP64 adds on this GPU: a third number, the fraction of the nominal
    # FP64 add rate (FP64_DADD_PER_S) at the kernel's FP64_ADDS_PER_ELEM adds per element
    rows["f64_1e8"].append(round(FP64_ADDS_PER_ELEM * N / (rows["f64_1e8"][0] * 1e-3) / FP64_DADD_PER_S, 3))
    del w_in, w_64, w_out
    # batched per-row fp32 inclusive scans: top-p over a 128,256-entry vocabulary, and short rows
    for r_, c_ in ((512, 128256), (262144, 256), (16384, 4096)):
        xr = torch.from_numpy(si.uniform_f32(r_ * c_, seed=82)).to(dev)
        orr = torch.empty_like(xr)
        rows[f"rows_{r_}x{c_}"] = entry(8 * r_ * c_, time_region(
            torch, stream, lambda: ss.ss_scan_rows(ss.SS_F32, True, xr, orr, r_, c_, stream=sh), 20))
        del xr, orr
    # segmented fp32 inclusive scans, n = 1e8, by mean segment length: [ms, frac on 2n
    # bytes, frac on 2n bytes plus the 8-byte segment starts that the call reads]
    xs_seg = torch.from_numpy(si.uniform_f32(N, seed=96)).to(dev)
    os_seg = torch.empty_like(xs_seg)
    for mean in (128256.0, 100.0, 4.0):
        off = torch.from_numpy(si.segment_offsets(N, mean, seed=98).astype(np.int64)).to(dev)
        ms = time_region(torch, stream, lambda: ss.ss_scan_segments(ss.SS_F32, True, xs_seg, os_seg, off, stream=sh), 20)
        rows[f"seg_mean{int(mean)}"] = entry(8 * N, ms) + entry(8 * N + 8 * (off.numel() - 1), ms)[1:]
        del off
    del xs_seg, os_seg, scratch

    # context only: torch.cumsum on the same int32 input, timed the same way
    def cumsum():
        with torch.cuda.stream(stream):  # torch ops run on torch's current stream
            torch.cumsum(xs_d, 0, dtype=torch.int32, out=out_d)
    rows["cumsum_1e8"] = entry(8 * N, time_region(torch, stream, cumsum, 20))
    return rows


def run_ours(args) -> None:
    import torch
    import seeded_inputs as si
    import stream_compaction_pass_gb300 as ss

    rank, world, local = dist_env()
    assert torch.cuda.is_available(), "bench.py needs a CUDA device"
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    ss.lib()  # fail loudly if the library is missing
    if args.config is not None:
        ss.ss_set_scan_config(args.config)

    xs = si.workload_int_pm1000(N, seed=2)
    xf = si.workload_f32_unit(N, seed=1)
    stream = torch.cuda.Stream(device=dev)
    sh = stream.cuda_stream
    with torch.cuda.stream(stream):
        xs_d = torch.from_numpy(xs).to(dev)
        xf_d = torch.from_numpy(xf).to(dev)
        out_i = torch.empty_like(xs_d)
        out_f = torch.empty_like(xf_d)
    torch.cuda.synchronize()

    launches = [
        lambda: ss.scan_exclusive_i32(xs_d, out_i, N, stream=sh),
        lambda: ss.scan_inclusive_i32(xs_d, out_i, N, stream=sh),
        lambda: ss.scan_exclusive_f32(xf_d, out_f, N, stream=sh),
        lambda: ss.scan_inclusive_f32(xf_d, out_f, N, stream=sh),
    ]

    def step():
        for f in launches:
            f()

    # correctness before timing: one step checked against the oracle (rank 0)
    if rank == 0 and not args.skip_check:
        import oracle as orc
        launches[0]()
        torch.cuda.synchronize()
        assert np.array_equal(out_i.cpu().numpy(), orc.scan_i32(xs, False)), "int32 scan mismatch"
        launches[3]()
        torch.cuda.synchronize()
        err = orc.fp32_normalised_error(out_f.cpu().numpy(), orc.scan_f32(xf, True), xf)
        assert err <= 1e-4, f"fp32 scan error {err}"

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    st, _ = ss.ss_stream_status(sh)
    assert st == ss.SS_OK

    # The timed region: K steps between two events on the launching stream.  No event sits
    # between launches (each one adds ~2 us of gap), so the mean launch duration of the scan
    # kernel is the region's time over its launches, inter-launch gaps included.
    sampler = ClockSampler(gpu_uuid(torch, dev)) if rank == 0 else None
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for _ in range(args.steps):
        for f in launches:
            f()
    t_end.record(stream)
    t_end.synchronize()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop() if sampler else None
    elapsed_ms = t_start.elapsed_time(t_end)
    mean_launch_ms = elapsed_ms / (len(launches) * args.steps)
    st, tile = ss.ss_stream_status(sh)
    assert st == ss.SS_OK, f"device status {st} at tile {tile}"

    elapsed_ms = max_over_ranks(elapsed_ms, dev)
    value = whole_job_rate(len(launches) * N * args.steps, world, elapsed_ms)
    ms_per_step = elapsed_ms / args.steps

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    # roofline of the dominant kernel (the look-back scan: every launch of the step)
    peak, peak_src = measured_hbm_peak()
    achieved = BYTES_PER_ELEM * N / (mean_launch_ms * 1e-3) / 1e9
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": recorded_traffic(), "kernel": "k_scan_lookback_pipe_sb",
                "mean_launch_ms": _sig(mean_launch_ms, 5), "peak_source": peak_src,
                "frac_of_nominal_8TBs": round(achieved / 8000.0, 4)}
    # the four variants one by one (after the timed region): each repeated back to back
    by_variant = {}
    for v, f in zip(VARIANTS, launches):
        by_variant[v] = time_region(torch, stream, f, 10)

    # end to end through the host-memory API: pinned host in, pinned host out
    e2e_steps = max(1, min(args.steps, args.e2e_steps))
    h_in_i = torch.from_numpy(xs).pin_memory()
    h_in_f = torch.from_numpy(xf).pin_memory()
    h_out_i = torch.empty_like(h_in_i).pin_memory()
    h_out_f = torch.empty_like(h_in_f).pin_memory()

    def e2e_step():
        ss.ss_scan_host(ss.SS_I32, False, h_in_i, h_out_i, N, stream=sh)
        ss.ss_scan_host(ss.SS_I32, True, h_in_i, h_out_i, N, stream=sh)
        ss.ss_scan_host(ss.SS_F32, False, h_in_f, h_out_f, N, stream=sh)
        ss.ss_scan_host(ss.SS_F32, True, h_in_f, h_out_f, N, stream=sh)

    e2e_step()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    e2e_s = time.perf_counter() - t0
    e2e = {"value": _sig(4 * N * e2e_steps / e2e_s / 1e9), "unit": UNIT,
           "h2d_bytes_per_step": 4 * N * 4, "d2h_bytes_per_step": 4 * N * 4, "steps": e2e_steps,
           "api": "ss_scan_host, pinned host buffers"}

    rows = {} if args.no_rows else row_rates(torch, ss, stream, dev, xs_d, xf_d, out_i, by_variant)
    cpu = None if args.no_cpu else cpu_baseline(xs, xf, budget_s=args.cpu_budget)

    emit({"metric": METRIC, "value": _sig(value, 5), "unit": UNIT, "n_gpus": world, "steps": args.steps,
          "warmup": args.warmup, "ms_per_step": _sig(ms_per_step, 5), "higher_is_better": True,
          "scaling": "weak", "vs_baseline": None, "dtype": "int32/fp32", "data": DATA,
          "config": {"workload": WORKLOAD, "n": N, "l2": "no flush: inputs > L2",
                     "parallelism": "replicas" if world > 1 else "single GPU",
                     "tile_elems": ss.ss_scan_tile_elems(),
                     "scan_config": "library default" if args.config is None else args.config},
          "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
          "gpu_launches": len(launches) * args.steps, "clocks": clocks,
          "rows_unit": "[ms, frac of HBM peak] unless named _us/_ms",
          "rows": rows})
    if world > 1:
        torch.distributed.destroy_process_group()


def profile_ablations(n: int) -> None:
    """One warm-up and one measured launch of each reduce-then-scan ablation
    (int32 exclusive, seeded [-1000, 1000] input), for a profiler to capture;
    checks the result of each against the oracle."""
    import torch
    import seeded_inputs as si
    import stream_compaction_pass_gb300 as ss
    import oracle as orc
    x = si.workload_int_pm1000(n, seed=2)
    ref = orc.scan_i32(x, False)
    d = torch.from_numpy(x).cuda()
    o = torch.empty_like(d)
    for algo in (ss.SS_ALGO_REDUCE_THEN_SCAN, ss.SS_ALGO_RTS_BLELLOCH, ss.SS_ALGO_RTS_BLELLOCH_PAD32,
                 ss.SS_ALGO_RTS_BLELLOCH_PAD2):
        for _ in range(2):
            ss.ss_scan(ss.SS_I32, False, algo, d, o)
        torch.cuda.synchronize()
        assert np.array_equal(o.cpu().numpy(), ref), f"ablation {algo} mismatch"
    print(f"ablations ok at n={n}")


def profile_compaction(n: int, p: float, predicate: bool = False) -> None:
    """Two launches of the default (flag) compaction at n keys, keep
    probability p (the compaction workload's generators), for a profiler to
    capture; checks the result against the oracle.  With `predicate`, the
    fp32 `v > 0` compaction of the predicate workload instead."""
    import torch
    import seeded_inputs as si
    import stream_compaction_pass_gb300 as ss
    import oracle as orc
    if predicate:
        x = si.workload_positive_f32(n, p, seed=5)
        ref = orc.compact_positive_f32(x)
        dx = torch.from_numpy(x).cuda()
        do = torch.empty_like(dx)
        cnt = torch.zeros(1, dtype=torch.int64, device="cuda")
        for _ in range(2):
            ss.compact_positive_f32(dx, do, cnt)
        torch.cuda.synchronize()
        c = int(cnt.item())
        assert c == ref.size and np.array_equal(do[:c].cpu().numpy().view(np.uint32), ref.view(np.uint32)), \
            "predicate compaction mismatch"
        print(f"predicate compaction ok at n={n}, p={p}, kept {c}")
        return
    keys, flags = si.workload_compaction(n, p, seed=3)
    ref = orc.compact_u32(keys, flags)
    dk = torch.from_numpy(keys.view(np.int32)).cuda()
    df = torch.from_numpy(flags).cuda()
    do = torch.empty_like(dk)
    cnt = torch.zeros(1, dtype=torch.int64, device="cuda")
    for _ in range(2):
        ss.compact_u32(dk, df, do, cnt)
    torch.cuda.synchronize()
    c = int(cnt.item())
    assert c == ref.size and np.array_equal(do[:c].cpu().numpy().view(np.uint32), ref), "compaction mismatch"
    print(f"compaction ok at n={n}, p={p}, kept {c}")


def profile_segments(n: int, mean: float) -> None:
    """Two launches of the fp32 inclusive segmented scan at n elements with
    segments of mean length `mean` (the segment workload's generators), for
    a profiler to capture; checks sampled segments against the oracle."""
    import torch
    import seeded_inputs as si
    import stream_compaction_pass_gb300 as ss
    import oracle as orc
    x = si.uniform_f32(n, seed=96)
    off = si.segment_offsets(n, mean, seed=98)
    dx = torch.from_numpy(x).cuda()
    do = torch.empty_like(dx)
    doff = torch.from_numpy(off.astype(np.int64)).cuda()
    for _ in range(2):
        ss.ss_scan_segments(ss.SS_F32, True, dx, do, doff)
    torch.cuda.synchronize()
    got = do.cpu().numpy()
    for s_ in np.linspace(0, off.size - 2, 5).astype(np.int64):  # whole segments, checked one by one
        a, b = int(off[s_]), int(off[s_ + 1])
        ref = orc.scan_f32(x[a:b], True)
        err = orc.fp32_normalised_error(got[a:b], ref, x[a:b]) if b > a else 0.0
        assert err <= 1e-4, f"segment {s_} error {err}"
    print(f"segmented scan ok at n={n}, mean {mean}, {off.size - 1} segments")


def profile_f64(n: int) -> None:
    """Two launches of the fp64 inclusive scan at n elements (seeded, values
    24-bit fractions scaled over 2^-10 .. 2^10), for a profiler to capture;
    checks the result against the oracle within the fp64 bound."""
    import torch
    import seeded_inputs as si
    import stream_compaction_pass_gb300 as ss
    import oracle as orc
    x = (si.uniform_f32(n, seed=64).astype(np.float64) - 0.5) * np.exp2(
        si.uniform_int32(n, -10, 10, seed=65).astype(np.float64))
    d = torch.from_numpy(x).cuda()
    o = torch.empty_like(d)
    for _ in range(2):
        ss.scan_inclusive_f64(d, o)
    torch.cuda.synchronize()
    err = float(np.max(np.abs(o.cpu().numpy() - orc.scan_f64(x, True)) / np.maximum(1.0, orc.abs_prefix_f64(x))))
    bound = (7 * ((n + 8191) // 8192) + 64) * 2.0 ** -53
    assert err <= bound, f"fp64 error {err} above {bound}"
    print(f"fp64 scan ok at n={n}, normalised error {err:.2e}")


def profile_wide(n: int) -> None:
    """Two launches each of the uint32 -> uint64 inclusive scan and the int64
    exclusive scan at n elements (seeded uniform words), for a profiler to
    capture; checks both against the oracle."""
    import torch
    import seeded_inputs as si
    import stream_compaction_pass_gb300 as ss
    import oracle as orc
    xu = si.uniform_u32(n, seed=60)
    x64 = ((si.uniform_u32(n, seed=62).astype(np.uint64) << np.uint64(32)) |
           si.uniform_u32(n, seed=63).astype(np.uint64)).view(np.int64)
    du = torch.from_numpy(xu.view(np.int32)).cuda()
    d64 = torch.from_numpy(x64).cuda()
    o = torch.empty(n, dtype=torch.int64, device="cuda")
    for _ in range(2):
        ss.ss_scan_wide(ss.SS_WIDE_U32_U64, True, du, o)
    torch.cuda.synchronize()
    assert np.array_equal(o.cpu().numpy().view(np.uint64), orc.scan_u32_u64(xu, True)), "uint32 -> uint64 mismatch"
    for _ in range(2):
        ss.ss_scan_wide(ss.SS_WIDE_I64, False, d64, o)
    torch.cuda.synchronize()
    assert np.array_equal(o.cpu().numpy(), orc.scan_i64(x64, False)), "int64 mismatch"
    print(f"64-bit sum scans ok at n={n}")


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=None,
                    help="single-pass tile configuration (default: the library's)")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--no-rows", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--skip-check", action="store_true")
    ap.add_argument("--profile-ablations", type=int, default=0, metavar="N",
                    help="only run each ablation twice at n=N (for a profiler) and exit")
    ap.add_argument("--profile-compaction", type=int, default=0, metavar="N",
                    help="only run the default compaction twice at n=N (for a profiler) and exit")
    ap.add_argument("--keep-p", type=float, default=0.5, help="keep probability for --profile-compaction")
    ap.add_argument("--predicate", action="store_true",
                    help="with --profile-compaction: the fp32 v > 0 compaction instead of the flag form")
    ap.add_argument("--profile-segments", type=int, default=0, metavar="N",
                    help="only run the fp32 segmented scan twice at n=N (for a profiler) and exit")
    ap.add_argument("--mean", type=float, default=128256.0, help="mean segment length for --profile-segments")
    ap.add_argument("--profile-f64", type=int, default=0, metavar="N",
                    help="only run the fp64 inclusive scan twice at n=N (for a profiler) and exit")
    ap.add_argument("--profile-wide", type=int, default=0, metavar="N",
                    help="only run the uint32 -> uint64 and int64 scans twice each at n=N (for a profiler) and exit")
    args = ap.parse_args()
    if args.profile_wide:
        profile_wide(args.profile_wide)
        return
    if args.profile_segments:
        profile_segments(args.profile_segments, args.mean)
        return
    if args.profile_f64:
        profile_f64(args.profile_f64)
        return
    if args.profile_compaction:
        profile_compaction(args.profile_compaction, args.keep_p, args.predicate)
        return
    if args.profile_ablations:
        profile_ablations(args.profile_ablations)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
