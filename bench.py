#!/usr/bin/env python
"""Benchmark of the tile-primitive matrix multiply D = A.B + beta.C on GB300.

One step is one call of the library's public C-ABI entry point (tpgemm_gemm)
on one batch of seeded synthetic operands already resident in HBM: the whole
hot path (TMA ring -> tcgen05.mma -> tensor-memory epilogue with beta.C) in
one kernel launch. The default workload is the 8192^3 bf16 problem with B
stored [N, K] and beta = 1, the shape the GEMM TFLOP/s metric is quoted on.

Prints ONE JSON line: metric, value (TFLOP/s), timing, clocks sampled during
the timed region, the roofline of the kernel, an end-to-end number through host
buffers, the other measured configurations (4096^3 f16, and the skinny
144 x 16392 x 4104 shape both with L2 flushed before every launch and back to
back), and the CPU oracle timed on a bounded sample of the same workload.
``--impl reference`` times that oracle alone, as the reference arm.

The design is single-GPU: the multiply has no exchange step, and more GPUs
would only run independent copies of it, which this program does not do.
``--gpus`` above 1 (or a launch with WORLD_SIZE above 1) is refused with a
message, except for the reference arm, whose ranks other than 0 exit quietly.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

METRIC = "GEMM TFLOP/s (fp16/bf16->fp32) at 4096^3/8192^3; % of tensor peak or HBM roof"
DEFAULT_WORKLOAD = "gemm_8192_bf16_transB_beta1"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# The device code of the tcgen05 kernel. What the planner chooses for a
# workload (tile, ring, grid, orientation, last-wave split, L2 policies) is in
# its plan string, recorded beside each traffic figure.
KERNEL_SOURCES = ["tile_primitive_tensor_gb300/csrc/tc_gemm.cu",
                  "tile_primitive_tensor_gb300/csrc/ptx.cuh",
                  "tile_primitive_tensor_gb300/csrc/tpgemm_internal.h"]


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--primitive", choices=["tcgen05_cp", "vcopy"], default=None,
                    help="measure a standalone primitive instead of the GEMM step")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(wl.BY_NAME))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU time of the oracle sample")
    ap.add_argument("--e2e-steps", type=int, default=30)
    ap.add_argument("--flush-l2", action="store_true",
                    help="overwrite a buffer larger than L2 before every timed step (the GEMM "
                         "alone is timed, with events around each launch)")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other configurations (4096^3, skinny cold and warm)")
    ap.add_argument("--config-steps", type=int, default=50,
                    help="timed launches per configuration of the configs block")
    return ap.parse_args(argv)


def code_only(src: str) -> str:
    """C/C++/CUDA source with comments removed and whitespace runs collapsed, so
    that the kernel hash changes with the code, not with its commentary."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":  # string or character literal, copied whole
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_hash() -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            h.update(code_only(f.read()).encode())
    return h.hexdigest()[:16]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def load_traffic(workload: str, plan=None):
    """DRAM bytes per launch from a committed ncu summary, if it was taken of
    this kernel (same device-code hash) running this plan (when one is given)."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(workload)
    if not e or e.get("kernel_hash") != kernel_hash():
        return None
    if plan is not None and e.get("plan") != plan:
        return None
    return e.get("traffic_bytes_per_launch")


# ------------------------------------------------------------------ clocks
# NVML clock-event reason bits (nvml.h, nvmlClocksEventReason*).
_NVML_REASONS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
                 "hw_thermal_slowdown": 0x40}


class _Nvml:
    """The few read-only NVML queries the sampler needs, through ctypes on the
    driver's libnvidia-ml (no Python NVML package is required)."""

    NVML_CLOCK_SM = 1

    def __init__(self, bus_id: str | None):
        import ctypes
        self.c = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.dev = ctypes.c_void_p()
        r = -1
        if bus_id:
            r = self.lib.nvmlDeviceGetHandleByPciBusId_v2(bus_id.encode(), ctypes.byref(self.dev))
        if r != 0:
            r = self.lib.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(self.dev))
        if r != 0:
            raise OSError("no NVML device handle")
        fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None)
        self.reasons_fn = fn or self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        self.max_sm = self._uint(self.lib.nvmlDeviceGetMaxClockInfo, self.NVML_CLOCK_SM)

    def _uint(self, fn, *args):
        v = self.c.c_uint()
        if fn(self.dev, *args, self.c.byref(v)) != 0:
            return None
        return v.value

    def sample(self) -> dict | None:
        sm = self._uint(self.lib.nvmlDeviceGetClockInfo, self.NVML_CLOCK_SM)
        if sm is None:
            return None
        mw = self._uint(self.lib.nvmlDeviceGetPowerUsage)
        rs = self.c.c_ulonglong()
        bits = rs.value if self.reasons_fn(self.dev, self.c.byref(rs)) == 0 else 0
        d = {"t": time.time(), "sm": float(sm), "sm_max": float(self.max_sm or sm),
             "power": None if mw is None else mw / 1000.0}
        d.update({k: bool(bits & m) for k, m in _NVML_REASONS.items()})
        return d

    def close(self):
        self.lib.nvmlShutdown()


class ClockSampler:
    """SM clock, power and clock-event reasons of one GPU during a timed region.

    NVML is polled about every millisecond from a thread, so even a region of
    a few milliseconds holds samples; when NVML cannot be loaded, nvidia-smi
    samples every 50 ms. The summary uses only samples taken inside the
    region; if none fell inside it the clocks are null, with the reason."""

    SMI_FIELDS = ("timestamp,pci.bus_id,clocks.sm,clocks.max.sm,power.draw,"
                  "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
                  "clocks_event_reasons.hw_thermal_slowdown,"
                  "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id: str | None, period_s: float = 0.001):
        self.bus_id = (bus_id or "").lower()
        self.period = period_s
        self.samples = []
        self.source = None
        self.proc = None
        self.thread = None
        self.stop_flag = threading.Event()

    def start(self):
        try:
            nvml = _Nvml(self.bus_id or None)
        except (OSError, AttributeError):
            nvml = None
        if nvml is not None:
            self.source = f"nvml every {self.period * 1e3:g} ms"
            self.thread = threading.Thread(target=self._poll, args=(nvml,), daemon=True)
            self.thread.start()
            return
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.SMI_FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.source = "nvidia-smi every 50 ms"
        self.thread = threading.Thread(target=self._read_smi, daemon=True)
        self.thread.start()

    def _poll(self, nvml):
        try:
            while not self.stop_flag.is_set():
                d = nvml.sample()
                if d is not None:
                    self.samples.append(d)
                time.sleep(self.period)
        finally:
            nvml.close()

    def _read_smi(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            bus = parts[1].lower()
            if self.bus_id and not bus.endswith(self.bus_id[-12:]):
                continue
            try:
                self.samples.append({
                    "t": time.time(), "sm": float(parts[2]), "sm_max": float(parts[3]),
                    "power": float(parts[4]) if parts[4] not in ("[N/A]", "N/A") else None,
                    "hw_slowdown": parts[6] == "Active",
                    "hw_thermal_slowdown": parts[7] == "Active",
                    "sw_thermal_slowdown": parts[8] == "Active",
                    "sw_power_cap": parts[9] == "Active",
                })
            except ValueError:
                continue

    def stop(self):
        self.stop_flag.set()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float) -> dict:
        return summarize_clocks(self.samples, t0, t1, self.source)


def summarize_clocks(samples, t0: float, t1: float, source) -> dict:
    """Median SM clock, max clock and active reasons of the samples taken in
    [t0, t1]; null clocks with a reason when no sample fell inside."""
    s = [x for x in samples if t0 <= x["t"] <= t1]
    if not s:
        why = ("no clock sampler could be started" if source is None else
               f"no sample ({source}) fell inside the {1e3 * (t1 - t0):.1f} ms timed region")
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                "source": source, "null_reason": why}
    reasons = [r for r in ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                           "sw_power_cap") if any(x[r] for x in s)]
    pw = [x["power"] for x in s if x["power"] is not None]
    return {"sm_mhz": statistics.median(x["sm"] for x in s),
            "sm_max_mhz": max(x["sm_max"] for x in s), "reasons": reasons,
            "samples": len(s), "power_w_max": max(pw) if pw else None, "source": source}


def host_cpu() -> dict:
    """Model name and logical CPU count of the host the oracle runs on."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=20).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.TimeoutExpired):
        pass
    return {"cpu_model": model, "logical_cpus": os.cpu_count()}


# -------------------------------------------------------------- CPU oracle
def oracle_sample_mx(w, A, B, C, seconds: float):
    """The block-scaled oracle on the first rows of workload w (whole rows of D,
    each entry a full K-long dot product); returns as oracle_sample."""
    import oracle
    oracle.build()
    SFA, SFB = wl.make_scales(w)
    Bb, sfb = wl.operand_bits(w, B), SFB.numpy()
    Ab, sfa = wl.operand_bits(w, A).reshape(w.M, w.K), SFA.numpy()
    Cn = None if C is None else C.numpy()

    def run(rows):
        t = time.perf_counter()
        oracle.gemm_mx(Ab[:rows], Bb, None if Cn is None else Cn[:rows], sfa[:rows], sfb, rows,
                       w.N, w.K, False, True, w.dtype, w.beta)
        return time.perf_counter() - t

    tp_ = run(1)
    rows = int(max(1, min(w.M, seconds / max(tp_, 1e-6))))
    el = run(rows)
    return 2.0 * rows * w.N * w.K / el / 1e12, rows * w.N, el, oracle.num_threads()


def oracle_sample(w, A, B, C, seconds: float, seed: int = 0):
    """Time the CPU oracle on a bounded sample of output entries of workload w.

    Returns (tflops, entries, elapsed, threads). Each entry is one full
    K-long dot product computed by the oracle from the 16-bit operands.
    """
    import numpy as np

    import oracle
    if isinstance(w, wl.MxWorkload):
        return oracle_sample_mx(w, A, B, C, seconds)
    oracle.build()
    Ab, Bb = wl.bits(A), wl.bits(B)
    Cn = None if C is None else C.numpy()
    rng = np.random.default_rng(seed)

    def run(n):
        r = rng.integers(0, w.M, n)
        c = rng.integers(0, w.N, n)
        t = time.perf_counter()
        oracle.gemm_entries(r, c, Ab, Bb, Cn, w.M, w.N, w.K, w.transA, w.transB, w.dtype, w.beta)
        return time.perf_counter() - t

    probe = max(16, oracle.num_threads() * 4)
    tp = run(probe)
    n = int(max(1, min(2_000_000, probe * seconds / max(tp, 1e-6))))
    el = run(n)
    return 2.0 * n * w.K / el / 1e12, n, el, oracle.num_threads()


def sample_text(n, w):
    if isinstance(w, wl.MxWorkload):
        return (f"{n} output entries (the first {n // w.N} rows of D), each a full {w.K}-long "
                "fp64 dot product of the block-scaled fp8 operands (oracle_gemm_mx)")
    return (f"{n} output entries of D at seeded uniform positions (of {w.M}x{w.N}), each a "
            f"full {w.K}-long fp64 dot product from the 16-bit operands (oracle_gemm_entries)")


def oracle_full(w, A, B, C):
    """Seconds the CPU oracle takes for the whole output of workload w."""
    import oracle
    oracle.build()
    Ab, Bb = wl.bits(A), wl.bits(B)
    Cn = None if C is None else C.numpy()
    t = time.perf_counter()
    oracle.gemm(Ab, Bb, Cn, w.M, w.N, w.K, w.transA, w.transB, w.dtype, w.beta)
    return time.perf_counter() - t


# Whole-output oracle runs reported beside the sampled baseline: the shapes the
# oracle finishes in seconds on the host cores.
FULL_ORACLE_WORKLOADS = ("atom_16x8x16_f16_int", "gemm_256_bf16_transB_beta1",
                         "skinny_144x16392x4104_f16_beta1")


# ---------------------------------------------------------------- our arm
class Problem:
    """One workload's operands resident on the device and its launch."""

    def __init__(self, tp, w, dev, stream):
        import torch
        self.tp, self.w = tp, w
        self.A, self.B, self.C = wl.make_inputs(w)
        self.Ad, self.Bd = self.A.to(dev), self.B.to(dev)
        self.Cd = None if self.C is None else self.C.to(dev)
        self.D = torch.empty(w.M, w.N, dtype=torch.float32, device=dev)
        self.sh = int(stream.cuda_stream)
        self.lib = tp.library()
        self.mx = isinstance(w, wl.MxWorkload)
        cp = None if self.Cd is None else self.Cd.data_ptr()
        if self.mx:
            # Block-scaled fp8: scales and the scale-packing workspace (the
            # packing runs inside every step, before the GEMM).
            self.SFA, self.SFB = wl.make_scales(w)
            self.sfa, self.sfb = self.SFA.to(dev), self.SFB.to(dev)
            wsb = tp.tpgemm_gemm_mx_workspace_bytes(w.M, w.N, w.K)
            self.ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
            self.fn = self.lib.tpgemm_gemm_mx
            self.args = (self.D.data_ptr(), self.Ad.data_ptr(), self.Bd.data_ptr(), cp,
                         self.sfa.data_ptr(), self.sfb.data_ptr(), w.M, w.N, w.K, w.dtype,
                         float(w.beta), self.ws.data_ptr(), wsb, self.sh)
            self.step()
            torch.cuda.synchronize()
            self.plan = tp.tpgemm_last_plan()[1]
        else:
            self.fn = self.lib.tpgemm_gemm
            self.args = (self.D.data_ptr(), self.Ad.data_ptr(), self.Bd.data_ptr(), cp, w.M, w.N,
                         w.K, int(w.transA), int(w.transB), w.dtype, float(w.beta), self.sh)
            self.plan = tp.tpgemm_describe_plan(w.M, w.N, w.K, w.transA, w.transB, w.dtype,
                                                w.beta)[1]

    def step(self):
        st = self.fn(*self.args)
        if st != 0:
            raise RuntimeError(f"tpgemm_gemm: {st} {self.tp.tpgemm_last_error_detail()}")

    def copies(self, n: int):
        """n launch argument sets, each on its own device copy of A, B, C and D
        (the first is this one): cycling through them, no launch finds its
        operands in L2 when their total exceeds it."""
        import torch
        sets, keep = [self.args], []
        if self.mx:
            raise ValueError("rotating copies are for the plain multiply")
        for _ in range(n - 1):
            t = (self.Ad.clone(), self.Bd.clone(), None if self.Cd is None else self.Cd.clone(),
                 torch.empty_like(self.D))
            keep.append(t)
            sets.append((t[3].data_ptr(), t[0].data_ptr(), t[1].data_ptr(),
                         None if t[2] is None else t[2].data_ptr()) + self.args[4:])
        self._copies = keep
        it = {"i": 0}

        def step():
            a = sets[it["i"]]
            it["i"] = (it["i"] + 1) % len(sets)
            st = self.lib.tpgemm_gemm(*a)
            if st != 0:
                raise RuntimeError(f"tpgemm_gemm: {st} {self.tp.tpgemm_last_error_detail()}")
        return step

    def release(self):
        del self.Ad, self.Bd, self.Cd, self.D
        self._copies = []
        if self.mx:
            del self.sfa, self.sfb, self.ws


def time_back_to_back(step, stream, steps: int) -> float:
    """Total ms of `steps` launches between two events. No event sits between
    launches: one there would stop the next launch's set-up from overlapping
    the previous launch (programmatic dependent launch)."""
    import torch
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    return ev0.elapsed_time(ev1)


def scrub_l2(scrub):
    """Leave L2 cold and clean: write a buffer larger than L2, then read it
    back, so L2 holds only clean lines of that buffer (a write alone would
    leave it full of dirty lines, whose write-back the next kernel would pay)."""
    scrub.fill_(1.0)
    return scrub.sum()


def time_cold(step, stream, steps: int, scrub) -> list:
    """ms of each launch timed alone after scrub_l2 (outside its events), so
    every launch starts from a cold, clean L2."""
    import torch
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for a, b in evs:
        scrub_l2(scrub)
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def roofline_of(w, launch_ms: float, peaks: dict, src: str) -> dict:
    """Achieved rate of one launch against the bound of its workload: tensor
    peak above the ridge point, HBM bandwidth below it."""
    # fp8 runs at twice the dense bf16 rate (nominal 4.5 / 2.25 PFLOP/s): its
    # peak is the measured bf16 one times that ratio. fp4 runs on the same
    # kind::f8f6f4 MMA at the fp8 rate.
    ratio = 2.0 if w.dtype in (wl.E4M3, wl.E5M2, wl.E2M1) else 1.0
    t_peak = peaks["bf16_tflops"] * ratio
    t_sust = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]) * ratio
    ridge = t_peak * 1e12 / (peaks["hbm_gbs"] * 1e9)  # flop per byte
    if w.flops / w.algorithmic_bytes > ridge:
        achieved = w.flops / (launch_ms * 1e-3) / 1e12
        return {"bound": "tensor", "achieved": round(achieved, 2), "peak": round(t_peak, 1),
                "unit": "TFLOP/s", "frac": round(achieved / t_peak, 4),
                "peak_kind": f"{src} bf16 dense burst" + (
                    " x 2 (nominal fp8 : bf16 ratio; fp4 runs at the fp8 rate)"
                    if ratio != 1.0 else ""),
                "frac_of_sustained": round(achieved / t_sust, 4)}
    achieved = w.algorithmic_bytes / (launch_ms * 1e-3) / 1e9
    return {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
            "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
            "peak_kind": f"{src} HBM copy bandwidth"}


def config_entry(w, ms: float, peaks: dict, src: str, how: str) -> dict:
    r = roofline_of(w, ms, peaks, src)
    return {"us": round(ms * 1e3, 2), "tflops": round(w.flops / (ms * 1e-3) / 1e12, 2),
            "gbs": round(w.algorithmic_bytes / (ms * 1e-3) / 1e9, 1), "bound": r["bound"],
            "frac": r["frac"], "of": r["peak_kind"], "timing": how}


# Device copies of the operands cycled through in the rotating cold mode: three
# sets of the skinny shape are 464 MB, over three times L2.
COLD_SETS = 3


def measure_configs(args, tp, dev, stream, scrub, peaks, src) -> dict:
    """The other targets: 4096^3 f16 (tensor-bound) back to back, and the skinny
    144 x 16392 x 4104 shape (HBM-bound) cold and warm. Cold is measured two
    ways: back to back over COLD_SETS device copies of the operands (each
    launch's operands were last touched two launches earlier, with over twice
    L2 of other traffic since), and each launch alone after an L2 scrub
    (which adds the grid's launch latency to every launch)."""
    import torch
    out = {}
    n = max(3, args.config_steps)
    for name, modes in (("gemm_4096_f16", ("warm",)),
                        ("skinny_144x16392x4104_f16_beta1", ("cold", "cold_alone", "warm")),
                        ("gemm_8192_e4m3_transB_beta1", ("warm",)),
                        ("mx_8192_e4m3_transB_beta1", ("warm",)),
                        ("mxfp4_8192_transB_beta1", ("warm",))):
        w = wl.BY_NAME[name]
        pr = Problem(tp, w, dev, stream)
        for _ in range(5):
            pr.step()
        torch.cuda.synchronize()
        e = {"plan": pr.plan}
        if "cold" in modes:
            rot = pr.copies(COLD_SETS)
            for _ in range(2 * COLD_SETS):
                rot()
            torch.cuda.synchronize()
            ms = time_back_to_back(rot, stream, n) / n
            e["cold"] = config_entry(w, ms, peaks, src,
                                     f"mean of {n} launches back to back over {COLD_SETS} device "
                                     f"copies of the operands "
                                     f"({COLD_SETS * w.algorithmic_bytes / 1e6:.0f} MB)")
        if "cold_alone" in modes:
            t = sorted(time_cold(pr.step, stream, n, scrub))
            e["cold_alone"] = config_entry(
                w, statistics.median(t), peaks, src,
                f"median of {n} launches, each alone after a {scrub.numel() * 4 >> 20} MB "
                "write and read-back of a scrub buffer")
            e["cold_alone"]["best_us"] = round(t[0] * 1e3, 2)
        if "warm" in modes:
            ms = time_back_to_back(pr.step, stream, n) / n
            e["warm"] = config_entry(w, ms, peaks, src,
                                     f"mean of {n} launches back to back, no L2 flush")
        tp.check(tp.tpgemm_last_device_error())
        pr.release()
        torch.cuda.empty_cache()
        out[name] = e
    return out


# Side-by-side (not a target): the same multiplies through torch's cuBLAS GEMM.
CUBLAS_WORKLOADS = ("gemm_8192_bf16_transB_beta1", "gemm_4096_f16",
                    "skinny_144x16392x4104_f16_beta1")


def measure_cublas(args, dev, stream, peaks, src) -> dict:
    """Each workload's D = A.B (+ C) through torch.addmm / torch.mm with an f32
    output (cuBLAS, f16/bf16 in, f32 accumulate), or with a 16-bit output where
    this torch has no f32-output form; back to back, warm L2."""
    import torch
    out = {}
    n = max(3, args.config_steps)
    for name in CUBLAS_WORKLOADS:
        w = wl.BY_NAME[name]
        A, B, C = (None if t is None else t.to(dev) for t in wl.make_inputs(w))
        a = A.t() if w.transA else A
        b = B.t() if w.transB else B
        form = "f32 out"

        def f32_call():
            if w.beta:
                return torch.addmm(C, a, b, out_dtype=torch.float32)
            return torch.mm(a, b, out_dtype=torch.float32)

        try:
            f32_call()
            call = f32_call
        except (RuntimeError, TypeError):
            form = "16-bit out, no C (no f32-output form in this torch)"
            call = lambda: torch.mm(a, b)  # noqa: E731
        for _ in range(5):
            call()
        torch.cuda.synchronize()
        ms = time_back_to_back(call, stream, n) / n
        e = config_entry(w, ms, peaks, src, f"mean of {n} calls back to back, no L2 flush")
        e["form"] = f"torch {'addmm' if (w.beta and form == 'f32 out') else 'mm'}, {form}"
        out[name] = e
        del A, B, C, a, b
        torch.cuda.empty_cache()
    return out


def run_ours(args):
    import torch

    import tile_primitive_tensor_gb300 as tp

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    w = wl.BY_NAME[args.workload]
    stream = torch.cuda.current_stream()
    pr = Problem(tp, w, dev, stream)
    A, B, C = pr.A, pr.B, pr.C

    for _ in range(args.warmup):
        pr.step()
    torch.cuda.synchronize()
    tp.check(tp.tpgemm_last_device_error())

    props = torch.cuda.get_device_properties(dev)
    bus = None
    if hasattr(props, "pci_bus_id"):
        bus = f"{getattr(props, 'pci_domain_id', 0):08x}:{props.pci_bus_id:02x}:" \
              f"{getattr(props, 'pci_device_id', 0):02x}.0"
    sampler = ClockSampler(bus)
    sampler.start()
    time.sleep(0.2)  # let the sampler start before the timed region
    # 512 MB: larger than L2 (129 MB), written before each launch in the cold modes.
    scrub = torch.empty(128 * 1024 * 1024, dtype=torch.float32, device=dev)

    torch.cuda.synchronize()
    t_wall0 = time.time()
    if args.flush_l2:
        total_ms = sum(time_cold(pr.step, stream, args.steps, scrub))
    else:
        total_ms = time_back_to_back(pr.step, stream, args.steps)
    t_wall1 = time.time()
    sampler.stop()
    tp.check(tp.tpgemm_last_device_error())
    ms_per_step = total_ms / args.steps
    launch_ms = ms_per_step  # one launch of the kernel per step
    value = w.flops * args.steps / (total_ms * 1e-3) / 1e12
    clocks = sampler.summary(t_wall0, t_wall1)
    plan = pr.plan
    pr.release()
    torch.cuda.empty_cache()

    peaks, src = load_peaks()
    configs = None if args.no_configs else measure_configs(args, tp, dev, stream, scrub, peaks,
                                                            src)
    cublas = None if args.no_configs else measure_cublas(args, dev, stream, peaks, src)
    del scrub
    torch.cuda.empty_cache()

    # ---- end to end through the host-buffer entry point: every step copies A,
    # B (and C) in from page-locked host memory and D back out, pipelined by
    # the library against the multiply of each row block. (The block-scaled
    # multiply has no host-buffer entry point.)
    if isinstance(w, wl.MxWorkload):
        return finish_line(args, w, value, ms_per_step, launch_ms, clocks, plan, peaks, src,
                           configs, A, B, C, None, cublas)
    lib = tp.library()
    sh = int(stream.cuda_stream)
    pin = lambda t: t.pin_memory()  # noqa: E731
    Ah, Bh = pin(A), pin(B)
    Ch = None if C is None else pin(C)
    Dh = torch.empty(w.M, w.N, dtype=torch.float32).pin_memory()
    h2d = A.numel() * A.element_size() + B.numel() * B.element_size() + \
        (0 if C is None else C.numel() * 4)
    d2h = w.M * w.N * 4
    ws_bytes = lib.tpgemm_gemm_host_workspace_bytes(w.M, w.N, w.K, w.dtype, float(w.beta))
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    hp = (Dh.data_ptr(), Ah.data_ptr(), Bh.data_ptr(), None if Ch is None else Ch.data_ptr())

    def e2e_step():
        st = lib.tpgemm_gemm_host(*hp, w.M, w.N, w.K, int(w.transA), int(w.transB), w.dtype,
                                  float(w.beta), ws.data_ptr(), ws_bytes, sh)
        if st != 0:
            raise RuntimeError(f"tpgemm_gemm_host: {st} {tp.tpgemm_last_error_detail()}")

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    ne = max(1, min(args.e2e_steps, args.steps))
    e2e_ms = time_back_to_back(e2e_step, stream, ne) / ne
    tp.check(tp.tpgemm_last_device_error())
    e2e_value = w.flops / (e2e_ms * 1e-3) / 1e12
    e2e = {"value": round(e2e_value, 2), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4)}
    return finish_line(args, w, value, ms_per_step, launch_ms, clocks, plan, peaks, src, configs,
                       A, B, C, e2e, cublas)


def finish_line(args, w, value, ms_per_step, launch_ms, clocks, plan, peaks, src, configs,
                A, B, C, e2e, cublas=None):
    """The JSON line: roofline of the (single) kernel of a step, configs, CPU baseline."""
    # ---- roofline of the (single) kernel of a step
    roof = roofline_of(w, launch_ms, peaks, src)
    roof["traffic"] = load_traffic(w.name, plan)
    roof["algorithmic"] = w.flops if roof["bound"] == "tensor" else w.algorithmic_bytes
    roof["kernel"] = plan

    out = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype":
            {wl.F16: "f16", wl.BF16: "bf16", wl.E4M3: "e4m3", wl.E5M2: "e5m2",
             wl.E2M1: "e2m1"}[w.dtype],
        "data": "synthetic (seeded, workloads.py)",
        "config": {**w.describe(), "l2": "flushed before every step (512 MB write + read)" if
                   args.flush_l2 else ("inputs larger than L2, no flush" if
                                       w.algorithmic_bytes > 129e6 else "warm L2 (inputs fit)"),
                   "parallelism": "single GPU"},
        "clocks": clocks,
        # block-scaled steps launch the scale-packing kernel before the GEMM
        "gpu_launches": args.steps * (2 if isinstance(w, wl.MxWorkload) else 1),
        "roofline": roof,
        "e2e": e2e,
    }
    if configs is not None:
        out["configs"] = configs
    if cublas is not None:
        out["cublas_side_by_side"] = cublas
    if not args.no_cpu_baseline:
        v, n, el, cores = oracle_sample(w, A, B, C, args.cpu_seconds)
        full = {}
        for name in FULL_ORACLE_WORKLOADS:
            fw = wl.BY_NAME[name]
            full[name] = round(oracle_full(fw, *wl.make_inputs(fw)), 4)
        out["cpu_baseline"] = {"value": v, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                               "omp_threads": cores, **host_cpu(),
                               "sample": sample_text(n, w), "seconds": round(el, 2),
                               "full_output_seconds": full}
    return out


# ------------------------------------------------------ tcgen05.cp primitive
CP_REGIONS = [  # (form, lane pattern, rows, row bits): 16 KB or less per CTA per copy
    ("128x256b", 1, 0, 128, 1024),
    ("4x256b", 2, 1, 128, 256),
    ("128x128b", 3, 0, 128, 1024),
    ("64x128b.warpx2::02_13", 4, 2, 64, 1024),
    ("64x128b.warpx2::01_23", 5, 3, 64, 1024),
    ("32x128b.warpx4", 6, 4, 32, 1024),
]


# Issuing threads measured per tcgen05.cp form (lane 0 of warps 0..n-1 of the
# round-trip kernel); the reported value is the largest count's.
CP_ISSUERS = (1, 4, 8)


def run_primitive_cp(args):
    """Shared-memory -> tensor-memory copy throughput of every tcgen05.cp form.

    One CTA per SM, each issuing its planned copy of a 128B-swizzled region
    `repeat` times before one commit; bytes = shared-memory bytes read. The
    derived peak is the shared-memory read port, 128 B per clock per SM, at the
    SM clock sampled during the run."""
    import torch

    import tile_primitive_tensor_gb300 as tp

    dev = torch.device("cuda", 0)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    repeat = 4096
    sampler = ClockSampler(None)
    sampler.start()
    time.sleep(0.4)
    t0 = time.time()
    forms = {}
    for name, shape, lanes, rows, bits in CP_REGIONS:
        groups = (rows + 7) // 8
        lbo, sbo = groups * 1024, 1024
        atoms = (bits // 128 + 7) // 8
        nbytes = atoms * lbo
        image = torch.randint(0, 256, (nbytes,), dtype=torch.uint8, device=dev)
        ncols = max(32, bits // 32)
        out = torch.empty(sms * 128 * ncols, dtype=torch.int32, device=dev)
        d = tp.cp_desc(rows, bits, swizzle=tp.TPGEMM_CP_SWIZZLE_128B, lbo=lbo, sbo=sbo,
                       lanes=lanes, shape=shape)

        def go(r, issuers):
            st = tp.tpgemm_cp_roundtrip_repeat(out, image, nbytes, d, 0, ncols, r, sms, issuers)
            if st != 0:
                raise RuntimeError(f"tpgemm_cp_roundtrip_repeat: {tp.tpgemm_last_error_detail()}")

        region = rows * bits // 8
        instr = (rows // 4 if lanes == 1 else 1) * (bits // (256 if shape in (1, 2) else 128))
        forms[name] = {"bytes_per_cta_copy": region, "instructions": instr}
        for issuers in CP_ISSUERS:
            for _ in range(3):
                go(repeat, issuers)
            torch.cuda.synchronize()
            times = {}
            for r in (1, repeat):  # the fixed cost of a launch (image, fill, read-back) subtracts
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                for _ in range(args.steps):
                    go(r, issuers)
                e1.record()
                torch.cuda.synchronize()
                times[r] = e0.elapsed_time(e1) / args.steps
            tp.check(tp.tpgemm_last_device_error())
            per_copy_s = (times[repeat] - times[1]) * 1e-3 / (repeat - 1)
            key = "" if issuers == 1 else f"_{issuers}_issuers"
            forms[name]["GB_per_s" + key] = round(sms * region / per_copy_s / 1e9, 1)
            forms[name]["ns_per_copy" + key] = round(per_copy_s * 1e9, 2)
    t1 = time.time()
    sampler.stop()
    clocks = sampler.summary(t0, t1)
    mhz = clocks["sm_mhz"] or 2070.0
    peak = sms * 128 * mhz * 1e6 / 1e9
    for f in forms.values():
        f["frac"] = round(f["GB_per_s"] / peak, 4)
        for i in CP_ISSUERS[1:]:
            f[f"frac_{i}_issuers"] = round(f[f"GB_per_s_{i}_issuers"] / peak, 4)
    best = forms["128x256b"]
    top = CP_ISSUERS[-1]
    # The oracle beside it: rebuilding the expected tensor memory of one CTA's
    # 128x256b copy on the host cores.
    import numpy as np

    from oracle import tmem_cp as ocp
    words = np.random.default_rng(0).integers(0, 2 ** 32, (128, 32), dtype=np.uint64).astype(
        np.uint32)
    n, c0 = 0, time.perf_counter()
    while time.perf_counter() - c0 < 2.0:
        ocp.tmem_image(words, ocp.LANES_ROWS, 0, 0, 32, 0)
        n += 1
    cpu_s = (time.perf_counter() - c0) / n
    cpu = {"value": round(128 * 128 / cpu_s / 1e9, 4), "unit": "GB/s", "cores": 1,
           "kind": "oracle", "sample": f"{n} rebuilds of one CTA's 128 x 1024-bit copy "
                                       "(oracle.tmem_cp.tmem_image)"}
    return {
        "metric": "tcgen05.cp shared->tensor memory copy bandwidth (shared-memory bytes read)",
        "value": best[f"GB_per_s_{top}_issuers"], "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
        "higher_is_better": True, "dtype": "b32", "data": "synthetic (random bytes)",
        "config": {"workload": "tcgen05_cp_128B_swizzle", "ctas": sms, "repeat": repeat},
        "clocks": clocks,
        "roofline": {"bound": "smem", "achieved": best[f"GB_per_s_{top}_issuers"],
                     "peak": round(peak, 1), "unit": "GB/s", "frac": best[f"frac_{top}_issuers"],
                     "issuers": top,
                     "single_issuer_frac": best["frac"],
                     "peak_kind": f"derived: {sms} SMs x 128 B/clk x {mhz:.0f} MHz (sampled)",
                     "traffic": None},
        "forms": forms,
        "cpu_baseline": cpu,
        "gpu_launches": 2 * len(CP_ISSUERS) * args.steps * len(CP_REGIONS),
    }


# ------------------------------------------- vectorised global <-> shared copy
def run_primitive_vcopy(args):
    """HBM round trip through shared memory with the vectorised copy.

    Every CTA (a warpgroup scope, 128 threads) moves one 32 x 512 fp16 region
    (32 KB) of a 1 GiB buffer global -> shared -> global; bytes = read + write,
    against the measured HBM copy bandwidth (which counts the same way)."""
    import numpy as np
    import torch

    import tile_primitive_tensor_gb300 as tp
    from oracle import vec_copy as ovc

    dev = torch.device("cuda", 0)
    rows, cols, eb, threads = 32, 512, 2, 128
    region = rows * cols
    total = 1 << 30
    ctas = total // (region * eb)
    src = torch.empty(total, dtype=torch.uint8, device=dev).random_(0, 256)
    dst = torch.empty_like(src)
    d = tp.vcopy_desc(rows, cols, eb, threads=threads)
    plan = tp.tpgemm_vcopy_plan(d)[1]

    def go():
        st = tp.tpgemm_vcopy_roundtrip(dst, src, total, d, ctas, region)
        if st != 0:
            raise RuntimeError(f"tpgemm_vcopy_roundtrip: {tp.tpgemm_last_error_detail()}")

    for _ in range(max(3, args.warmup)):
        go()
    torch.cuda.synchronize()
    if not torch.equal(dst, src):
        raise RuntimeError("vectorised copy round trip differs from its source")
    sampler = ClockSampler(None)
    sampler.start()
    time.sleep(0.4)
    t0 = time.time()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        go()
    e1.record()
    torch.cuda.synchronize()
    t1 = time.time()
    sampler.stop()
    ms = e0.elapsed_time(e1) / args.steps
    gbs = 2 * total / (ms * 1e-3) / 1e9
    peaks, src_kind = load_peaks()
    # The oracle beside it: the identity copy of one CTA's region on the host.
    rng = np.random.default_rng(0)
    host = rng.integers(0, 256, region * eb, dtype=np.uint8)
    dd = {"rows": rows, "cols": cols, "elem_bytes": eb, "g_row_stride": cols, "g_offset": 0,
          "s_row_stride": cols, "s_offset": 0, "s_swizzle": 0}
    n, c0 = 0, time.perf_counter()
    while time.perf_counter() - c0 < 2.0:
        ovc.expected_dst(host, host, dd, 1, 0)
        n += 1
    cpu_s = (time.perf_counter() - c0) / n
    return {
        "metric": "vectorised global->shared->global copy bandwidth (bytes read + written)",
        "value": round(gbs, 1), "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True,
        "dtype": "f16", "data": "synthetic (random bytes)",
        "config": {"workload": "vcopy_32x512_f16_warpgroup", "buffer_bytes": total, "ctas": ctas,
                   "plan": plan, "l2": "inputs larger than L2, no flush"},
        "clocks": sampler.summary(t0, t1),
        "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": round(gbs / peaks["hbm_gbs"], 4),
                     "peak_kind": f"{src_kind} HBM copy bandwidth", "traffic": None},
        "cpu_baseline": {"value": round(2 * region * eb / cpu_s / 1e9, 4), "unit": "GB/s",
                         "cores": 1, "kind": "oracle",
                         "sample": f"{n} host copies of one CTA's region (oracle.vec_copy)"},
        "gpu_launches": args.steps,
    }


# ---------------------------------------------------------- reference arm
def run_reference(args):
    w = wl.BY_NAME[args.workload]
    A, B, C = wl.make_inputs(w)
    total = args.steps + args.warmup
    budget = 150.0  # seconds for the whole run
    per_step = max(0.02, budget / max(total, 1))
    # calibrate the number of entries per step
    _, n0, el0, _ = oracle_sample(w, A, B, C, 0.5, seed=1)
    per_entry = el0 / n0
    n_step = max(1, int(per_step / per_entry))
    import numpy as np

    import oracle
    Ab, Bb = wl.bits(A), wl.bits(B)
    Cn = None if C is None else C.numpy()
    rng = np.random.default_rng(2)

    def step():
        r = rng.integers(0, w.M, n_step)
        c = rng.integers(0, w.N, n_step)
        oracle.gemm_entries(r, c, Ab, Bb, Cn, w.M, w.N, w.K, w.transA, w.transB, w.dtype, w.beta)

    for _ in range(args.warmup):
        step()
    t = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t
    value = 2.0 * n_step * w.K * args.steps / el / 1e12
    cores = oracle.num_threads()
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic (seeded, workloads.py)",
        "config": {**w.describe(), "parallelism": "cpu oracle"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"per step: {sample_text(n_step, w)}"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


SINGLE_GPU = ("bench.py: single-GPU design; the multiply has no exchange step and this "
              "program runs no replicas, so --gpus must be 1 (WORLD_SIZE 1)")


def main(argv=None):
    args = parse_args(argv)
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args)), flush=True)
        return 0
    if args.gpus != 1 or world != 1:
        log(SINGLE_GPU)
        return 2
    if args.primitive:
        fn = {"tcgen05_cp": run_primitive_cp, "vcopy": run_primitive_vcopy}[args.primitive]
        print(json.dumps(fn(args)), flush=True)
        return 0
    print(json.dumps(run_ours(args)), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
