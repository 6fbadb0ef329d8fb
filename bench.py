#!/usr/bin/env python
"""Benchmark of the tile-primitive matrix multiply D = A.B + beta.C on GB300.

One step is one call of the library's public C-ABI entry point (tpgemm_gemm)
on one batch of seeded synthetic operands already resident in HBM: the whole
hot path (TMA ring -> tcgen05.mma -> tensor-memory epilogue with beta.C) in
one kernel launch. The default workload is the 8192^3 bf16 problem with B
stored [N, K] and beta = 1, the shape the GEMM TFLOP/s metric is quoted on.

Prints ONE JSON line (rank 0): metric, value (whole-job TFLOP/s), timing,
clocks sampled during the timed region, the roofline of the kernel, an
end-to-end number through host buffers, and the CPU oracle timed on a bounded
sample of the same workload. ``--impl reference`` times that oracle alone, as
the reference arm. With several GPUs (torchrun) every rank runs an independent
replica: the method has no exchange step.
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
KERNEL_SOURCES = ["tile_primitive_tensor_gb300/csrc/tc_gemm.cu",
                  "tile_primitive_tensor_gb300/csrc/ptx.cuh",
                  "tile_primitive_tensor_gb300/csrc/tpgemm_api.cu"]


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def parse_args():
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
    return ap.parse_args()


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


def load_traffic(workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it matches this kernel."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(workload)
    if not e or e.get("kernel_hash") != kernel_hash():
        return None
    return e.get("traffic_bytes_per_launch")


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons for one GPU."""

    FIELDS = ("timestamp,pci.bus_id,clocks.sm,clocks.max.sm,power.draw,"
              "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id: str | None):
        self.bus_id = (bus_id or "").lower()
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
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
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float):
        s = [x for x in self.samples if t0 <= x["t"] <= t1]
        if not s:
            s = self.samples[-3:]
        if not s:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        reasons = [r for r in ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                               "sw_power_cap") if any(x[r] for x in s)]
        pw = [x["power"] for x in s if x["power"] is not None]
        return {"sm_mhz": statistics.median(x["sm"] for x in s),
                "sm_max_mhz": max(x["sm_max"] for x in s), "reasons": reasons,
                "samples": len(s), "power_w_max": max(pw) if pw else None}


# ---------------------------------------------------------- across ranks
def max_over_ranks(ms: float, world: int, device="cpu") -> float:
    """The slowest rank's time, on every rank (one replica per GPU: the job
    takes as long as its slowest replica)."""
    if world <= 1:
        return ms
    import torch
    t = torch.tensor([ms], device=device, dtype=torch.float64)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_tflops(world: int, flops_per_step: float, steps: int, total_ms: float) -> float:
    """Whole-job throughput: the work of all replicas over the slowest one's time."""
    return world * flops_per_step * steps / (total_ms * 1e-3) / 1e12


# -------------------------------------------------------------- CPU oracle
def oracle_sample(w, A, B, C, seconds: float, seed: int = 0):
    """Time the CPU oracle on a bounded sample of output entries of workload w.

    Returns (tflops, entries, elapsed, threads). Each entry is one full
    K-long dot product computed by the oracle from the 16-bit operands.
    """
    import numpy as np

    import oracle
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
    return (f"{n} output entries of D at seeded uniform positions (of {w.M}x{w.N}), each a "
            f"full {w.K}-long fp64 dot product from the 16-bit operands (oracle_gemm_entries)")


# ---------------------------------------------------------------- our arm
def run_ours(args, rank, world, local_rank):
    import torch

    import tile_primitive_tensor_gb300 as tp

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    w = wl.BY_NAME[args.workload]
    A, B, C = wl.make_inputs(w)
    Ad, Bd = A.to(dev), B.to(dev)
    Cd = None if C is None else C.to(dev)
    D = torch.empty(w.M, w.N, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    sh = int(stream.cuda_stream)
    lib = tp.library()
    plan = tp.tpgemm_describe_plan(w.M, w.N, w.K, w.transA, w.transB, w.dtype, w.beta)[1]
    dp, ap_, bp = D.data_ptr(), Ad.data_ptr(), Bd.data_ptr()
    cp = None if Cd is None else Cd.data_ptr()

    def step():
        st = lib.tpgemm_gemm(dp, ap_, bp, cp, w.M, w.N, w.K, int(w.transA), int(w.transB),
                             w.dtype, float(w.beta), sh)
        if st != 0:
            raise RuntimeError(f"tpgemm_gemm: {st} {tp.tpgemm_last_error_detail()}")

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    tp.check(tp.tpgemm_last_device_error())

    props = torch.cuda.get_device_properties(dev)
    bus = None
    if hasattr(props, "pci_bus_id"):
        bus = f"{getattr(props, 'pci_domain_id', 0):08x}:{props.pci_bus_id:02x}:" \
              f"{getattr(props, 'pci_device_id', 0):02x}.0"
    sampler = ClockSampler(bus)
    sampler.start()
    time.sleep(0.4)  # let nvidia-smi start before the timed region

    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    if args.flush_l2:
        # Cold L2 for every step: a 512 MB write between launches, outside the
        # per-launch events.
        scrub = torch.empty(128 * 1024 * 1024, dtype=torch.float32, device=dev)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        for a, b in evs:
            scrub.fill_(1.0)
            a.record(stream)
            step()
            b.record(stream)
        torch.cuda.synchronize()
        total_ms = sum(a.elapsed_time(b) for a, b in evs)
    else:
        # Events only around the whole timed loop: an event between two launches
        # would stop the next launch's set-up from overlapping the previous one.
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize()
        total_ms = ev0.elapsed_time(ev1)
    t_wall1 = time.time()
    if world > 1:
        torch.distributed.barrier()
    sampler.stop()
    tp.check(tp.tpgemm_last_device_error())
    total_ms = max_over_ranks(total_ms, world, dev)
    ms_per_step = total_ms / args.steps
    launch_ms = ms_per_step  # one launch of the kernel per step
    value = job_tflops(world, w.flops, args.steps, total_ms)
    clocks = sampler.summary(t_wall0, t_wall1)

    # ---- end to end through the host-buffer entry point: every step copies A,
    # B (and C) in from page-locked host memory and D back out, pipelined by
    # the library against the multiply of each row block.
    pin = lambda t: t.pin_memory()  # noqa: E731
    Ah, Bh = pin(A), pin(B)
    Ch = None if C is None else pin(C)
    Dh = torch.empty(w.M, w.N, dtype=torch.float32).pin_memory()
    h2d = A.numel() * A.element_size() + B.numel() * B.element_size() + \
        (0 if C is None else C.numel() * 4)
    d2h = w.M * w.N * 4
    del Ad, Bd, Cd, D
    torch.cuda.empty_cache()
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
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(ne):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / ne
    e2e_ms = max_over_ranks(e2e_ms, world, dev)
    e2e_value = job_tflops(world, w.flops, 1, e2e_ms)

    # ---- roofline of the (single) kernel of a step
    peaks, src = load_peaks()
    # fp8 runs at twice the dense bf16 rate (nominal 4.5 / 2.25 PFLOP/s): its
    # peak is the measured bf16 one times that ratio.
    ratio = 2.0 if w.dtype in (wl.E4M3, wl.E5M2) else 1.0
    t_peak = peaks["bf16_tflops"] * ratio
    t_sust = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]) * ratio
    ridge = t_peak * 1e12 / (peaks["hbm_gbs"] * 1e9)  # flop per byte
    tensor_bound = w.flops / w.algorithmic_bytes > ridge
    if tensor_bound:
        achieved = w.flops / (launch_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": round(achieved, 2),
                "peak": round(t_peak, 1), "unit": "TFLOP/s",
                "frac": round(achieved / t_peak, 4),
                "peak_kind": f"{src} bf16 dense burst" + (
                    " x 2 (nominal fp8 : bf16 ratio)" if ratio != 1.0 else ""),
                "frac_of_sustained": round(achieved / t_sust, 4)}
    else:
        achieved = w.algorithmic_bytes / (launch_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                "peak_kind": f"{src} HBM copy bandwidth"}
    roof["traffic"] = load_traffic(w.name)
    roof["algorithmic"] = w.flops if tensor_bound else w.algorithmic_bytes
    roof["kernel"] = plan

    out = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype":
            {wl.F16: "f16", wl.BF16: "bf16", wl.E4M3: "e4m3", wl.E5M2: "e5m2"}[w.dtype],
        "data": "synthetic (seeded, workloads.py)",
        "config": {**w.describe(), "l2": "flushed before every step (512 MB write)" if
                   args.flush_l2 else ("inputs larger than L2, no flush" if
                                       w.algorithmic_bytes > 129e6 else "warm L2 (inputs fit)"),
                   "parallelism": f"replicas x{world}"},
        "clocks": clocks,
        "gpu_launches": args.steps,
        "roofline": roof,
        "e2e": {"value": round(e2e_value, 2), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4)},
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, n, el, cores = oracle_sample(w, A, B, C, args.cpu_seconds)
        out["cpu_baseline"] = {"value": v, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                               "sample": sample_text(n, w), "seconds": round(el, 2)}
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


def main():
    args = parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args)), flush=True)
        return 0
    if args.primitive:
        if rank == 0:
            fn = {"tcgen05_cp": run_primitive_cp, "vcopy": run_primitive_vcopy}[args.primitive]
            print(json.dumps(fn(args)), flush=True)
        return 0
    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    try:
        out = run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(out), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
