#!/usr/bin/env python3
"""Throughput of the batched Walsh-Hadamard transform on GB300.

Metric: FWT vectors/s (plus effective and per-kernel HBM GB/s against the
measured copy bandwidth).  One step = one full transform of every vector of the
workload's batch, with inputs resident in HBM.  The default workload is the
largest specified one, n = 24 (2^24 amplitudes), batch 16, split complex fp64
*and* the same states in split complex fp32 (6 GiB of input, out of place), the
multi-pass Kronecker path.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle, timed the same way

Multi-GPU runs (torchrun, one rank per GPU) replicate the per-rank workload
with no collective on the data path (weak scaling); rank 0 prints one JSON line.

The line: `value` (vectors/s, inputs resident in HBM), `kernels` (per-pass device
times from the library's event trace), `roofline` (the dominant pass against the
measured copy bandwidth, with its ncu DRAM traffic while the sources match the
committed capture), `per_config` (every specified shape on its own, beside the
time of a plain streaming kernel over the same bytes, and checked against the CPU
oracle), `e2e` (the same metric from pinned host arrays through the host-buffer
entry points, beside plain copies of the same bytes), `cpu_baseline` (the oracle on
the host cores) and `clocks` (sampled during the timed region).
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "FWT vectors/sec and achieved HBM GB/s vs n (fraction of GB300 ~8 TB/s peak)"
UNIT = "vectors/s"
FALLBACK_HBM_GBS = 6800.0
# named step workloads: each is a list of input shapes transformed once per step
STEP_WORKLOADS = {
    "n24_b16": ["n24_b16_c64", "n24_b16_c32"],
    "n18_b256_i32": ["n18_b256_i32"],
    "n14_b64_c32": ["n14_b64_c32"],
    "n12_b64_c32": ["n12_b64_c32"],
    "n10_b64_c32": ["n10_b64_c32"],
    "n24_b16_c64": ["n24_b16_c64"],
    "n24_b16_c32": ["n24_b16_c32"],
}
DEFAULT_WORKLOAD = "n24_b16"


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(STEP_WORKLOADS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--bits", default="",
                    help="LO,NBITS: time the transform over index bits [LO, LO+NBITS) only")
    ap.add_argument("--phase", action="store_true",
                    help="time the fused phase + transform (fp32 parts; random per-vector angles)")
    ap.add_argument("--batch", type=int, default=0,
                    help="override the batch of every part (small cases for profiling; 0 = as specified)")
    ap.add_argument("--e2e-steps", type=int, default=25)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-sample", type=int, default=8,
                    help="vectors per part in the cpu_baseline sample of our arm")
    ap.add_argument("--ref-sample", type=int, default=0,
                    help="vectors per part in each step of the reference (CPU oracle) arm "
                         "(0 = enough to keep every host core busy)")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the per-configuration measurements (all specified shapes)")
    return ap.parse_args(argv)


# ---- distributed helpers (also exercised on CPU with gloo by the tests) ------------------

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, local, world


def rank_seed(base: int, rank: int) -> int:
    """Rank 0 draws the specified states; other ranks draw their own batch."""
    return base if rank == 0 else base + 1000 * rank


def dist_max(value: float, device=None) -> float:
    """Maximum of a float over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()):
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(device=None):
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized():
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# ---- clocks during the timed region ------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(1.0)  # let the sampler start before the timed region

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def mark(self):
        return len(self.lines)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)

    def summary(self, first: int, last: int):
        rows = []
        for line in self.lines[first:last]:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), parts[3:]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        reasons = set()
        for _, _, flags in rows:
            for name, flag in zip(self.REASONS, flags[1:]):
                if flag.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r[0] for r in rows),
                "sm_max_mhz": max(r[1] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows)}


class NvmlSampler:
    """The same clock record from NVML (the driver's libnvidia-ml) through ctypes, read
    every few milliseconds in a thread, so a timed region of ~100 ms still holds tens
    of samples.  Reads only; changes no setting."""

    # clocks event reason bits (nvml.h)
    REASON_BITS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
                   "hw_thermal_slowdown": 0x40, "hw_power_brake_slowdown": 0x80}

    def __init__(self, gpu_uuid: str, period_s: float = 0.005):
        import ctypes

        self.period = period_s
        self.samples = []  # (sm_mhz, sm_max_mhz, reasons bits, power_w)
        self._stop = threading.Event()
        self.thread = None
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.dev = ctypes.c_void_p()
        if self.lib.nvmlDeviceGetHandleByUUID(gpu_uuid.encode(), ctypes.byref(self.dev)) != 0:
            raise OSError("no NVML device for " + gpu_uuid)
        self._reasons = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        if self._read() is None:
            raise OSError("NVML clock query failed")

    def _read(self):
        import ctypes

        sm, mx, pw = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.dev, 1, ctypes.byref(sm)) != 0:  # NVML_CLOCK_SM
            return None
        if self.lib.nvmlDeviceGetMaxClockInfo(self.dev, 1, ctypes.byref(mx)) != 0:
            return None
        if self._reasons(self.dev, ctypes.byref(rs)) != 0:
            return None
        power = pw.value / 1000.0 if self.lib.nvmlDeviceGetPowerUsage(self.dev, ctypes.byref(pw)) == 0 else None
        return (float(sm.value), float(mx.value), int(rs.value), power)

    def start(self):
        def run():
            while not self._stop.is_set():
                r = self._read()
                if r is not None:
                    self.samples.append(r)
                self._stop.wait(self.period)

        self.thread = threading.Thread(target=run, daemon=True)
        self.thread.start()
        time.sleep(0.05)

    def mark(self):
        return len(self.samples)

    def stop(self):
        self._stop.set()
        if self.thread is not None:
            self.thread.join(timeout=2)

    def summary(self, first: int, last: int):
        rows = self.samples[first:last]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0,
                    "source": "nvml"}
        reasons = sorted({name for r in rows for name, bit in self.REASON_BITS.items() if r[2] & bit})
        powers = [r[3] for r in rows if r[3] is not None]
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows),
                "power_w_max": round(max(powers), 1) if powers else None, "source": "nvml, 5 ms"}


def clock_sampler(uuid: str):
    """NVML sampler when the driver library answers, else nvidia-smi at 100 ms."""
    uid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    try:
        return NvmlSampler(uid)
    except (OSError, AttributeError):
        return ClockSampler(uid)


# ---- roofline inputs ---------------------------------------------------------------

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs: torch copy, burst)"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback (6.8 TB/s, one earlier GB300 copy measurement)"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "walsh_hadamard_transform_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh")):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def ncu_record(kernel_key: str):
    """The committed ncu DRAM record of `kernel_key` (profiles/ncu_traffic.json), or
    None when there is none or the kernel sources changed since it was captured."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    rec = d.get(kernel_key)
    if not rec or rec.get("source_sha") != kernel_source_hash():
        return None
    return rec


def ncu_traffic(kernel_key: str):
    """DRAM bytes (read + write) of one launch of `kernel_key` at the specified batch."""
    rec = ncu_record(kernel_key)
    return None if rec is None else rec.get("dram_bytes_per_launch")


def ncu_bytes_per_vector(kernel_key: str):
    """DRAM bytes (read + write) a launch of `kernel_key` moves per vector: the slope of a
    fit over two batch sizes when captured that way (the L2's fixed share of dirty
    lines at the end of a launch drops out), else one capture divided by its batch."""
    rec = ncu_record(kernel_key)
    return None if rec is None else rec.get("dram_bytes_per_vector")


# ---- our CUDA path ---------------------------------------------------------------

def pass_names(w, fwt):
    f = fwt.plan_factors(w.n, w.dtype)
    names = []
    for i, k in enumerate(f):
        kind = "single" if len(f) == 1 else ("row" if i == 0 else "col")
        names.append(f"{w.dtype} {kind} pass K={k} (n={w.n})")
    return names


def run_ours(args):
    import numpy as np
    import torch

    import walsh_hadamard_transform_gb300 as fwt
    from walsh_hadamard_transform_gb300 import inputs

    rank, local, world = dist_env()
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    fwt.library()

    parts = [inputs.WORKLOADS[name] for name in STEP_WORKLOADS[args.workload]]
    if args.batch > 0:
        parts = [dataclasses.replace(w, batch=args.batch) for w in parts]
    host, dev_in, dev_out = [], [], []
    for w in parts:
        re, im = inputs.draw(w.values, w.n, w.batch, rank_seed(w.seed, rank), w.dtype)
        host.append((re, im))
        dev_in.append((torch.from_numpy(re).to(device), torch.from_numpy(im).to(device)))
        dev_out.append((torch.empty_like(dev_in[-1][0]), torch.empty_like(dev_in[-1][1])))
    torch.cuda.synchronize(device)

    bits = tuple(int(v) for v in args.bits.split(",")) if args.bits else None
    if args.phase:
        parts_idx = [i for i, w in enumerate(parts) if w.dtype in ("c32", "c64")]
        if not parts_idx or bits is not None:
            raise SystemExit("--phase needs a floating-point workload and no --bits")
        parts = [parts[i] for i in parts_idx]
        host = [host[i] for i in parts_idx]
        dev_in = [dev_in[i] for i in parts_idx]
        dev_out = [dev_out[i] for i in parts_idx]
        gen = torch.Generator(device=device).manual_seed(rank_seed(11, rank))
        thetas = [torch.rand(w.batch, w.N, device=device, generator=gen,
                             dtype=torch.float64 if w.dtype == "c64" else torch.float32) * (2 * np.pi)
                  for w in parts]

    def step():
        for pi, (w, (a, b), (c, d)) in enumerate(zip(parts, dev_in, dev_out)):
            if args.phase:
                fwt.phase_transform(a, b, thetas[pi], c, d, normalize=w.normalize)
            else:
                fwt.transform(a, b, c, d, normalize=w.normalize, bits=bits)

    names, owners = [], []  # one entry per pass launched by a step, and its part
    for pi, (w, (a, b), (c, d)) in enumerate(zip(parts, dev_in, dev_out)):
        if bits is None and not args.phase:
            part_names = pass_names(w, fwt)
        else:  # count the passes of a bit-range or phase transform from one traced call
            tr = fwt.PassTrace([torch.cuda.Event(enable_timing=True) for _ in range(16)])
            with tr:
                if args.phase:
                    fwt.phase_transform(a, b, thetas[pi], c, d, normalize=w.normalize)
                else:
                    fwt.transform(a, b, c, d, normalize=w.normalize, bits=bits)
            what = "phase+transform" if args.phase else f"bits [{bits[0]}, {bits[0] + bits[1]})"
            part_names = [f"{w.dtype} {what} pass {i + 1} (n={w.n})" for i in range(tr.count // 2)]
        names += part_names
        owners += [pi] * len(part_names)
    launches_per_step = len(names)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(device)

    uuid = str(torch.cuda.get_device_properties(device).uuid)
    sampler = clock_sampler(uuid)
    sampler.start()
    events = [torch.cuda.Event(enable_timing=True) for _ in range(2 * launches_per_step * args.steps)]
    trace = fwt.PassTrace(events)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    barrier(device)
    torch.cuda.synchronize(device)
    mark0 = sampler.mark()
    with trace:
        t0.record()
        for _ in range(args.steps):
            step()
        t1.record()
    torch.cuda.synchronize(device)
    barrier(device)
    mark1 = sampler.mark()
    elapsed_ms = t0.elapsed_time(t1)
    elapsed_ms = dist_max(elapsed_ms, device)
    sampler.stop()
    clocks = sampler.summary(mark0, mark1)

    durs = trace.durations_ms()
    assert len(durs) == launches_per_step * args.steps, "pass trace incomplete"
    per_kernel = {}
    for i, d in enumerate(durs):
        per_kernel.setdefault(i % launches_per_step, []).append(d)

    vectors_per_rank = sum(w.batch for w in parts)
    total_vectors = vectors_per_rank * world * args.steps
    value = total_vectors / (elapsed_ms / 1e3)
    algo_bytes_step = sum(2 * w.bytes_in for w in parts)  # 1 read + 1 write of every vector
    peak, peak_src = measured_peaks()

    # dominant kernel: largest share of device time
    kernels = []
    for li, (nm, pi) in enumerate(zip(names, owners)):
        mean_ms = statistics.mean(per_kernel[li])
        algo = 2 * parts[pi].bytes_in  # every pass reads and writes the whole batch once
        if args.phase and li == [i for i, o in enumerate(owners) if o == pi][0]:
            algo += algo // 4  # the first pass also reads the angles (one per amplitude)
        kernels.append({"kernel": nm, "mean_ms": mean_ms,
                        "median_ms": statistics.median(per_kernel[li]), "min_ms": min(per_kernel[li]),
                        "total_ms": sum(per_kernel[li]),
                        "algo_bytes_per_launch": algo, "gbs": algo / (mean_ms * 1e-3) / 1e9})
    top = max(kernels, key=lambda k: k["total_ms"])
    # the committed ncu traffic is per launch of the default batch
    traffic_of = (lambda key: ncu_traffic(key)) if args.batch <= 0 else (lambda key: None)
    traffic = traffic_of(top["kernel"])
    # DRAM bytes per vector: the pass model (each pass reads and writes the vector
    # once), the one-round-trip ideal, and the ncu-measured bytes when every pass of
    # the part has a current capture
    per_vector = []
    for pi, w in enumerate(parts):
        ks = [k for k, o in zip(kernels, owners) if o == pi]
        vec = w.bytes_in // w.batch  # re + im of one vector
        meas = [ncu_bytes_per_vector(k["kernel"]) if args.batch <= 0 else None for k in ks]
        per_vector.append({"part": w.name, "passes": len(ks), "model": 2 * len(ks) * vec,
                           "one_round_trip": 2 * vec,
                           "measured": (int(sum(meas))
                                        if meas and all(m is not None for m in meas) else None)})
    roofline = {"bound": "hbm", "achieved": round(top["gbs"], 1), "peak": peak, "unit": "GB/s",
                "frac": round(top["gbs"] / peak, 4), "traffic": traffic,
                "kernel": top["kernel"], "peak_source": peak_src,
                "algo_bytes_per_launch": top["algo_bytes_per_launch"]}

    result = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(elapsed_ms / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "+".join(sorted({{"c64": "int64", "c32": "f32", "i32": "int32"}[w.dtype] for w in parts})),
        "data": "synthetic (seeded PCG64; Gaussian unit-L2 states / uniform ints, per the workload)",
        "config": {
            "workload": (args.workload if args.batch <= 0 else "%s (batch %d)" % (args.workload, args.batch))
                        + ("" if bits is None else " bits [%d, %d)" % (bits[0], bits[0] + bits[1]))
                        + (" phase+transform" if args.phase else ""),
            "parts": [{"name": w.name, "n": w.n, "batch": w.batch, "dtype": w.dtype,
                       "normalize": w.normalize, "factors": fwt.plan_factors(w.n, w.dtype)}
                      for w in parts],
            "layout": "split re/im arrays, batch-major, out of place",
            "l2": "inputs larger than L2 (%.1f GiB in per step), no flush" % (
                sum(w.bytes_in for w in parts) / 2 ** 30),
            "arith": {"c64": "exact int64 fixed-point butterflies, one fp64 rounding per pass",
                      "c32": "fp32", "i32": "int32 wrap"},
        },
        # algorithmic bytes (one read + one write of every vector) over the step time
        "hbm_gbs_effective_per_gpu": round(algo_bytes_step * args.steps / (elapsed_ms / 1e3) / 1e9, 1),
        "kernels": [{k: (round(v, 4) if isinstance(v, float) else v) for k, v in kk.items()} for kk in kernels],
        "roofline": roofline,
        "dram_bytes_per_vector": per_vector,
        "clocks": clocks,
        "gpu_launches": launches_per_step * args.steps,
    }

    if not args.no_e2e and not args.phase and not args.bits:
        # the host-buffer entry points cover the whole transform only
        result["e2e"] = run_e2e(args, parts, host, device, fwt, world)
    checks = []
    if (rank == 0 and world == 1 and not args.no_per_config and args.batch <= 0
            and bits is None and not args.phase):
        mine = {w.name: (i, w) for i, w in enumerate(parts)}
        entries = []
        for label, name in CONFIGS:
            w = inputs.WORKLOADS[name]
            reuse = None
            if name in mine:  # the step's own buffers (same seeded states)
                i = mine[name][0]
                reuse = (dev_in[i], dev_out[i])
            entry, check = measure_config(label, w, fwt, device, peak, reuse)
            if reuse is not None:
                check["host_in"] = host[mine[name][0]]
            entries.append(entry)
            checks.append(check)
        result["per_config"] = entries
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"], errors = cpu_leg(parts, host, args.cpu_sample, checks)
        for entry in result.get("per_config", []):
            entry.update(errors.get(entry["config"], {}))
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


# The five specified configurations (the last in fp64 and fp32), in order of n.
CONFIGS = [("c1", "n10_b64_c32"), ("c2", "n12_b64_c32"), ("c3", "n14_b64_c32"),
           ("c4", "n18_b256_i32"), ("c5a", "n24_b16_c64"), ("c5b", "n24_b16_c32")]


def copy_floor_s(nbytes, reps, replays, device):
    """Seconds per step of the simplest kernel that reads and writes `nbytes` once (one
    launch of torch's elementwise negation, src -> dst), back to back from a CUDA graph
    over `reps` buffer pairs: the timing harness of measure_config applied to a plain
    one-launch streaming step.  (A captured copy_ becomes a graph memcpy node, which
    measured at half the kernel's rate for large buffers, so it is not used.)"""
    import torch

    n = nbytes // 4
    src = [torch.ones(n, dtype=torch.float32, device=device) for _ in range(reps)]
    dst = [torch.empty_like(src[0]) for _ in range(reps)]
    side = torch.cuda.Stream(device)
    side.wait_stream(torch.cuda.current_stream(device))
    with torch.cuda.stream(side):
        for r in range(reps):
            torch.neg(src[r], out=dst[r])
    torch.cuda.synchronize(device)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        for r in range(reps):
            torch.neg(src[r], out=dst[r])
    graph.replay()
    torch.cuda.synchronize(device)
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g0.record()
    for _ in range(replays):
        graph.replay()
    g1.record()
    torch.cuda.synchronize(device)
    t = g0.elapsed_time(g1) / 1e3 / (replays * reps)
    del graph, src, dst
    return t


def measure_config(label, w, fwt, device, peak, reuse=None):
    """Throughput of one specified configuration on its own, inputs in HBM.

    Configurations whose in + out buffers fit in L2 cycle through R copies of them
    (R x buffers >= 4 x L2, so each transform reads its inputs from HBM); the steps
    run back to back from a CUDA graph of R transforms (launch overhead stripped;
    the eager per-step time through the Python binding is reported beside it).
    Per-kernel device times come from the library's pass trace over eager steps.
    Returns the entry and, for the CPU leg's oracle check, the inputs and the GPU
    results of the vectors it checks."""
    import numpy as np
    import torch

    l2 = int(getattr(torch.cuda.get_device_properties(device), "L2_cache_size", 128 << 20))
    set_bytes = 2 * w.bytes_in  # inputs and outputs
    reps = 1 if set_bytes >= l2 else -(-4 * l2 // set_bytes)
    if reuse is not None:
        (a, b), (c, d) = reuse
        host_in = None
    else:
        host_in = w.generate()
        a = torch.from_numpy(host_in[0]).to(device)
        b = torch.from_numpy(host_in[1]).to(device)
        c, d = torch.empty_like(a), torch.empty_like(b)
    sets = [((a, b), (c, d))]
    for _ in range(reps - 1):
        sets.append(((a.clone(), b.clone()), (torch.empty_like(a), torch.empty_like(b))))

    def step(r):
        (x, y), (u, v) = sets[r]
        fwt.transform(x, y, u, v, normalize=w.normalize)

    for r in range(min(reps, 3)):
        step(r)
    torch.cuda.synchronize(device)
    small = set_bytes < l2
    names = pass_names(w, fwt)
    npass = len(names)
    # per-kernel device times, eager launches under the pass trace
    k_eager = max(reps, 300) if small else 20
    events = [torch.cuda.Event(enable_timing=True) for _ in range(2 * npass * k_eager)]
    trace = fwt.PassTrace(events)
    with trace:
        for i in range(k_eager):
            step(i % reps)
    torch.cuda.synchronize(device)
    durs = trace.durations_ms()
    kernels = []
    algo = 2 * w.bytes_in  # every pass reads and writes the whole batch once
    for li, nm in enumerate(names):
        ds = durs[li::npass]
        mean = statistics.mean(ds)
        kernels.append({"kernel": nm, "mean_us": round(mean * 1e3, 2),
                        "median_us": round(statistics.median(ds) * 1e3, 2),
                        "min_us": round(min(ds) * 1e3, 2),
                        "gbs": round(algo / (mean * 1e-3) / 1e9, 1)})
    # eager steps through the Python binding (host launch overhead included)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(k_eager):
        step(i % reps)
    e1.record()
    torch.cuda.synchronize(device)
    eager_us = e0.elapsed_time(e1) * 1e3 / k_eager
    # back-to-back steps from a CUDA graph
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream(device)
    with torch.cuda.graph(graph, stream=side):
        for r in range(reps):
            step(r)
    replays = max(1, -(-3000 // reps)) if small else 20
    graph.replay()
    torch.cuda.synchronize(device)
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g0.record()
    for _ in range(replays):
        graph.replay()
    g1.record()
    torch.cuda.synchronize(device)
    steps = replays * reps
    step_s = g0.elapsed_time(g1) / 1e3 / steps
    gbs = algo / step_s / 1e9
    copy_s = copy_floor_s(w.bytes_in, reps, replays, device)
    entry = {
        "config": label, "workload": w.name, "n": w.n, "batch": w.batch, "dtype": w.dtype,
        "normalize": w.normalize, "factors": fwt.plan_factors(w.n, w.dtype), "passes": npass,
        "vectors_per_s": round(w.batch / step_s, 1), "us_per_step": round(step_s * 1e6, 3),
        "effective_gbs": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4),
        "algo_bytes_per_step": algo,
        "timing": ("CUDA graph of %d back-to-back transforms over %d buffer sets (%.0f MiB, "
                   "inputs read from HBM), replayed %d times" % (reps, reps, reps * set_bytes / 2 ** 20, replays)
                   if small else "CUDA graph of one transform, replayed %d times (inputs larger than L2)" % replays),
        "eager_us_per_step": round(eager_us, 3),
        # the same bytes read and written once by a plain streaming kernel (torch.neg, one
        # launch a step, same graph harness): the floor of a one-launch step of this size
        "copy_floor_us_per_step": round(copy_s * 1e6, 3),
        "speed_vs_copy": round(copy_s / step_s, 3),
        "kernels": kernels,
    }
    meas = [ncu_bytes_per_vector(k["kernel"]) for k in kernels]
    entry["dram_bytes_per_vector"] = {
        "model": 2 * npass * (w.bytes_in // w.batch), "one_round_trip": 2 * (w.bytes_in // w.batch),
        "measured": int(sum(meas)) if all(m is not None for m in meas) else None}
    # the vectors the CPU leg checks against the oracle: all of them up to n = 18, the
    # first and the last at n = 24
    rows = list(range(w.batch)) if w.n <= 18 else [0, w.batch - 1]
    got = (c[rows].cpu().numpy(), d[rows].cpu().numpy())
    check = {"label": label, "workload": w, "rows": rows, "host_in": host_in, "got": got}
    del sets
    return entry, check


def run_e2e(args, parts, host, device, fwt, world):
    """Same metric through the public host-buffer API (fwt_host_* via
    transform_host): every step copies its inputs in from pinned host memory,
    transforms them and copies the results back, chunk by chunk with the copies of
    neighbouring chunks overlapping the transform.  The parts are independent
    batches, so each goes on its own stream with its own workspace: one part's
    first copies in overlap the other's last copies out."""
    import torch

    pin_in, pin_out = [], []
    for (re, im) in host:
        a = torch.from_numpy(re).pin_memory()
        b = torch.from_numpy(im).pin_memory()
        pin_in.append((a, b))
        pin_out.append((torch.empty_like(a).pin_memory(), torch.empty_like(b).pin_memory()))
    h2d = sum(a.numel() * a.element_size() + b.numel() * b.element_size() for a, b in pin_in)
    ws_each = [fwt.fwt_host_workspace_bytes(fwt.DTYPES[w.dtype], w.n, w.batch) for w in parts]
    wss = [torch.empty(nb, dtype=torch.uint8, device=device) for nb in ws_each]
    streams = [torch.cuda.Stream(device) for _ in parts]

    def step():
        for w, s, ws, (a, b), (ha, hb) in zip(parts, streams, wss, pin_in, pin_out):
            fwt.transform_host(a, b, ha, hb, normalize=w.normalize, workspace=ws, stream=s,
                               synchronize=False)

    main = torch.cuda.current_stream(device)
    # at least as many untimed steps as the main timed region (the first transfers of freshly
    # pinned buffers are several times slower than later ones)
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(device)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    ends = [[torch.cuda.Event(enable_timing=True) for _ in range(args.e2e_steps)] for _ in streams]
    barrier(device)
    t0.record(main)
    for s in streams:
        s.wait_event(t0)
    for i in range(args.e2e_steps):
        step()
        for p, s in enumerate(streams):
            ends[p][i].record(s)
    for s in streams:
        main.wait_stream(s)
    t1.record(main)
    torch.cuda.synchronize(device)
    barrier(device)
    ms = dist_max(t0.elapsed_time(t1), device)
    # a step's time: the later of the parts, each from its previous step's end
    per_step = [max((ends[p][i - 1] if i else t0).elapsed_time(ends[p][i]) for p in range(len(streams)))
                for i in range(args.e2e_steps)]
    vectors = sum(w.batch for w in parts) * world * args.e2e_steps
    floor = copies_only(args, pin_in, pin_out, device)
    return {"value": round(vectors / (ms / 1e3), 2), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": h2d, "steps": args.e2e_steps, "warmup": max(3, args.warmup),
            "ms_per_step": round(ms / args.e2e_steps, 3),
            "step_ms": {"median": round(statistics.median(per_step), 3), "min": round(min(per_step), 3),
                        "max": round(max(per_step), 3)},
            "copies_only": floor,
            "workspace_bytes": sum(ws_each), "streams": len(streams)}


def copies_only(args, pin_in, pin_out, device):
    """The host link's floor for the same step: the same bytes copied host -> device on
    one stream and device -> host on another (whole arrays, no transform), timed like the
    end-to-end steps.  Its per-step median against e2e's shows how much of the link time
    the pipelined transform adds; long steps in both come from the link, not the pipeline."""
    import torch

    # separate device buffers for the two directions, so the concurrent copies touch
    # disjoint memory
    dbuf = [(torch.empty_like(a, device=device), torch.empty_like(b, device=device)) for a, b in pin_in]
    dsrc = [(torch.zeros_like(a, device=device), torch.zeros_like(b, device=device)) for a, b in pin_in]
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
    main = torch.cuda.current_stream(device)

    def step():
        s_in.wait_stream(main)
        s_out.wait_stream(main)
        with torch.cuda.stream(s_in):
            for (a, b), (da, db) in zip(pin_in, dbuf):
                da.copy_(a, non_blocking=True)
                db.copy_(b, non_blocking=True)
        with torch.cuda.stream(s_out):
            for (ha, hb), (da, db) in zip(pin_out, dsrc):
                ha.copy_(da, non_blocking=True)
                hb.copy_(db, non_blocking=True)
        main.wait_stream(s_in)
        main.wait_stream(s_out)

    for _ in range(3):
        step()
    torch.cuda.synchronize(device)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.e2e_steps + 1)]
    ev[0].record(main)
    for i in range(args.e2e_steps):
        step()
        ev[i + 1].record(main)
    torch.cuda.synchronize(device)
    per = [ev[i].elapsed_time(ev[i + 1]) for i in range(args.e2e_steps)]
    del dbuf, dsrc
    return {"ms_per_step": round(sum(per) / len(per), 3), "median_ms": round(statistics.median(per), 3),
            "max_ms": round(max(per), 3)}


def oracle_step(orc, parts, host, threads):
    """Every real array of every part through the CPU oracle, the arrays run
    concurrently (ctypes releases the GIL) and each split over whole vectors."""
    from concurrent.futures import ThreadPoolExecutor

    jobs = [(arr, w.normalize) for w, pair in zip(parts, host) for arr in pair]
    per_job = max(1, threads // len(jobs))
    with ThreadPoolExecutor(max_workers=len(jobs)) as pool:
        list(pool.map(lambda j: orc.fwt(j[0], normalize=j[1], nthreads=per_job), jobs))
    return min(threads, sum(min(per_job, arr.shape[0]) for arr, _ in jobs))


def cpu_info():
    """Host core count and CPU model (lscpu, else /proc/cpuinfo)."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
        arch = next((ln.split(":", 1)[1].strip() for ln in out.splitlines()
                     if ln.startswith("Architecture:")), None)
        if model and arch:
            model = f"{model} ({arch})"
    except (OSError, subprocess.SubprocessError):
        pass
    if not model:
        try:
            for line in open("/proc/cpuinfo"):
                if line.lower().startswith(("model name", "cpu part")):
                    model = line.split(":", 1)[1].strip()
                    break
        except OSError:
            pass
    return {"nproc": os.cpu_count() or 1, "model": model or "unknown"}


def cpu_baseline(parts, host, sample):
    """The CPU oracle as it stands, timed twice on the host: one thread on the first
    vector of each part, and every core on the first `sample` vectors of each part
    (the arrays run concurrently, each split over whole vectors)."""
    import oracle

    orc = oracle.default()
    info = cpu_info()
    threads = max(1, info["nproc"])
    one = [(re[:1], im[:1]) for re, im in host]
    t = time.perf_counter()
    for w, (re, im) in zip(parts, one):
        for arr in (re, im):
            orc.fwt(arr, normalize=w.normalize, nthreads=1)
    secs1 = time.perf_counter() - t
    v1 = sum(min(1, w.batch) for w in parts)
    cut = [(re[:sample], im[:sample]) for re, im in host]
    t = time.perf_counter()
    used = oracle_step(orc, parts, cut, threads)
    secs = time.perf_counter() - t
    vectors = sum(min(sample, w.batch) for w in parts)
    names = ", ".join(w.name for w in parts)
    return {"value": round(vectors / secs, 4), "unit": UNIT, "cores": used, "kind": "oracle",
            "sample": "first %d vectors of each part (%s), %.1f s wall on %d threads" % (
                sample, names, secs, used),
            "single_thread": {"value": round(v1 / secs1, 4), "unit": UNIT, "cores": 1,
                              "sample": "first vector of each part (%s), %.1f s wall" % (names, secs1)},
            "all_cores": {"value": round(vectors / secs, 4), "unit": UNIT, "cores": used},
            "nproc": info["nproc"], "cpu_model": info["model"]}


def cpu_leg(parts, host, sample, checks):
    """The CPU oracle's leg of the run: its timed baseline, then the check of the
    per-configuration GPU results it was handed against the oracle (per-vector
    complex relative L2 error, max over the checked vectors; int32 bit for bit)."""
    import numpy as np

    import oracle

    base = cpu_baseline(parts, host, sample)
    threads = max(1, os.cpu_count() or 1)
    errors = {}
    for ch in checks:
        w, rows = ch["workload"], ch["rows"]
        re, im = ch["host_in"]
        ore, oim = oracle.fwt_complex(re[rows], im[rows], normalize=w.normalize, nthreads=threads)
        gre, gim = ch["got"]
        desc = "all %d vectors" % w.batch if len(rows) == w.batch else "vectors %s" % rows
        if w.dtype == "i32":
            errors[ch["label"]] = {"oracle_check": desc, "bit_exact": bool(
                np.array_equal(gre, ore) and np.array_equal(gim, oim))}
            continue
        worst = 0.0
        for k in range(len(rows)):
            ref = np.concatenate([ore[k], oim[k]])
            got = np.concatenate([gre[k], gim[k]]).astype(np.float64)
            scale = max(float(np.max(np.abs(ref))), 1e-300)
            num = float(np.linalg.norm((got - ref) / scale))
            den = float(np.linalg.norm(ref / scale)) or 1.0
            worst = max(worst, num / den)
        errors[ch["label"]] = {"oracle_check": desc, "max_rel_l2_err": float("%.3e" % worst),
                               "tolerance": 2e-6 if w.dtype == "c32" else 1e-12}
    return base, errors


# ---- the reference arm: the CPU oracle -------------------------------------------------

def run_reference(args):
    rank, _, world = dist_env()
    if rank != 0:
        return  # rank 0 alone runs the CPU reference
    import oracle
    from walsh_hadamard_transform_gb300 import inputs

    parts = [inputs.WORKLOADS[name] for name in STEP_WORKLOADS[args.workload]]
    info = cpu_info()
    threads = max(1, info["nproc"])
    # each step runs the 2 arrays of every part at once, each over its vectors: enough
    # vectors that every core has one
    want = args.ref_sample if args.ref_sample > 0 else -(-threads // (2 * len(parts)))
    sample = max(1, min(want, min(w.batch for w in parts)))
    host = [w.generate(batch=sample) for w in parts]
    orc = oracle.default()
    for _ in range(args.warmup):
        oracle_step(orc, parts, host, threads)
    t = time.perf_counter()
    for _ in range(args.steps):
        used = oracle_step(orc, parts, host, threads)
    secs = time.perf_counter() - t
    vectors = sample * len(parts) * args.steps
    value = vectors / secs
    desc = "first %d vectors of each part (%s) per step" % (sample, ", ".join(w.name for w in parts))
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(secs / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64+uint32 (oracle)",
        "data": "synthetic (seeded PCG64)",
        "config": {"workload": args.workload, "sample": desc},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": used, "kind": "oracle",
                         "sample": desc, "nproc": info["nproc"], "cpu_model": info["model"]},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.steps < 1 or args.warmup < 0:
        raise SystemExit("--steps must be >= 1 and --warmup >= 0")
    if args.impl == "reference":
        # fewer, bounded CPU steps: each is seconds of host work
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
