#!/usr/bin/env python3
"""Benchmark: symmetric-window AllReduce(sum), R=8 rank windows of 256 MiB fp32
(67,108,864 elements per rank, seeded U(-1,1)), two-shot, on one GB300.

One step = one sym_allreduce call over the whole workload (inputs resident in
HBM).  Prints ONE JSON line (rank 0):

  value      algbw = bytes per rank / step time, summed over replicas (GB/s)
  roofline   HBM-bound: compulsory bytes of the dominant kernel per launch
             (read R*S + write R*S) / its average CUDA-event duration, against
             the measured copy bandwidth; traffic = ncu DRAM bytes per launch
  e2e        the same metric through the C ABI with pinned HOST buffers: every
             step copies the R inputs in and the result (the reduced vector every
             rank holds, read from rank 0's window) out
  cpu_baseline  the CPU oracle (test infrastructure) timed on a bounded sample

  --impl reference  times the CPU oracle as the reference arm (rank 0 only).

Multi-GPU (torchrun, --gpus N): every rank runs an independent replica of the
one-GPU emulation (no data-path collective); barrier + max over ranks.
"""
from __future__ import annotations

import argparse
import ctypes
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

METRIC = "AllReduce algbw GB/s and HBM GB/s (% of peak) at R=8, 256 MB/rank fp32, 1 GB300"
R_DEFAULT, N_DEFAULT = 8, 1 << 26
FALLBACK_HBM_GBS = 6800.0
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "twoshot_st_f32_R8_traffic.json")
KERNEL_SRC = [os.path.join(ROOT, "symmetric_memory_allreduce_gb300", "csrc", f)
              for f in ("allreduce_kernels.cuh", "allreduce_f32.cu", "symar_internal.cuh")]


# ----------------------------------------------------------------- pure helpers (CPU-testable)

def algo_bytes(algo: str, R: int, S: int) -> dict:
    """Per-launch byte models of one AllReduce of S bytes per rank over R windows.

    compulsory: the HBM bytes the emulation cannot avoid (each input read once,
    each output written once).  logical: bytes the algorithm's loads and stores
    name (repeated reads of one line by several rank-slots counted each time).
    """
    logical = {"oneshot": R * (R + 1) * S, "twoshot": 2 * R * S,
               "twoshot_pull": (3 * R - 1) * S, "twoshot_split": (3 * R - 1) * S}[algo]
    return {"compulsory": 2 * R * S, "logical": logical}


def measured_peak() -> tuple[float, str]:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for p in KERNEL_SRC:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(R: int, S: int) -> float | None:
    """DRAM bytes per launch from the committed ncu summary, if the kernel is unchanged."""
    try:
        with open(TRAFFIC_FILE) as f:
            t = json.load(f)
    except Exception:
        return None
    if t.get("source_sha256") != kernel_source_hash():
        return None
    per_byte = float(t["dram_bytes_per_launch"]) / float(t["bytes_per_rank"])
    return per_byte * S if int(t["R"]) == R else None


def _size(nbytes: int) -> str:
    """1 KiB, 64 MiB, 1 GiB ..."""
    for unit, shift in (("GiB", 30), ("MiB", 20), ("KiB", 10)):
        if nbytes >= 1 << shift and nbytes % (1 << shift) == 0:
            return f"{nbytes >> shift} {unit}"
    return f"{nbytes} B"


def percentile(xs, q):
    xs = sorted(xs)
    if not xs:
        return float("nan")
    k = (len(xs) - 1) * q
    lo, hi = int(k), min(int(k) + 1, len(xs) - 1)
    return xs[lo] + (xs[hi] - xs[lo]) * (k - lo)


def summarize_clocks(samples: list[dict], max_mhz: float | None) -> dict:
    reasons = set()
    for s in samples:
        reasons.update(s.get("reasons", []))
    busy = [s["sm_mhz"] for s in samples if "gpu_idle" not in s.get("reasons", [])] or \
           [s["sm_mhz"] for s in samples]
    return {"sm_mhz": statistics.median(busy) if busy else None, "sm_max_mhz": max_mhz,
            "reasons": sorted(reasons), "samples": len(samples)}


def max_over_ranks(value: float) -> float:
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier():
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.barrier()


# ----------------------------------------------------------------- clocks (read-only NVML)

_REASON_BITS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
                0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
                0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
                0x100: "display_clock_setting"}


class ClockSampler(threading.Thread):
    """Samples SM clock and clock-event reasons every ~20 ms (reads only)."""

    def __init__(self, pci_bus_id: str | None):
        super().__init__(daemon=True)
        self.samples: list[dict] = []
        self.max_mhz = None
        self._halt = threading.Event()
        self._nvml = None
        self._h = None
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                raise OSError("nvmlInit")
            h = ctypes.c_void_p()
            ok = False
            if pci_bus_id:
                ok = nv.nvmlDeviceGetHandleByPciBusId_v2(pci_bus_id.encode(), ctypes.byref(h)) == 0
            if not ok:
                ok = nv.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(h)) == 0
            if not ok:
                raise OSError("nvml handle")
            m = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(m)) == 0:
                self.max_mhz = float(m.value)
            self._nvml, self._h = nv, h
        except OSError:
            self._nvml = None

    def _sample(self):
        nv, h = self._nvml, self._h
        mhz, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(mhz)) != 0:
            return
        fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(nv, "nvmlDeviceGetCurrentClocksThrottleReasons")
        reasons = []
        if fn(h, ctypes.byref(rs)) == 0:
            reasons = [n for b, n in _REASON_BITS.items() if rs.value & b]
        self.samples.append({"t": time.time(), "sm_mhz": float(mhz.value), "reasons": reasons})

    def run(self):
        if self._nvml is None:
            return
        while not self._halt.is_set():
            self._sample()
            time.sleep(0.02)

    def stop(self):
        self._halt.set()
        self.join(timeout=2)

    def window(self, t0: float, t1: float) -> list[dict]:
        return [s for s in self.samples if t0 <= s["t"] <= t1]


def nvidia_smi_clocks() -> dict | None:
    """One-shot fallback when NVML is not loadable."""
    try:
        out = subprocess.run(["nvidia-smi", "--query-gpu=clocks.sm,clocks.max.sm",
                              "--format=csv,noheader,nounits"], capture_output=True, text=True,
                             timeout=10).stdout.split("\n")[0].split(",")
        return {"sm_mhz": float(out[0]), "sm_max_mhz": float(out[1]), "reasons": [],
                "samples": 1, "note": "nvidia-smi after the timed region"}
    except Exception:
        return None


# ----------------------------------------------------------------- CPU oracle legs

def cpu_oracle_rate(x_sample, budget_s: float) -> dict:
    """Times the oracle (test infrastructure) over a bounded sample; returns GB/s of algbw."""
    import oracle

    oracle.build()
    R, n = x_sample.shape
    nthreads = os.cpu_count() or 1
    passes, used = 0, 1
    t0 = time.perf_counter()
    while True:
        _, used = oracle.allreduce_sum_mt(x_sample, nthreads)
        passes += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    S = n * x_sample.itemsize
    # the same rank-order sum on one thread, over a quarter of the budget
    p1 = 0
    t1 = time.perf_counter()
    while True:
        oracle.allreduce_sum_mt(x_sample, 1)
        p1 += 1
        el1 = time.perf_counter() - t1
        if el1 >= budget_s / 4:
            break
    return {"value": S * passes / el / 1e9, "unit": "GB/s", "cores": used, "kind": "oracle",
            "sample": f"the whole workload: R={R} x {n} fp32 elements ({S >> 20} MiB) per rank, "
                      f"{passes} passes in {el:.1f} s, {used} threads",
            "seconds_per_pass": el / passes, "single_thread_value": S * p1 / el1 / 1e9,
            "cpu_model": cpu_model()}


def cpu_model() -> str:
    """The host CPU's name from /proc/cpuinfo (x86 'model name'; Arm implementer/part)."""
    try:
        with open("/proc/cpuinfo") as f:
            text = f.read()
    except OSError:
        return "unknown"
    fields = {}
    for line in text.splitlines():
        if ":" in line:
            k, v = line.split(":", 1)
            fields.setdefault(k.strip(), v.strip())
    if "model name" in fields:
        return fields["model name"]
    if "CPU part" in fields:
        return f"Arm implementer {fields.get('CPU implementer', '?')} part {fields['CPU part']}"
    return "unknown"


def run_reference(args) -> int:
    """The reference arm: the CPU oracle, rank 0 only, over the whole workload every step."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    from symmetric_memory_allreduce_gb300 import workloads as wl

    R, n = args.ranks, args.count
    x = wl.uniform_f32(3, R, n) if n == N_DEFAULT else wl.normal_f32(4, R, n)
    import oracle

    oracle.build()
    nthreads = os.cpu_count() or 1
    for _ in range(args.warmup):
        oracle.allreduce_sum_mt(x, nthreads)
    times = []
    used = 1
    for _ in range(args.steps):
        t0 = time.perf_counter()
        _, used = oracle.allreduce_sum_mt(x, nthreads)
        times.append(time.perf_counter() - t0)
    t = sum(times) / len(times)
    S = n * 4
    value = S / t / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": t * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": DATA,
            "algo": "CPU oracle (rank-order fp32 sum per element, host threads)",
            "config": _config(R, n),
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": used, "kind": "oracle",
                             "sample": f"the whole workload every step: R={R} x {n} fp32 elements "
                                       f"per rank, {used} threads",
                             "cpu_model": cpu_model()},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


DATA = "synthetic (seeded U(-1,1) fp32 per rank, numpy PCG64)"


def _config(R, n):
    """The workload, identical in both arms (how it is computed is the line's `algo`)."""
    return {"workload": f"AllReduce(sum) R={R} rank windows x {n} fp32 elements "
                        f"({n * 4 >> 20} MiB) per rank, seeded U(-1,1)",
            "R": R, "count_per_rank": n, "bytes_per_rank": n * 4,
            "l2": "inputs 2 GiB > 126 MiB L2 (no flush needed)", "parallelism": "replicas"}


# ----------------------------------------------------------------- our arm

def run_ours(args) -> int:
    import numpy as np
    import torch
    import torch.distributed as dist

    import symmetric_memory_allreduce_gb300 as sm
    from symmetric_memory_allreduce_gb300 import workloads as wl

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)               # one replica per GPU, bound before any allocation
    if world > 1 and not dist.is_initialized():
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    sm.load()
    R, n = args.ranks, args.count
    S = n * 4
    x = wl.uniform_f32(3, R, n) if n == N_DEFAULT else wl.normal_f32(4, R, n)
    send, recv = sm.Window(R, S), sm.Window(R, S)
    stream = torch.cuda.current_stream()
    for r in range(R):
        send.write(r, x[r])
    stream.synchronize()

    def step():
        sm.sym_allreduce(send, recv, n, "f32", "sum", args.algo)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if sm.sym_stream_status() != sm.SYM_OK:
        raise RuntimeError("warm-up reported a device status: " + sm.sym_last_error())

    props = torch.cuda.get_device_properties(local)
    try:
        bus = f"{props.pci_domain_id:08X}:{props.pci_bus_id:02X}:{props.pci_device_id:02X}.0"
    except AttributeError:
        bus = None
    sampler = ClockSampler(bus)
    sampler.start()
    time.sleep(0.05)

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize()
    launches0 = sm.sym_launch_count()
    w0 = time.time()
    t_all0 = torch.cuda.Event(enable_timing=True)
    t_all1 = torch.cuda.Event(enable_timing=True)
    t_all0.record(stream)
    for i in range(args.steps):
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    t_all1.record(stream)
    torch.cuda.synchronize()
    w1 = time.time()
    barrier()
    launches = sm.sym_launch_count() - launches0
    sampler.stop()
    if sm.sym_stream_status() != sm.SYM_OK:
        raise RuntimeError("timed region reported a device status: " + sm.sym_last_error())
    total_ms = t_all0.elapsed_time(t_all1)
    per = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    kern_ms = sum(per) / len(per)
    total_ms = max_over_ranks(total_ms)
    ms_per_step = total_ms / args.steps
    value = world * S / (ms_per_step * 1e-3) / 1e9

    peak, peak_kind = measured_peak()
    bytes_model = algo_bytes(args.algo if args.algo != "auto" else
                             sm.sym_allreduce_algo(send, n, "f32"), R, S)
    achieved = bytes_model["compulsory"] / (kern_ms * 1e-3) / 1e9
    clk_samples = sampler.window(w0, w1)
    clocks = summarize_clocks(clk_samples, sampler.max_mhz) if clk_samples else nvidia_smi_clocks()

    # e2e: pinned host buffers through the C ABI, copies inside the timed region.
    # Every step copies its R inputs host -> device (sym_window_write), runs the
    # AllReduce, and copies the result device -> host (sym_window_read of rank
    # 0's window: every rank holds the same reduced vector, which the oracle
    # produces once).  Two window pairs and three streams let step k+1's inputs
    # cross the host link while step k's result comes back.
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(sm, send, recv, x, R, n, args, world, stream)

    secondary = None
    if rank == 0 and world == 1 and not args.no_secondary and (R, n) == (R_DEFAULT, N_DEFAULT):
        secondary = run_secondary(sm, stream, x, peak)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_oracle_rate(x, args.cpu_seconds)

    traffic = recorded_traffic(R, S)
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": DATA,
        "algo": args.algo, "config": _config(R, n),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": "k_twoshot_st<F32T,8,1>" if args.algo in ("twoshot", "auto")
                     else args.algo, "peak_kind": f"{peak_kind} HBM copy bandwidth",
                     "bytes_per_launch": bytes_model["compulsory"],
                     "kernel_ms": kern_ms, "kernel_ms_p10": percentile(per, 0.1),
                     "kernel_ms_p90": percentile(per, 0.9)},
        # bytes actually read and written (ncu DRAM counters of this kernel) over its time
        "hbm_gbs": traffic / (kern_ms * 1e-3) / 1e9 if traffic else None,
        "hbm_pct_of_peak": 100.0 * traffic / (kern_ms * 1e-3) / 1e9 / peak if traffic else None,
        "compulsory_gbs": achieved,
        "logical_gbs": bytes_model["logical"] / (kern_ms * 1e-3) / 1e9,
        "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches, "clocks": clocks,
        "secondary": secondary,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    send.free()
    recv.free()
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_e2e(sm, send, recv, x, R, n, args, world, stream) -> dict:
    """End to end through the C ABI with pinned host buffers (see run_ours)."""
    import numpy as np
    import torch

    S = n * 4
    steps = max(3, args.e2e_steps)
    h_in = torch.empty((R, S), dtype=torch.uint8, pin_memory=True)
    h_in.numpy()[:] = x.view(np.uint8)
    # the step's result: the reduced vector (every rank's window holds the same bytes; the oracle
    # produces it once), read back from rank 0's window
    h_out = [torch.empty((S,), dtype=torch.uint8, pin_memory=True) for _ in range(2)]
    sends = [send, sm.Window(R, S)]
    recvs = [recv, sm.Window(R, S)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    for e in ev_done + ev_out:
        e.record(stream)

    def e2e_step(k):
        b = k % 2
        s_in.wait_event(ev_done[b])                 # the AllReduce of step k-2 has read sends[b]
        for r in range(R):
            sends[b].write(r, (h_in.data_ptr() + r * S, S), stream=s_in)
        ev_in[b].record(s_in)
        stream.wait_event(ev_in[b])
        stream.wait_event(ev_out[b])                # the copy-out of step k-2 has read recvs[b]
        sm.sym_allreduce(sends[b], recvs[b], n, "f32", "sum", args.algo, stream=stream)
        ev_done[b].record(stream)
        s_out.wait_event(ev_done[b])
        recvs[b].read(0, (h_out[b].data_ptr(), S), stream=s_out)
        ev_out[b].record(s_out)

    for k in range(2):                              # warm-up
        e2e_step(k)
    torch.cuda.synchronize()
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_event(e0)
    s_out.wait_event(e0)
    for k in range(steps):
        e2e_step(k)
    stream.wait_event(ev_out[(steps - 1) % 2])
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    if sm.sym_stream_status() != sm.SYM_OK:
        raise RuntimeError("e2e reported a device status: " + sm.sym_last_error())
    e_ms = max_over_ranks(e0.elapsed_time(e1)) / steps
    # the result that came back equals the device result of the last step (bytes)
    check = bool(torch.equal(h_out[(steps - 1) % 2], recvs[(steps - 1) % 2].tensor()[0, :S].cpu()))
    for w in (sends[1], recvs[1]):
        w.free()
    return {"value": world * S / (e_ms * 1e-3) / 1e9, "unit": "GB/s",
            "h2d_bytes_per_step": R * S, "d2h_bytes_per_step": S, "steps": steps,
            "ms_per_step": e_ms,
            "host_link_gbs": (R * S + S) / (e_ms * 1e-3) / 1e9, "result_read_back_matches": check,
            "pipeline": "2 window pairs, 3 streams: copy-in of the R inputs || AllReduce || "
                        "copy-out of the result (rank 0's window)"}


def run_secondary(sm, stream, x3, peak) -> list[dict]:
    """The other measured rows, each timed over >= 20 launches (CUDA events per launch on the
    library's stream, after 5 warm-ups) and checked against the oracle in the same run:
    R=8 x 128 MiB bf16 (two-shot, pull) and 256 MiB fp32 pull, R=8 x 64 MiB one-shot and two-shot, the
    put + signal AllGather at 8 chunks per signal, and the AUTO crossover (64 to 512 KiB per rank).
    x3: the R=8 x 256 MiB fp32 inputs already on the host."""
    import numpy as np
    import torch

    import oracle
    from symmetric_memory_allreduce_gb300 import workloads as wl

    oracle.build()
    nthr = os.cpu_count() or 1
    rows = []

    def row(name, algo, dtype, R, S, ts, comp, parity, check, logical=None):
        mean = sum(ts) / len(ts)
        d = {"row": name, "algo": algo, "dtype": dtype, "R": R, "bytes_per_rank": S,
             "launches": len(ts), "kernel_ms": mean, "kernel_ms_median": statistics.median(ts),
             "bytes_model": "compulsory: every input read once, every output written once",
             "bytes_per_launch": comp, "achieved_gbs": comp / (mean * 1e-3) / 1e9,
             "frac": comp / (mean * 1e-3) / 1e9 / peak, "parity": bool(parity), "check": check}
        if logical:
            d["logical_gbs"] = logical / (mean * 1e-3) / 1e9
        rows.append(d)

    def allreduce_rows(name, x, dtype, algos):
        R, n = x.shape
        S = n * x.itemsize
        send, recv = sm.Window(R, S), sm.Window(R, S)
        try:
            for r in range(R):
                send.write(r, x[r])
            stream.synchronize()
            want, _ = oracle.allreduce_sum_mt(x, nthr)
            y = np.empty(n, x.dtype)
            for algo in algos:
                ts = _time_launches(lambda: sm.sym_allreduce(send, recv, n, dtype, "sum", algo), 20,
                                    stream)
                if sm.sym_stream_status() != sm.SYM_OK:
                    raise RuntimeError(f"{name} {algo}: " + sm.sym_last_error())
                ok = True
                for r in range(R):
                    recv.read(r, y)
                    stream.synchronize()
                    ok &= bool(np.array_equal(y.view(np.uint8), want.view(np.uint8)))
                m = algo_bytes(algo, R, S)
                row(name, algo, dtype, R, S, ts, m["compulsory"], ok,
                    "every element of every rank equals the oracle (bit-exact)", m["logical"])
        finally:
            send.free()
            recv.free()

    allreduce_rows("allreduce R=8 x 128 MiB bf16 U(-1,1)", wl.to_bf16_bits(x3), "bf16",
                   ["twoshot", "twoshot_pull"])
    allreduce_rows("allreduce R=8 x 256 MiB fp32 U(-1,1)", x3, "f32", ["twoshot_pull"])
    allreduce_rows("allreduce R=8 x 64 MiB fp32 N(0,1)", wl.workload_inputs(2), "f32", ["oneshot", "twoshot"])

    # put + signal AllGather, R=16 x 32 MiB, 64 KiB chunks, 8 chunks per signal
    c5 = wl.PUT_SIGNAL
    R, S, chunk, batch = c5["R"], c5["nbytes"], c5["chunk"], c5["batch"]
    xb = wl.random_bytes(5, R, S)
    send, recv = sm.Window(R, S, ncounters=1), sm.Window(R, R * S, nsignals=R)
    try:
        for r in range(R):
            send.write(r, xb[r])
        stream.synchronize()
        ts = _time_launches(lambda: sm.sym_allgather(send, recv, S // 4, "f32", "put_signal", chunk,
                                                     batch), 20, stream)
        if sm.sym_stream_status() != sm.SYM_OK:
            raise RuntimeError("put + signal allgather: " + sm.sym_last_error())
        want, sig, cnt = oracle.put_signal_allgather(xb, chunk, batch)
        del xb
        ok = True
        out = np.empty(R * S, np.uint8)
        for p in range(R):
            recv.read(p, out)
            stream.synchronize()
            ok &= bool(np.array_equal(out, want))
            ok &= all(sm.sym_signal_read(recv, p, q) == int(sig[p, q]) for q in range(R))
            ok &= sm.sym_counter_read(send, p, 0) == int(cnt[p])
        row("put+signal allgather R=16 x 32 MiB random bytes", "put_signal (64 KiB chunks, 8 per signal)",
            "bytes", R, S,
            ts, R * S + R * R * S, ok,
            "every rank's gathered bytes, all R*R signal counts and R counters equal the oracle's "
            "sequential put + signal model")
    finally:
        send.free()
        recv.free()

    # AUTO crossover: device time per call from 100 calls in a CUDA graph, replayed 10 times
    points = []
    for nbytes in (64 << 10, 128 << 10, 256 << 10, 512 << 10):
        R, n = 8, nbytes // 4
        x = wl.workload_inputs(4, n=n)
        send, recv = sm.Window(R, nbytes), sm.Window(R, nbytes)
        try:
            for r in range(R):
                send.write(r, x[r])
            stream.synchronize()
            pt = {"bytes_per_rank": nbytes, "auto": sm.sym_allreduce_algo(send, n, "f32")}
            for algo in ("oneshot", "twoshot"):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    for _ in range(100):
                        sm.sym_allreduce(send, recv, n, "f32", "sum", algo)
                g.replay()
                torch.cuda.synchronize()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for _ in range(10):
                    g.replay()
                e1.record(stream)
                torch.cuda.synchronize()
                pt[f"{algo}_us"] = e0.elapsed_time(e1) * 1e3 / 1000
                del g
            want = oracle.allreduce_sum_f32(x)
            sm.sym_allreduce(send, recv, n, "f32", "sum", "auto")
            ok = sm.sym_stream_status() == sm.SYM_OK
            y = np.empty(n, np.float32)
            for r in range(R):
                recv.read(r, y)
                stream.synchronize()
                ok &= bool(np.array_equal(y.view(np.uint32), want.view(np.uint32)))
            pt["faster"] = "oneshot" if pt["oneshot_us"] < pt["twoshot_us"] else "twoshot"
            # AUTO's pick against the faster of the two at this size (1.0 = it picked the faster)
            pt["auto_over_best"] = pt[pt["auto"] + "_us"] / min(pt["oneshot_us"], pt["twoshot_us"])
            pt["parity"] = bool(ok)
            points.append(pt)
        finally:
            send.free()
            recv.free()
    rows.append({"row": "allreduce R=8 fp32 N(0,1) AUTO crossover", "R": 8, "dtype": "f32",
                 "threshold": "SYM_ONESHOT_MAX_BYTES (128 KiB per rank)", "points": points,
                 "auto_over_best_max": max(p["auto_over_best"] for p in points),
                 "parity": all(p["parity"] for p in points),
                 "check": "AUTO's result on every rank equals the oracle (bit-exact)"})
    return rows


def run_sweep(args) -> int:
    """Message-size sweep (R=8, 1 KiB .. 1 GiB per rank, fp32 N(0,1)): median kernel time of
    every algorithm per size, one JSON object per (size, algo) on stdout."""
    import torch

    import symmetric_memory_allreduce_gb300 as sm
    from symmetric_memory_allreduce_gb300 import workloads as wl

    torch.cuda.set_device(0)
    sm.load()
    stream = torch.cuda.current_stream()
    R = args.ranks
    peak, _ = measured_peak()
    sizes = [s for s in wl.SWEEP_BYTES if s <= args.sweep_max]
    algos = ["oneshot", "twoshot", "twoshot_pull", "twoshot_split"]
    flush = _l2_flush_buffer()
    for nbytes in sizes:
        n = nbytes // 4
        x = wl.normal_f32(4, R, n)
        send, recv = sm.Window(R, nbytes), sm.Window(R, nbytes)
        for r in range(R):
            send.write(r, x[r])
        stream.synchronize()
        for algo in algos:
            # >= 20 launches and >= 200 ms of timed launches, after 5 warm-ups
            iters = max(20, min(2000, int(2e9 / max(nbytes * 2 * R, 1))))
            ts = _time_launches(lambda: sm.sym_allreduce(send, recv, n, "f32", "sum", algo), iters,
                                stream, None, 200.0)
            iters = len(ts)
            assert sm.sym_stream_status() == sm.SYM_OK
            med = statistics.median(ts)
            comp = algo_bytes(algo, R, nbytes)["compulsory"]
            row = {"bytes_per_rank": nbytes, "algo": algo, "iters": iters,
                   "us_median": med * 1e3, "us_p10": percentile(ts, 0.1) * 1e3,
                   "us_p90": percentile(ts, 0.9) * 1e3,
                   "algbw_gbs": nbytes / (med * 1e-3) / 1e9,
                   "hbm_gbs": comp / (med * 1e-3) / 1e9,
                   "hbm_frac": comp / (med * 1e-3) / 1e9 / peak,
                   "auto": sm.sym_allreduce_algo(send, n, "f32")}
            if 2 * R * nbytes <= L2_FLUSH_BYTES // 2:
                # inputs + outputs fit in L2: also time with L2 flushed before each launch
                cold = _time_launches(lambda: sm.sym_allreduce(send, recv, n, "f32", "sum", algo),
                                      min(iters, 50), stream, flush)
                row["us_median_cold"] = statistics.median(cold) * 1e3
            if nbytes <= (16 << 20):
                # device-side latency: 100 calls recorded in a CUDA graph, replayed
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    for _ in range(100):
                        sm.sym_allreduce(send, recv, n, "f32", "sum", algo)
                g.replay()
                torch.cuda.synchronize()
                g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                g0.record(stream)
                for _ in range(10):
                    g.replay()
                g1.record(stream)
                torch.cuda.synchronize()
                assert sm.sym_stream_status() == sm.SYM_OK
                row["us_per_call_graph"] = g0.elapsed_time(g1) * 1e3 / 1000
                del g
            print(json.dumps(row), flush=True)
        send.free()
        recv.free()
    return 0


def _time_launches(fn, iters: int, stream, flush=None, min_ms: float = 0.0) -> list[float]:
    """Per-launch CUDA-event times (ms) of fn() on `stream`, after 5 warm-ups.

    At least `iters` launches, repeated in batches of `iters` until the timed
    launches add up to `min_ms`.  flush: a device buffer larger than L2,
    overwritten before every timed launch (outside its events) so that the
    launch starts with a cold L2."""
    import torch

    for _ in range(5):
        fn()
    torch.cuda.synchronize()
    out: list[float] = []
    while True:
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(iters)]
        for s, e in ev:
            if flush is not None:
                flush.zero_()
            s.record(stream)
            fn()
            e.record(stream)
        torch.cuda.synchronize()
        out += [s.elapsed_time(e) for s, e in ev]
        if sum(out) >= min_ms or len(out) >= 100 * iters:
            return out


L2_FLUSH_BYTES = 256 << 20       # about twice the 126 MiB L2


def _l2_flush_buffer():
    import torch

    return torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")


def run_suite(args) -> int:
    """Every hot-path row on its workload: one JSON object per (row, variant).

    --rows picks row groups, --scale divides every per-rank size (small cases
    for profiler runs), --suite-iters fixes the timed launches per row."""
    import torch

    import symmetric_memory_allreduce_gb300 as sm
    from symmetric_memory_allreduce_gb300 import workloads as wl

    torch.cuda.set_device(0)
    sm.load()
    stream = torch.cuda.current_stream()
    peak, peak_kind = measured_peak()
    flush = _l2_flush_buffer()

    def report(row, variant, ts, per_rank, hbm_bytes, logical_bytes=None, extra=None):
        med = statistics.median(ts)
        d = {"row": row, "variant": variant, "iters": len(ts), "us_median": med * 1e3,
             "us_p10": percentile(ts, 0.1) * 1e3, "us_p90": percentile(ts, 0.9) * 1e3,
             "algbw_gbs": per_rank / (med * 1e-3) / 1e9,
             "hbm_model_gbs": hbm_bytes / (med * 1e-3) / 1e9,
             "frac_of_peak": hbm_bytes / (med * 1e-3) / 1e9 / peak, "peak_gbs": peak,
             "peak_kind": peak_kind}
        if logical_bytes:
            d["logical_gbs"] = logical_bytes / (med * 1e-3) / 1e9
        if extra:
            d.update(extra)
        print(json.dumps(d), flush=True)
        assert sm.sym_stream_status() == sm.SYM_OK, sm.sym_last_error()

    def iters_for(nbytes):
        if args.suite_iters:
            return args.suite_iters
        return max(20, min(1000, int(4e9 / max(nbytes, 1))))

    def its(n):
        return args.suite_iters or n

    # every row: >= 20 launches and >= 200 ms of timed launches (fixed count with --suite-iters)
    min_ms = 0.0 if args.suite_iters else 200.0

    def timed(fn, iters, stream_, flush=None):
        return _time_launches(fn, iters, stream_, flush, min_ms)

    scale = max(1, args.scale)
    wanted = [w.strip() for w in args.rows.split(",") if w.strip()]

    def want(group):
        return not wanted or group in wanted

    # AllReduce rows: R=4 x 4 MiB, R=8 x 64 MiB and R=8 x 256 MiB (fp32, and 128 MiB bf16),
    # every algorithm
    cases = [(1, "f32", ["oneshot", "twoshot", "twoshot_pull", "twoshot_split"]),
             (2, "f32", ["oneshot", "twoshot", "twoshot_pull", "twoshot_split"]),
             (3, "f32", ["twoshot", "twoshot_pull", "twoshot_split"]),
             (3, "bf16", ["twoshot", "twoshot_pull"])]
    for cfg, dt, algos in cases if want("allreduce") else []:
        x = wl.workload_inputs(cfg, n=wl.WORKLOADS[cfg].count // scale)
        if dt == "bf16":
            x = wl.to_bf16_bits(x)
        R, n = x.shape
        S = n * x.itemsize
        send, recv = sm.Window(R, S), sm.Window(R, S)
        for r in range(R):
            send.write(r, x[r])
        stream.synchronize()
        for algo in algos:
            ts = timed(lambda: sm.sym_allreduce(send, recv, n, dt, "sum", algo),
                                iters_for(2 * R * S), stream)
            m = algo_bytes(algo, R, S)
            resident = 2 * R * S < (126 << 20)
            report(f"allreduce R={R} x {_size(S)} {wl.WORKLOADS[cfg].dist}", f"{algo} {dt}", ts, S,
                   m["compulsory"], m["logical"],
                   {"R": R, "bytes_per_rank": S, "l2_resident": resident})
            if resident:
                # the same launches with L2 flushed before each one (cold column)
                ts = timed(lambda: sm.sym_allreduce(send, recv, n, dt, "sum", algo),
                                    its(50), stream, flush)
                report(f"allreduce R={R} x {_size(S)} {wl.WORKLOADS[cfg].dist}", f"{algo} {dt} cold L2",
                       ts, S, m["compulsory"],
                       m["logical"], {"R": R, "bytes_per_rank": S, "l2_resident": False})
        send.free()
        recv.free()
        del x

    # AllGather (copy, CE) and put+signal AllGather: R=16 x 32 MiB of random bytes
    if want("allgather") or want("put_signal"):
        cfg5 = wl.PUT_SIGNAL
        R, S = cfg5["R"], cfg5["nbytes"] // scale
        xb = wl.random_bytes(5, R, S)
        send, recv = sm.Window(R, S, ncounters=1), sm.Window(R, R * S, nsignals=R)
        for r in range(R):
            send.write(r, xb[r])
        stream.synchronize()
        comp = R * S + R * R * S
        for algo in ("copy", "ce") if want("allgather") else ():
            ts = timed(lambda: sm.sym_allgather(send, recv, S // 4, "f32", algo), its(50),
                                stream)
            kern = os.environ.get("SYM_ALLGATHER_KERNEL", "bulk") if algo == "copy" else "copy engines"
            report(f"allgather R={R} x {_size(S)} bytes", algo, ts, S, comp,
                   extra={"R": R, "bytes_per_rank": S, "kernel": kern})
        nchunks = -(-S // cfg5["chunk"])
        for batch in (8, 1, 64) if want("put_signal") else ():
            ts = timed(lambda: sm.sym_allgather(send, recv, S // 4, "f32", "put_signal",
                                                         cfg5["chunk"], batch), its(50), stream)
            report(f"put_signal allgather R={R} x {_size(S)} bytes", f"chunk 64KiB, {batch} chunks/signal",
                   ts, S, comp,
                   extra={"R": R, "bytes_per_rank": S, "signals_per_pair": -(-nchunks // batch)})
        send.free()
        recv.free()

    # AlltoAll: R=8, 32 MiB per rank (R segments of 4 MiB)
    if want("alltoall"):
        R, B = 8, (4 << 20) // scale
        xa = wl.random_bytes(6, R, R * B)
        send, recv = sm.Window(R, R * B), sm.Window(R, R * B, nsignals=1)
        for r in range(R):
            send.write(r, xa[r])
        stream.synchronize()
        for algo in ("copy", "put_signal"):
            ts = timed(lambda: sm.sym_alltoall(send, recv, B // 4, "f32", algo), its(100),
                                stream)
            report("alltoall", algo, ts, R * B, 2 * R * R * B, extra={"R": R, "bytes_per_segment": B})
        send.free()
        recv.free()

    # fused producer + AllReduce: R=8 x 256 MiB fp32
    if want("fused"):
        x = wl.workload_inputs(3, n=wl.WORKLOADS[3].count // scale)
        R, n = x.shape
        S = n * 4
        win_in, send, recv = sm.Window(R, S), sm.Window(R, S), sm.Window(R, S)
        for r in range(R):
            win_in.write(r, x[r])
        stream.synchronize()
        alpha = [1.0 + 0.25 * r for r in range(R)]
        ts = timed(lambda: sm.sym_scale_allreduce(win_in, send, recv, alpha, n), its(100),
                            stream)
        report("fused producer + allreduce", "scale then two-shot, counter relay", ts, S,
               3 * R * S, extra={"R": R, "bytes_per_rank": S,
                                 "bytes_model": "read in RS + write contributions RS + write "
                                                "results RS"})
        for w in (win_in, send, recv):
            w.free()

    # practical ceilings on this GPU (library kernels, calibration only): an SM
    # copy (reads = writes), a copy-engine copy, and a write-only fill, 2 GiB each
    if want("ceiling"):
        nb = (2 << 30) // scale
        src = torch.empty(nb // 4, dtype=torch.float32, device="cuda").normal_()
        dst = torch.empty_like(src)
        ts = timed(lambda: torch.mul(src, 1.0, out=dst), its(50), stream)
        report("ceiling", "SM copy (torch elementwise)", ts, nb, 2 * nb, extra={"bytes": nb})
        ts = timed(lambda: dst.copy_(src), its(50), stream)
        report("ceiling", "device copy (torch copy_)", ts, nb, 2 * nb, extra={"bytes": nb})
        ts = timed(lambda: dst.fill_(1.0), its(50), stream)
        report("ceiling", "write only (torch fill_)", ts, nb, nb, extra={"bytes": nb})
        del src, dst
    return 0


# ----------------------------------------------------------------- results table

# kernel-name patterns of each row's main launch, for matching an ncu launch list to the rows
_MAIN_KERNEL = {"oneshot": "k_oneshot", "twoshot": "k_twoshot_st", "twoshot_pull": "k_twoshot_pull_ws",
                "put_signal": "k_put_signal_allgather"}


def table_rows():
    """(label, workload index, algo, dtype, count or bytes, extra) of every results-table row."""
    rows = []
    for dist in ("rankfill", "normal"):
        for algo in ("oneshot", "twoshot"):
            rows.append((f"R=4 × 4 MiB, {'rank fill' if dist == 'rankfill' else 'N(0,1)'}", 1, algo,
                         "f32", 1 << 20, dist))
    for algo in ("oneshot", "twoshot", "twoshot_pull"):
        rows.append(("R=8 × 64 MiB, N(0,1)", 2, algo, "f32", 1 << 24, None))
    for dt in ("f32", "bf16"):
        for algo in ("twoshot", "twoshot_pull"):
            rows.append((f"R=8 × {_size((1 << 26) * (4 if dt == 'f32' else 2))}, U(-1,1)", 3, algo, dt,
                         1 << 26, None))
    for k in range(11):
        nbytes = 1024 * 4 ** k
        for algo in ("oneshot", "twoshot"):
            rows.append((f"R=8 × {_size(nbytes)}, N(0,1) (sweep)", 4, algo, "f32", nbytes // 4, None))
    for batch in (8, 1, 64):
        rows.append((f"R=16 × 32 MiB bytes, 64 KiB chunks, {batch}/signal", 5, "put_signal", "bytes",
                     32 << 20, batch))
    return rows


def _table_inputs(cfg, dt, n, extra):
    from symmetric_memory_allreduce_gb300 import workloads as wl

    if cfg == 5:
        return wl.random_bytes(5, wl.PUT_SIGNAL["R"], n)
    x = wl.workload_inputs(cfg, n=n, dist=extra) if cfg != 4 else wl.workload_inputs(4, n=n)
    return wl.to_bf16_bits(x) if dt == "bf16" else x


def parse_dram_csv(path: str) -> list[tuple[str, float]]:
    """(kernel name, DRAM bytes read + written) of every launch in an ncu --csv launch list."""
    import csv

    per = {}
    order = []
    with open(path) as f:
        lines = [l for l in f if l.startswith('"')]
    for rec in csv.DictReader(lines):
        key = rec.get("ID")
        if key not in per:
            per[key] = [rec.get("Kernel Name", ""), 0.0]
            order.append(key)
        if rec.get("Metric Name") in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
            v = float(rec["Metric Value"].replace(",", ""))
            unit = rec.get("Metric Unit", "byte")
            scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}.get(unit, 1)
            per[key][1] += v * scale
    return [(per[k][0], per[k][1]) for k in order]


def run_table(args) -> int:
    """The benchmark results table: every config x algo x dtype row timed (CUDA events, >= 20
    launches and >= 200 ms after 5 warm-ups), every rank's output compared with the oracle, the
    oracle timed on 1 and on all host threads.  --table-dram-pass instead launches each row's call
    once (run it under ncu with the one-pass DRAM metrics); --dram-csv reads that launch list back
    into the table's DRAM column.  Markdown on stdout."""
    import numpy as np
    import torch

    import symmetric_memory_allreduce_gb300 as sm
    from symmetric_memory_allreduce_gb300 import workloads as wl

    torch.cuda.set_device(0)
    sm.load()
    stream = torch.cuda.current_stream()
    peak, peak_kind = measured_peak()
    dram = parse_dram_csv(args.dram_csv) if args.dram_csv else None
    dram_pos = 0
    nthr = os.cpu_count() or 1
    out = []
    if not args.table_dram_pass:
        import oracle

        oracle.build()
    for label, cfg, algo, dt, n, extra in table_rows():
        x = _table_inputs(cfg, dt, n, extra)
        R = x.shape[0]
        if cfg == 5:
            S = x.shape[1]
            c5 = wl.PUT_SIGNAL
            send, recv = sm.Window(R, S, ncounters=1), sm.Window(R, R * S, nsignals=R)
            call = (lambda: sm.sym_allgather(send, recv, S // 4, "f32", "put_signal", c5["chunk"], extra))
            comp, logical = R * S + R * R * S, 2 * R * R * S
        else:
            S = x.shape[1] * x.itemsize
            send, recv = sm.Window(R, S), sm.Window(R, S)
            call = (lambda: sm.sym_allreduce(send, recv, x.shape[1], dt, "sum", algo))
            m = algo_bytes(algo, R, S)
            comp, logical = m["compulsory"], m["logical"]
        try:
            for r in range(R):
                send.write(r, x[r])
            stream.synchronize()
            if args.table_dram_pass:
                call()
                torch.cuda.synchronize()
                continue
            iters = max(20, min(2000, int(4e9 / max(comp, 1))))
            ts = _time_launches(call, iters, stream, None, 200.0)
            if sm.sym_stream_status() != sm.SYM_OK:
                raise RuntimeError(f"{label} {algo}: " + sm.sym_last_error())
            med = statistics.median(ts)
            # parity: every rank's output against the oracle; oracle timed on 1 and nthr threads
            if cfg == 5:
                t0 = time.perf_counter()
                want, sig, cnt = oracle.put_signal_allgather(x, wl.PUT_SIGNAL["chunk"], extra)
                t1_ms, tn_ms = (time.perf_counter() - t0) * 1e3, None
                ok = True
                buf = np.empty(R * S, np.uint8)
                for p in range(R):
                    recv.read(p, buf)
                    stream.synchronize()
                    ok &= bool(np.array_equal(buf, want))
                    ok &= all(sm.sym_signal_read(recv, p, q) == int(sig[p, q]) for q in range(R))
                    ok &= sm.sym_counter_read(send, p, 0) == int(cnt[p])
            else:
                t0 = time.perf_counter()
                oracle.allreduce_sum_mt(x, 1)
                t1_ms = (time.perf_counter() - t0) * 1e3
                t0 = time.perf_counter()
                want, _ = oracle.allreduce_sum_mt(x, nthr)
                tn_ms = (time.perf_counter() - t0) * 1e3
                ok = True
                y = np.empty(x.shape[1], x.dtype)
                for r in range(R):
                    recv.read(r, y)
                    stream.synchronize()
                    ok &= bool(np.array_equal(y.view(np.uint8), want.view(np.uint8)))
            row = {"label": label, "algo": algo, "dtype": dt, "R": R, "bytes_per_rank": S,
                   "t_ms": med, "launches": len(ts), "algbw": S / (med * 1e-3) / 1e9,
                   "logical_gbs": logical / (med * 1e-3) / 1e9,
                   "compulsory_gbs": comp / (med * 1e-3) / 1e9, "parity": ok,
                   "oracle_1t_ms": t1_ms, "oracle_nt_ms": tn_ms, "l2_resident": 2 * R * S < (126 << 20),
                   "oracle_threads": nthr, "cpu_model": cpu_model()}
            if dram is not None:
                pat = _MAIN_KERNEL[algo]
                while dram_pos < len(dram) and pat not in dram[dram_pos][0]:
                    dram_pos += 1
                if dram_pos < len(dram):
                    row["dram_bytes"] = dram[dram_pos][1]
                    row["dram_gbs"] = dram[dram_pos][1] / (med * 1e-3) / 1e9
                    dram_pos += 1
            out.append(row)
            print(json.dumps(row), file=sys.stderr, flush=True)
        finally:
            send.free()
            recv.free()
    if args.table_dram_pass:
        return 0
    print(format_table(out, peak, peak_kind, nthr, cpu_model()))
    return 0


def format_table(rows: list[dict], peak: float, peak_kind: str, nthr: int, cpu: str) -> str:
    """Markdown of the results table from its JSON rows (as run_table writes them to stderr).
    A row is flagged L2-served when its logical bytes exceed the DRAM bytes by more than 10 %:
    repeated reads of the same lines came from L2, not HBM."""
    lines = [f"| Workload | Algo | dtype | t median (ms) | algbw GB/s | logical GB/s | compulsory GB/s "
             f"| HBM GB/s (ncu DRAM bytes / t) | % of measured peak | logical / DRAM | parity "
             f"| oracle 1-thread (ms) | oracle {nthr}-thread (ms) |",
             "|---|---|---|---|---|---|---|---|---|---|---|---|---|"]
    for r in rows:
        ratio = "—"
        if "dram_gbs" in r:
            hbm = f"{r['dram_gbs']:,.0f}"
            pct = ("L2-resident (n/m)" if r["l2_resident"] else f"{100 * r['dram_gbs'] / peak:.1f} %")
            if not r["l2_resident"]:
                q = r["logical_gbs"] / r["dram_gbs"]
                ratio = f"{q:.2f}" + (" (L2-served)" if q > 1.1 else "")
        else:
            hbm, pct = "—", ("L2-resident (n/m)" if r["l2_resident"] else
                             f"{100 * r['compulsory_gbs'] / peak:.1f} % (compulsory)")
        parity = "bit-exact" if r["parity"] else "**MISMATCH**"
        tn = f"{r['oracle_nt_ms']:.1f}" if r["oracle_nt_ms"] is not None else "—"
        lines.append(f"| {r['label']} | {r['algo']} | {r['dtype']} | {r['t_ms']:.4f} | {r['algbw']:,.1f} "
                     f"| {r['logical_gbs']:,.0f} | {r['compulsory_gbs']:,.0f} | {hbm} | {pct} | {ratio} "
                     f"| {parity} | {r['oracle_1t_ms']:.1f} | {tn} |")
    lines.append(f"\nPeak: {peak:,.0f} GB/s ({peak_kind} HBM copy bandwidth, MEASURED_PEAKS.json); "
                 f"host: {cpu}, {nthr} threads.")
    return "\n".join(lines)


def run_table_from_json(args) -> int:
    """Re-render the results table from the JSON rows a --table run wrote (no GPU); the host's
    thread count and CPU come from the rows, else from --table-threads / --table-cpu."""
    rows = [json.loads(l) for l in open(args.table_from_json) if l.startswith("{")]
    peak, peak_kind = measured_peak()
    nthr = rows[0].get("oracle_threads", args.table_threads) if rows else args.table_threads
    cpu = rows[0].get("cpu_model", args.table_cpu) if rows else args.table_cpu
    print(format_table(rows, peak, peak_kind, nthr, cpu))
    return 0


def parse(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--algo", default="twoshot",
                    choices=["auto", "oneshot", "twoshot", "twoshot_pull", "twoshot_split"])
    ap.add_argument("--ranks", type=int, default=R_DEFAULT)
    ap.add_argument("--count", type=int, default=N_DEFAULT)
    ap.add_argument("--e2e-steps", type=int, default=40,
                    help="end-to-end steps (the pipeline's fill and drain amortise over them)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the other rows (bf16 and pull at R=8 x 256 MiB, R=8 x 64 MiB, "
                         "put + signal AllGather, AUTO crossover)")
    ap.add_argument("--sweep", action="store_true",
                    help="message-size sweep of every algorithm instead of the contract line")
    ap.add_argument("--sweep-max", type=int, default=1 << 30)
    ap.add_argument("--suite", action="store_true",
                    help="time every hot-path row on its workload instead of the contract line")
    ap.add_argument("--rows", default="",
                    help="--suite: comma-separated row groups (allreduce, allgather, put_signal, "
                         "alltoall, fused, ceiling); default all")
    ap.add_argument("--scale", type=int, default=1,
                    help="--suite: divide every per-rank size by this (small profiling cases)")
    ap.add_argument("--suite-iters", type=int, default=0,
                    help="--suite: timed launches per row (0: by size); small for profiler runs")
    ap.add_argument("--table", action="store_true",
                    help="the results table (every config x algo x dtype) as markdown")
    ap.add_argument("--table-dram-pass", action="store_true",
                    help="--table: launch each row's call once (for an ncu one-pass DRAM launch list)")
    ap.add_argument("--dram-csv", default="",
                    help="--table: ncu --csv launch list of a --table-dram-pass run (DRAM column)")
    ap.add_argument("--table-from-json", default="",
                    help="re-render the table from the JSON rows (stderr) of a --table run; no GPU")
    ap.add_argument("--table-threads", type=int, default=os.cpu_count() or 1,
                    help="--table-from-json: oracle threads of the recorded run, if the rows lack it")
    ap.add_argument("--table-cpu", default="(not recorded)",
                    help="--table-from-json: host CPU of the recorded run, if the rows lack it")
    a = ap.parse_args(argv)
    a.warmup = max(a.warmup, 3)          # at least three untimed warm-up steps
    return a


def main(argv=None) -> int:
    args = parse(argv)
    if args.impl == "reference":
        return run_reference(args)
    if args.sweep:
        return run_sweep(args)
    if args.suite:
        return run_suite(args)
    if args.table_from_json:
        return run_table_from_json(args)
    if args.table or args.table_dram_pass:
        return run_table(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
