"""Benchmark: SSD forward tokens/s on the Mamba-2 2.7B-shaped layer.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--algo auto|fused|chunked]

One step = one full forward pass (all four steps of the method) over one
batch of synthetic inputs that already sit in HBM.  Prints ONE JSON line.

* value      B·L / time, device-timed with CUDA events over K steps (inputs of
             709 MB exceed the 126 MB L2, so no flush is needed between steps).
* e2e        the same metric through the public call with pinned host buffers:
             every step copies its inputs host→device and reads y and the final
             state back, inside the timed region.
* roofline   algorithmic bytes of one launch / the dominant kernel's average
             launch time (events around each call on its stream), against the
             measured HBM copy bandwidth.
* cpu_baseline  the fp64 CPU oracle timed on the host cores on a bounded
             sample of the same workload.
* --impl reference  times the oracle itself as the reference arm.

Multi-GPU: the scan has no cross-GPU exchange on one node, so N ranks run N
independent replicas (weak scaling); rank 0 prints max-over-ranks timing.
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
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "SSD fwd tokens/s (B·L/s) on 1 B300 & % of roofline (HBM GB/s or TC TFLOP/s)"
DEFAULT_WORKLOAD = "mamba2_2p7b"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def _dist():
    """(rank, world, local_rank) from torchrun's environment, else (0, 1, 0)."""
    if "RANK" in os.environ and "WORLD_SIZE" in os.environ:
        return int(os.environ["RANK"]), int(os.environ["WORLD_SIZE"]), int(os.environ.get("LOCAL_RANK", 0))
    return 0, 1, 0


def _kernel_source_hash(algo_used: str) -> str:
    name = "fused.cu" if algo_used == "fused" else "chunked.cu"
    with open(os.path.join(ROOT, "ssd_scan_fwd_b300", "csrc", name), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def _recorded_traffic(workload: str, algo_used: str):
    """DRAM bytes per launch of the dominant kernel from a committed ncu
    summary, or None if none exists or the kernel source changed since."""
    kern = "ssd_fused" if algo_used == "fused" else "ssd_chunk_scan"
    path = os.path.join(ROOT, "profiles", f"{kern}_{workload}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m_b = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    m_h = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text)
    if not m_b or not m_h or m_h.group(1) != _kernel_source_hash(algo_used):
        return None
    return float(m_b.group(1))


class _NvmlPoller:
    """SM clock and clock-event reasons (and, less often, power) read through
    NVML (libnvidia-ml, loaded with ctypes) on a thread every fraction of a
    millisecond, so that a timed region of a few milliseconds still gets
    samples."""

    # clock-event reason bits (nvml.h)
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, uuid: str | None):
        import ctypes
        import threading
        self.ct = ctypes
        self.nv = ctypes.CDLL("libnvidia-ml.so.1")
        if self.nv.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        ok = False
        if uuid:
            u = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
            ok = self.nv.nvmlDeviceGetHandleByUUID(u.encode(), ctypes.byref(self.h)) == 0
        if not ok:
            raise RuntimeError("no NVML handle for the device")
        self.reason_fn = getattr(self.nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(self.nv, "nvmlDeviceGetCurrentClocksThrottleReasons", None)
        self.rows = []
        self.stop = threading.Event()
        self.th = threading.Thread(target=self._run, daemon=True)

    def _run(self):
        ct = self.ct
        clk, mx, pw, rs = ct.c_uint(), ct.c_uint(), ct.c_uint(), ct.c_ulonglong()
        self.nv.nvmlDeviceGetMaxClockInfo(self.h, 1, ct.byref(mx))
        i = 0
        while not self.stop.is_set():
            self.nv.nvmlDeviceGetClockInfo(self.h, 1, ct.byref(clk))      # NVML_CLOCK_SM
            if self.reason_fn is not None:
                self.reason_fn(self.h, ct.byref(rs))
            if i % 16 == 0:  # the power reading is the slow one
                self.nv.nvmlDeviceGetPowerUsage(self.h, ct.byref(pw))
            self.rows.append((clk.value, mx.value, pw.value / 1000.0, rs.value))
            i += 1
            time.sleep(0.0002)

    def start(self):
        self.th.start()

    def finish(self):
        self.stop.set()
        self.th.join()
        return self.rows


class ClockSampler:
    """SM clock and throttle reasons while the timed region runs: NVML polled
    on a thread (a timed region of a few milliseconds still gets samples),
    else nvidia-smi samples every 200 ms."""

    FIELDS = ("index,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.proc = None
        self.path = None
        self.nvml = None
        self.nvml_rows = None

    def __enter__(self):
        try:
            self.nvml = _NvmlPoller(self.uuid)
            self.nvml.start()
            time.sleep(0.005)
            return self
        except Exception:
            self.nvml = None
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.nvml is not None:
            self.nvml_rows = self.nvml.finish()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.nvml_rows is not None:
            rows = self.nvml_rows
            if not rows:
                return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
            sm = sorted(r[0] for r in rows)
            loaded = sm[len(sm) // 2:]
            reasons = sorted({name for r in rows for bit, name in _NvmlPoller.REASONS.items() if r[3] & bit})
            return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(r[1] for r in rows),
                    "reasons": reasons, "samples": len(rows), "source": "nvml poll",
                    "power_w_max": max(r[2] for r in rows)}
        if self.proc is None or not self.path:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            if self.uuid and self.uuid not in parts[1]:
                continue
            rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None

        sm = [num(r[2]) for r in rows if num(r[2]) is not None]
        mx = [num(r[3]) for r in rows if num(r[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[6 + i].lower() == "active"})
        loaded = sorted(sm)[len(sm) // 2:] if sm else []
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows), "source": "nvidia-smi 200 ms",
                "power_w_max": max((num(r[4]) or 0.0) for r in rows)}


def _device_uuid(torch, dev):
    try:
        return str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        return None


# ---------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline and the reference arm)
# ---------------------------------------------------------------------------
def _oracle_sample(w, inp, budget_s: float):
    """Time the fp64 oracle on whole batch rows (all heads, full length) of
    the workload, adding rows while the budget allows.  Returns
    (tokens/s, threads, description, seconds)."""
    import oracle
    threads = len(os.sched_getaffinity(0))
    oracle.set_threads(threads)
    rows, tok, secs = 0, 0, 0.0
    while rows < w.batch:
        b = rows
        row = [None if v is None else v.double().numpy()
               for v in (inp["x"][b:b + 1], inp["dt"][b:b + 1], inp["A"], inp["Bm"][b:b + 1],
                         inp["Cm"][b:b + 1], inp["D"],
                         None if inp["init_state"] is None else inp["init_state"][b:b + 1])]
        t0 = time.perf_counter()
        oracle.ssd_recurrent(*row)
        secs += time.perf_counter() - t0
        rows += 1
        tok += w.seqlen
        if secs >= budget_s:
            break
    desc = (f"fp64 sequential-recurrence oracle (OpenMP over heads) on {rows} of {w.batch} batch rows "
            f"x {w.seqlen} tokens x {w.nheads} heads of the workload")
    return tok / secs, threads, desc, secs


def run_reference(args, w):
    rank, world, _ = _dist()
    if rank != 0:
        return 0
    from ssd_scan_fwd_b300.inputs import generate
    inp = generate(w)
    import oracle
    threads = len(os.sched_getaffinity(0))
    oracle.set_threads(threads)
    b = 0
    sl = slice(b, b + 1)
    L_s = min(w.seqlen, max(256, int(args.ref_tokens)))

    def step():
        oracle.ssd_recurrent(inp["x"][sl, :L_s], inp["dt"][sl, :L_s], inp["A"], inp["Bm"][sl, :L_s],
                             inp["Cm"][sl, :L_s], inp["D"],
                             None if inp["init_state"] is None else inp["init_state"][sl])

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    value = L_s / dt
    desc = (f"each step: the fp64 oracle on 1 batch row x {L_s} tokens x {w.nheads} heads "
            f"of the workload (bounded sample)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": _config(w),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def _config(w):
    from ssd_scan_fwd_b300.inputs import algorithmic_bytes
    return {"workload": f"{w.name}: B={w.batch} L={w.seqlen} H={w.nheads} P={w.headdim} "
                        f"N={w.dstate} G={w.ngroups} io={w.io_dtype}"
                        + (" init_state" if w.has_init else ""),
            "batch": w.batch, "seqlen": w.seqlen, "nheads": w.nheads, "headdim": w.headdim,
            "dstate": w.dstate, "ngroups": w.ngroups, "io_dtype": w.io_dtype,
            "accumulate": "fp32", "state": "fp32",
            "algorithmic_bytes_per_step": algorithmic_bytes(w),
            "l2": f"inputs larger than L2 ({algorithmic_bytes(w) / 1e6:.0f} MB moved per step vs 126 MB L2); no flush"}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
def run_ours(args, w):
    import torch
    import torch.distributed as dist

    import ssd_scan_fwd_b300 as ssd
    from ssd_scan_fwd_b300 import _lib
    from ssd_scan_fwd_b300.inputs import algorithmic_bytes, algorithmic_flops, generate

    rank, world, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    inp = generate(w)
    d = {k: (None if v is None else v.to(dev)) for k, v in inp.items()}
    B, L, H, P, N = w.batch, w.seqlen, w.nheads, w.headdim, w.dstate
    y = torch.empty_like(d["x"])
    fs = torch.empty(B, H, P, N, dtype=torch.float32, device=dev)
    cargs = ssd.make_args(d["x"], d["dt"], d["A"], d["Bm"], d["Cm"], d["D"], d["init_state"], y, fs,
                          algo=args.algo)
    need = ssd.workspace_size(cargs)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    cargs.workspace = ws.data_ptr()
    cargs.workspace_bytes = need
    lib = _lib.lib()
    import ctypes
    stream = torch.cuda.current_stream(dev)
    sh = ctypes.c_void_p(stream.cuda_stream)
    algo_used = "fused" if (args.algo in ("fused",) or (args.algo == "auto" and _fused_chosen(cargs))) else "chunked"
    launches_per_step = 1 if algo_used == "fused" else 4

    def step():
        _lib.check(lib.ssd_fwd(ctypes.byref(cargs), sh), "ssd_fwd")

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()

    # timed region: K steps, events per call on the launching stream
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(_device_uuid(torch, dev)) as clk:
        torch.cuda.synchronize(dev)
        if world > 1:
            dist.barrier()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for i in range(args.steps):
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        t1.record(stream)
        torch.cuda.synchronize(dev)
        if world > 1:
            dist.barrier()
    total_ms = t0.elapsed_time(t1)
    per_launch_ms = statistics.mean(s.elapsed_time(e) for s, e in zip(starts, ends))
    ms_per_step, value = whole_job(total_ms, args.steps, B * L, world,
                                   lambda v: _reduce_max(dist, torch, v, dev) if world > 1 else v)

    # end to end through the public call with pinned host buffers
    e2e = None if args.no_e2e else _e2e(args, w, inp, dev, world)

    peaks, src = _peaks()
    alg_bytes = algorithmic_bytes(w)
    achieved = alg_bytes / (per_launch_ms / 1e3) / 1e9
    peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    traffic = _recorded_traffic(w.name, algo_used)
    # the tensor-pipe side of the same launch: algorithmic flops (bf16
    # operands, fp32 accumulation) against the measured dense bf16 burst peak
    tc_peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    tc_achieved = algorithmic_flops(w) / (per_launch_ms / 1e3) / 1e12
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        v, thr, desc, secs = _oracle_sample(w, inp, args.cpu_budget)
        cpu = {"value": v, "unit": "tokens/s", "cores": thr, "kind": "oracle",
               "sample": desc + f" ({secs:.1f} s)"}
    lps, lps_how = _launches_per_step(torch, step, launches_per_step)
    if rank == 0:
        clocks = clk.summary()
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if w.io_dtype == "bf16" else "f32",
            "data": "synthetic", "config": dict(_config(w), algo=algo_used),
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic,
                         "kernel": "ssd_fused" if algo_used == "fused" else "ssd_chunked (4 kernels)",
                         "peak_source": f"{src} hbm_gbs (MEASURED_PEAKS.json)" if src == "measured" else "fallback",
                         "per_launch_ms": per_launch_ms,
                         "tc": {"achieved": tc_achieved, "peak": tc_peak, "unit": "TFLOP/s",
                                "frac": tc_achieved / tc_peak, "flops_per_launch": algorithmic_flops(w),
                                "peak_source": (f"{src} bf16_tflops (MEASURED_PEAKS.json, burst)"
                                                if src == "measured" else "fallback")}},
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": lps * args.steps,
            "gpu_launches_how": lps_how,
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def _reduce_max(dist, torch, v: float, dev) -> float:
    """Maximum of v over all ranks of the process group."""
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _launches_per_step(torch, step, static: int):
    """Kernels one step launches, counted on one more, untimed step run under
    torch.profiler's CUDA activity trace after the timed region (memsets and
    copies are not kernels); the path's static count when the trace is not
    available.  Returns (count, how it was obtained)."""
    try:
        from torch.profiler import ProfilerActivity, profile
        torch.cuda.synchronize()
        with profile(activities=[ProfilerActivity.CUDA]) as prof:
            step()
            torch.cuda.synchronize()
        n = 0
        for e in prof.events():
            if e.device_type != torch.autograd.DeviceType.CUDA:
                continue
            if any(t in e.name for t in ("Memset", "Memcpy", "memset", "memcpy")):
                continue
            n += 1
        if n > 0:
            return n, "counted: CUDA kernels of one untimed step under torch.profiler"
    except Exception:  # noqa: BLE001 - the static count stands in
        pass
    return static, "static: kernels the path launches per call"


def whole_job(total_ms: float, steps: int, tokens_per_rank: int, world: int, reduce_max):
    """Whole-job throughput of N replicas: the slowest rank's time (max over
    ranks) for K steps, and the tokens of all ranks over that time.
    Returns (ms_per_step, tokens/s)."""
    slowest = reduce_max(total_ms)
    ms_per_step = slowest / steps
    return ms_per_step, world * tokens_per_rank / (ms_per_step / 1e3)


def _fused_chosen(cargs) -> bool:
    import ctypes

    from ssd_scan_fwd_b300 import _lib
    a = _lib.SsdFwdArgs.from_buffer_copy(cargs)
    a.algo = _lib.SSD_ALGO_FUSED
    return _lib.lib().ssd_fwd_workspace_size(ctypes.byref(a)) != ctypes.c_size_t(-1).value


def _e2e(args, w, inp, dev, world):
    """Same metric through the C ABI on host buffers: ssd_fwd_host copies the
    step's inputs from pinned host memory and y / final_state back, every
    step, inside the timed region (overlapping the copies of one group of
    batch rows with the compute of another)."""
    import ctypes

    import torch

    import ssd_scan_fwd_b300 as ssd
    from ssd_scan_fwd_b300 import _lib
    host = {k: (None if v is None else v.pin_memory()) for k, v in inp.items()}
    B, L, H, P, N = w.batch, w.seqlen, w.nheads, w.headdim, w.dstate
    y_host = torch.empty(inp["x"].shape, dtype=inp["x"].dtype).pin_memory()
    f_host = torch.empty(B, H, P, N, dtype=torch.float32).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in host.values() if v is not None)
    d2h = y_host.numel() * y_host.element_size() + f_host.numel() * 4
    cargs = ssd.make_args(host["x"], host["dt"], host["A"], host["Bm"], host["Cm"], host["D"], host["init_state"],
                          y_host, f_host, algo=args.algo)
    lib = _lib.lib()
    need = lib.ssd_fwd_host_workspace_size(ctypes.byref(cargs))
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    cargs.workspace = ws.data_ptr()
    cargs.workspace_bytes = need
    s = torch.cuda.current_stream(dev)
    sh = ctypes.c_void_p(s.cuda_stream)

    def step():
        _lib.check(lib.ssd_fwd_host(ctypes.byref(cargs), sh), "ssd_fwd_host")

    for _ in range(max(1, args.warmup // 2)):
        step()
    torch.cuda.synchronize(dev)
    k = max(1, min(args.steps, args.e2e_steps))
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(s)
    for _ in range(k):
        step()
    t1.record(s)
    torch.cuda.synchronize(dev)
    ms = t0.elapsed_time(t1) / k
    link = _link_bandwidth(torch, dev)
    # the copies alone, at the measured link rates, overlapping in the two directions
    ideal_ms = max(h2d / link["h2d_gbs"], d2h / link["d2h_gbs"], (h2d + d2h) / link["bidir_gbs"]) / 1e6
    return {"value": world * B * L / (ms / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms, "steps": k, "api": "ssd_fwd_host (C ABI, host buffers)",
            "link": dict(link, copy_bound_ms=ideal_ms, frac=ideal_ms / ms)}


def _link_bandwidth(torch, dev, nbytes: int = 256 << 20, reps: int = 3):
    """Pinned host <-> device copy bandwidth (GB/s): host to device, device to
    host, and both at once on two streams (the sum of the bytes over the time)."""
    h_src = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    h_dst = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    d_a = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    d_b = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    s1, s2 = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def timed(fn):
        best = float("inf")
        for _ in range(reps):
            torch.cuda.synchronize(dev)
            t = time.perf_counter()
            fn()
            torch.cuda.synchronize(dev)
            best = min(best, time.perf_counter() - t)
        return best

    def h2d():
        with torch.cuda.stream(s1):
            d_a.copy_(h_src, non_blocking=True)

    def d2h():
        with torch.cuda.stream(s2):
            h_dst.copy_(d_b, non_blocking=True)

    def both():
        h2d()
        d2h()

    t_in, t_out, t_both = timed(h2d), timed(d2h), timed(both)
    return {"h2d_gbs": nbytes / t_in / 1e9, "d2h_gbs": nbytes / t_out / 1e9, "bidir_gbs": 2 * nbytes / t_both / 1e9,
            "bytes_per_copy": nbytes, "how": "pinned torch copies, best of 3, host wall clock around a synchronise"}


# ---------------------------------------------------------------------------
# Recurrent (decode) step: one token per sequence, the state updated in place.
# Not the headline line; run with --op step.
# ---------------------------------------------------------------------------
STEP_METRIC = "SSD decode step: tokens/s (one token per (batch row) per call) on 1 B300 & % of HBM roofline"


def step_bytes(B, H, P, N, G, io_bytes) -> int:
    """Bytes one ssd_step call must move: the fp32 state read and written,
    x in and y out, Bm and Cm in, dt in."""
    return 2 * B * H * P * N * 4 + 2 * B * H * P * io_bytes + 2 * B * G * N * io_bytes + B * H * 4


def run_step(args, w):
    import torch

    import ssd_scan_fwd_b300 as ssd
    from ssd_scan_fwd_b300.inputs import generate

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    B = args.decode_batch
    wl = w.with_(batch=B, seqlen=1, has_init=True)
    inp = generate(wl)
    d = {k: (None if v is None else v.to(dev)) for k, v in inp.items()}
    x, dt, Bm, Cm = (d[k][:, 0].contiguous() for k in ("x", "dt", "Bm", "Cm"))
    state = d["init_state"].clone()
    y = torch.empty_like(x)
    args_c = ssd.make_step_args(x, dt, d["A"], Bm, Cm, d["D"], state, y)
    import ctypes

    from ssd_scan_fwd_b300 import _lib
    lib = _lib.lib()
    stream = torch.cuda.current_stream(dev)
    sh = ctypes.c_void_p(stream.cuda_stream)

    def step():
        _lib.check(lib.ssd_step(ctypes.byref(args_c), sh), "ssd_step")

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(_device_uuid(torch, dev)) as clk:
        torch.cuda.synchronize(dev)
        for i in range(args.steps):
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
    ms = statistics.mean(a.elapsed_time(b) for a, b in zip(starts, ends))
    io = 2 if wl.io_dtype == "bf16" else 4
    nbytes = step_bytes(B, wl.nheads, wl.headdim, wl.dstate, wl.ngroups, io)
    peaks, src = _peaks()
    peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    achieved = nbytes / (ms / 1e3) / 1e9
    cpu = None
    if not args.no_cpu_baseline:
        import oracle
        threads = len(os.sched_getaffinity(0))
        oracle.set_threads(threads)
        nb = min(B, 8)
        t0 = time.perf_counter()
        reps = 0
        while True:
            oracle.ssd_recurrent(inp["x"][:nb], inp["dt"][:nb], inp["A"], inp["Bm"][:nb], inp["Cm"][:nb], inp["D"],
                                 inp["init_state"][:nb])
            reps += 1
            if time.perf_counter() - t0 >= args.cpu_budget:
                break
        secs = time.perf_counter() - t0
        cpu = {"value": reps * nb / secs, "unit": "tokens/s", "cores": threads, "kind": "oracle",
               "sample": f"fp64 recurrence oracle, one token of {nb} of {B} batch rows x {wl.nheads} heads, "
                         f"{reps} repetitions ({secs:.1f} s)"}
    lps, lps_how = _launches_per_step(torch, step, 1)
    line = {
        "metric": STEP_METRIC, "value": B / (ms / 1e3), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if wl.io_dtype == "bf16" else "f32", "data": "synthetic",
        "config": {"workload": f"decode step, {w.name} head shapes: B={B} H={wl.nheads} P={wl.headdim} "
                               f"N={wl.dstate} G={wl.ngroups} io={wl.io_dtype}",
                   "state_bytes": B * wl.nheads * wl.headdim * wl.dstate * 4,
                   "l2": "state larger than L2; no flush" if B * wl.nheads * wl.headdim * wl.dstate * 4 > 126e6
                         else "state smaller than L2"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": None, "kernel": "ssd_step_kernel",
                     "peak_source": f"{src} hbm_gbs (MEASURED_PEAKS.json)" if src == "measured" else "fallback",
                     "bytes_per_call": nbytes},
        "cpu_baseline": cpu, "e2e": None, "gpu_launches": lps * args.steps,
        "gpu_launches_how": lps_how, "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# Backward pass (gradients of every input for a given dy, dfinal).  Not the
# headline line; run with --op bwd.
# ---------------------------------------------------------------------------
BWD_METRIC = "SSD bwd tokens/s (B·L/s, all gradients) on 1 B300 & % of HBM roofline"


def bwd_bytes(B, L, H, P, N, G, io_bytes, has_init) -> int:
    """Bytes one ssd_bwd call must move at least: x, dy and dx; dt and ddt;
    Bm, Cm, dBm, dCm; dfinal and dinit (and init_state when given)."""
    per_tok_head = 3 * P * io_bytes + 2 * 4
    per_tok_group = 4 * N * io_bytes
    per_head = (3 if has_init else 2) * P * N * 4
    return B * L * (H * per_tok_head + G * per_tok_group) + B * H * per_head


def run_bwd(args, w):
    import torch

    import ssd_scan_fwd_b300 as ssd
    from ssd_scan_fwd_b300.inputs import generate, torch_dtype

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    inp = generate(w)
    d = {k: (None if v is None else v.to(dev)) for k, v in inp.items()}
    B, L, H, P, N, G = w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups
    g = torch.Generator().manual_seed(4242)
    dy = torch.randn(B, L, H, P, generator=g).to(torch_dtype(w.io_dtype)).to(dev)
    dfinal = torch.randn(B, H, P, N, generator=g).to(dev)
    ws = torch.empty(1, dtype=torch.uint8, device=dev)
    out = ssd.ssd_bwd(d["x"], d["dt"], d["A"], d["Bm"], d["Cm"], d["D"], d["init_state"], dy=dy, dfinal=dfinal)
    a = ssd.make_args(d["x"], d["dt"], d["A"], d["Bm"], d["Cm"], d["D"], d["init_state"])
    import ctypes

    from ssd_scan_fwd_b300 import _lib
    ba = _lib.SsdBwdArgs()
    ba.fwd = a
    ba.dy, ba.dfinal = dy.data_ptr(), dfinal.data_ptr()
    for k in ("dx", "ddt", "dA", "dBm", "dCm", "dD", "dinit"):
        setattr(ba, k, None if out[k] is None else out[k].data_ptr())
    lib = _lib.lib()
    need = lib.ssd_bwd_workspace_size(ctypes.byref(ba))
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    ba.fwd.workspace, ba.fwd.workspace_bytes = ws.data_ptr(), need
    stream = torch.cuda.current_stream(dev)
    sh = ctypes.c_void_p(stream.cuda_stream)

    def step():
        _lib.check(lib.ssd_bwd(ctypes.byref(ba), sh), "ssd_bwd")

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(_device_uuid(torch, dev)) as clk:
        torch.cuda.synchronize(dev)
        for i in range(args.steps):
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
    ms = statistics.mean(s.elapsed_time(e) for s, e in zip(starts, ends))
    io = 2 if w.io_dtype == "bf16" else 4
    nbytes = bwd_bytes(B, L, H, P, N, G, io, d["init_state"] is not None)
    # tensor-core per-chunk gradients (bf16 operands, fp32 accumulation) on
    # this shape unless forced onto the fp32 CUDA-core kernels
    tc = (w.io_dtype == "bf16" and P == 64 and N == 128 and os.environ.get("SSD_BWD_CUDA_CORES") != "1")
    peaks, src = _peaks()
    peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    achieved = nbytes / (ms / 1e3) / 1e9
    cpu = None
    if not args.no_cpu_baseline:
        import oracle
        threads = len(os.sched_getaffinity(0))
        oracle.set_threads(threads)
        # one batch row, a slice of heads: the oracle runs (batch, group) pairs in parallel
        hs = max(1, min(H, 8))
        sub = {k: inp[k] for k in inp}
        t0 = time.perf_counter()
        oracle.ssd_recurrent_bwd(sub["x"][:1, :, :hs], sub["dt"][:1, :, :hs], sub["A"][:hs],
                                 sub["Bm"][:1], sub["Cm"][:1], None if sub["D"] is None else sub["D"][:hs],
                                 None, dy=dy[:1, :, :hs].cpu(), dfinal=dfinal[:1, :hs].cpu())
        secs = time.perf_counter() - t0
        cpu = {"value": L * hs / H / secs, "unit": "tokens/s", "cores": min(threads, G), "kind": "oracle",
               "sample": f"fp64 backward oracle on 1 of {B} batch rows x {hs} of {H} heads x {L} tokens "
                         f"({secs:.1f} s; tokens/s scaled to all {H} heads; groups run in parallel, "
                         f"{G} here)"}
    lps, lps_how = _launches_per_step(torch, step, 5)
    line = {
        "metric": BWD_METRIC, "value": B * L / (ms / 1e3), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if tc else "f32", "data": "synthetic",
        "config": {"workload": f"backward pass, {w.name}: B={B} L={L} H={H} P={P} N={N} G={G} io={w.io_dtype}",
                   "algorithmic_bytes_per_step": nbytes,
                   "l2": f"inputs larger than L2 ({nbytes / 1e6:.0f} MB moved per step vs 126 MB L2); no flush"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": None, "kernel": "ssd_bwd (all launches)",
                     "peak_source": f"{src} hbm_gbs (MEASURED_PEAKS.json)" if src == "measured" else "fallback"},
        "cpu_baseline": cpu, "e2e": None, "gpu_launches": lps * args.steps,
        "gpu_launches_how": lps_how, "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# Forward pass with the complex (rotational) decay.  Not the headline line;
# run with --op rot.
# ---------------------------------------------------------------------------
ROT_METRIC = "SSD fwd with complex (rotational) decay: tokens/s (B·L/s) on 1 B300 & % of HBM roofline"


def run_rot(args, w):
    import torch

    import ssd_scan_fwd_b300 as ssd
    from ssd_scan_fwd_b300.inputs import algorithmic_bytes, generate

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    inp = generate(w)
    d = {k: (None if v is None else v.to(dev)) for k, v in inp.items()}
    B, L, H, P, N, G = w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups
    g = torch.Generator().manual_seed(4343)
    theta = ((torch.rand(B, L, H, generator=g) * 2 - 1) * 0.5).to(dev)
    y = torch.empty_like(d["x"])
    fr = torch.empty(B, H, P, N, device=dev)
    fi = torch.empty(B, H, P, N, device=dev)
    import ctypes

    from ssd_scan_fwd_b300 import _lib
    ra = _lib.SsdFwdRotArgs()
    ra.base = ssd.make_args(d["x"], d["dt"], d["A"], d["Bm"], d["Cm"], d["D"], d["init_state"], y, fr,
                            algo=args.algo)
    ra.theta, ra.init_state_im, ra.final_state_im = theta.data_ptr(), None, fi.data_ptr()
    lib = _lib.lib()
    need = lib.ssd_fwd_rot_workspace_size(ctypes.byref(ra))
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    ra.base.workspace, ra.base.workspace_bytes = ws.data_ptr(), need
    stream = torch.cuda.current_stream(dev)
    sh = ctypes.c_void_p(stream.cuda_stream)
    # the fused kernel takes bf16 io, headdim 64, dstate 128 (one launch a
    # step); otherwise, or with --algo chunked, the chunked path (five launches)
    fused = args.algo != "chunked" and w.io_dtype == "bf16" and P == 64 and N == 128

    def step():
        _lib.check(lib.ssd_fwd_rot(ctypes.byref(ra), sh), "ssd_fwd_rot")

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(_device_uuid(torch, dev)) as clk:
        torch.cuda.synchronize(dev)
        for i in range(args.steps):
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
    ms = statistics.mean(s.elapsed_time(e) for s, e in zip(starts, ends))
    # the forward pass's bytes plus θ in and the imaginary final state out
    nbytes = algorithmic_bytes(w) + B * L * H * 4 + B * H * P * N * 4
    peaks, src = _peaks()
    peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    achieved = nbytes / (ms / 1e3) / 1e9
    cpu = None
    if not args.no_cpu_baseline:
        import oracle
        threads = len(os.sched_getaffinity(0))
        oracle.set_threads(threads)
        hs = max(1, min(H, threads))
        t0 = time.perf_counter()
        oracle.ssd_recurrent_rot(inp["x"][:1, :, :hs], inp["dt"][:1, :, :hs], theta[:1, :, :hs].cpu(), inp["A"][:hs],
                                 inp["Bm"][:1], inp["Cm"][:1], None if inp["D"] is None else inp["D"][:hs])
        secs = time.perf_counter() - t0
        cpu = {"value": L * hs / H / secs, "unit": "tokens/s", "cores": min(threads, hs), "kind": "oracle",
               "sample": f"fp64 complex-decay oracle on 1 of {B} batch rows x {hs} of {H} heads x {L} tokens "
                         f"({secs:.1f} s; tokens/s scaled to all {H} heads)"}
    lps, lps_how = _launches_per_step(torch, step, (1 if fused else 5))
    line = {
        "metric": ROT_METRIC, "value": B * L / (ms / 1e3), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"complex decay, {w.name}: B={B} L={L} H={H} P={P} N={N} G={G} io={w.io_dtype}, "
                               f"θ ~ U(-0.5, 0.5)",
                   "algorithmic_bytes_per_step": nbytes,
                   "l2": f"inputs larger than L2 ({nbytes / 1e6:.0f} MB moved per step vs 126 MB L2); no flush"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": None,
                     "kernel": "ssd_fused_kernel (complex decay)" if fused else "ssd_fwd_rot (all launches)",
                     "peak_source": f"{src} hbm_gbs (MEASURED_PEAKS.json)" if src == "measured" else "fallback"},
        "cpu_baseline": cpu, "e2e": None, "gpu_launches": lps * args.steps,
        "gpu_launches_how": lps_how, "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# Forward pass with the steps around the scan in a Mamba block: Δ =
# softplus(dt + dt_bias) and the output gate y · silu(z).  Not the headline
# line; run with --op ex.
# ---------------------------------------------------------------------------
EX_METRIC = "SSD fwd with softplus(dt + dt_bias) and y·silu(z): tokens/s (B·L/s) on 1 B300 & % of HBM roofline"


def run_ex(args, w):
    import torch

    import ssd_scan_fwd_b300 as ssd
    from ssd_scan_fwd_b300.inputs import algorithmic_bytes, generate, torch_dtype

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    inp = generate(w)
    d = {k: (None if v is None else v.to(dev)) for k, v in inp.items()}
    B, L, H, P, N, G = w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups
    g = torch.Generator().manual_seed(4545)
    dt_raw = (torch.randn(B, L, H, generator=g) - 1.0).to(dev)  # raw dt: Δ = softplus(dt + dt_bias)
    dt_bias = (torch.rand(H, generator=g) * 0.5).to(dev)
    z = torch.randn(B, L, H, P, generator=g).to(torch_dtype(w.io_dtype)).to(dev)
    y = torch.empty_like(d["x"])
    fs = torch.empty(B, H, P, N, device=dev)
    # the workspace once, outside the timed region
    need = ssd.workspace_size(ssd.make_args(d["x"], dt_raw, d["A"], d["Bm"], d["Cm"], d["D"], d["init_state"],
                                            y, fs))
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        ssd.ssd_fwd_ex(d["x"], dt_raw, d["A"], d["Bm"], d["Cm"], d["D"], d["init_state"], dt_bias=dt_bias,
                       dt_softplus=True, z=z, y=y, final_state=fs, workspace=ws)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(_device_uuid(torch, dev)) as clk:
        torch.cuda.synchronize(dev)
        for i in range(args.steps):
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
    ms = statistics.mean(s.elapsed_time(e) for s, e in zip(starts, ends))
    # the forward pass's bytes plus z in (dt_bias is negligible)
    nbytes = algorithmic_bytes(w) + B * L * H * P * (2 if w.io_dtype == "bf16" else 4)
    peaks, src = _peaks()
    peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    achieved = nbytes / (ms / 1e3) / 1e9
    lps, lps_how = _launches_per_step(torch, step, 1)
    line = {
        "metric": EX_METRIC, "value": B * L / (ms / 1e3), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"Δ pre-processing and gate, {w.name}: B={B} L={L} H={H} P={P} N={N} G={G} "
                               f"io={w.io_dtype}, dt ~ N(-1, 1), dt_bias ~ U(0, 0.5), z ~ N(0, 1)",
                   "algorithmic_bytes_per_step": nbytes,
                   "l2": f"inputs larger than L2 ({nbytes / 1e6:.0f} MB moved per step vs 126 MB L2); no flush"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": _recorded_traffic("ex_" + w.name, "fused"),
                     "kernel": "ssd_fused_kernel (Δ pre-processing and gate instantiation)",
                     "peak_source": f"{src} hbm_gbs (MEASURED_PEAKS.json)" if src == "measured" else "fallback"},
        "cpu_baseline": None, "e2e": None, "gpu_launches": lps * args.steps,
        "gpu_launches_how": lps_how, "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# Forward pass with retrieval rank R (MIMO).  Not the headline line; run with
# --op mimo.  The workload keeps its rows: seqlen / R tokens of R ranks each.
# ---------------------------------------------------------------------------
MIMO_METRIC = "SSD fwd with retrieval rank R (MIMO): tokens/s (B·L/s) on 1 B300 & % of HBM roofline"


def run_mimo(args, w):
    import ctypes

    import torch

    import ssd_scan_fwd_b300 as ssd
    from ssd_scan_fwd_b300 import _lib
    from ssd_scan_fwd_b300.inputs import generate_mimo

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    R = args.rank
    w = w.with_(seqlen=w.seqlen // R)
    inp = generate_mimo(w, R)
    d = {k: (None if v is None else v.to(dev)) for k, v in inp.items()}
    B, L, H, P, N, G = w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups
    y = torch.empty_like(d["x"])
    fs = torch.empty(B, H, P, N, device=dev)
    ws = [None]
    stream = torch.cuda.current_stream(dev)

    def step():
        _, _ = ssd.ssd_fwd_mimo(d["x"], d["dt"], d["A"], d["Bm"], d["Cm"], d["D"], d["init_state"], y=y,
                                final_state=fs, workspace=ws[0])

    # the workspace once, outside the timed region
    m = _lib.SsdFwdMimoArgs()
    m.base.batch, m.base.seqlen, m.base.nheads, m.base.headdim, m.base.ngroups, m.base.dstate = B, L, H, P, G, N
    m.base.io_dtype, m.rank = 1, R
    for name in ("x", "dt", "A", "Bm", "Cm", "y"):
        setattr(m.base, name, {"y": y}.get(name, d.get(name)).data_ptr())
    m.base.final_state = fs.data_ptr()
    need = _lib.lib().ssd_fwd_mimo_workspace_size(ctypes.byref(m))
    ws[0] = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(_device_uuid(torch, dev)) as clk:
        torch.cuda.synchronize(dev)
        for i in range(args.steps):
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
    ms = statistics.mean(s.elapsed_time(e) for s, e in zip(starts, ends))
    # x, y: B·L·R·H·P bf16 each; dt: B·L·H fp32; Bm, Cm: B·L·R·G·N bf16 each;
    # final state (and init) B·H·P·N fp32
    nbytes = B * L * R * H * P * 2 * 2 + B * L * H * 4 + B * L * R * G * N * 2 * 2 + B * H * P * N * 4 * (
        2 if w.has_init else 1)
    peaks, src = _peaks()
    peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    achieved = nbytes / (ms / 1e3) / 1e9
    cpu = None
    if not args.no_cpu_baseline:
        import oracle
        threads = len(os.sched_getaffinity(0))
        oracle.set_threads(threads)
        hs = max(1, min(H, threads))
        t0 = time.perf_counter()
        oracle.ssd_recurrent_mimo(inp["x"][:1, :, :, :hs], inp["dt"][:1, :, :hs], inp["A"][:hs], inp["Bm"][:1],
                                  inp["Cm"][:1], inp["D"][:hs])
        secs = time.perf_counter() - t0
        cpu = {"value": L * hs / H / secs, "unit": "tokens/s", "cores": min(threads, hs), "kind": "oracle",
               "sample": f"fp64 retrieval-rank oracle on 1 of {B} batch rows x {hs} of {H} heads x {L} tokens "
                         f"({secs:.1f} s; tokens/s scaled to all {H} heads)"}
    lps, lps_how = _launches_per_step(torch, step, 1)
    line = {
        "metric": MIMO_METRIC, "value": B * L / (ms / 1e3), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"retrieval rank R={R}, {w.name} rows: B={B} L={L} tokens x R={R} H={H} P={P} "
                               f"N={N} G={G} io={w.io_dtype}",
                   "algorithmic_bytes_per_step": nbytes,
                   "l2": f"inputs larger than L2 ({nbytes / 1e6:.0f} MB moved per step vs 126 MB L2); no flush"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": None, "kernel": "ssd_fused_kernel (one launch a step)",
                     "peak_source": f"{src} hbm_gbs (MEASURED_PEAKS.json)" if src == "measured" else "fallback"},
        "cpu_baseline": cpu, "e2e": None, "gpu_launches": lps * args.steps,
        "gpu_launches_how": lps_how, "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--algo", choices=["auto", "fused", "chunked"], default="auto")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--cpu-budget", type=float, default=10.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--ref-tokens", type=int, default=1024, help="tokens per reference-arm step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--op", choices=["fwd", "step", "bwd", "rot", "mimo", "ex"], default="fwd",
                    help="fwd: the forward pass (headline); step: the recurrent decode step; bwd: the backward "
                         "pass; rot: the forward pass with the complex (rotational) decay; mimo: the forward "
                         "pass with retrieval rank --rank; ex: the forward pass with Δ = softplus(dt + dt_bias) "
                         "and the gate y·silu(z)")
    ap.add_argument("--rank", type=int, default=4, help="retrieval rank R (--op mimo)")
    ap.add_argument("--decode-batch", type=int, default=64, help="sequences per decode step (--op step)")
    ap.add_argument("--batch", type=int, default=0,
                    help="override the workload's batch (smaller profiling cases only)")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)  # at least 3 untimed warm-up steps
    from ssd_scan_fwd_b300.inputs import WORKLOADS
    w = WORKLOADS[args.workload]
    if args.batch > 0:
        w = w.with_(batch=args.batch)
    if args.impl == "reference":
        return run_reference(args, w)
    if args.op == "step":
        return run_step(args, w)
    if args.op == "bwd":
        return run_bwd(args, w)
    if args.op == "rot":
        return run_rot(args, w)
    if args.op == "mimo":
        return run_mimo(args, w)
    if args.op == "ex":
        return run_ex(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
