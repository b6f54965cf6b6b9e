"""Benchmark of the GB300 FlashAttention-2 forward (one JSON line on rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one forward pass (one kernel launch of the library) over the whole
workload: by default bf16, causal, GQA, B=2, H_q=32, H_kv=8, qL=kL=4096,
D=128, inputs resident in HBM.  L2 is flushed (a 512 MiB write) before every
timed step, outside the timed kernel.  The device time of each launch is taken
with CUDA events on the stream the kernel runs on; ``value`` is TFLOP/s =
4*B*H_q*qL*kL*D (halved when causal) / mean launch time, summed over ranks
(each rank runs its own copy of the workload: weak scaling, no collective on
the data path).  ``e2e`` repeats the measurement through the C ABI with the
inputs in pinned host memory: host->device copies of Q, K, V, the forward,
and device->host copies of O and L are all inside the timed region.
``cpu_baseline`` times the fp64 oracle (test infrastructure, CPU) on a
bounded sample of query rows of the same workload.
``--impl reference`` times that oracle alone (the CPU reference arm).

``--pass bwd`` measures the backward instead: a step is one ``fa_bwd_full``
call (D pre-pass, dK/dV kernel, dQ kernel, plus the keep-mask and mask
pre-passes where the workload has dropout or a mask, or the tf32 copies and
separate dV, dK, dQ kernels for fp32) on the forward's own O and L, and
``value`` is TFLOP/s = 2.5x the forward's count (the five products of the
FA-2 backward) / mean call time; its ``cpu_baseline`` times the fp64
gradient oracle on whole GQA groups of the same workload.
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
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

L2_FLUSH_BYTES = 512 << 20
CSRC = "attention_forward_08_gb300/csrc/"
KERNEL_SOURCES = [CSRC + f for f in ("fa_kernel.cuh", "fa_ptx.cuh", "fa_launch.cuh", "fa_params.h")]


def kernel_sources(w: workloads.Workload, kind: str = "fwd") -> list:
    """The sources the plan of `w` compiles from (the hash that marks a committed ncu summary as
    taken on the current code covers these, so an edit to another plan leaves it valid)."""
    if kind == "fwd":
        extra = ("fa_tf32_prep.cu", "fa_tf32_ops.cuh") if w.dtype == "f32" else ()
        return KERNEL_SOURCES + [CSRC + f for f in extra]
    common = ("fa_bwd_kernel.cuh", "fa_bwd_impl.cuh", "fa_bwd_launch.h", "fa_bwd.cu")
    if w.dtype == "f32":
        plan = ("fa_bwd_tf32_kernel.cuh", "fa_bwd_tf32.cu", "fa_tf32_ops.cuh")
    elif w.D == 256:
        plan = ("fa_bwd256_kernel.cuh", "fa_bwd256.cu")
    elif w.mask_kind:
        plan = ("fa_bwd_mask.cu",) if w.mask_kind == 1 else ("fa_bwd_mask_add.cu",)
    elif w.dropout_p > 0:
        plan = ("fa_bwd_drop.cu",) + (("fa_bwd_drop_cap.cu",) if w.softcap else ())
    elif w.window or w.softcap or w.q_offset:
        plan = ("fa_bwd_feat.cu",) + (("fa_bwd_feat_cap.cu",) if w.softcap else ())
    else:
        plan = ()
    return KERNEL_SOURCES + [CSRC + f for f in common + plan]


FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ----------------------------------------------------------------------------- helpers

def kernel_source_hash(sources=None) -> str:
    h = hashlib.sha256()
    for rel in sources or KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def peak_for(w: workloads.Workload, peaks: dict) -> float:
    """Dense tensor peak for the workload's MMA kind (TF32 = bf16 x 1/2, the nominal ratio)."""
    bf16 = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    return bf16 if w.dtype in ("bf16", "f16") else bf16 * 0.5


def algorithmic_bytes(w: workloads.Workload) -> int:
    esz = 4 if w.dtype == "f32" else 2
    qo = 2 * w.B * w.H_q * w.qL * w.D * esz
    kv = 2 * w.B * w.H_kv * w.kL * w.D * esz
    lse = 4 * w.B * w.H_q * w.qL
    mask = 0 if w.mask_kind == 0 else w.B * w.H_q * w.qL * w.kL * (1 if w.mask_kind == 1 else esz)
    return qo + kv + lse + mask


EX2_PER_CLK_PER_SM = 32  # special-function-unit exponentials per clock per SM on this GPU generation


def exp_roofline(w: workloads.Workload, mean_ms: float, sms: int, sm_mhz):
    """Secondary roofline of the softmax's exponentials: one ex2 per allowed score (the FLOP
    count's 4 D per score) per call, against SMs x 32 ex2 per clock x the median SM clock sampled
    during the timed region -- a derived peak, not a measured one (None without a clock sample)."""
    achieved = w.flops() / (4.0 * w.D) / (mean_ms * 1e-3) / 1e9
    peak = sms * EX2_PER_CLK_PER_SM * sm_mhz * 1e-3 if sm_mhz else None
    return {"bound": "sfu", "achieved": achieved, "peak": peak, "unit": "Gexp/s",
            "frac": achieved / peak if peak else None,
            "peak_source": f"derived: {sms} SMs x {EX2_PER_CLK_PER_SM} ex2/clk x median sampled SM clock"}


def traffic_from_profiles(w: workloads.Workload, kind: str = "fwd"):
    """DRAM bytes per launch (per call for the backward) from a committed ncu summary, if it was
    taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", f"fa_{kind}_{w.name}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    s = re.search(r"kernel_source_sha:\s*([0-9a-f]+)", text)
    if not m or not s or s.group(1) != kernel_source_hash(kernel_sources(w, kind)):
        return None
    return float(m.group(1))


class CopyPipeline:
    """End-to-end steps: upload the step's inputs from pinned host memory, make the
    call, download its results to pinned host memory, with uploads, calls and
    downloads on three streams and two device buffer sets, so that step s+1's
    upload and step s-1's download overlap step s's call.  (Splitting the copies
    over more streams measured no faster: one upload stream already saturates
    the host link.)  Each set is (device inputs, device outputs, pinned host
    outputs, launch(stream_handle))."""

    def __init__(self, dev, host_in, sets):
        import torch
        self.torch = torch
        self.host_in, self.sets = host_in, sets
        self.up, self.compute, self.down = (torch.cuda.Stream(dev) for _ in range(3))
        self.ev = {k: [torch.cuda.Event() for _ in sets] for k in ("up", "comp", "down")}

    def step(self, s):
        torch = self.torch
        b = s % len(self.sets)
        din, dout, hout, launch = self.sets[b]
        with torch.cuda.stream(self.up):
            self.up.wait_event(self.ev["comp"][b])      # the last call reading this set's inputs is done
            for d_, h_ in zip(din, self.host_in):
                d_.copy_(h_, non_blocking=True)
            self.ev["up"][b].record(self.up)
        self.compute.wait_event(self.ev["up"][b])
        self.compute.wait_event(self.ev["down"][b])     # this set's last outputs have left the device
        launch(self.compute.cuda_stream)
        self.ev["comp"][b].record(self.compute)
        with torch.cuda.stream(self.down):
            self.down.wait_event(self.ev["comp"][b])
            for h_, d_ in zip(hout, dout):
                h_.copy_(d_, non_blocking=True)
            self.ev["down"][b].record(self.down)

    def time_ms(self, steps, warmup, dev, world):
        torch = self.torch
        for s in range(warmup):
            self.step(s)
        torch.cuda.synchronize(dev)
        barrier(world)
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(self.compute)
        for s in range(steps):
            self.step(s)
        self.compute.wait_stream(self.up)
        self.compute.wait_stream(self.down)
        e1.record(self.compute)
        torch.cuda.synchronize(dev)
        barrier(world)
        return e0.elapsed_time(e1) / steps


class ClockSampler:
    """Samples the SM clock, power and clock-event (throttle) reasons of one GPU while running:
    read-only NVML queries (libnvidia-ml through ctypes) every ``period`` seconds, or nvidia-smi
    every 100 ms where NVML cannot be loaded.  Samples are tagged with the phase they fall in
    (``mark(phase)``): the summary of a phase uses that phase's samples only."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    # clock-event reason bits of nvmlDeviceGetCurrentClocksEventReasons
    REASON_BITS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
                   "hw_thermal_slowdown": 0x40, "hw_power_brake_slowdown": 0x80}

    def __init__(self, gpu_index: int, uuid: str | None = None, period: float = 0.001):
        self.gpu = gpu_index
        self.period = period
        self.samples = []   # (phase, sm_mhz, max_mhz, power_w, [reasons])
        self.phase = None
        self._stop = threading.Event()
        self._thread = None
        self.source = "nvidia-smi"
        self._nvml = self._open_nvml(gpu_index, uuid)

    def _open_nvml(self, index, uuid):
        import ctypes
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return None
            h = ctypes.c_void_p()
            ok = False
            if uuid:
                for u in (uuid, "GPU-" + uuid):
                    if lib.nvmlDeviceGetHandleByUUID(u.encode(), ctypes.byref(h)) == 0:
                        ok = True
                        break
            if not ok and lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(h)) != 0:
                return None
            reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                lib.nvmlDeviceGetCurrentClocksThrottleReasons
            self.source = "nvml"
            return lib, h, reasons
        except (OSError, AttributeError):
            return None

    def _sample_nvml(self):
        import ctypes
        lib, h, reasons_fn = self._nvml
        sm, mx, mw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        if lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(sm)) != 0:  # NVML_CLOCK_SM
            return None
        lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))
        lib.nvmlDeviceGetPowerUsage(h, ctypes.byref(mw))
        reasons_fn(h, ctypes.byref(rs))
        names = [n for n, bit in self.REASON_BITS.items() if rs.value & bit]
        return float(sm.value), float(mx.value), mw.value / 1000.0, names

    def _sample_smi(self):
        out = subprocess.run(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                              "--format=csv,noheader,nounits"], capture_output=True, text=True,
                             timeout=5).stdout.strip()
        parts = [p.strip() for p in out.split(",")]
        if len(parts) < 8:
            return None
        num = lambda x: float(x) if x.replace(".", "", 1).isdigit() else None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        return (num(parts[0]), num(parts[1]), num(parts[2]),
                [names[i] for i in range(4) if parts[4 + i].lower() == "active"])

    def _run(self):
        while not self._stop.is_set():
            try:
                smp = self._sample_nvml() if self._nvml else self._sample_smi()
                if smp is not None and smp[0] is not None:
                    self.samples.append((self.phase, *smp))
            except Exception:
                pass
            self._stop.wait(self.period if self._nvml else 0.1)

    def mark(self, phase):
        self.phase = phase

    def sample_now(self):
        """One sample from the calling thread (NVML only), tagged with the current phase."""
        if not self._nvml:
            return
        try:
            smp = self._sample_nvml()
            if smp is not None:
                self.samples.append((self.phase, *smp))
        except Exception:
            pass

    def sample_until(self, event, period=0.0002, limit=30.0):
        """Sample every `period` seconds until the CUDA event has completed (the timed steps have run)."""
        t0 = time.perf_counter()
        while not event.query() and time.perf_counter() - t0 < limit:
            self.sample_now()
            time.sleep(period)

    def start(self):
        self._thread = threading.Thread(target=self._run, daemon=True)
        self._thread.start()

    def stop(self):
        self._stop.set()
        if self._thread:
            self._thread.join(timeout=10)
        if self._nvml:
            self._nvml[0].nvmlShutdown()

    def summary(self, phase="timed"):
        """Median SM clock, max clock and active reasons over the samples of ``phase`` only (never
        idle time: a phase without samples reports none)."""
        inside = [smp for smp in self.samples if smp[0] == phase]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "source": self.source}
        sm = [x[1] for x in inside]
        mx = [x[2] for x in inside if x[2]]
        pw = [x[3] for x in inside if x[3] is not None]
        reasons = sorted({r for x in inside for r in x[4]})
        return {"sm_mhz": statistics.median(sm), "sm_min_mhz": min(sm), "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None, "reasons": reasons, "samples": len(inside),
                "source": self.source}


def make_sampler(dev):
    """A ClockSampler for torch device ``dev`` (matched to NVML by UUID where torch reports it)."""
    import torch
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")[0]
    index = int(vis) if vis.isdigit() else dev.index
    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    return ClockSampler(index, uuid)


SOAK_SECONDS = 1.0  # back-to-back steps, sampled, right before the timed steps (--soak-seconds)
SOAK = {"seconds": SOAK_SECONDS}


def soak(step_fn, sampler, dev):
    """Run ``step_fn`` back to back for about SOAK_SECONDS (untimed), so the clock record covers the
    kernel at a sustained load, not only the few milliseconds of the timed steps."""
    import torch
    sampler.mark("soak")
    t0 = time.perf_counter()
    n = 0
    while n == 0 or time.perf_counter() - t0 < SOAK["seconds"]:
        for _ in range(8):
            step_fn()
        n += 8
        torch.cuda.synchronize(dev)
    sampler.mark(None)
    return n


def clocks_record(sampler):
    """The line's ``clocks``: the timed steps' own samples, plus the soak's beside them."""
    timed, soaked = sampler.summary("timed"), sampler.summary("soak")
    rec = {k: timed[k] for k in ("sm_mhz", "sm_max_mhz", "reasons", "samples")}
    rec.update({"sm_min_mhz": timed.get("sm_min_mhz"), "power_w_max": timed.get("power_w_max"),
                "source": timed["source"], "window": "timed steps only",
                "soak": {k: soaked.get(k) for k in ("sm_mhz", "sm_min_mhz", "sm_max_mhz", "power_w_max", "reasons",
                                                    "samples")}})
    rec["soak"]["seconds"] = SOAK["seconds"]
    return rec


# ----------------------------------------------------------------------------- CPU oracle timing

def oracle_sample(w: workloads.Workload, q, k, v, m, seconds: float):
    """Time the fp64 oracle on evenly spaced query rows (~`seconds` of CPU work).

    Returns (algorithmic FLOP of the sampled rows, wall seconds, rows, threads)."""
    import numpy as np
    import oracle
    qo, ko, vo = q.double().numpy(), k.double().numpy(), v.double().numpy()
    mo = None if m is None else m.double().numpy()
    total_rows = w.B * w.H_q * w.qL
    threads = os.cpu_count() or 1
    scale = float(np.float32(w.sm_scale))

    def rows_flops(rows):
        i = np.asarray(rows) % w.qL
        hi = np.minimum(i + w.q_offset, w.kL - 1) if w.causal else np.full(len(rows), w.kL - 1)
        lo = np.maximum(0, i + w.q_offset - w.window + 1) if w.window > 0 else np.zeros(len(rows), dtype=np.int64)
        return float(np.sum(4.0 * w.D * np.maximum(0, hi - lo + 1)))

    def run(n):
        rows = np.linspace(0, total_rows - 1, n).astype(np.int64).tolist()
        t0 = time.perf_counter()
        oracle.attention(qo, ko, vo, scale, causal=w.causal, mask=mo, mask_kind=w.mask_kind, rows=rows,
                         n_threads=threads, window=w.window, softcap=float(np.float32(w.softcap)),
                         q_offset=w.q_offset, dropout_p=float(np.float32(w.dropout_p)), seed=w.dropout_seed,
                         offset=w.dropout_offset)
        return rows, time.perf_counter() - t0

    n = max(threads, 16)
    rows, dt = run(n)
    while dt < 0.5 and n < total_rows:
        n = min(total_rows, n * 4)
        rows, dt = run(n)
    if dt < seconds and n < total_rows:
        n = min(total_rows, max(n, int(n * seconds / max(dt, 1e-6))))
        rows, dt = run(n)
    return rows_flops(rows), dt, len(rows), threads


# ----------------------------------------------------------------------------- distributed plumbing

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x: float, world: int, device=None) -> float:
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ----------------------------------------------------------------------------- arms

def run_reference_bwd(args, w):
    """The reference arm of ``--pass bwd``: the fp64 gradient oracle, timed on a bounded sample of
    the workload each step (``oracle_bwd_sample``), on the backward's metric."""
    check_bwd_workload(w)
    q, k, v, m = workloads.make_inputs(w)
    do = workloads.make_dout(w)
    per_step = max(2.0, min(15.0, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_bwd_sample(w, q, k, v, do, per_step / 4, m)
    flops = secs = 0.0
    threads, sample = 1, ""
    for _ in range(args.steps):
        f, dt, sample, threads = oracle_bwd_sample(w, q, k, v, do, per_step, m)
        flops += f
        secs += dt
    value = flops / secs / 1e12
    line = {
        "impl": "reference", "metric": "attention bwd TFLOP/s", "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": secs / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": dict(config_of(w, args), **{"pass": "bwd", "layout": "BHSD"}),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": f"per step: {sample}, fp64 C gradient oracle"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_reference(args, w):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    if args.pass_ == "bwd":
        return run_reference_bwd(args, w)
    q, k, v, m = workloads.make_inputs(w)
    per_step = max(2.0, min(15.0, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_sample(w, q, k, v, m, seconds=per_step / 4)
    flops = secs = 0.0
    rows_total = 0
    threads = 1
    for _ in range(args.steps):
        f, dt, nrows, threads = oracle_sample(w, q, k, v, m, seconds=per_step)
        flops += f
        secs += dt
        rows_total += nrows
    value = flops / secs / 1e12
    sample = (f"{rows_total} evenly spaced query rows over {args.steps} steps "
              f"({rows_total / args.steps:.0f} of {w.B * w.H_q * w.qL} per step), fp64 C oracle")
    line = {
        "impl": "reference", "metric": "attention fwd TFLOP/s", "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": secs / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(w, args),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def config_of(w, args):
    extra = {k: getattr(w, k) for k in ("window", "softcap", "q_offset", "dropout_p") if getattr(w, k)}
    return {"workload": w.name, "B": w.B, "H_q": w.H_q, "H_kv": w.H_kv, "seq_len": w.qL, "kL": w.kL, "D": w.D,
            **extra,
            "causal": w.causal, "mask": ["none", "bool", "additive"][w.mask_kind],
            "layout": "token-major O" if w.layout == "dit" else "BHSD",
            "global_batch": w.B * max(1, args.gpus), "parallelism": f"replicas x{max(1, args.gpus)}",
            "l2": "flushed (512 MiB write) before every timed step"}


def run_ours(args, w):
    import torch
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    import attention_forward_08_gb300 as fa
    fa.load_library()

    q, k, v, m = workloads.make_inputs(w)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    md = None if m is None else m.to(dev)
    B, H, qL, D = q.shape
    if w.layout == "dit":
        o_tok = torch.empty((qL, H * D), dtype=q.dtype, device=dev)
        od = o_tok.view(qL, H, D).permute(1, 0, 2).unsqueeze(0)
    else:
        od = torch.empty((B, H, qL, D), dtype=q.dtype, device=dev)
    lsed = torch.empty((B, H, qL), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    fargs = fa.make_args(qd, kd, vd, od, lsed, scale=w.sm_scale, causal=w.causal, mask=md,
                         mask_kind=None if md is None else w.mask_kind, stream=stream.cuda_stream,
                         window=w.window, q_offset=w.q_offset, softcap=w.softcap, dropout_p=w.dropout_p,
                         dropout_seed=w.dropout_seed, dropout_offset=w.dropout_offset)
    # the library's scratch for plans that want one (fp32: the tf32 pre-pass), allocated once
    workspace = fa.attach_workspace(fargs, dev)  # noqa: F841 (kept alive for every launch)
    launches_per_call = 4 if fargs.workspace else 1
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def launch():
        rc = fa.fa_fwd_ex(fargs)
        if rc != 0:
            raise fa.FaError(rc, fa.fa_last_error())

    for _ in range(args.warmup):
        flush.fill_(1)
        launch()
    torch.cuda.synchronize(dev)
    assert fa.fa_sync_status(None) == 0, fa.fa_last_error()

    sampler = make_sampler(dev)
    sampler.start()

    def soak_step():
        flush.fill_(1)
        launch()
    soak(soak_step, sampler, dev)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize(dev)
    sampler.mark("timed")
    t_wall = time.perf_counter()
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        starts[i].record(stream)
        launch()
        ends[i].record(stream)
    sampler.sample_until(ends[-1])  # clock samples while the timed steps run, however short they are
    torch.cuda.synchronize(dev)
    barrier(world)
    wall = time.perf_counter() - t_wall
    sampler.mark(None)
    sampler.stop()
    rc = fa.fa_sync_status(None)
    assert rc == 0, fa.fa_last_error()
    kernel_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    mean_ms = sum(kernel_ms) / len(kernel_ms)
    mean_ms = max_over_ranks(mean_ms, world, dev)
    flops = w.flops()
    value = flops * world / (mean_ms * 1e-3) / 1e12

    # ---- end to end through the C ABI: pinned host inputs -> device -> forward -> host outputs,
    # uploads / calls / downloads pipelined over three streams (CopyPipeline)
    host_in = [t.pin_memory() for t in ((q, k, v) if m is None else (q, k, v, m))]
    h2d = sum(t.numel() * t.element_size() for t in host_in)

    def make_set():
        din = [t.to(dev) for t in host_in]
        if w.layout == "dit":
            o_t = torch.empty((qL, H * D), dtype=q.dtype, device=dev)
            o_v = o_t.view(qL, H, D).permute(1, 0, 2).unsqueeze(0)
        else:
            o_t = o_v = torch.empty((B, H, qL, D), dtype=q.dtype, device=dev)
        l_t = torch.empty((B, H, qL), dtype=torch.float32, device=dev)
        sargs = fa.make_args(din[0], din[1], din[2], o_v, l_t, scale=w.sm_scale, causal=w.causal,
                             mask=None if m is None else din[3], mask_kind=None if m is None else w.mask_kind,
                             window=w.window, q_offset=w.q_offset, softcap=w.softcap, dropout_p=w.dropout_p,
                             dropout_seed=w.dropout_seed, dropout_offset=w.dropout_offset)
        sws = fa.attach_workspace(sargs, dev)

        def launch_on(stream_handle, sargs=sargs, sws=sws):
            sargs.stream = stream_handle
            rc = fa.fa_fwd_ex(sargs)
            if rc != 0:
                raise fa.FaError(rc, fa.fa_last_error())
        hout = [torch.empty(o_t.shape, dtype=o_t.dtype).pin_memory(), torch.empty(l_t.shape).pin_memory()]
        return din, [o_t, l_t], hout, launch_on

    pipe = CopyPipeline(dev, host_in, [make_set(), make_set()])
    d2h = sum(t.numel() * t.element_size() for t in pipe.sets[0][2])
    e_steps = max(3, min(args.steps, 50))
    e2e_ms = max_over_ranks(pipe.time_ms(e_steps, max(2, min(args.warmup, 4)), dev, world), world, dev)
    e2e_value = flops * world / (e2e_ms * 1e-3) / 1e12

    peaks, peak_src = load_peaks()
    peak = peak_for(w, peaks)
    achieved = flops / (mean_ms * 1e-3) / 1e12
    traffic = traffic_from_profiles(w)
    clocks = clocks_record(sampler)

    line = {
        "metric": "attention fwd TFLOP/s", "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": mean_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": config_of(w, argparse.Namespace(gpus=world)),
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "peak_source": (f"{peak_src} bf16 dense (burst; f16 runs at the same rate)"
                                     if w.dtype in ("bf16", "f16")
                                     else f"{peak_src} bf16 dense (burst) x 0.5 nominal tf32 ratio"),
                     "kernels": ("tf32 pre-pass (Q, K rounded; V rounded and transposed) + forward"
                                 if fargs.workspace else "forward"),
                     "algorithmic_bytes": algorithmic_bytes(w),
                     "hbm_gbs": algorithmic_bytes(w) / (mean_ms * 1e-3) / 1e9},
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms},
        "clocks": clocks,
        "gpu_launches": launches_per_call * args.steps,
        "timed_region_s": wall,
        "kernel_ms": {"min": min(kernel_ms), "median": statistics.median(kernel_ms), "max": max(kernel_ms)},
        "exp_roofline": exp_roofline(w, mean_ms, torch.cuda.get_device_properties(dev).multi_processor_count,
                                     clocks["sm_mhz"]),
    }
    if rank == 0 and not args.no_cpu_baseline:
        f, dt, nrows, threads = oracle_sample(w, q, k, v, m, seconds=args.cpu_seconds)
        line["cpu_baseline"] = {"value": f / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                                "sample": f"{nrows} evenly spaced query rows of {w.B * w.H_q * w.qL} "
                                          f"({dt:.1f} s, fp64 C oracle, {threads} threads)"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def oracle_bwd_sample(w, q, k, v, do, seconds, m=None):
    """Time the fp64 gradient oracle on a bounded sample of the workload: whole GQA groups of batch
    0 (as many kv heads as host threads), on the leading Ls positions of the sequence, Ls grown from
    256 until one run takes about `seconds`."""
    import numpy as np

    import oracle
    threads = os.cpu_count() or 1
    group = w.H_q // w.H_kv
    n_kv = max(1, min(w.H_kv, threads))

    def run(Ls):
        qs = q[:1, :n_kv * group, :Ls].double().numpy()
        ks, vs = k[:1, :n_kv, :Ls].double().numpy(), v[:1, :n_kv, :Ls].double().numpy()
        dos = do[:1, :n_kv * group, :Ls].double().numpy()
        mk = {}
        if m is not None:
            ms = m.expand(w.B, w.H_q, w.qL, w.kL)[:1, :n_kv * group, :Ls, :Ls]
            mk = dict(mask=(ms.numpy().astype(np.uint8) if w.mask_kind == 1 else ms.double().numpy()),
                      mask_kind=w.mask_kind)
        t0 = time.perf_counter()
        oracle.attention_bwd(qs, ks, vs, dos, float(np.float32(w.sm_scale)), causal=w.causal, n_threads=threads, **mk,
                             window=w.window, q_offset=w.q_offset, softcap=float(np.float32(w.softcap)),
                             dropout_p=float(np.float32(w.dropout_p)), seed=w.dropout_seed, offset=w.dropout_offset)
        return time.perf_counter() - t0

    Ls = min(256, w.qL, w.kL)
    dt = run(Ls)
    if dt < seconds / 4 and Ls < min(w.qL, w.kL):
        Ls = min(w.qL, w.kL, max(Ls, int(Ls * (seconds / max(dt, 1e-6)) ** 0.5) // 128 * 128))
        dt = run(Ls)
    sub = w.with_(B=1, H_q=n_kv * group, H_kv=n_kv, qL=Ls, kL=Ls)
    return 2.5 * sub.flops(), dt, f"{n_kv} whole GQA groups of batch 0 on the first {Ls} positions", min(threads, n_kv)


def check_bwd_workload(w):
    """The backward's scope: bf16 / fp16 at D 64 and 128 with every forward option (a mask not with a
    softcap); D 256 and fp32 (D 64, 128) with causal or full attention only."""
    feats = w.window or w.q_offset or w.softcap or w.dropout_p
    if w.dtype == "f32":
        ok = w.D in (64, 128) and not feats and w.mask_kind == 0
    elif w.D == 256:
        ok = not feats and w.mask_kind == 0
    else:
        ok = w.D in (64, 128) and not (w.mask_kind and w.softcap)
    if not ok:
        raise SystemExit(f"--pass bwd does not cover this workload ({w.name}): bf16/fp16 D 64 or 128 with any "
                         "forward option, D 256 and fp32 D 64 or 128 without a mask, window, offset, softcap or "
                         "dropout")


def bwd_args(fa, w, ptrs, mask, stream_handle):
    """fa_bwd_args for one call: ptrs = q, k, v, o, dout, lse, dq, dk, dv (device addresses)."""
    a = fa.FaBwdArgs()
    a.q, a.k, a.v, a.o, a.dout, a.lse, a.dq, a.dk, a.dv = ptrs
    a.B, a.H_q, a.H_kv, a.qL, a.kL, a.D = w.B, w.H_q, w.H_kv, w.qL, w.kL, w.D
    a.scale, a.causal = w.sm_scale, int(w.causal)
    a.window, a.q_offset, a.softcap = w.window, w.q_offset, w.softcap
    a.dropout_p, a.dropout_seed, a.dropout_offset = w.dropout_p, w.dropout_seed, w.dropout_offset
    a.dtype = {"f16": fa.FA_DTYPE_F16, "f32": fa.FA_DTYPE_F32}.get(w.dtype, fa.FA_DTYPE_BF16)
    if mask is not None:
        a.mask, a.mask_kind = mask.data_ptr(), w.mask_kind
        a.mask_strides[:] = (mask.stride(0), mask.stride(1), mask.stride(2))
    a.stream = stream_handle
    return a


def bwd_launches(w) -> int:
    """Kernel launches of one backward call."""
    if w.dtype == "f32":
        return 11  # row-dot, four tf32 copies, three transposes, dV, dK, dQ
    return 3 + (1 if w.dropout_p else 0) + (1 if w.mask_kind else 0)


def run_ours_bwd(args, w):
    import torch
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    import attention_forward_08_gb300 as fa
    fa.load_library()
    check_bwd_workload(w)
    q, k, v, m = workloads.make_inputs(w)
    do = workloads.make_dout(w)
    qd, kd, vd, dod = q.to(dev), k.to(dev), v.to(dev), do.to(dev)
    md = None if m is None else m.to(dev)
    # the forward's O in BHSD (the DiT workload's token-major O is a forward output layout)
    od, lsed = fa.attention(qd, kd, vd, scale=w.sm_scale, causal=w.causal, window=w.window, q_offset=w.q_offset,
                            softcap=w.softcap, dropout_p=w.dropout_p, dropout_seed=w.dropout_seed,
                            dropout_offset=w.dropout_offset, mask=md, mask_kind=w.mask_kind or None)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    stream = torch.cuda.current_stream(dev)
    args_c = bwd_args(fa, w, [t.data_ptr() for t in (qd, kd, vd, od, dod, lsed, dq, dk, dv)], md, stream.cuda_stream)
    ws_bytes = fa.fa_bwd_full_workspace_bytes(args_c)
    if ws_bytes < 0:
        raise fa.FaError(fa.FA_ERR_INVALID_ARGUMENT, fa.fa_last_error())
    ws = torch.empty(ws_bytes + 256, dtype=torch.uint8, device=dev)
    args_c.workspace, args_c.workspace_bytes = (ws.data_ptr() + 255) // 256 * 256, ws_bytes
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def launch():
        rc = fa.fa_bwd_full(args_c)
        if rc != 0:
            raise fa.FaError(rc, fa.fa_last_error())

    for _ in range(args.warmup):
        flush.fill_(1)
        launch()
    torch.cuda.synchronize(dev)
    assert fa.fa_sync_status(None) == 0, fa.fa_last_error()
    sampler = make_sampler(dev)
    sampler.start()

    def soak_step():
        flush.fill_(1)
        launch()
    soak(soak_step, sampler, dev)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize(dev)
    sampler.mark("timed")
    t_wall = time.perf_counter()
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        starts[i].record(stream)
        launch()
        ends[i].record(stream)
    sampler.sample_until(ends[-1])  # clock samples while the timed steps run, however short they are
    torch.cuda.synchronize(dev)
    barrier(world)
    wall = time.perf_counter() - t_wall
    sampler.mark(None)
    sampler.stop()
    assert fa.fa_sync_status(None) == 0, fa.fa_last_error()
    call_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    mean_ms = max_over_ranks(sum(call_ms) / len(call_ms), world, dev)
    flops = 2.5 * w.flops()
    value = flops * world / (mean_ms * 1e-3) / 1e12

    # end to end: pinned host inputs (q, k, v, o, dO, L) -> device -> fa_bwd -> host dq, dk, dv,
    # uploads / calls / downloads pipelined over three streams (CopyPipeline)
    host_in = [t.cpu().pin_memory() for t in (qd, kd, vd, od, dod, lsed)]
    h2d = sum(t.numel() * t.element_size() for t in host_in)

    def make_set():
        din = [torch.empty_like(t) for t in (qd, kd, vd, od, dod, lsed)]
        dout = [torch.empty_like(t) for t in (qd, kd, vd)]
        sws = torch.empty(ws_bytes + 256, dtype=torch.uint8, device=dev)
        sptrs = [t.data_ptr() for t in din] + [t.data_ptr() for t in dout]

        def launch_on(stream_handle, sptrs=sptrs, sws=sws):
            a = bwd_args(fa, w, sptrs, md, stream_handle)  # the mask stays resident, as the bench's K/V would not
            a.workspace, a.workspace_bytes = (sws.data_ptr() + 255) // 256 * 256, ws_bytes
            rc = fa.fa_bwd_full(a)
            if rc != 0:
                raise fa.FaError(rc, fa.fa_last_error())
        return din, dout, [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in dout], launch_on

    pipe = CopyPipeline(dev, host_in, [make_set(), make_set()])
    d2h = sum(t.numel() * t.element_size() for t in pipe.sets[0][2])
    e_steps = max(3, min(args.steps, 20))
    e2e_ms = max_over_ranks(pipe.time_ms(e_steps, 3, dev, world), world, dev)

    peaks, peak_src = load_peaks()
    peak = peak_for(w, peaks)
    clocks = clocks_record(sampler)
    line = {
        "metric": "attention bwd TFLOP/s", "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": mean_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": dict(config_of(w, argparse.Namespace(gpus=world)), **{"pass": "bwd", "layout": "BHSD"}),
        "roofline": {"bound": "tensor", "achieved": flops / (mean_ms * 1e-3) / 1e12, "peak": peak,
                     "unit": "TFLOP/s", "frac": flops / (mean_ms * 1e-3) / 1e12 / peak,
                     "traffic": traffic_from_profiles(w, "bwd"),
                     "peak_source": f"{peak_src} bf16 dense (burst)" + (", x0.5 for TF32" if w.dtype == "f32" else ""),
                     "kernels": "one fa_bwd_full call: D pre-pass + "
                                + ("tf32 copies and transposes + dV + dK + dQ" if w.dtype == "f32" else
                                   ("keep-mask pre-pass + " if w.dropout_p else "")
                                   + ("mask transpose + " if w.mask_kind else "") + "dK/dV + dQ")},
        "e2e": {"value": flops * world / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "clocks": clocks,
        "gpu_launches": bwd_launches(w) * args.steps,
        "timed_region_s": wall,
        "call_ms": {"min": min(call_ms), "median": statistics.median(call_ms), "max": max(call_ms)},
    }
    if rank == 0 and not args.no_cpu_baseline:
        f, dt, what, threads = oracle_bwd_sample(w, q, k, v, do, args.cpu_seconds, m)
        line["cpu_baseline"] = {"value": f / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                                "sample": f"{what} ({dt:.1f} s, fp64 C gradient oracle, {threads} threads)"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=workloads.BENCH_WORKLOAD, choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--pass", dest="pass_", default="fwd", choices=["fwd", "bwd"])
    ap.add_argument("--soak-seconds", type=float, default=SOAK_SECONDS,
                    help="sampled back-to-back steps before the timed ones (0: one batch of 8, e.g. under ncu)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    w = workloads.WORKLOADS[args.workload]
    SOAK.update(seconds=max(0.0, args.soak_seconds))
    if args.impl == "reference":
        return run_reference(args, w)
    if args.pass_ == "bwd":
        return run_ours_bwd(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
