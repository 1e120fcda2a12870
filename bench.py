"""Benchmark of the KDA core on one GB300 (or N replicas under torchrun).

One step = one ``kda_chunk_fwd`` prefill of the largest workload that fits one
GPU: 1,048,576 tokens packed as 16 sequences (lengths log-uniform in [1024,
262144]), H=8, d_k=d_v=128, bf16 q/k/v, fp32 g/beta, a random fp32 initial
state per sequence and the final states returned: the headline prefill
tokens/s.  The same JSON line also carries the B=2, H=16, T=4096 prefill, the
96-head 32768-token prefill, the decode half of the metric (256 requests x 96
heads x 128 x 128, fp32 state in place, 64 consecutive ``kda_recurrent_step``
calls) and the other entry points.

Timing: inputs are resident in HBM; every timed step is bracketed by CUDA
events on the launching stream, and L2 is flushed (a 256 MiB write, outside
the events) between prefill steps (the headline's inputs, 12.9 GB, are larger
than L2 anyway).  ``e2e`` repeats the headline prefill through the C ABI with
the inputs in pinned host memory: host->device copies, the call and the
device->host copy of out and the final states are inside the timed region.
``--impl reference`` times the CPU oracle instead.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
"""
from __future__ import annotations

import argparse
import contextlib
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import kda_inputs as ki  # noqa: E402

METRIC = "KDA prefill tokens/s & % bf16 TC roofline; decode steps/s & % HBM BW (1×GB300)"
HEADLINE_W = 4         # 1M-token varlen prefill (16 sequences): the headline
PREFILL_W = 1          # B=2 H16 T4096 prefill, reported alongside (and the backward's workload)
K3_W = 2               # 96-head prefill, reported alongside
DECODE_W = 3
L2_FLUSH_BYTES = 256 << 20
SLEEP_CYCLES = 200_000  # about 0.1 ms at 2 GHz, spent before each timed step


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sus=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


# ---------------------------------------------------------------------------
# algorithmic work per token-head (d = head dim): FLOPs 6 d_k d_v + 2 C (d_k + d_v);
# bytes of q, k, v, out (input dtype), g and beta (fp32), plus each state read or
# written

def prefill_flops(token_heads, dk, dv, C=64):
    return token_heads * (6 * dk * dv + 2 * C * (dk + dv))


def prefill_bytes(token_heads, dk, dv, n_states_read, n_states_written, in_bytes=2):
    per = in_bytes * (2 * dk + dv) + 4 * dk + 4 + in_bytes * dv
    return token_heads * per + 4 * dk * dv * (n_states_read + n_states_written)


def prefill_kernel_bytes(token_heads, dk, dv, n_states_read, n_states_written, in_bytes=2):
    """The same algorithmic bytes split by the kernel that moves them: the chunk
    prep kernel reads q, k, g, beta; the serial kernel reads v and the initial
    states and writes out and the final states."""
    return {"kda_chunk_prep_kernel": token_heads * (in_bytes * 2 * dk + 4 * dk + 4),
            "kda_chunk_serial_kernel": token_heads * 2 * in_bytes * dv
            + 4 * dk * dv * (n_states_read + n_states_written)}


def chunk_kernels(varlen, count):
    """Kernels of one bf16 kda_chunk_fwd call, in launch order, from how many it
    launched: [cu_seqlens check, chunk offsets,] prep, serial pass 0[, segment
    combine][, serial pass 1] (the last two only when some sequence is longer
    than one 512-chunk segment)."""
    head = ["kda_seqlens_kernel", "kda_chunk_offsets_kernel"] if varlen else []
    rest = count - len(head)
    tail = {2: [], 3: ["kda_chunk_serial_kernel_pass1"],
            4: ["kda_segment_combine_kernel", "kda_chunk_serial_kernel_pass1"]}[rest]
    return head + ["kda_chunk_prep_kernel", "kda_chunk_serial_kernel"] + tail


def decode_bytes(NH, dk, dv, in_bytes=2):
    return NH * (2 * 4 * dk * dv + in_bytes * (2 * dk + dv) + 4 * dk + 4 + in_bytes * dv)


# ---------------------------------------------------------------------------

class ClockSampler:
    """SM clock and throttle reasons while the timed loop runs.

    Polls NVML (the counters nvidia-smi reports) from a thread about once per
    millisecond, so that even a timed region of a few milliseconds has samples;
    falls back to ``nvidia-smi -lms 200`` where libnvidia-ml cannot be loaded.
    Reads only; changes no setting."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    # nvmlClocksEventReasons bits (nvml.h)
    BITS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
            0x40: "hw_thermal_slowdown"}

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.nvml = None
        self.lines = []
        self.sm = []
        self.mx = None
        self.reasons = set()
        self.source = None

    def _nvml_open(self):
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            return None
        h = ctypes.c_void_p()
        ok = False
        try:
            uuid = "GPU-" + str(torch.cuda.get_device_properties(self.index).uuid)
            ok = lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(h)) == 0
        except (AttributeError, RuntimeError):
            ok = False
        if not ok and lib.nvmlDeviceGetHandleByIndex_v2(self.index, ctypes.byref(h)) != 0:
            lib.nvmlShutdown()
            return None
        v = ctypes.c_uint()
        if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(v)) == 0:  # NVML_CLOCK_SM
            self.mx = float(v.value)
        try:
            reasons = lib.nvmlDeviceGetCurrentClocksEventReasons
        except AttributeError:
            reasons = lib.nvmlDeviceGetCurrentClocksThrottleReasons
        return lib, h, reasons

    def _poll(self):
        import ctypes
        lib, h, get_reasons = self.nvml
        v, r = ctypes.c_uint(), ctypes.c_ulonglong()
        while not self.stop.is_set():
            if lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(v)) == 0:
                self.sm.append(float(v.value))
            if get_reasons(h, ctypes.byref(r)) == 0:
                for bit, name in self.BITS.items():
                    if r.value & bit:
                        self.reasons.add(name)
            self.stop.wait(0.001)

    def __enter__(self):
        self.stop = threading.Event()
        try:
            self.nvml = self._nvml_open()
        except OSError:
            self.nvml = None
        if self.nvml:
            self.source = "nvml, ~1 ms polling"
            self.t = threading.Thread(target=self._poll, daemon=True)
            self.t.start()
            return self
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.source = "nvidia-smi -lms 200"
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        self.stop.set()
        if self.nvml:
            self.t.join(timeout=5)
            self.nvml[0].nvmlShutdown()
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = list(self.sm), self.mx, set(self.reasons)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0,
                    "source": self.source}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm), "source": self.source}


def dist_setup(gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def whole_job_rate(units_per_rank, ms_slowest, world):
    """Units per second of the whole job: every rank processes `units_per_rank`
    (weak scaling, independent replicas) and the job takes as long as the
    slowest rank."""
    return units_per_rank * world / (ms_slowest * 1e-3)


def graph_ms_over_ranks(ms, world):
    """Job-wide CUDA-graph step time from each rank's ``ms`` (-1 where that rank's
    capture or replay failed): (None, True) if any rank failed, else (the slowest
    rank's ms, False)."""
    failed = max_over_ranks(1.0 if ms <= 0 else 0.0, world) > 0
    return (None, True) if failed else (max_over_ranks(ms, world), False)


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# source files each kernel is compiled from (their hash dates a traffic record)
_BWD_TC = ["kda_backward_tc.cu", "kda_backward_chunk.cuh", "kda_sm100.cuh", "kda_internal.h"]
KERNEL_SOURCES = {
    "kda_chunk_prep_kernel": ["kda_prefill_tc.cu", "kda_sm100.cuh", "kda_internal.h"],
    "kda_chunk_serial_kernel": ["kda_prefill_tc.cu", "kda_sm100.cuh", "kda_internal.h"],
    "kda_decode_kernel": ["kda_recurrent.cu", "kda_internal.h"],
    "kda_recurrent_kernel": ["kda_recurrent.cu", "kda_internal.h"],
    "kda_bwd_prep_tc_kernel": _BWD_TC,
    "kda_bwd_pass_tc_kernel<0>": _BWD_TC,
    "kda_bwd_pass_tc_kernel<1>": _BWD_TC,
    "kda_bwd_grad_tc_kernel": _BWD_TC,
}


def source_sha(kernel):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "gated_delta_rule_gb300", "csrc")
    for f in KERNEL_SOURCES[kernel]:
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def committed_traffic(kernel, workload):
    """DRAM bytes (read + write) per launch of `kernel` on `workload` from the
    committed ncu summary (profiles/traffic.json), if it was taken on the kernel's
    current sources; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p) or kernel not in KERNEL_SOURCES:
        return None
    d = json.load(open(p)).get(kernel, {}).get(workload)
    if not d or d.get("source_sha") != source_sha(kernel):
        return None
    return d.get("bytes_per_launch")


# ---------------------------------------------------------------------------

def bench_prefill(kda, idx, steps, warmup, flush, stream, clk=None, world=1, gated=False):
    w = ki.WORKLOADS[idx]
    d = ki.workload_inputs(idx)
    if gated:  # decay logits + per-head scale instead of the fp32 log-decay
        d = ki.gate_logits(d, seed=ki.SEED_BASE + idx)
    dev = torch.device("cuda")
    t = {k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in d.items()}
    B, T, H, dk = t["q"].shape
    dv = t["v"].shape[-1]
    N = B if t["cu_seqlens"] is None else t["cu_seqlens"].shape[0] - 1
    out = torch.empty(B, T, H, dv, dtype=t["q"].dtype, device=dev)
    sT = torch.empty(N, H, dk, dv, dtype=torch.float32, device=dev)

    def step():
        if gated:
            kda.kda_chunk_fwd_gated(t["q"], t["k"], t["v"], t["z"], t["gate_scale"], t["beta"],
                                    t["initial_state"], t["scale"], cu_seqlens=t["cu_seqlens"], out=out,
                                    final_state=sT, stream=stream)
        else:
            kda.kda_chunk_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["initial_state"],
                              t["scale"], cu_seqlens=t["cu_seqlens"], out=out, final_state=sT,
                              stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(warmup):
            step()
            flush.zero_()
    stream.synchronize()
    step()
    stream.synchronize()
    names = chunk_kernels(t["cu_seqlens"] is not None, kda.kda_last_launch_count())
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    kev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)]
           for _ in range(steps)]
    for e in [x for row in kev for x in row]:
        e.record(stream)  # creates the CUDA handles before the timed loop
    stream.synchronize()
    launches = 0
    barrier(world)
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    # timed steps: events only around each whole call, so nothing sits between
    # the library's own launches (its kernels may overlap one another)
    with (clk or contextlib.nullcontext()), torch.cuda.stream(stream):
        for e0, e1 in evs:
            flush.zero_()
            # keep the GPU busy while the host enqueues the step, so no host-side
            # gap falls between the events
            torch.cuda._sleep(SLEEP_CYCLES)
            e0.record(stream)
            step()
            launches += kda.kda_last_launch_count()
            e1.record(stream)
        stream.synchronize()
    torch.cuda.synchronize()
    barrier(world)
    wall = time.perf_counter() - wall0
    kda.kda_get_device_error(stream)
    ms = [e0.elapsed_time(e1) for e0, e1 in evs]
    # the same steps again with the library recording an event between its
    # kernels: the per-kernel split (these events serialise the kernels)
    with torch.cuda.stream(stream):
        for ke in kev:
            flush.zero_()
            torch.cuda._sleep(SLEEP_CYCLES)
            kda.kda_set_launch_events(ke)
            step()
        stream.synchronize()
    if launches != steps * len(names):
        raise RuntimeError(f"expected {len(names)} kernels per step, counted {launches / steps}")
    kernel_ms = {}
    for i, n in enumerate(names):
        kernel_ms[n] = kernel_ms.get(n, 0.0) + statistics.mean(ke[i].elapsed_time(ke[i + 1]) for ke in kev)
    th = B * T * H if t["cu_seqlens"] is None else T * H
    n_read = N if t["initial_state"] is not None else 0
    g_saving = th * 2 * dk if gated else 0  # bf16 logits instead of fp32 log-decay
    return dict(ms=ms, token_heads=th, tokens=B * T, dk=dk, dv=dv, H=H,
                flops=prefill_flops(th, dk, dv),
                bytes=prefill_bytes(th, dk, dv, n_read * H, N * H) - g_saving,
                kernel_bytes=prefill_kernel_bytes(th, dk, dv, n_read * H, N * H),
                kernel_ms=kernel_ms, launches=launches, wall=wall, d=d, t=t, out=out, sT=sT,
                name=w["name"])


def kernel_roofline(r, pk, world):
    """Roofline of the kernel that takes the most device time per step (the serial
    kernel's time counts both of its passes when sequences are segment-split: its
    algorithmic bytes are moved over the two)."""
    timed = {n: ms for n, ms in r["kernel_ms"].items() if n in r["kernel_bytes"]}
    if "kda_chunk_serial_kernel_pass1" in r["kernel_ms"]:
        timed["kda_chunk_serial_kernel"] += r["kernel_ms"]["kda_chunk_serial_kernel_pass1"]
    name = max(timed, key=timed.get)
    ms = max_over_ranks(timed[name], world)
    gbs = r["kernel_bytes"][name] / (ms * 1e-3) / 1e9
    return {"bound": "hbm", "kernel": name, "achieved": gbs, "peak": pk["hbm"], "unit": "GB/s",
            "frac": gbs / pk["hbm"], "traffic": committed_traffic(name, r["name"]),
            "peak_source": pk["src"] + " (burst copy)",
            "algorithmic_bytes_per_launch": r["kernel_bytes"][name],
            "launch_ms": ms,
            "kernel_ms": {n: max_over_ranks(v, world) for n, v in r["kernel_ms"].items()}}


def gpu_local_cpus(index):
    """The CPUs NVML names as closest to GPU ``index`` (nvmlDeviceGetCpuAffinity),
    within this process's allowed set; None when NVML cannot say."""
    try:
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            return None
        try:
            h = ctypes.c_void_p()
            ok = False
            try:
                uuid = "GPU-" + str(torch.cuda.get_device_properties(index).uuid)
                ok = lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(h)) == 0
            except (AttributeError, RuntimeError):
                ok = False
            if not ok and lib.nvmlDeviceGetHandleByIndex_v2(index, ctypes.byref(h)) != 0:
                return None
            words = (max(os.cpu_count() or 1, max(os.sched_getaffinity(0)) + 1) + 63) // 64
            mask = (ctypes.c_ulong * words)()
            if lib.nvmlDeviceGetCpuAffinity(h, words, mask) != 0:
                return None
            cpus = {64 * i + b for i in range(words) for b in range(64) if (mask[i] >> b) & 1}
            cpus &= os.sched_getaffinity(0)
            return cpus or None
        finally:
            lib.nvmlShutdown()
    except (OSError, AttributeError):
        return None


def bench_prefill_e2e(kda, r, steps, warmup, stream):
    """Same prefill through the C ABI from pinned host buffers (H2D + call + D2H timed).
    The pinned buffers are allocated (and first touched) from the CPUs closest to the
    GPU, so that they sit in that CPU's memory; the process's CPU set is restored
    afterwards."""
    d = r["d"]
    prev = os.sched_getaffinity(0)
    local = gpu_local_cpus(torch.cuda.current_device())
    if local:
        os.sched_setaffinity(0, local)
    try:
        host = {k: v.pin_memory() for k, v in d.items() if torch.is_tensor(v)}
        out_h = torch.empty(r["out"].shape, dtype=r["out"].dtype).pin_memory()
        sT_h = torch.empty(r["sT"].shape, dtype=torch.float32).pin_memory()
    finally:
        os.sched_setaffinity(0, prev)
    dev = r["t"]
    names = [k for k in ("q", "k", "v", "g", "beta", "initial_state", "cu_seqlens")
             if host.get(k) is not None]
    h2d = sum(host[k].numel() * host[k].element_size() for k in names)
    d2h = out_h.numel() * out_h.element_size() + sT_h.numel() * 4

    def step():
        for k in names:
            dev[k].copy_(host[k], non_blocking=True)
        kda.kda_chunk_fwd(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"],
                          dev.get("initial_state"), dev["scale"], cu_seqlens=dev.get("cu_seqlens"),
                          out=r["out"], final_state=r["sT"], stream=stream)
        out_h.copy_(r["out"], non_blocking=True)
        sT_h.copy_(r["sT"], non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(warmup):
            step()
        stream.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            step()
        e1.record(stream)
    stream.synchronize()
    ms = e0.elapsed_time(e1) / steps
    return dict(ms=ms, h2d=h2d, d2h=d2h, host_cpus=len(local) if local else None)


def bench_decode(kda, steps_total, warmup, stream, clk=None):
    w = ki.WORKLOADS[DECODE_W]
    N, H, dk, dv = w["N"], w["H"], w["dk"], w["dv"]
    seed = ki.SEED_BASE + DECODE_W
    dev = torch.device("cuda")
    S = ki.decode_state(N, H, dk, dv, seed=seed).to(dev)
    n_in = w["steps"]
    ins = []
    for s in range(n_in):
        x = ki.decode_inputs(N, H, dk, dv, "bf16", seed=seed, step=s)
        ins.append({k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in x.items()})
    out = torch.empty(N, H, dv, dtype=torch.bfloat16, device=dev)

    def step(x):
        kda.kda_recurrent_step(S, x["q"], x["k"], x["v"], x["g"], x["beta"], scale=x["scale"],
                               out=out, stream=stream)

    with torch.cuda.stream(stream):
        for i in range(warmup):
            step(ins[i % n_in])
    stream.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches = 0
    with (clk or contextlib.nullcontext()), torch.cuda.stream(stream):
        torch.cuda._sleep(SLEEP_CYCLES)
        e0.record(stream)
        for i in range(steps_total):
            step(ins[i % n_in])
            launches += kda.kda_last_launch_count()
        e1.record(stream)
        stream.synchronize()
    ms = e0.elapsed_time(e1) / steps_total
    graph = decode_graph_timing(kda, S, ins, out, stream, reps=4)
    return dict(ms=ms, NH=N * H, N=N, H=H, dk=dk, dv=dv, bytes=decode_bytes(N * H, dk, dv),
                name=w["name"], steps=steps_total, launches=launches, graph=graph)


def decode_graph_timing(kda, S, ins, out, stream, reps):
    """The decode steps of ``ins`` captured once in a CUDA graph and replayed ``reps``
    times on ``stream``: ms per step and kernels per replay, or (ms = -1) the error
    that stopped the capture or the replay."""
    try:
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream()
        cap.wait_stream(stream)
        captured = 0
        with torch.cuda.graph(g, stream=cap):
            for x in ins:
                kda.kda_recurrent_step(S, x["q"], x["k"], x["v"], x["g"], x["beta"], scale=x["scale"], out=out,
                                       stream=cap)
                captured += kda.kda_last_launch_count()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            stream.wait_stream(cap)
            g.replay()  # untimed first replay
            stream.synchronize()
            torch.cuda._sleep(SLEEP_CYCLES)
            e0.record(stream)
            for _ in range(reps):
                g.replay()
            e1.record(stream)
            stream.synchronize()
        kda.kda_get_device_error(stream)
        return dict(ms=e0.elapsed_time(e1) / (reps * len(ins)), launches_per_replay=captured, replays=reps,
                    steps_per_replay=len(ins), error=None)
    except Exception as e:  # reported in the JSON line; the eager numbers stand
        return dict(ms=-1.0, launches_per_replay=0, replays=0, steps_per_replay=len(ins),
                    error=f"{type(e).__name__}: {e}"[:300])


def bench_multi_step(kda, n_tok, warmup, stream, clk=None, iters=20):
    """kda_recurrent_multi_step on the decode batch (256 requests x 96 heads), n_tok
    tokens per request, all accepted: the state is read and written once per call."""
    w = ki.WORKLOADS[DECODE_W]
    N, H, dk, dv = w["N"], w["H"], w["dk"], w["dv"]
    seed = ki.SEED_BASE + DECODE_W
    dev = torch.device("cuda")
    S = ki.decode_state(N, H, dk, dv, seed=seed).to(dev)
    d = ki.prefill_inputs(N, n_tok, H, dk, dv, "bf16", seed=seed + 100)
    t = {k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in d.items()}
    out = torch.empty(N, n_tok, H, dv, dtype=torch.bfloat16, device=dev)

    def step():
        kda.kda_recurrent_multi_step(S, t["q"], t["k"], t["v"], t["g"], t["beta"], scale=t["scale"],
                                     out=out, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(warmup):
            step()
    stream.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches = 0
    with (clk or contextlib.nullcontext()), torch.cuda.stream(stream):
        torch.cuda._sleep(SLEEP_CYCLES)
        e0.record(stream)
        for _ in range(iters):
            step()
            launches += kda.kda_last_launch_count()
        e1.record(stream)
        stream.synchronize()
    ms = e0.elapsed_time(e1) / iters
    per_tok = 2 * (2 * dk + dv) + 4 * dk + 4 + 2 * dv
    nbytes = N * H * (8 * dk * dv + n_tok * per_tok)
    return dict(ms=ms, N=N, H=H, n=n_tok, bytes=nbytes, launches=launches, iters=iters)


def bench_decode_fused(kda, steps_total, warmup, stream, clk=None):
    """kda_decode_step_fused on the decode batch: short convolutions, SiLU, L2 norm,
    the step, RMSNorm and the output gate per token."""
    w = ki.WORKLOADS[DECODE_W]
    N, H, dk, dv = w["N"], w["H"], w["dk"], w["dv"]
    seed = ki.SEED_BASE + DECODE_W
    dev = torch.device("cuda")
    S = ki.decode_state(N, H, dk, dv, seed=seed).to(dev)
    x = {k: v.to(dev) for k, v in ki.fused_decode_extras(N, H, dk, dv, "bf16", seed=seed).items()}
    d = {k: (v.to(dev) if torch.is_tensor(v) else v)
         for k, v in ki.decode_inputs(N, H, dk, dv, "bf16", seed=seed, step=0).items()}
    out = torch.empty(N, H, dv, dtype=torch.bfloat16, device=dev)

    def step():
        kda.kda_decode_step_fused(S, x["conv_q"], x["conv_k"], x["conv_v"], d["q"], d["k"], d["v"], x["w_q"],
                                  x["w_k"], x["w_v"], d["g"], d["beta"], x["out_gate"], x["norm_weight"],
                                  scale=d["scale"], eps=1e-6, out=out, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(warmup):
            step()
    stream.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches = 0
    with (clk or contextlib.nullcontext()), torch.cuda.stream(stream):
        torch.cuda._sleep(SLEEP_CYCLES)
        e0.record(stream)
        for _ in range(steps_total):
            step()
            launches += kda.kda_last_launch_count()
        e1.record(stream)
        stream.synchronize()
    ms = e0.elapsed_time(e1) / steps_total
    # state read + write, raw q/k/v, g, beta, gate logits, out, three cache slots read
    # and written per q/k/v channel
    per_head = 8 * dk * dv + 2 * (2 * dk + dv) + 4 * dk + 4 + 2 * dv + 2 * dv + 6 * 2 * (2 * dk + dv)
    return dict(ms=ms, N=N, H=H, bytes=N * H * per_head, launches=launches, steps=steps_total)


CHUNK_BWD_KERNELS = ["kda_bwd_prep_tc_kernel", "kda_bwd_pass_tc_kernel<0>", "kda_bwd_pass_tc_kernel<1>",
                     "kda_bwd_grad_tc_kernel"]
def chunk_bwd_bytes(dk, dv, C=64):
    """Algorithmic bytes per (chunk, head) of the four tensor-core kernels of the
    chunked backward (each tensor counted once per chunk and head).
    Prep: reads the bf16 q, k, v and dO rows, g and beta; writes the record (four
    [C][d_k] and two [C][d_v] matrices, e^{G_C}, the [d_k][d_v] Z_q, the [C][C] A).
    Forward pass (kda_bwd_pass_tc_kernel<0>): reads W, K_end, U_bar, e^{G_C}; writes S and U.
    Reverse pass (<1>): reads W_y, diag(beta) K+, V_y, Z_q, e^{G_C}, beta; writes X, dY, dv.
    Gradient kernel: reads S, X, U, dY, A, the bf16 q, k, v, dO rows, g and beta; writes
    fp32 dq, dk, dg and dbeta."""
    inputs = 2 * C * (2 * dk + 2 * dv) + 4 * C * dk + 4 * C
    rec = 4 * (4 * C * dk + 2 * C * dv + dk + dk * dv + C * C)
    state = 4 * (dk * dv + C * dv)
    fwd = 4 * (2 * C * dk + C * dv + dk) + state
    rev = 4 * (2 * C * dk + C * dv + dk * dv + dk + C) + state + 4 * C * dv
    grad = inputs + 2 * state + 4 * C * C + 4 * (3 * C * dk + C)
    return {"kda_bwd_prep_tc_kernel": inputs + rec, "kda_bwd_pass_tc_kernel<0>": fwd,
            "kda_bwd_pass_tc_kernel<1>": rev, "kda_bwd_grad_tc_kernel": grad}


def chunk_bwd_roofline(bw, ms, kernel_ms, hbm_peak, workload):
    """``roofline`` of the chunked backward for its dominant kernel (bound "hbm",
    algorithmic bytes over the kernel's event time), every kernel's rate beside it."""
    by = {n: b * bw["chunk_heads"] for n, b in chunk_bwd_bytes(bw["dk"], bw["dv"]).items()}
    rates = {}
    for n, t in kernel_ms.items():
        if n in by:
            x = by[n] / (t * 1e-3) / 1e9
            rates[n] = {"achieved": x, "unit": "GB/s", "frac": x / hbm_peak}
    k = max(kernel_ms, key=kernel_ms.get)
    call = sum(by.values()) / (ms * 1e-3) / 1e9
    return {"bound": "hbm", "kernel": k, "achieved": rates[k]["achieved"], "peak": hbm_peak, "unit": "GB/s",
            "frac": rates[k]["frac"], "traffic": committed_traffic(k, workload), "peak_source": "measured (burst copy)",
            "bytes_per_launch": by[k], "call_gbs": call, "call_frac": call / hbm_peak, "kernel_rates": rates}


def bench_backward(kda, steps, warmup, stream, entry="kda_chunk_bwd", names=None):
    """``entry`` (kda_chunk_bwd or kda_backward) on the headline prefill workload (B=2,
    H=16, T=4096): gradients of every input given random output and final-state
    gradients.  With ``names`` (the call's kernels in launch order), a second set of
    calls records an event between the kernels for the per-kernel split."""
    d = ki.workload_inputs(PREFILL_W)
    dev = torch.device("cuda")
    t = {k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in d.items()}
    B, T, H, dk = t["q"].shape
    dv = t["v"].shape[-1]
    gen = torch.Generator().manual_seed(1)
    do = torch.randn(B, T, H, dv, generator=gen).to(torch.bfloat16).to(dev)
    dST = torch.randn(B, H, dk, dv, generator=gen).to(dev)

    fn = getattr(kda, entry)

    def step():
        fn(t["q"], t["k"], t["v"], t["g"], t["beta"], t["initial_state"], t["scale"], do, dST, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(warmup):
            step()
    stream.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches = 0
    with torch.cuda.stream(stream):
        torch.cuda._sleep(SLEEP_CYCLES)
        e0.record(stream)
        for _ in range(steps):
            step()
            launches += kda.kda_last_launch_count()
        e1.record(stream)
        stream.synchronize()
    ms = e0.elapsed_time(e1) / steps
    kernel_ms = {}
    if names:
        kev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)] for _ in range(steps)]
        with torch.cuda.stream(stream):
            for ke in kev:
                for ev in ke:
                    ev.record(stream)
            stream.synchronize()
            for ke in kev:
                torch.cuda._sleep(SLEEP_CYCLES)
                kda.kda_set_launch_events(ke)
                step()
            stream.synchronize()
        if launches != steps * len(names):
            raise RuntimeError(f"expected {len(names)} kernels per call, counted {launches / steps}")
        for i, n in enumerate(names):
            kernel_ms[n] = statistics.mean(ke[i].elapsed_time(ke[i + 1]) for ke in kev)
    th = B * T * H
    # inputs (q, k, v, d_out bf16; g fp32; beta) and fp32 gradients, plus the states
    per = 2 * (2 * dk + 2 * dv) + 4 * dk + 4 + 4 * (3 * dk + dv) + 4
    nbytes = th * per + 4 * dk * dv * B * H * 4
    return dict(ms=ms, tokens=B * T, bytes=nbytes, launches=launches, kernel_ms=kernel_ms, dk=dk, dv=dv,
                chunk_heads=B * H * ((T + 63) // 64), name=ki.WORKLOADS[PREFILL_W]["name"])


ORACLE_MIN_CPU_S = 12.0  # CPU-seconds (wall x threads) of oracle work behind each rate
ORACLE_SEQ_TOKENS = 2048  # varlen sample: this many leading tokens of every sequence


def oracle_sample(idx, d=None, threads=None):
    """A bounded sample of workload ``idx`` for the CPU oracle, with the workload's
    shapes and distributions: fixed-length workloads keep every token of the first
    heads (enough heads to give every oracle thread one (sequence, head) problem);
    the varlen workload keeps the first ORACLE_SEQ_TOKENS tokens of each sequence
    (each from its own initial state) on the first heads.  ``d``: the workload's
    full inputs if already generated (a subset of heads is generated otherwise).
    Returns (inputs, description)."""
    w = ki.WORKLOADS[idx]
    H = w["H"]
    nseq = w.get("nseq", w.get("B", 1))
    nh = max(1, min(H, -(-int(threads or 1) // nseq)))
    heads = list(range(nh))
    if d is None:
        d = ki.workload_inputs(idx, heads=heads)
    sub = {x: (d[x][:, :, heads] if d[x] is not None and d[x].shape[2] != nh else d[x])
           for x in ("q", "k", "v", "g", "beta")}
    s0 = d["initial_state"]
    if s0 is not None and s0.shape[1] != nh:
        s0 = s0[:, heads]
    if d["cu_seqlens"] is None:
        text = f"{w['name']}: all {w.get('B', 1)}x{w['T']} tokens on {nh} of {H} heads"
        return dict(sub, initial_state=s0, scale=d["scale"], cu_seqlens=None), text
    import torch as _t
    cu = d["cu_seqlens"].numpy()
    spans = [(int(cu[n]), min(int(cu[n + 1]), int(cu[n]) + ORACLE_SEQ_TOKENS)) for n in range(len(cu) - 1)]
    cat = {x: _t.cat([sub[x][:, a:b] for a, b in spans], dim=1).contiguous() for x in sub}
    new_cu = _t.from_numpy(ki.cu_seqlens_from_lengths([b - a for a, b in spans]))
    text = (f"{w['name']}: the first {ORACLE_SEQ_TOKENS} tokens of each of its {len(spans)} sequences "
            f"({int(new_cu[-1])} tokens) on {nh} of {H} heads")
    return dict(cat, initial_state=s0, scale=d["scale"], cu_seqlens=new_cu), text


def oracle_prefill_rate(idx, d=None, min_cpu_s=ORACLE_MIN_CPU_S):
    """CPU oracle on a bounded sample of workload ``idx`` (oracle_sample), repeated
    until it has done about ``min_cpu_s`` of CPU work: returns (tokens/s, threads,
    sample text, seconds).  Tokens/s counts whole tokens (every head of a token)."""
    import oracle
    w = ki.WORKLOADS[idx]
    x, text = oracle_sample(idx, d, oracle.threads())
    Hs = x["q"].shape[2]
    nprob = Hs * (x["q"].shape[0] if x["cu_seqlens"] is None else x["cu_seqlens"].shape[0] - 1)
    used = min(oracle.threads(), nprob)
    passes = 0
    t0 = time.perf_counter()
    while True:
        oracle.prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], x["initial_state"], x["scale"],
                       cu_seqlens=x["cu_seqlens"])
        passes += 1
        dt = time.perf_counter() - t0
        if dt * used >= min_cpu_s or passes >= 256:
            break
    token_heads = x["q"].shape[0] * x["q"].shape[1] * Hs
    tokens_per_s = passes * token_heads / dt / w["H"]   # whole-token rate: every token has H heads
    sample = f"{text} ({token_heads} token-heads) x {passes} passes, {dt:.2f} s wall on {used} threads"
    return tokens_per_s, used, sample, dt


# ---------------------------------------------------------------------------

def headline_config(world):
    """``config`` of the JSON line: the headline workload, named by what it is."""
    w = ki.WORKLOADS[HEADLINE_W]
    return {"workload": w["name"], "tokens": w["T"], "sequences": w["nseq"],
            "lengths": f"log-uniform in [{w['lo']}, {w['hi']}], rescaled to the total",
            "H": w["H"], "d_k": w["dk"], "d_v": w["dv"], "chunk": 64,
            "initial_state": "random fp32 per sequence", "final_state": "returned",
            "parallelism": f"replicas x{world}",
            "l2": "inputs (12.9 GB) larger than L2; also flushed (256 MiB write) between timed steps, "
                  "outside the events"}


def run_reference(args, world, rank):
    """The reference arm: the CPU oracle on bounded samples of the headline workload."""
    if rank != 0:
        return
    rates, sample, threads = [], "", 1
    w = ki.WORKLOADS[HEADLINE_W]
    import oracle
    d, _ = oracle_sample(HEADLINE_W, None, oracle.threads())
    for _ in range(min(args.warmup, 1)):
        oracle_prefill_rate(HEADLINE_W, d, min_cpu_s=ORACLE_MIN_CPU_S / 4)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        r, threads, sample, _ = oracle_prefill_rate(HEADLINE_W, d)
        rates.append(r)
    wall = time.perf_counter() - t0
    val = statistics.median(rates)
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * w["T"] / val, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": dict(headline_config(world), parallelism="none (CPU oracle)"),
            "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "wall_s": wall}
    print(json.dumps(line), flush=True)


def ncu_case(which):
    """Two untimed launches of one workload, for profiler captures: ``prefill`` (B2
    H16 T4096), ``prefill96`` (96 heads x 32768), ``varlen`` (the 1M-token headline),
    ``bwd`` (kda_chunk_bwd on B2 H16 T4096), ``decode32`` / ``decode`` (32 or 256
    requests x 96 heads), ``multi32`` / ``multi`` (4-token multi-step decode on 32 or
    256 requests x 96 heads)."""
    import gated_delta_rule_gb300 as kda
    kda.build()
    kda.load_library()
    dev = torch.device("cuda")
    if which.startswith("prefill") or which in ("varlen", "bwd"):
        idx = {"prefill": PREFILL_W, "prefill96": K3_W, "varlen": HEADLINE_W, "bwd": PREFILL_W}[which]
        d = ki.workload_inputs(idx)
        t = {k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in d.items()}
        if which == "bwd":
            B, T, H, dk = t["q"].shape
            gen = torch.Generator().manual_seed(1)
            do = torch.randn(B, T, H, t["v"].shape[-1], generator=gen).to(torch.bfloat16).to(dev)
            dST = torch.randn(B, H, dk, t["v"].shape[-1], generator=gen).to(dev)
        for _ in range(2):
            if which == "bwd":
                kda.kda_chunk_bwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["initial_state"], t["scale"],
                                  do, dST)
            else:
                kda.kda_chunk_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["initial_state"],
                                  t["scale"], cu_seqlens=t["cu_seqlens"])
    else:
        w = ki.WORKLOADS[DECODE_W]
        N = 32 if which in ("decode32", "multi32") else w["N"]
        S = ki.decode_state(N, w["H"], w["dk"], w["dv"], seed=1).to(dev)
        x = ki.decode_inputs(N, w["H"], w["dk"], w["dv"], "bf16", seed=1, step=0)
        x = {k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in x.items()}
        if which.startswith("multi"):
            x = ki.prefill_inputs(N, 4, w["H"], w["dk"], w["dv"], "bf16", seed=2)
            x = {k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in x.items()}
        for _ in range(2):
            if which.startswith("multi"):
                kda.kda_recurrent_multi_step(S, x["q"], x["k"], x["v"], x["g"], x["beta"], scale=x["scale"])
            else:
                kda.kda_recurrent_step(S, x["q"], x["k"], x["v"], x["g"], x["beta"], scale=x["scale"])
    torch.cuda.synchronize()
    kda.kda_get_device_error()
    print(json.dumps({"ncu_case": which, "ok": True}))


def prefill_summary(r, pk, world):
    """A prefill workload's sub-key: step time, rates, per-kernel split and the
    fractions of both peaks."""
    ms = max_over_ranks(statistics.mean(r["ms"]), world)
    return {"workload": r["name"], "ms_per_step": ms,
            "kernel_ms": {n: max_over_ranks(v, world) for n, v in r["kernel_ms"].items()},
            "kernel_hbm_frac": {n: r["kernel_bytes"][n] / (r["kernel_ms"][n] * 1e-3) / 1e9 / pk["hbm"]
                                for n in r["kernel_bytes"] if n in r["kernel_ms"]},
            "tokens_per_s": world * r["tokens"] / (ms * 1e-3),
            "hbm_frac": r["bytes"] / (ms * 1e-3) / 1e9 / pk["hbm"],
            "tc_frac": r["flops"] / (ms * 1e-3) / 1e12 / pk["bf16"],
            "t_roof_over_t": max(r["flops"] / (pk["bf16"] * 1e12), r["bytes"] / (pk["hbm"] * 1e9)) / (ms * 1e-3),
            "gpu_launches": r["launches"]}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-k3", action="store_true")
    ap.add_argument("--ncu-case", choices=["prefill", "prefill96", "varlen", "bwd", "decode32", "decode", "multi32", "multi"],
                    help="run two untimed launches of one workload (for ncu captures) and exit")
    args = ap.parse_args()
    if args.ncu_case:
        ncu_case(args.ncu_case)
        return
    world, rank, local = dist_setup(args.gpus)
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    if args.warmup < 3:
        args.warmup = 3

    import gated_delta_rule_gb300 as kda
    kda.build()
    kda.load_library()
    pk = peaks()
    stream = torch.cuda.Stream()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")

    clk = ClockSampler(local)
    pre = bench_prefill(kda, HEADLINE_W, args.steps, args.warmup, flush, stream, clk, world)
    wall = pre["wall"]

    ms = statistics.mean(pre["ms"])
    ms = max_over_ranks(ms, world)
    tokens_all = pre["tokens"] * world
    value = whole_job_rate(pre["tokens"], ms, world)
    ach_gbs = pre["bytes"] / (ms * 1e-3) / 1e9
    ach_tf = pre["flops"] / (ms * 1e-3) / 1e12
    roof = kernel_roofline(pre, pk, world)
    path_roof = {"bound": "hbm", "achieved": ach_gbs, "peak": pk["hbm"], "unit": "GB/s",
                 "frac": ach_gbs / pk["hbm"], "algorithmic_bytes_per_step": pre["bytes"],
                 "note": "whole step (all kernels of one kda_chunk_fwd call)"}
    tc = {"achieved": ach_tf, "peak": pk["bf16"], "unit": "TFLOP/s", "frac": ach_tf / pk["bf16"],
          "algorithmic_flops_per_launch": pre["flops"]}
    t_roof = max(pre["flops"] / (pk["bf16"] * 1e12), pre["bytes"] / (pk["hbm"] * 1e9))
    head_summary = prefill_summary(pre, pk, world)
    step_ms = {"mean": ms, "median": max_over_ranks(statistics.median(pre["ms"]), world),
               "best": max_over_ranks(min(pre["ms"]), world), "reps": len(pre["ms"])}

    # warm-up: the first device reads of freshly pinned host pages run several
    # times slower (one or two calls), so eight untimed calls precede the timed five
    e2e = bench_prefill_e2e(kda, pre, 5, 8, stream)
    e2e_val = tokens_all / (max_over_ranks(e2e["ms"], world) * 1e-3)
    cpu_d = pre["d"] if rank == 0 and world == 1 and not args.no_cpu_baseline else None
    del pre

    extra = {}
    clk_p1 = ClockSampler(local)
    p1 = bench_prefill(kda, PREFILL_W, args.steps, 3, flush, stream, clk_p1, world)
    extra["prefill_B2_H16_T4096"] = dict(prefill_summary(p1, pk, world), roofline=kernel_roofline(p1, pk, world),
                                         clocks=clk_p1.summary())
    del p1
    clk_dec = ClockSampler(local)
    dec = bench_decode(kda, 64, args.warmup, stream, clk_dec)
    dms = max_over_ranks(dec["ms"], world)
    d_gbs = dec["bytes"] / (dms * 1e-3) / 1e9
    extra["decode"] = {
        "workload": dec["name"], "ms_per_step": dms, "steps_timed": dec["steps"],
        "steps_per_s": world * 1e3 / dms, "tokens_per_s": world * dec["N"] * 1e3 / dms,
        "roofline": {"bound": "hbm", "kernel": "kda_decode_kernel", "achieved": d_gbs,
                     "peak": pk["hbm"], "unit": "GB/s", "frac": d_gbs / pk["hbm"],
                     "traffic": committed_traffic("kda_decode_kernel", dec["name"]),
                     "algorithmic_bytes_per_launch": dec["bytes"]},
        "clocks": clk_dec.summary(), "gpu_launches": dec["launches"]}
    gr = dec["graph"]
    g_ms, g_failed = graph_ms_over_ranks(gr["ms"], world)
    extra["decode"]["cuda_graph"] = {
        "ms_per_step": g_ms, "steps_per_replay": gr["steps_per_replay"],
        "replays_timed": gr["replays"], "launches_per_replay": gr["launches_per_replay"],
        "hbm_frac": dec["bytes"] / (g_ms * 1e-3) / 1e9 / pk["hbm"] if g_ms else None,
        "error": gr["error"] or ("the capture failed on another rank" if g_failed else None)}
    del dec
    fz = bench_decode_fused(kda, 64, args.warmup, stream)
    f_ms = max_over_ranks(fz["ms"], world)
    f_gbs = fz["bytes"] / (f_ms * 1e-3) / 1e9
    extra["decode_fused"] = {
        "workload": f"kda_decode_fused_N{fz['N']}_H{fz['H']}_d128", "ms_per_step": f_ms,
        "steps_per_s": world * 1e3 / f_ms,
        # the whole call (front-end, step and back-end kernels) against its algorithmic bytes
        "roofline": {"bound": "hbm", "kernel": "kda_decode_front_kernel + kda_decode_kernel + kda_decode_back_kernel",
                     "achieved": f_gbs, "peak": pk["hbm"], "unit": "GB/s", "frac": f_gbs / pk["hbm"],
                     "algorithmic_bytes_per_call": fz["bytes"]},
        "gpu_launches": fz["launches"]}
    del fz
    clk_ms = ClockSampler(local)
    ms4 = bench_multi_step(kda, 4, args.warmup, stream, clk_ms)
    m_ms = max_over_ranks(ms4["ms"], world)
    m_gbs = ms4["bytes"] / (m_ms * 1e-3) / 1e9
    m_wl = f"kda_multi_step_N{ms4['N']}_H{ms4['H']}_n{ms4['n']}_d128"
    extra["decode_multi_token"] = {
        "workload": m_wl, "ms_per_call": m_ms,
        "tokens_per_s": world * ms4["N"] * ms4["n"] * 1e3 / m_ms,
        "roofline": {"bound": "hbm", "kernel": "kda_recurrent_kernel", "achieved": m_gbs,
                     "peak": pk["hbm"], "unit": "GB/s", "frac": m_gbs / pk["hbm"],
                     "traffic": committed_traffic("kda_recurrent_kernel", m_wl),
                     "algorithmic_bytes_per_launch": ms4["bytes"]},
        "clocks": clk_ms.summary(), "gpu_launches": ms4["launches"]}
    del ms4
    if not args.no_k3:
        clk_k3 = ClockSampler(local)
        k3 = bench_prefill(kda, K3_W, max(3, args.steps // 4), 3, flush, stream, clk_k3, world)
        extra["prefill_96heads"] = dict(prefill_summary(k3, pk, world), clocks=clk_k3.summary())
        del k3

    gp = bench_prefill(kda, PREFILL_W, args.steps, 3, flush, stream, None, world, gated=True)
    gms = max_over_ranks(statistics.mean(gp["ms"]), world)
    extra["prefill_gated"] = {
        "workload": gp["name"] + "_gate_logits", "ms_per_step": gms,
        "kernel_ms": {n: max_over_ranks(v, world) for n, v in gp["kernel_ms"].items()},
        "tokens_per_s": world * gp["tokens"] / (gms * 1e-3),
        "hbm_frac": gp["bytes"] / (gms * 1e-3) / 1e9 / pk["hbm"], "gpu_launches": gp["launches"]}
    del gp
    bw = bench_backward(kda, max(3, args.steps // 4), 3, stream, "kda_chunk_bwd", CHUNK_BWD_KERNELS)
    bms = max_over_ranks(bw["ms"], world)
    extra["backward"] = {
        "workload": bw["name"] + "_backward", "entry": "kda_chunk_bwd", "ms_per_call": bms,
        "kernel_ms": {n: max_over_ranks(v, world) for n, v in bw["kernel_ms"].items()},
        "tokens_per_s": world * bw["tokens"] / (bms * 1e-3),
        "hbm_frac": bw["bytes"] / (bms * 1e-3) / 1e9 / pk["hbm"], "gpu_launches": bw["launches"]}
    extra["backward"]["roofline"] = chunk_bwd_roofline(bw, bms, extra["backward"]["kernel_ms"], pk["hbm"],
                                                       extra["backward"]["workload"])
    bw = bench_backward(kda, 3, 3, stream, "kda_backward")
    bms = max_over_ranks(bw["ms"], world)
    extra["backward_token_loop"] = {
        "workload": bw["name"] + "_backward", "entry": "kda_backward", "ms_per_call": bms,
        "tokens_per_s": world * bw["tokens"] / (bms * 1e-3), "gpu_launches": bw["launches"]}
    del bw

    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": headline_config(world),
            "roofline": roof, "path_roofline": path_roof, "tc_roofline": tc,
            "t_roof_over_t": t_roof / (ms * 1e-3),
            "kernel_ms": head_summary["kernel_ms"], "kernel_hbm_frac": head_summary["kernel_hbm_frac"],
            "e2e": {"value": e2e_val, "unit": "tokens/s", "h2d_bytes_per_step": e2e["h2d"],
                    "d2h_bytes_per_step": e2e["d2h"],
                    "pinned_on": (f"memory of the {e2e['host_cpus']} CPUs NVML names closest to the GPU"
                                  if e2e["host_cpus"] else "the allocating thread's memory node")},
            "gpu_launches": head_summary["gpu_launches"], "clocks": clk.summary(), "wall_s_timed_region": wall,
            "step_ms": step_ms}
    line.update(extra)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        r, threads, sample, _ = oracle_prefill_rate(HEADLINE_W, cpu_d)
        line["cpu_baseline"] = {"value": r, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                                "sample": sample}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
