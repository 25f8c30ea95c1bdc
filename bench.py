#!/usr/bin/env python3
"""Benchmark of the W4A16 hot path on one B300 (or N independent replicas).

One step = w4_quantize_pack(W) followed by w4_matmul(A, qweight, scales, zeros) on
the 70B-scale MLP layer (W fp16 [28672, 8192] ~ N(0, 0.015^2) with 0.1% of entries
x10, group 128; A bf16 [1, 8192] ~ N(0, 1)); another step workload via --workload.

value      algorithmic GB/s of the whole step (quantize bytes W + qweight + scales +
           zeros, plus matmul bytes qweight + scales + zeros + A + Y) over the device
           time of K steps, inputs resident in HBM.  The K quantize launches and then the
           K matmul launches run as CUDA graphs (no host work between launches) between
           CUDA events on the launching stream; step i's matmul reads the packed weights
           step i's quantize wrote.
kernels    every workload's kernels timed the same way (K launches each): the decode
           GEMV on the Llama-7B shape, the M = 8 skinny GEMM, the prefill tcgen05 GEMM
           and their quantize launches, plus the symmetric quantizer and the explicit
           dequantize on the step workload; each with its fraction of the measured peak
           and the bar it is held to.
roofline   the step's dominant kernel (the larger share of the step's device time): its
           algorithmic bytes per launch over its average launch duration, against the
           measured HBM copy bandwidth.  roofline_tensor: the same for the prefill GEMM's
           flops against the measured dense-bf16 peak.
e2e        the same step metric through the public API with host buffers: every step
           copies W and A from pinned host memory, runs both calls, and reads Y back.
cpu_baseline  the CPU oracle (plain C, one thread) on a bounded sample of the workload.

Timing of one phase (K launches of one kernel): the launches are captured as CUDA
graphs (one graph of exactly K launches, or repeats of one graph plus a remainder
graph when K is large); every graph that is timed is replayed untimed first; then
L2 is flushed by writing a buffer twice its size, a sleep kernel holds the stream
while the host enqueues the events and the replays (so no host delay falls inside
the event window), and CUDA events on the launching stream bracket the replays.
L2 never serves a launch's inputs: they rotate through copies spanning >= 3x L2
(launch i uses copy i mod C).

--impl reference times that oracle alone (the reference arm).  Under torchrun each
rank runs its own replica (weak scaling; no data-path collective); rank 0 prints the
max-over-ranks time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "W4A16 matmul HBM GB/s & TFLOP/s vs B300 roofline; quantize-pack GB/s"
DEFAULT_WORKLOAD = "mlp70b"
OTHER_WORKLOADS = ["llama7b_gemv", "skinny_m8", "prefill_gemm"]
ROTATE_L2 = 3              # rotating input copies span >= 3x the L2 size
MAX_COPIES = 64            # cap for tiny inputs (the correctness-only configuration)
MAX_GRAPH = 1000           # launches per captured CUDA graph at most
MSE_LAUNCHES = 5           # the MSE-search calibrator (~30 ms a launch) is timed over this many
GPTQ_LAUNCHES = 3          # GPTQ (O(N K^2) fused multiply-adds, ms a launch) likewise
GPTQ_WORKLOAD = "llama7b_gemv"
SLEEP_CYCLES = 4_000_000   # ~2 ms sleep kernel ahead of each event window
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
PROFILE_DIR = os.path.join(ROOT, "profiles")
CSRC = "w4a16_matmul_asym_b300/csrc/"
# The files that hold each kernel family's device code: its own header and the device
# headers it includes.  Their digest dates a profile.  Left out: the public header (error
# codes only) and gemm_tcgen05.cuh in the warp-MMA family, which takes only its host-side
# tensor-map helpers from there.
KERNEL_SOURCES = {
    "quantize_pack": [CSRC + "quantize_pack.cuh", CSRC + "common.cuh", CSRC + "prefetch.cuh"],
    "gemv": [CSRC + "gemv_dp4a.cuh", CSRC + "gemv.cuh", CSRC + "common.cuh", CSRC + "prefetch.cuh"],
    "gemv_mma": [CSRC + "gemv_mma.cuh", CSRC + "common.cuh", CSRC + "prefetch.cuh"],
    "quantize_calib": [CSRC + "quantize_calib.cuh", CSRC + "common.cuh"],
    "act_quant": [CSRC + "act_quant.cuh", CSRC + "common.cuh"],
    "gptq": [CSRC + "gptq.cuh", CSRC + "common.cuh"],
    "gemm_tcgen05": [CSRC + "gemm_tcgen05.cuh", CSRC + "common.cuh"],
    "dequantize": [CSRC + "dequantize.cuh", CSRC + "common.cuh"],
}
# The target fraction of each kernel's roofline per workload: (fraction, of which peak)
BARS = {
    ("quantize_pack", "mlp70b"): (0.60, "hbm"),
    ("quantize_pack", "llama7b_gemv"): (0.60, "hbm"),
    ("quantize_pack", "skinny_m8"): (0.60, "hbm"),
    ("quantize_pack", "prefill_gemm"): (0.60, "hbm"),
    ("matmul", "mlp70b"): (0.70, "hbm"),
    ("matmul", "llama7b_gemv"): (0.70, "hbm"),
    ("matmul", "skinny_m8"): (0.70, "hbm"),
    ("matmul", "prefill_gemm"): (0.50, "bf16"),
}


# ---- accounting -----------------------------------------------------------------------
def quantize_bytes(N: int, K: int, w_itemsize: int) -> int:
    """W read + qweight, scales (fp16) and zeros (uint8) written."""
    ng = K // 128
    return N * K * w_itemsize + N * K // 2 + N * ng * 2 + N * ng


def matmul_bytes(M: int, N: int, K: int) -> int:
    """qweight + scales + zeros + A read, Y written."""
    ng = K // 128
    return N * K // 2 + N * ng * 2 + N * ng + M * K * 2 + M * N * 2


def matmul_flops(M: int, N: int, K: int) -> int:
    return 2 * M * N * K


def dequantize_bytes(N: int, K: int) -> int:
    """qweight + scales + zeros read, bf16 W_hat written."""
    ng = K // 128
    return N * K // 2 + 3 * N * ng + 2 * N * K


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def matmul_kernel_name(M: int, K: int) -> str:
    """Which kernel family w4_matmul runs for this shape (mirrors the dispatch)."""
    if 2 <= M <= 16 and K % 2048 == 0 and M * K * 2 <= 128 * 1024:
        return "gemv_mma"
    if M > 8:
        return "gemm_tcgen05"
    return "gemv"


def source_digest(kernel: str) -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kernel]:
        path = os.path.join(ROOT, rel)
        if os.path.exists(path):
            with open(path, "rb") as f:
                h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the
    current kernel source (else None)."""
    path = os.path.join(PROFILE_DIR, f"{kernel}_{workload}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    m_src = re.search(r"^source_sha256_16:\s*([0-9a-f]+)", text, re.M)
    m_tr = re.search(r"^dram_bytes_per_launch:\s*([0-9]+)", text, re.M)
    if not m_src or not m_tr or m_src.group(1) != source_digest(kernel):
        return None
    return int(m_tr.group(1))


def host_cpu():
    """(cores this process may run on, CPU model name)."""
    try:
        cores = len(os.sched_getaffinity(0))
    except AttributeError:
        cores = os.cpu_count() or 1
    model = "unknown"
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    return cores, model


# ---- distributed control plane (CPU gloo; no data-path collective) ---------------------
def dist_info():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def dist_init(ws: int):
    if ws <= 1:
        return None
    import torch.distributed as dist
    if not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("gloo")
    return dist


def aggregate(local_seconds: float, local_units: float, dist=None):
    """(max seconds over ranks, sum of units over ranks)."""
    if dist is None:
        return local_seconds, local_units
    import torch
    t = torch.tensor([local_seconds], dtype=torch.float64)
    u = torch.tensor([local_units], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


# ---- graph sizing ------------------------------------------------------------------------
def graph_plan(count: int, period: int, max_graph: int = MAX_GRAPH):
    """How `count` launches are split into captured graphs: (n, reps, rest) with
    reps graphs of n launches and one of `rest` (n a multiple of `period`, so every
    replay continues the copy rotation, unless count itself fits one graph)."""
    if count <= 0:
        return 0, 0, 0
    if count <= max_graph:
        return count, 1, 0
    n = period * max(1, max_graph // period)
    reps, rest = divmod(count, n)
    return n, reps, rest


# ---- clocks ---------------------------------------------------------------------------
class ClockSampler:
    """Samples the SM clock and the clock-event (throttle) reasons while running:
    through NVML if it loads, else by polling nvidia-smi."""

    REASONS = {
        0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
        0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
        0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
        0x100: "display_clock_setting",
    }

    def __init__(self, device_index: int, period_s: float = 0.02):
        self.period = period_s
        self.index = device_index
        self.samples, self.reasons = [], set()
        self.max_mhz = None
        self.error = None
        self.source = None
        self._stop = threading.Event()
        self._first = threading.Event()
        self._thread = None
        self.nv = None
        try:
            import pynvml
            pynvml.nvmlInit()
            self.h = pynvml.nvmlDeviceGetHandleByIndex(device_index)
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(self.h, pynvml.NVML_CLOCK_SM)
            self.nv = pynvml
            self.source = "nvml"
        except Exception as e:  # fall back to nvidia-smi
            self.error = f"nvml: {type(e).__name__}: {e}"
            self.source = "nvidia-smi"

    def _sample_nvml(self):
        self.samples.append(self.nv.nvmlDeviceGetClockInfo(self.h, self.nv.NVML_CLOCK_SM))
        bits = self.nv.nvmlDeviceGetCurrentClocksEventReasons(self.h)
        for b, name in self.REASONS.items():
            if bits & b:
                self.reasons.add(name)

    def _sample_smi(self):
        import subprocess
        q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")
        out = subprocess.run(["nvidia-smi", "-i", str(self.index), f"--query-gpu={q}",
                              "--format=csv,noheader,nounits"], capture_output=True, text=True,
                             timeout=5).stdout.strip().split(",")
        self.samples.append(float(out[0]))
        self.max_mhz = float(out[1])
        for name, val in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                              "sw_power_cap"), out[2:]):
            if val.strip().lower() == "active":
                self.reasons.add(name)

    def _run(self):
        while not self._stop.is_set():
            try:
                self._sample_nvml() if self.nv is not None else self._sample_smi()
            except Exception as e:
                self.error = f"{type(e).__name__}: {e}"
            self._first.set()
            time.sleep(self.period)

    def start(self):
        """Starts sampling and returns once the first sample is taken, so that the
        sampler's start-up never overlaps an event window."""
        self._thread = threading.Thread(target=self._run, daemon=True)
        self._thread.start()
        self._first.wait(timeout=10)

    def stop(self):
        if self._thread is not None:
            self._stop.set()
            self._thread.join()
        out = {"sm_mhz": statistics.median(self.samples) if self.samples else None,
               "sm_max_mhz": self.max_mhz, "reasons": sorted(self.reasons),
               "samples": len(self.samples), "source": self.source}
        if self.error:
            out["note"] = self.error
        return out


# ---- CPU oracle timing --------------------------------------------------------------------
def oracle_sample_rate(workload: str, budget_s: float, max_rows: int | None = None):
    """Time the CPU oracle (quantize + matmul, as it stands) on the first rows of the
    workload's W until `budget_s` of CPU time is spent.  Returns (GB/s, description,
    seconds per pass, bytes per pass)."""
    import oracle
    import synth
    oracle.build()
    wl = synth.WORKLOADS[workload]
    rows = wl.N if max_rows is None else max(1, min(wl.N, max_rows))
    W, A = synth.make_workload(workload, N=rows)
    isz = W.dtype.itemsize
    nbytes = quantize_bytes(rows, wl.K, isz) + matmul_bytes(A.shape[0], rows, wl.K)
    passes, spent = 0, 0.0
    while spent < budget_s or passes == 0:
        t0 = time.perf_counter()
        q, s, z = oracle.quantize_pack(W)
        oracle.matmul(A, q, s, z)
        spent += time.perf_counter() - t0
        passes += 1
    desc = (f"oracle quantize+matmul on the first {rows} of {wl.N} rows of the {workload} "
            f"workload (K={wl.K}, M={A.shape[0]}), {passes} pass(es), 1 thread")
    return passes * nbytes / spent / 1e9, desc, spent / passes, nbytes


def oracle_prefill_rate(budget_s: float, threads: int, workload: str = "prefill_gemm"):
    """Time the CPU oracle's fp64 matmul (as it stands) on a compute-bound workload with
    every host thread busy: each of `threads` threads runs one oracle.matmul call on its
    own block of R rows of W against all M activation rows (the C call releases the
    GIL, so the blocks run in parallel).  R is sized so that a thread spends about
    `budget_s` seconds.  Returns (TFLOP/s, description, threads)."""
    import concurrent.futures
    import oracle
    import synth
    oracle.build()
    wl = synth.WORKLOADS[workload]
    threads = max(1, min(threads, wl.N))
    probe = min(8, wl.N)
    Wp, Ap = synth.make_workload(workload, N=probe)
    qp, sp, zp = oracle.quantize_pack(Wp)
    t0 = time.perf_counter()
    oracle.matmul(Ap, qp, sp, zp)
    per_row = max((time.perf_counter() - t0) / probe, 1e-6)
    rows = max(1, min(wl.N // threads, int(budget_s / per_row)))
    W, A = synth.make_workload(workload, N=threads * rows)
    q, s, z = oracle.quantize_pack(W)
    M, K = A.shape
    blocks = [(q[i * rows:(i + 1) * rows], s[i * rows:(i + 1) * rows], z[i * rows:(i + 1) * rows])
              for i in range(threads)]
    with concurrent.futures.ThreadPoolExecutor(max_workers=threads) as pool:
        t0 = time.perf_counter()
        list(pool.map(lambda b: oracle.matmul(A, *b), blocks))
        wall = time.perf_counter() - t0
    flops = 2.0 * M * threads * rows * K
    desc = (f"oracle fp64 matmul of the {workload} workload (M={M}, K={K}) on {threads} x {rows} "
            f"of its {wl.N} rows of W, one row block per host thread, {threads} threads at once")
    return flops / wall / 1e12, desc, threads


# ---- our arm --------------------------------------------------------------------------
class PhaseTimer:
    """Times `count` back-to-back launches of one kernel (see the module docstring)."""

    def __init__(self, torch, dev, stream, l2_bytes: int):
        self.torch = torch
        self.dev = dev
        self.stream = stream
        self.cap = torch.cuda.Stream(dev)
        self.flush_buf = torch.empty(2 * l2_bytes, dtype=torch.uint8, device=dev)
        self.launches = 0          # our kernels launched inside event windows

    def time(self, launch, count: int, warmup: int, period: int):
        """Seconds per launch; launch(i, stream) enqueues launch i on `stream`."""
        torch = self.torch
        n, reps, rest = graph_plan(count, period)

        def graph_of(k):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=self.cap):
                for i in range(k):
                    launch(i, self.cap)
            return g

        g_main = graph_of(n)
        g_rest = graph_of(rest) if rest else None
        done = 0
        while True:                      # every timed graph replayed, >= warmup launches
            g_main.replay()
            done += n
            if g_rest is not None:
                g_rest.replay()
                done += rest
            if done >= warmup:
                break
        self.flush_buf.zero_()
        torch.cuda.synchronize(self.dev)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(SLEEP_CYCLES)
        a.record(self.stream)
        for _ in range(reps):
            g_main.replay()
        if g_rest is not None:
            g_rest.replay()
        b.record(self.stream)
        torch.cuda.synchronize(self.dev)
        self.launches += count
        del g_main, g_rest
        return a.elapsed_time(b) / 1e3 / count, {"graph_launches": n, "replays": reps, "remainder": rest}


def copies_for(nbytes: int, l2: int) -> int:
    return min(MAX_COPIES, max(2, -(-ROTATE_L2 * l2 // max(1, nbytes))))


def hbm_entry(us_s: float, nbytes: int, peaks, bar=None, **extra):
    gbs = nbytes / us_s / 1e9
    d = {"us": us_s * 1e6, "bytes": nbytes, "GB/s": gbs, "frac_hbm": gbs / peaks["hbm_gbs"]}
    if bar is not None:
        d["bar"] = bar
        d["meets_bar"] = d["frac_hbm"] >= bar
    d.update(extra)
    return d


def run_workload(w4, torch, np, synth, timer, wl_name, steps, warmup, l2, peaks, step_workload,
                 extras):
    """Quantize and matmul launches of one workload (and, for the step workload, the
    extra kernels).  Returns (kernels dict, phase seconds, info)."""
    dev = timer.dev
    wl = synth.WORKLOADS[wl_name]
    N, K = wl.N, wl.K
    W, A = synth.make_workload(wl_name)
    M = A.shape[0]
    qb, mb = quantize_bytes(N, K, W.dtype.itemsize), matmul_bytes(M, N, K)
    qsz = N * K // 2 + 3 * N * (K // 128)
    cw, cm = copies_for(W.nbytes, l2), copies_for(qsz, l2)
    period = cw * cm // math.gcd(cw, cm)
    Wds = [torch.from_numpy(W).to(dev) for _ in range(cw)]
    Ad = torch.from_numpy(A.view(np.int16)).to(dev).view(torch.bfloat16)
    qs = [torch.empty((N, K // 2), dtype=torch.uint8, device=dev) for _ in range(cm)]
    ss = [torch.empty((N, K // 128), dtype=torch.float16, device=dev) for _ in range(cm)]
    zs = [torch.empty((N, K // 128), dtype=torch.uint8, device=dev) for _ in range(cm)]
    Y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    for i in range(cm):
        w4.quantize_pack(Wds[i % cw], out=(qs[i], ss[i], zs[i]))
    torch.cuda.synchronize(dev)

    def q_launch(i, s_):
        w4.quantize_pack(Wds[i % cw], out=(qs[i % cm], ss[i % cm], zs[i % cm]), stream=s_)

    def m_launch(i, s_):
        w4.matmul(Ad, qs[i % cm], ss[i % cm], zs[i % cm], out=Y, stream=s_)

    q_s, q_graph = timer.time(q_launch, steps, warmup, period)
    m_s, m_graph = timer.time(m_launch, steps, warmup, period)
    mk = matmul_kernel_name(M, K)
    rot = f"{cw} copies of W ({cw * W.nbytes / 1e6:.0f} MB), {cm} packed copies ({cm * qsz / 1e6:.0f} MB)"
    ks = {"quantize_pack": hbm_entry(q_s, qb, peaks, BARS.get(("quantize_pack", wl_name), (None,))[0],
                                     launches=steps, graphs=q_graph,
                                     traffic=profiled_traffic("quantize_pack", wl_name))}
    bar = BARS.get(("matmul", wl_name))
    if mk == "gemm_tcgen05":
        fl = matmul_flops(M, N, K)
        tf = fl / m_s / 1e12
        ent = {"kernel": mk, "us": m_s * 1e6, "flops": fl, "TFLOP/s": tf,
               "frac_bf16_burst": tf / peaks["bf16_tflops"],
               "frac_bf16_sustained": tf / peaks["bf16_tflops_sustained"],
               "GB/s": mb / m_s / 1e9, "launches": steps, "graphs": m_graph,
               "traffic": profiled_traffic(mk, wl_name)}
        if bar:
            ent["bar"] = bar[0]
            ent["meets_bar"] = ent["frac_bf16_burst"] >= bar[0]
    else:
        ent = hbm_entry(m_s, mb, peaks, bar[0] if bar else None, kernel=mk, launches=steps,
                        graphs=m_graph, traffic=profiled_traffic(mk, wl_name))
    ks["matmul"] = ent
    info = {"N": N, "K": K, "M": M, "w_dtype": wl.w_dtype, "rotation": rot, "qb": qb, "mb": mb}

    if extras and wl_name == step_workload:
        out_bytes = N * K * 2
        co = copies_for(out_bytes, l2)
        outs = [torch.empty((N, K), dtype=torch.bfloat16, device=dev) for _ in range(co)]
        sym_s, _ = timer.time(lambda i, s_: w4.quantize_pack(
            Wds[i % cw], out=(qs[i % cm], ss[i % cm], zs[i % cm]), stream=s_, symmetric=True),
            steps, warmup, period)
        dq_period = cm * co // math.gcd(cm, co)
        dq_s, _ = timer.time(lambda i, s_: w4.dequantize(
            qs[i % cm], ss[i % cm], zs[i % cm], dtype=torch.bfloat16, out=outs[i % co], stream=s_),
            steps, warmup, dq_period)
        ks["quantize_pack_sym"] = hbm_entry(sym_s, qb, peaks, launches=steps)
        ks["dequantize_bf16"] = hbm_entry(dq_s, dequantize_bytes(N, K), peaks, launches=steps,
                                          rotation=f"{cm} packed copies, {co} output copies",
                                          traffic=profiled_traffic("dequantize", wl_name))
        del outs
        # Clip-range calibration: the percentile calibrator over K launches; the MSE
        # search (1000 candidates, n * 128 divisions per group: arithmetic-bound) over
        # MSE_LAUNCHES launches on the first rows that make ~1/8 of the matrix.
        pc_s, _ = timer.time(lambda i, s_: w4.quantize_pack(
            Wds[i % cw], out=(qs[i % cm], ss[i % cm], zs[i % cm]), stream=s_, calibration="percentile", param=99.9),
            steps, warmup, period)
        ks["quantize_pack_percentile"] = hbm_entry(pc_s, qb, peaks, launches=steps, p=99.9,
                                                   groups_per_s=N * K / 128 / pc_s)
        rows = max(1, N // 8)
        Wsub = [w[:rows] for w in Wds]
        outs_sub = [(q[:rows], s[:rows], z[:rows]) for q, s, z in zip(qs, ss, zs)]
        n_mse = min(steps, MSE_LAUNCHES)
        mse_s, _ = timer.time(lambda i, s_: w4.quantize_pack(
            Wsub[i % cw], out=outs_sub[i % cm], stream=s_, calibration="mse", param=1000),
            n_mse, 1, period)
        ks["quantize_pack_mse"] = {"us": mse_s * 1e6, "rows": rows, "candidates": 1000, "launches": n_mse,
                                   "groups_per_s": rows * K / 128 / mse_s,
                                   "GB/s": quantize_bytes(rows, K, W.dtype.itemsize) / mse_s / 1e9,
                                   "bound": "alu (1000 candidates x 128 divisions per group)"}
    if extras and wl_name == GPTQ_WORKLOAD:
        # GPTQ on synthetic calibration activations X [2K, K] ~ N(0, 1) with neighbouring
        # inputs correlated (x_k += 0.9 x_(k-1)); the kernel's input U, the upper Cholesky
        # factor of the damped H^-1, is prepared on the host with numpy in fp64.
        rng = np.random.default_rng(11)
        X = rng.standard_normal((2 * K, K))
        X[:, 1:] += 0.9 * X[:, :-1]
        H = X.T @ X / X.shape[0]
        H += 1e-4 * np.mean(np.diag(H)) * np.eye(K)
        U = np.ascontiguousarray(np.linalg.cholesky(np.linalg.inv(H)).T, dtype=np.float32)
        Ud = torch.from_numpy(U).to(dev)
        del X, H, U
        n_g = min(steps, GPTQ_LAUNCHES)
        g_s, _ = timer.time(lambda i, s_: w4.gptq_quantize(Wds[i % cw], Ud, out=(qs[i % cm], ss[i % cm], zs[i % cm]),
                                                           stream=s_), n_g, 1, period)
        ks["gptq_quantize"] = {"us": g_s * 1e6, "launches": n_g, "fma": N * K * (K - 1) // 2,
                               "TFMA/s": N * K * (K - 1) / 2 / g_s / 1e12,
                               "bound": "fp32 fused multiply-adds (O(N K^2), sequential per element)"}
        del Ud
    if extras:
        # W4A8: the per-token INT8 activation quantizer, then the W4A8 matmul on the same
        # packed copies (the GEMM path widens a_q into a workspace; the decode path needs none).
        aq, sa = w4.quantize_act_int8(Ad)
        actq_s, _ = timer.time(lambda i, s_: w4.quantize_act_int8(Ad, stream=s_, out=(aq, sa)), steps, warmup, 1)
        need = w4.w4_matmul_w4a8_workspace_size(M, K)
        ws = torch.empty((max(need, 1),), dtype=torch.uint8, device=dev)
        w8_s, w8_graph = timer.time(lambda i, s_: w4.matmul_w4a8(
            aq, sa, qs[i % cm], ss[i % cm], zs[i % cm], out=Y, stream=s_, workspace=ws), steps, warmup, cm)
        ks["quantize_act_int8"] = hbm_entry(actq_s, 3 * M * K + 4 * M, peaks, launches=steps,
                                            note="A is read twice and may stay in L2 between launches")
        fl = matmul_flops(M, N, K)
        w8b = N * K // 2 + 3 * N * (K // 128) + M * K + 4 * M + 2 * M * N
        ent = hbm_entry(w8_s, w8b, peaks, launches=steps, workspace_bytes=need, graphs=w8_graph)
        ent["TFLOP/s"] = fl / w8_s / 1e12
        ent["frac_bf16_burst"] = ent["TFLOP/s"] / peaks["bf16_tflops"]
        ks["matmul_w4a8"] = ent
        del ws
    del Wds, qs, ss, zs, Y, Ad
    torch.cuda.empty_cache()
    return ks, (q_s, m_s), info


def run_ours(args, ws, rank, local, dist):
    import numpy as np
    import torch
    import synth
    import w4a16_matmul_asym_b300 as w4

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 126 << 20) or (126 << 20)
    peaks, peak_src = measured_peaks()
    timer = PhaseTimer(torch, dev, stream, l2)
    steps, warmup = args.steps, args.warmup
    step_wl = args.workload

    sampler = ClockSampler(torch.cuda.current_device())
    barrier(dist)
    sampler.start()
    kernels, step_info = {}, None
    plan = [step_wl] + ([w for w in OTHER_WORKLOADS if w != step_wl] if not args.no_extra else [])
    for name in plan:
        ks, (q_s, m_s), info = run_workload(w4, torch, np, synth, timer, name, steps, warmup, l2,
                                            peaks, step_wl, not args.no_extra)
        kernels[name] = ks
        if name == step_wl:
            step_info, step_q, step_m = info, q_s, m_s
    clocks = sampler.stop()
    barrier(dist)

    N, K, M = step_info["N"], step_info["K"], step_info["M"]
    step_bytes = step_info["qb"] + step_info["mb"]
    local_s = (step_q + step_m) * steps
    tot_s, tot_bytes = aggregate(local_s, step_bytes * steps, dist)
    value = tot_bytes / tot_s / 1e9

    sk = kernels[step_wl]
    if step_q >= step_m:
        dom, ent = "quantize_pack", sk["quantize_pack"]
    else:
        dom, ent = sk["matmul"].get("kernel", "matmul"), sk["matmul"]
    if "TFLOP/s" in ent:
        roofline = {"bound": "tensor", "kernel": dom, "workload": step_wl, "achieved": ent["TFLOP/s"],
                    "peak": peaks["bf16_tflops"], "unit": "TFLOP/s", "frac": ent["frac_bf16_burst"],
                    "peak_source": peak_src, "traffic": ent.get("traffic")}
    else:
        roofline = {"bound": "hbm", "kernel": dom, "workload": step_wl, "achieved": ent["GB/s"],
                    "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": ent["frac_hbm"],
                    "peak_source": peak_src, "traffic": ent.get("traffic")}
    roofline_tensor = None
    if "prefill_gemm" in kernels:
        g = kernels["prefill_gemm"]["matmul"]
        roofline_tensor = {"bound": "tensor", "kernel": g.get("kernel"), "workload": "prefill_gemm",
                           "achieved": g.get("TFLOP/s"), "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                           "frac": g.get("frac_bf16_burst"), "peak_source": peak_src,
                           "peak_sustained": peaks["bf16_tflops_sustained"],
                           "frac_sustained": g.get("frac_bf16_sustained"), "traffic": g.get("traffic")}

    # End to end through the public API with host buffers (pinned), copies inside.
    wl = synth.WORKLOADS[step_wl]
    W, A = synth.make_workload(step_wl)
    Wh = torch.from_numpy(W).pin_memory()
    Ah = torch.from_numpy(A.view(np.int16)).pin_memory()
    Yh = torch.empty((M, N), dtype=torch.bfloat16).pin_memory()
    Wd = torch.empty_like(Wh, device=dev)
    Ad = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
    q = torch.empty((N, K // 2), dtype=torch.uint8, device=dev)
    s = torch.empty((N, K // 128), dtype=torch.float16, device=dev)
    z = torch.empty((N, K // 128), dtype=torch.uint8, device=dev)
    Y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    e2e_steps = max(3, min(args.steps, 50))
    h2d = Wh.numel() * Wh.element_size() + Ah.numel() * Ah.element_size()
    d2h = Yh.numel() * Yh.element_size()

    def e2e_step():
        Wd.copy_(Wh, non_blocking=True)
        Ad.view(torch.int16).copy_(Ah, non_blocking=True)
        w4.quantize_pack(Wd, out=(q, s, z), stream=stream)
        w4.matmul(Ad, q, s, z, out=Y, stream=stream)
        Yh.copy_(Y, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(dist)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_s, e2e_units = aggregate(e0.elapsed_time(e1) / 1e3, step_bytes * e2e_steps, dist)
    e2e = {"value": e2e_units / e2e_s / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "steps": e2e_steps}

    result = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws,
        "steps": steps, "warmup": warmup, "ms_per_step": tot_s / steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "w4a16: int4 weights with fp16 scales, bf16 activations, fp32 accumulation "
                 "(quantize in fp32)",
        "data": "synthetic",
        "config": {
            "workload": f"{step_wl}: {wl.desc}; group 128",
            "N": N, "K": K, "M": M, "group": 128, "w_dtype": wl.w_dtype,
            "step": "w4_quantize_pack + w4_matmul",
            "l2": (f"inputs larger than L2 and rotated, each set >= {ROTATE_L2}x the "
                   f"{l2 / 2**20:.0f} MiB L2 (step: {step_info['rotation']}); L2 flushed before "
                   f"every event window"),
            "timing": (f"per kernel: CUDA events around {steps} back-to-back launches replayed from "
                       f"CUDA graphs (graphs of <= {MAX_GRAPH} launches, each replayed untimed before "
                       f"the window); step = the quantize phase then the matmul phase, step i's matmul "
                       f"reading what step i's quantize wrote"),
            "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
        },
        "roofline": roofline,
        "roofline_tensor": roofline_tensor,
        "kernels": kernels,
        "e2e": e2e,
        "gpu_launches": timer.launches,
        "clocks": clocks,
    }
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        rate, desc, _, _ = oracle_sample_rate(step_wl, budget_s=args.cpu_budget, max_rows=args.cpu_rows)
        cores, model = host_cpu()
        result["cpu_baseline"] = {"value": rate, "unit": "GB/s", "cores": 1, "kind": "oracle",
                                  "sample": desc, "host_cores": cores, "cpu_model": model}
        if args.cpu_prefill_budget > 0:
            # The compute-bound case on every host core: the context for roofline_tensor.
            tf, pdesc, used = oracle_prefill_rate(args.cpu_prefill_budget, cores)
            result["cpu_baseline_tensor"] = {"value": tf, "unit": "TFLOP/s", "cores": used, "kind": "oracle",
                                             "sample": pdesc, "host_cores": cores, "cpu_model": model}
    return result


# ---- one launch of one kernel (for profiler captures) ------------------------------------
ONCE_KERNELS = ("quantize_pack", "quantize_pack_sym", "quantize_pack_percentile", "quantize_pack_mse",
                "dequantize", "matmul", "quantize_act_int8", "matmul_w4a8", "gptq_quantize")


def run_once(args):
    """Two launches of one kernel on the workload's inputs (the first warms up), then a
    device sync: a small, self-contained command for profiler captures.  No timing."""
    import numpy as np
    import torch
    import synth
    import w4a16_matmul_asym_b300 as w4
    dev = torch.device("cuda", 0)
    W, A = synth.make_workload(args.workload)
    M, N, K = A.shape[0], W.shape[0], W.shape[1]
    Wd = torch.from_numpy(W).to(dev)
    Ad = torch.from_numpy(A.view(np.int16)).to(dev).view(torch.bfloat16)
    q, s, z = w4.quantize_pack(Wd)
    name = args.once
    if name == "gptq_quantize":
        rng = np.random.default_rng(11)
        X = rng.standard_normal((2 * K, K))
        X[:, 1:] += 0.9 * X[:, :-1]
        H = X.T @ X / X.shape[0]
        H += 1e-4 * np.mean(np.diag(H)) * np.eye(K)
        Ud = torch.from_numpy(np.ascontiguousarray(np.linalg.cholesky(np.linalg.inv(H)).T, dtype=np.float32)).to(dev)
    aq, sa = w4.quantize_act_int8(Ad)
    for _ in range(2):
        if name == "quantize_pack":
            w4.quantize_pack(Wd, out=(q, s, z))
        elif name == "quantize_pack_sym":
            w4.quantize_pack(Wd, out=(q, s, z), symmetric=True)
        elif name == "quantize_pack_percentile":
            w4.quantize_pack(Wd, out=(q, s, z), calibration="percentile", param=99.9)
        elif name == "quantize_pack_mse":
            w4.quantize_pack(Wd[: max(1, N // 8)], calibration="mse", param=1000)
        elif name == "dequantize":
            w4.dequantize(q, s, z)
        elif name == "matmul":
            w4.matmul(Ad, q, s, z)
        elif name == "quantize_act_int8":
            w4.quantize_act_int8(Ad, out=(aq, sa))
        elif name == "matmul_w4a8":
            w4.matmul_w4a8(aq, sa, q, s, z)
        elif name == "gptq_quantize":
            w4.gptq_quantize(Wd, Ud, out=(q, s, z))
    torch.cuda.synchronize(dev)
    rc = w4.w4_check_device_error(0)
    print(json.dumps({"once": name, "workload": args.workload, "M": M, "N": N, "K": K, "status": rc}))
    return 0 if rc == 0 else 1


# ---- reference arm: the CPU oracle alone ------------------------------------------------
def run_reference(args, ws, rank):
    import synth
    wl = synth.WORKLOADS[args.workload]
    # Size the per-step sample so warmup + steps stay within about two minutes.
    _, _, sec_per_pass, _ = oracle_sample_rate(args.workload, budget_s=0.0, max_rows=64)
    per_row = sec_per_pass / 64
    budget_per_step = 120.0 / max(1, args.steps + args.warmup)
    rows = int(max(1, min(wl.N, budget_per_step / per_row)))
    import oracle
    W, A = synth.make_workload(args.workload, N=rows)
    nbytes = quantize_bytes(rows, wl.K, W.dtype.itemsize) + matmul_bytes(A.shape[0], rows, wl.K)

    def step():
        q, s, z = oracle.quantize_pack(W)
        oracle.matmul(A, q, s, z)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    secs = time.perf_counter() - t0
    value = nbytes * args.steps / secs / 1e9
    cores, model = host_cpu()
    desc = (f"oracle quantize+matmul on the first {rows} of {wl.N} rows of the {args.workload} "
            f"workload per step (K={wl.K}, M={A.shape[0]}), 1 thread")
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32 quantize, f64 matmul", "data": "synthetic",
        "config": {"workload": f"{args.workload}: {wl.desc}; group 128", "N": wl.N, "K": wl.K,
                   "M": wl.M, "group": 128, "sample_rows": rows},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": desc, "host_cores": cores, "cpu_model": model},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    import synth
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=list(synth.WORKLOADS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--cpu-budget", type=float, default=10.0,
                    help="seconds of CPU time for the oracle baseline")
    ap.add_argument("--cpu-rows", type=int, default=1024,
                    help="rows of W in the oracle baseline sample")
    ap.add_argument("--cpu-prefill-budget", type=float, default=5.0,
                    help="seconds per host thread for the all-core oracle matmul on the prefill "
                         "workload (0 skips it)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="time the step workload only (no other workloads or extra kernels)")
    ap.add_argument("--once", choices=ONCE_KERNELS,
                    help="run one kernel twice on the workload and exit (for profiler captures)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.steps < 1:
        ap.error("--steps must be at least 1")
    if args.once:
        return run_once(args)
    ws, rank, local = dist_info()
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, ws, rank)), flush=True)
        return 0
    dist = dist_init(ws)
    res = run_ours(args, ws, rank, local, dist)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
