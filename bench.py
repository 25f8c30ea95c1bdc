#!/usr/bin/env python3
"""Benchmark of the W4A16 hot path on one B300 (or N independent replicas).

One step = w4_quantize_pack(W) followed by w4_matmul(A, qweight, scales, zeros) on
the Llama-7B-shaped decode workload (W fp16 [11008, 4096] ~ N(0, 0.02) with 0.1% of
entries x10, group 128; A bf16 [1, 4096] ~ N(0, 1)); other workloads via --workload.

value      algorithmic GB/s of the whole step (quantize bytes W + qweight + scales +
           zeros, plus matmul bytes qweight + scales + zeros + A + Y) over the device
           time of K steps, inputs resident in HBM.  The K quantize launches and then the
           K matmul launches run as CUDA graphs (no host work between launches) between
           CUDA events on the launching stream; L2 never serves a launch's weights: the
           inputs rotate through copies spanning >= 3x the L2 size (launch i uses copy
           i mod C), and step i's matmul reads the packed weights step i's quantize wrote.
roofline   the kernel with the largest share of the step: its algorithmic bytes (or
           flops for the tensor-core GEMM) per launch over its average launch duration
           (its phase's event time / K), against the measured HBM (or bf16) peak.
e2e        the same metric through the public API with host buffers: every step
           copies W and A from pinned host memory, runs both calls, and reads Y back.
cpu_baseline  the CPU oracle (plain C, one thread) on a bounded sample of the workload.

--impl reference times that oracle alone (the reference arm).  Under torchrun each
rank runs its own replica (weak scaling; no data-path collective); rank 0 prints the
max-over-ranks time.
"""
from __future__ import annotations

import argparse
import hashlib
import math
import json
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
DEFAULT_WORKLOAD = "llama7b_gemv"
ROTATE_L2 = 3              # rotating input copies span >= 3x the L2 size
MAX_COPIES = 64            # cap for tiny inputs (the correctness-only configuration)
LAUNCHES_PER_GRAPH = 50    # launches per captured CUDA graph (rounded to the copy cycle)
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
PROFILE_DIR = os.path.join(ROOT, "profiles")
KERNEL_SOURCES = {  # every file a kernel is compiled from (its digest dates a profile)
    "quantize_pack": ["w4a16_matmul_asym_b300/csrc/quantize_pack.cuh", "w4a16_matmul_asym_b300/csrc/common.cuh"],
    "gemv": ["w4a16_matmul_asym_b300/csrc/gemv_dp4a.cuh", "w4a16_matmul_asym_b300/csrc/gemv.cuh",
             "w4a16_matmul_asym_b300/csrc/common.cuh"],
    "gemm_tcgen05": ["w4a16_matmul_asym_b300/csrc/gemm_tcgen05.cuh", "w4a16_matmul_asym_b300/csrc/common.cuh"],
    "dequantize": ["w4a16_matmul_asym_b300/csrc/dequantize.cuh", "w4a16_matmul_asym_b300/csrc/common.cuh"],
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


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def source_digest(kernel: str) -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, rel), "rb") as f:
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

    def __init__(self, device_index: int, period_s: float = 0.01):
        self.period = period_s
        self.index = device_index
        self.samples, self.reasons = [], set()
        self.max_mhz = None
        self.error = None
        self.source = None
        self._stop = threading.Event()
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
            time.sleep(self.period)

    def start(self):
        self._thread = threading.Thread(target=self._run, daemon=True)
        self._thread.start()

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


# ---- our arm --------------------------------------------------------------------------
def run_ours(args, ws, rank, local, dist):
    import numpy as np
    import torch
    import synth
    import w4a16_matmul_asym_b300 as w4

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = synth.WORKLOADS[args.workload]
    N, K = wl.N, wl.K
    W, A = synth.make_workload(args.workload)
    M = A.shape[0]
    isz = W.dtype.itemsize
    qb, mb = quantize_bytes(N, K, isz), matmul_bytes(M, N, K)
    step_bytes = qb + mb
    gemm = M > 8
    mm_name = "gemm_tcgen05" if gemm else "gemv"

    # L2 must not serve the timed launches: every launch reads a copy of its inputs that
    # the launches before it have evicted.  W is replicated for the quantize launches and
    # the packed weights for the matmul launches, each set >= 3x the L2 size, and launch
    # i uses copy i mod C.  Step i's quantize writes the packed copy its matmul reads.
    l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 126 << 20) or (126 << 20)
    w_bytes = W.nbytes
    qsz_bytes = N * K // 2 + 3 * N * (K // 128)
    cw = min(MAX_COPIES, max(2, -(-ROTATE_L2 * l2 // w_bytes)))
    cm = min(MAX_COPIES, max(2, -(-ROTATE_L2 * l2 // qsz_bytes)))
    l2_defeated = cw * w_bytes >= ROTATE_L2 * l2 and cm * qsz_bytes >= ROTATE_L2 * l2
    lcm = cw * cm // math.gcd(cw, cm)
    R = lcm * max(1, -(-LAUNCHES_PER_GRAPH // lcm))          # launches per captured graph
    steps = args.steps
    n_rep, rem = divmod(steps, R)

    Wh = torch.from_numpy(W)
    Wds = [Wh.to(dev) for _ in range(cw)]
    Ad = torch.from_numpy(A.view(np.int16)).to(dev).view(torch.bfloat16)
    qs = [torch.empty((N, K // 2), dtype=torch.uint8, device=dev) for _ in range(cm)]
    ss = [torch.empty((N, K // 128), dtype=torch.float16, device=dev) for _ in range(cm)]
    zs = [torch.empty((N, K // 128), dtype=torch.uint8, device=dev) for _ in range(cm)]
    Y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    Wd, q, s, z = Wds[0], qs[0], ss[0], zs[0]
    stream = torch.cuda.current_stream(dev)

    def step():
        w4.quantize_pack(Wd, out=(q, s, z), stream=stream)
        w4.matmul(Ad, q, s, z, out=Y, stream=stream)

    # Both phases as CUDA graphs of R launches (no host work between launches).
    for i in range(cm):
        w4.quantize_pack(Wds[i % cw], out=(qs[i], ss[i], zs[i]), stream=stream)
    w4.matmul(Ad, qs[0], ss[0], zs[0], out=Y, stream=stream)
    torch.cuda.synchronize(dev)
    cap = torch.cuda.Stream(dev)

    def capture(n):
        """(quantize graph, matmul graph) of n launches starting at copy 0."""
        g_q, g_m = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_q, stream=cap):
            for i in range(n):
                w4.quantize_pack(Wds[i % cw], out=(qs[i % cm], ss[i % cm], zs[i % cm]), stream=cap)
        with torch.cuda.graph(g_m, stream=cap):
            for i in range(n):
                w4.matmul(Ad, qs[i % cm], ss[i % cm], zs[i % cm], out=Y, stream=cap)
        return g_q, g_m

    # R is a multiple of both copy counts, so every replay continues the rotation.
    g_q, g_m = capture(R)
    g_qr, g_mr = capture(rem) if rem else (None, None)
    for _ in range(max(1, -(-args.warmup // R))):   # >= warmup untimed steps
        g_q.replay()
        g_m.replay()
    torch.cuda.synchronize(dev)

    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    sampler = ClockSampler(torch.cuda.current_device())
    barrier(dist)
    torch.cuda.synchronize(dev)
    sampler.start()
    ev[0].record(stream)
    for _ in range(n_rep):
        g_q.replay()
    if g_qr is not None:
        g_qr.replay()
    ev[1].record(stream)
    for _ in range(n_rep):
        g_m.replay()
    if g_mr is not None:
        g_mr.replay()
    ev[2].record(stream)
    torch.cuda.synchronize(dev)
    barrier(dist)
    clocks = sampler.stop()
    launches = 2 * steps
    q_total = ev[0].elapsed_time(ev[1]) / 1e3
    m_total = ev[1].elapsed_time(ev[2]) / 1e3
    local_s = q_total + m_total
    tot_s, tot_bytes = aggregate(local_s, step_bytes * steps, dist)
    value = tot_bytes / tot_s / 1e9

    peaks, peak_src = measured_peaks()
    q_avg = q_total / steps
    m_avg = m_total / steps
    kernels = {
        "quantize_pack": {"us": q_avg * 1e6, "bytes": qb, "GB/s": qb / q_avg / 1e9,
                          "frac_hbm": qb / q_avg / 1e9 / peaks["hbm_gbs"]},
        mm_name: {"us": m_avg * 1e6, "bytes": mb, "GB/s": mb / m_avg / 1e9,
                  "frac_hbm": mb / m_avg / 1e9 / peaks["hbm_gbs"]},
    }
    if gemm:
        fl = matmul_flops(M, N, K)
        kernels[mm_name]["TFLOP/s"] = fl / m_avg / 1e12
        kernels[mm_name]["frac_bf16_burst"] = fl / m_avg / 1e12 / peaks["bf16_tflops"]
        kernels[mm_name]["frac_bf16_sustained"] = fl / m_avg / 1e12 / peaks["bf16_tflops_sustained"]
    # Dominant kernel: the larger share of the step's device time.
    if q_avg >= m_avg:
        dom, ach, unit, peak, bound = "quantize_pack", qb / q_avg / 1e9, "GB/s", peaks["hbm_gbs"], "hbm"
    elif gemm:
        dom, unit, bound = mm_name, "TFLOP/s", "tensor"
        ach, peak = matmul_flops(M, N, K) / m_avg / 1e12, peaks["bf16_tflops"]
    else:
        dom, ach, unit, peak, bound = mm_name, mb / m_avg / 1e9, "GB/s", peaks["hbm_gbs"], "hbm"
    roofline = {"bound": bound, "kernel": dom, "achieved": ach, "peak": peak, "unit": unit,
                "frac": ach / peak, "peak_source": peak_src,
                "traffic": profiled_traffic(dom, args.workload)}

    # The two further kernels (not part of the step): the symmetric quantizer on the
    # same W copies, and the explicit dequantize of the packed copies into rotating
    # bf16 outputs; same method (CUDA graphs of back-to-back launches, events around
    # `steps` launches per kernel, inputs and outputs rotated over >= 3x L2).
    if not args.no_extra:
        out_bytes = N * K * 2
        co = min(MAX_COPIES, max(2, -(-ROTATE_L2 * l2 // out_bytes)))
        outs = [torch.empty((N, K), dtype=torch.bfloat16, device=dev) for _ in range(co)]

        def time_phase(launch_i, period):
            n = period * max(1, -(-LAUNCHES_PER_GRAPH // period))
            reps, rest = divmod(steps, n)

            def graph_of(count):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=cap):
                    for i in range(count):
                        launch_i(i, cap)
                return g
            g_full = graph_of(n)
            g_rest = graph_of(rest) if rest else None
            g_full.replay()
            torch.cuda.synchronize(dev)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(reps):
                g_full.replay()
            if g_rest is not None:
                g_rest.replay()
            b.record(stream)
            torch.cuda.synchronize(dev)
            return a.elapsed_time(b) / 1e3 / steps

        sym_s = time_phase(lambda i, s_: w4.quantize_pack(Wds[i % cw], out=(qs[i % cm], ss[i % cm], zs[i % cm]),
                                                          stream=s_, symmetric=True), R)
        dq_period = cm * co // math.gcd(cm, co)
        dq_s = time_phase(lambda i, s_: w4.dequantize(qs[i % cm], ss[i % cm], zs[i % cm], dtype=torch.bfloat16,
                                                      out=outs[i % co], stream=s_), dq_period)
        dqb = qsz_bytes + out_bytes
        kernels["quantize_pack_sym"] = {"us": sym_s * 1e6, "bytes": qb, "GB/s": qb / sym_s / 1e9,
                                        "frac_hbm": qb / sym_s / 1e9 / peaks["hbm_gbs"], "launches": steps}
        kernels["dequantize_bf16"] = {"us": dq_s * 1e6, "bytes": dqb, "GB/s": dqb / dq_s / 1e9,
                                      "frac_hbm": dqb / dq_s / 1e9 / peaks["hbm_gbs"], "launches": steps,
                                      "rotation": f"{cm} packed copies, {co} output copies",
                                      "traffic": profiled_traffic("dequantize", args.workload)}
        del outs

    # End to end through the public API with host buffers (pinned), copies inside.
    Wh = torch.from_numpy(W).pin_memory()
    Ah = torch.from_numpy(A.view(np.int16)).pin_memory()
    Yh = torch.empty((M, N), dtype=torch.bfloat16).pin_memory()
    e2e_steps = max(3, min(args.steps, 50))
    h2d = Wh.numel() * Wh.element_size() + Ah.numel() * Ah.element_size()
    d2h = Yh.numel() * Yh.element_size()

    def e2e_step():
        Wd.copy_(Wh, non_blocking=True)
        Ad.view(torch.int16).copy_(Ah, non_blocking=True)
        step()
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
        "steps": steps, "warmup": args.warmup, "ms_per_step": tot_s / steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {
            "workload": f"{args.workload}: {wl.desc}; group 128",
            "N": N, "K": K, "M": M, "group": 128, "w_dtype": wl.w_dtype,
            "step": "w4_quantize_pack + w4_matmul",
            "l2": (f"not serving the timed launches: inputs larger than L2, rotated: {cw} copies of W "
                   f"({cw * w_bytes / 1e6:.0f} MB) for the quantize launches, {cm} copies of the packed "
                   f"weights ({cm * qsz_bytes / 1e6:.0f} MB) for the matmul launches, each set >= "
                   f"{ROTATE_L2}x the {l2 / 2**20:.0f} MiB L2; launch i uses copy i mod C"
                   if l2_defeated else
                   f"tiny workload: {cw} / {cm} rotating copies do not span {ROTATE_L2}x L2 (correctness config)"),
            "timing": (f"CUDA events around {steps} quantize launches, then around {steps} matmul launches "
                       f"(CUDA graphs of {R} launches each; step i's matmul reads what step i's quantize "
                       f"wrote); per-kernel time = phase time / steps"),
            "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
        },
        "roofline": roofline,
        "kernels": kernels,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clocks,
    }
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        rate, desc, _, _ = oracle_sample_rate(args.workload, budget_s=args.cpu_budget,
                                              max_rows=args.cpu_rows)
        result["cpu_baseline"] = {"value": rate, "unit": "GB/s", "cores": 1, "kind": "oracle",
                                  "sample": desc}
    return result


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
                         "sample": desc},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    import synth
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=list(synth.WORKLOADS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--cpu-budget", type=float, default=10.0,
                    help="seconds of CPU time for the oracle baseline")
    ap.add_argument("--cpu-rows", type=int, default=2048,
                    help="rows of W in the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip timing the symmetric quantizer and the explicit dequantize")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
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
