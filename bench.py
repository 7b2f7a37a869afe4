"""Benchmark of the MX quantized linear on one or more GB300s (replicas).

Headline workload: the MXFP8 decode linear N=7168, K=2048 with 32x32-block E8M0
scales, bf16 activations quantized inside each call; one step = one call at each
of M = 1, 4, 16, 32 tokens.  value = algorithmic bytes of the step (weight bytes
+ codes + bf16 x + bf16 out, unpadded K) / device time of the step, summed over
ranks (each rank runs its own replica; there is no data-path collective).

Weights rotate over enough packed copies (> 4x L2) that every call streams its
weight from HBM.  Steps are CUDA-graph replays queued behind a short device
sleep, timed with CUDA events on the launching stream.

Also reported: the roofline of the dominant call (event-timed graph of
back-to-back M=32 calls over the rotated copies), the block-scaled prefill GEMM
M=4096 N=K=7168 in TFLOP/s, the MXFP4 MoE gate/up (E=64, T=64, top-8) in GB/s,
the oracle timed on the host cores (cpu_baseline), and an end-to-end figure
through the Python API with pinned host copies each step.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
"""
import argparse
import ctypes
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

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "MX linear HBM GB/s at M<=32 and block-scaled TFLOPS at M=4096 (1 GB300)"
N_DEC, K_DEC, MS = 7168, 2048, (1, 4, 16, 32)
WORKLOAD = "MXFP8 decode linear N=7168 K=2048, 32x32 E8M0 blocks (codes 118..132), bf16 x N(0,1) quantized per token in the call, M in {1,4,16,32}"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS = 6800.0, 1900.0


def linear_bytes(M, N, K, block=True):
    codes = (N // 32) * (K // 32) if block else N * (K // 32)
    return N * K + codes + 2 * M * K + 2 * M * N


def moe_bytes(D, N, K, T, topk):
    return D * N * (K // 2 + K // 32) + 2 * T * K + 2 * T * topk * N + 4 * T * topk


TRAFFIC_PROFILE = os.path.join(ROOT, "profiles", "gemv_tc_kernel_decode_7168x2048.md")
GEMV_SOURCE = os.path.join(ROOT, "mxfp4_quantized_linear_gb300", "csrc", "gemv_tc.cu")


def profiled_traffic():
    """DRAM bytes (read + write) a gemv_tc_kernel launch of the step moved, averaged
    over the 4 launches of a step, from the committed ncu summary; None when the
    kernel source has changed since that capture."""
    import hashlib
    try:
        text = open(TRAFFIC_PROFILE).read()
        want = hashlib.sha256(open(GEMV_SOURCE, "rb").read()).hexdigest()
    except OSError:
        return None
    sha = traffic = None
    for line in text.splitlines():
        line = line.replace("`", "").strip()
        if line.startswith("source sha256:"):
            sha = line.split(":", 1)[1].strip()
        elif line.startswith("traffic_bytes_per_launch:"):
            traffic = int(line.split(":", 1)[1].strip())
    return traffic if sha == want else None


def peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(ms: float, ws: int, device) -> float:
    """The slowest rank's time: every rank's timed region ends at the same
    barrier, so the job took the maximum."""
    if ws <= 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(ws: int, bytes_per_rank_step: int, ms_step: float) -> float:
    """Whole-job GB/s: every rank streams its own replica's bytes each step
    (weak scaling: the work per GPU is fixed as the GPU count grows)."""
    return ws * bytes_per_rank_step / (ms_step * 1e-3) / 1e9


# ------------------------------------------------------------------- clocks

REASON_BITS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
               0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
               0x100: "display_clocks_setting"}


class ClockSampler:
    """SM clock and clock-event (throttle) reasons sampled while the timed
    region runs: NVML through ctypes every millisecond (read-only queries),
    else nvidia-smi every 50 ms.  Nothing here changes a GPU setting."""

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.samples = []
        self._stop = threading.Event()
        self._thread = None

    def _nvml(self):
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return None
            h = ctypes.c_void_p()
            found = False
            try:  # the NVML device of this CUDA device, by PCI address
                pr = torch.cuda.get_device_properties(self.index)
                bus = f"{pr.pci_domain_id:08x}:{pr.pci_bus_id:02x}:{pr.pci_device_id:02x}.0"
                found = lib.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(h)) == 0
            except Exception:
                found = False
            if not found:
                found = lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.index), ctypes.byref(h)) == 0
            if not found:
                return None
            reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                lib.nvmlDeviceGetCurrentClocksThrottleReasons
            return lib, h, reasons
        except Exception:
            return None

    def _loop(self, lib, h, reasons):
        NVML_CLOCK_SM = 1
        cur, mx, r = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        if lib.nvmlDeviceGetMaxClockInfo(h, NVML_CLOCK_SM, ctypes.byref(mx)) != 0:
            mx.value = 0
        while not self._stop.is_set():
            if lib.nvmlDeviceGetClockInfo(h, NVML_CLOCK_SM, ctypes.byref(cur)) == 0 and \
                    reasons(h, ctypes.byref(r)) == 0:
                self.samples.append((float(cur.value), float(mx.value), int(r.value)))
            time.sleep(0.001)

    def __enter__(self):
        nv = self._nvml()
        if nv is not None:
            self._thread = threading.Thread(target=self._loop, args=nv, daemon=True)
            self._thread.start()
            while not self.samples and self._thread.is_alive():  # the first sample precedes the region
                time.sleep(0.001)
            return self
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index),
                 "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.active",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self._thread is not None:
            self._stop.set()
            self._thread.join(timeout=5)
            return
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                return
            for l in out.splitlines():
                parts = [p.strip() for p in l.split(",")]
                try:
                    self.samples.append((float(parts[0]), float(parts[1]), int(parts[2], 16)))
                except Exception:
                    continue

    def summary(self):
        sm = [c for c, _, _ in self.samples]
        mx = [m for _, m, _ in self.samples if m > 0]
        reasons = set()
        for _, _, bits in self.samples:
            for b, name in REASON_BITS.items():
                if bits & b and name != "gpu_idle":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm),
                "source": "nvml" if self._thread is not None else "nvidia-smi"}


# ------------------------------------------------------------------- our arm

def run_ours(args, ws, rank, local):
    import mxfp4_quantized_linear_gb300 as mx
    from mxfp4_quantized_linear_gb300 import inputs

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    lib = mx.load_library()
    _ = lib
    stream = torch.cuda.Stream(dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    # ---- weights: one packed copy per rotation slot, > 4x L2 in total
    c = inputs.decode_linear(K=K_DEC, Ms=MS, N=N_DEC)
    wdev, cdev = c["w"].to(dev), c["codes"].to(dev)
    per_copy = mx.mx_pack_size("e4m3", 1, N_DEC, K_DEC)
    ncopies = max(8, -(-4 * l2 // per_copy))
    ncopies = -(-ncopies // len(MS)) * len(MS)
    with torch.cuda.stream(stream):
        packed = [mx.mx_pack_weights(wdev, cdev, "e4m3") for _ in range(ncopies)]
    xs = {M: c["xs"][M].to(dev) for M in MS}
    outs = {M: torch.empty((M, N_DEC), dtype=torch.bfloat16, device=dev) for M in MS}
    wsz = max(mx.mxfp8_linear_workspace_size(M, packed[0]) for M in MS)
    work = torch.empty(max(wsz, 256), dtype=torch.uint8, device=dev)
    step_bytes = sum(linear_bytes(M, N_DEC, K_DEC, True) for M in MS)
    kernels_per_step = len(MS)  # one gemv_tc_kernel launch a call (M <= 32)

    def call(M, w):
        mx.mxfp8_linear(xs[M], w, out=outs[M], workspace=work)

    # ---- graphs of whole steps (4 calls on 4 different weight copies each;
    # step s uses rotation slot s % nslots).  The timed steps run as ONE graph
    # of exactly --steps steps, so every step boundary overlaps through
    # programmatic dependent launch the same way whatever the step count; past
    # CHUNK steps a CHUNK-step graph (a multiple of the rotation, so slots
    # continue across replays) is replayed and a remainder graph ends the run.
    nslots = ncopies // len(MS)
    CHUNK = nslots * max(1, 1800 // nslots)

    def capture(n_steps):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for s in range(n_steps):
                for i, M in enumerate(MS):
                    call(M, packed[(s % nslots) * len(MS) + i])
        return g

    with torch.cuda.stream(stream):
        for M in MS:  # warm up (PDL / cluster launch set-up) before capture
            call(M, packed[0])
        torch.cuda.synchronize()
        g_warm = capture(args.warmup)
        q, r = divmod(args.steps, CHUNK) if args.steps > CHUNK else (0, args.steps)
        g_chunk = capture(CHUNK) if q else None
        g_rest = capture(r) if r else None
    torch.cuda.synchronize()

    def timed_steps():
        for _ in range(q):
            g_chunk.replay()
        if g_rest is not None:
            g_rest.replay()

    def barrier():
        if ws > 1:
            torch.distributed.barrier()

    with torch.cuda.stream(stream):
        g_warm.replay()
    torch.cuda.synchronize()
    # ---- timed region
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev.index if dev.index is not None else 0) as clk:
        with torch.cuda.stream(stream):
            torch.cuda._sleep(int(2e6))  # keep the queue ahead of the device
            e0.record(stream)
            timed_steps()
            e1.record(stream)
        torch.cuda.synchronize()
    barrier()
    ms_total = max_over_ranks(e0.elapsed_time(e1), ws, dev)
    ms_step = ms_total / args.steps
    value = job_throughput(ws, step_bytes, ms_step)

    # ---- roofline of the dominant (and only) kernel of the step, gemv_tc_kernel:
    # algorithmic bytes of a launch (averaged over its 4 launches a step) over
    # its average launch duration in the timed region, on this rank
    hbm_peak, bf16_peak, peak_kind = peaks()
    launch_ms = ms_step / kernels_per_step
    achieved = (step_bytes / kernels_per_step) / (launch_ms * 1e-3) / 1e9
    # context: each M alone, back-to-back over the rotated copies
    per_m = {}
    for M in MS:
        gm = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(gm, stream=stream):
                for w in packed:
                    call(M, w)
            gm.replay()
            torch.cuda.synchronize()
            torch.cuda._sleep(int(1e6))
            e0.record(stream)
            gm.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        t = e0.elapsed_time(e1) / ncopies
        per_m[str(M)] = {"us_per_call": round(t * 1e3, 3),
                         "GB/s": round(linear_bytes(M, N_DEC, K_DEC, True) / (t * 1e-3) / 1e9, 1)}
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                "frac": round(achieved / hbm_peak, 4), "traffic": profiled_traffic(),
                "kernel": "gemv_tc_kernel (in-kernel activation quant + tcgen05 split-K GEMV), "
                          f"{kernels_per_step} launches a step, {step_bytes // kernels_per_step} "
                          "algorithmic bytes a launch on average",
                "peak_source": f"{peak_kind} HBM copy bandwidth", "per_call": per_m}

    result = {"metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": ws,
              "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 6),
              "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3",
              "data": "synthetic",
              "config": {"workload": WORKLOAD, "N": N_DEC, "K": K_DEC, "Ms": list(MS),
                         "l2": f"weights rotated over {ncopies} packed copies "
                               f"({ncopies * per_copy / 1e6:.0f} MB > 4x L2 {l2 / 1e6:.0f} MB)",
                         "graph": f"timed steps in one graph of exactly {args.steps} steps"
                                  if args.steps <= CHUNK else
                                  f"timed steps as {q} replays of a {CHUNK}-step graph + {r}",
                         "parallelism": f"replicas x{ws}"},
              "roofline": roofline, "gpu_launches": kernels_per_step * args.steps,
              "clocks": clk.summary()}
    if rank == 0 and not args.no_extras:
        with ClockSampler(dev.index if dev.index is not None else 0) as clk_x:
            result["mxf8_peak"] = mx_peak(mx, stream)
            mx8 = result["mxf8_peak"]["TFLOP/s"]
            result["gemm_m4096"] = bench_prefill(mx, inputs, dev, stream, bf16_peak, peak_kind, mx8)
            result["moe_gate_up"] = bench_moe(mx, inputs, dev, stream, hbm_peak)
            result["moe_expert"] = bench_expert(mx, inputs, dev, stream, hbm_peak)
            result["moe_w4a8_prefill"] = bench_w4a8(mx, inputs, dev, stream, bf16_peak, peak_kind, mx8)
            result["configs"] = bench_configs(mx, inputs, dev, stream, hbm_peak, bf16_peak, peak_kind)
        result["extras_clocks"] = clk_x.summary()
        result["e2e"] = bench_e2e(mx, packed, dev, stream, args)
    del g_warm, g_chunk, g_rest
    return result


def mx_peak(mx, stream):
    """The dense MXFP8 tensor peak measured now, on this GPU: every SM runs a
    block-scaled tcgen05 MMA-only loop (burst: 5 launches of about 1 ms)."""
    with torch.cuda.stream(stream):
        tf = mx.mx_measure_mxf8_peak(iters=2000, reps=5)
    return {"TFLOP/s": round(tf, 1), "how": "tcgen05.mma kind::mxf8f6f4 block_scale (M=128 N=224 K=32, e4m3 "
            "operands in shared memory) from two issuing threads on every SM, 5 x 1 ms launches, CUDA events"}


def bench_prefill(mx, inputs, dev, stream, bf16_peak, peak_kind, mx8_peak=None):
    c = inputs.prefill_gemm()
    x = c["x"].to(dev)
    wd, cd = c["w"].to(dev), c["codes"].to(dev)
    with torch.cuda.stream(stream):
        ws = [mx.mx_pack_weights(wd, cd, "e4m3") for _ in range(4)]
        out = torch.empty((4096, 7168), dtype=torch.bfloat16, device=dev)
        work = torch.empty(mx.mxfp8_linear_workspace_size(4096, ws[0]), dtype=torch.uint8, device=dev)
        for w in ws:
            mx.mxfp8_linear(x, w, out=out, workspace=work)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 8
        e0.record(stream)
        for r in range(reps):
            mx.mxfp8_linear(x, ws[r % 4], out=out, workspace=work)
        e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    flops = 2.0 * 4096 * 7168 * 7168
    tf = flops / (ms * 1e-3) / 1e12
    return {"workload": "MXFP8 prefill GEMM M=4096 N=7168 K=7168, x quantized in the call",
            "ms": round(ms, 4), "TFLOP/s": round(tf, 1),
            "frac_tensor": round(tf / mx8_peak, 4) if mx8_peak else None,
            "peak_source": "dense MXFP8 peak measured in this run (mxf8_peak)",
            "frac_2x_bf16": round(tf / (2 * bf16_peak), 4),
            "note": f"frac_2x_bf16: against 2 x the {peak_kind} bf16 dense peak (nominal 8-bit ratio)"}


def bench_linear_shape(mx, inputs, dev, stream, hbm_peak, N, K, M):
    """One MXFP8 linear shape, graph-timed: calls back to back over packed
    weight copies rotated past 4x L2 (us a call, GB/s of algorithmic bytes)."""
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    c = inputs.decode_linear(K=K, Ms=(M,), N=N)
    wd, cd = c["w"].to(dev), c["codes"].to(dev)
    ncopies = max(4, -(-4 * l2 // mx.mx_pack_size("e4m3", 1, N, K)))
    with torch.cuda.stream(stream):
        packed = [mx.mx_pack_weights(wd, cd, "e4m3") for _ in range(ncopies)]
    x = c["xs"][M].to(dev)
    out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    work = torch.empty(max(256, mx.mxfp8_linear_workspace_size(M, packed[0])), dtype=torch.uint8, device=dev)
    fns = [lambda i=i: mx.mxfp8_linear(x, packed[i % ncopies], out=out, workspace=work) for i in range(2 * ncopies)]
    ms = graph_ms(stream, fns)
    b = linear_bytes(M, N, K, True)
    return {"workload": f"MXFP8 linear N={N} K={K} M={M}, 32x32 codes", "us": round(ms * 1e3, 3),
            "GB/s": round(b / (ms * 1e-3) / 1e9, 1), "frac_hbm": round(b / (ms * 1e-3) / 1e9 / hbm_peak, 4),
            "TFLOP/s": round(2.0 * M * N * K / (ms * 1e-3) / 1e12, 1)}


def bench_moe(mx, inputs, dev, stream, hbm_peak):
    m = inputs.moe_gate_up()
    with torch.cuda.stream(stream):
        p = mx.mx_pack_weights(m["w"].to(dev), m["codes"].to(dev), "e2m1")
        x, ids = m["x"].to(dev), m["ids"].to(dev)
        out = torch.empty((64, 8, 4096), dtype=torch.bfloat16, device=dev)
        work = torch.empty(mx.mxfp4_moe_workspace_size(64, 8, 64, 4096, 4096), dtype=torch.uint8, device=dev)
        for _ in range(3):
            mx.mxfp4_moe_linear(x, ids, p, out=out, workspace=work)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 10
        e0.record(stream)
        for _ in range(reps):
            mx.mxfp4_moe_linear(x, ids, p, out=out, workspace=work)
        e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    D = int(torch.unique(m["ids"]).numel())
    b = moe_bytes(D, 4096, 4096, 64, 8)
    gbs = b / (ms * 1e-3) / 1e9
    return {"workload": "MXFP4 A16W4 MoE gate/up E=64 N=4096 K=4096 T=64 top-8 (weights 0.5 GB > L2)",
            "ms": round(ms, 4), "GB/s": round(gbs, 1), "frac_hbm": round(gbs / hbm_peak, 4),
            "experts_touched": D}


def bench_expert(mx, inputs, dev, stream, hbm_peak):
    """The full routed expert (gate/up + SiLU-and-mul, down projection, combine),
    E=64 I=2048 H=4096 T=64 top-8, graph-replayed back to back."""
    E, I, H, T, topk = 64, 2048, 4096, 64, 8
    m = inputs.moe_expert(E=E, I=I, H=H, T=T, topk=topk)
    reps = 10
    with torch.cuda.stream(stream):
        w13 = mx.mx_pack_weights(m["w13"].to(dev), m["c13"].to(dev), "e2m1", mx.MX_PACK_GATE_UP)
        w2 = mx.mx_pack_weights(m["w2"].to(dev), m["c2"].to(dev), "e2m1", 0)
        x, ids, wts = m["x"].to(dev), m["ids"].to(dev), m["weights"].to(dev)
        out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        work = torch.empty(mx.mxfp4_moe_expert_workspace_size(T, topk, E, H, I, H), dtype=torch.uint8, device=dev)
        for _ in range(3):
            mx.mxfp4_moe_expert(x, ids, wts, w13, w2, out=out, workspace=work)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(reps):
                mx.mxfp4_moe_expert(x, ids, wts, w13, w2, out=out, workspace=work)
        g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(int(1e6))
        e0.record(stream)
        g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    D = int(torch.unique(m["ids"]).numel())
    b = D * (2 * I * (H // 2 + H // 32) + H * (I // 2 + I // 32)) + 2 * T * H * 2 + 8 * T * topk
    gbs = b / (ms * 1e-3) / 1e9
    del g
    return {"workload": "MXFP4 routed expert E=64 I=2048 H=4096 T=64 top-8: gate/up + SiLU-and-mul, "
                        "down projection, top-k combine", "ms": round(ms, 4), "GB/s": round(gbs, 1),
            "frac_hbm": round(gbs / hbm_peak, 4), "experts_touched": D}


def bench_w4a8(mx, inputs, dev, stream, bf16_peak, peak_kind, mx8_peak=None):
    """The routed expert GEMM with MXFP8 activations (MXFP4 x MXFP8, the prefill
    form): E=64 N=4096 K=4096, T=4096 tokens top-8, TFLOP/s against twice the
    bf16 dense peak (the nominal 8-bit ratio)."""
    E, N, K, T, topk = 64, 4096, 4096, 4096, 8
    m = inputs.moe_gate_up(E=E, N=N, K=K, T=T, topk=topk, seed=3, device=dev)
    torch.cuda.synchronize()  # drawn on the default stream; packed and used on `stream`
    with torch.cuda.stream(stream):
        p = mx.mx_pack_weights(m["w"], m["codes"], "e2m1")
        out = torch.empty((T, topk, N), dtype=torch.bfloat16, device=dev)
        work = torch.empty(mx.mxfp4_moe_workspace_size(T, topk, E, N, K), dtype=torch.uint8, device=dev)
        for _ in range(2):
            mx.mxfp4_moe_linear_w4a8(m["x"], m["ids"], p, out=out, workspace=work)
        torch.cuda.synchronize()
        reps = 5
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(int(1e6))
        e0.record(stream)
        for _ in range(reps):
            mx.mxfp4_moe_linear_w4a8(m["x"], m["ids"], p, out=out, workspace=work)
        e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    tflops = 2.0 * T * topk * N * K / (ms * 1e-3) / 1e12
    peak8 = 2.0 * bf16_peak
    del p, m, out, work
    return {"workload": "MXFP4 x MXFP8 routed expert GEMM E=64 N=4096 K=4096 T=4096 top-8 "
                        "(activations quantized per token in the call)",
            "ms": round(ms, 4), "TFLOP/s": round(tflops, 1),
            "frac_tensor": round(tflops / mx8_peak, 4) if mx8_peak else None,
            "peak_source": "dense MXFP8 peak measured in this run (mxf8_peak)",
            "frac_2x_bf16": round(tflops / peak8, 4),
            "note": f"frac_2x_bf16: against 2 x the {peak_kind} bf16 dense peak (nominal 8-bit ratio)"}


def graph_ms(stream, fns, reps=5):
    """Median over ``reps`` replays of one graph holding every call of ``fns``
    back to back, divided by the number of calls (ms a call).  Each replay is
    queued behind a short device sleep and timed with CUDA events on
    ``stream``."""
    with torch.cuda.stream(stream):
        for f in fns[:2]:
            f()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for f in fns:
                f()
        g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        times = []
        for _ in range(reps):
            torch.cuda._sleep(int(1e6))
            e0.record(stream)
            g.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1) / len(fns))
    del g
    return statistics.median(times)


def bench_configs(mx, inputs, dev, stream, hbm_peak, bf16_peak, peak_kind):
    """The other workloads of the layer, each timed as a graph of back-to-back
    calls whose weights (or routed experts) rotate over more than 4x L2:
    the small GEMV M=1 N=512 K=1024 with 1x32 row codes; the decode linear at
    K=2080 (K % 128 != 0, padded) for M = 1 and 32; the sweep linears N=24576
    K=1536 and N=7168 K=8192 at M = 1, 32 and 256; the sweep experts E=256
    N=4096 K=7168 top-8 at T = 1, 8, 64 and 256 (A16W4), the top-k ids
    rotating over 16 draws so consecutive calls touch different experts."""
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    lines = []

    def linear_lines(name, c, Ms, block):
        N, K = c["N"], c["K"]
        wd, cd = c["w"].to(dev), c["codes"].to(dev)
        per_copy = mx.mx_pack_size("e4m3", 1, N, K)
        ncopies = max(8, -(-4 * l2 // per_copy))
        with torch.cuda.stream(stream):
            packed = [mx.mx_pack_weights(wd, cd, "e4m3") for _ in range(ncopies)]
        calls = max(ncopies, 64)
        work = torch.empty(max(256, max(mx.mxfp8_linear_workspace_size(M, packed[0]) for M in Ms)),
                           dtype=torch.uint8, device=dev)
        for M in Ms:
            x = c["xs"][M].to(dev) if "xs" in c else c["x"][:M].to(dev)
            out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            fns = [lambda w=packed[i % ncopies]: mx.mxfp8_linear(x, w, out=out, workspace=work)
                   for i in range(calls)]
            ms = graph_ms(stream, fns)
            b = linear_bytes(M, N, K, block)
            gbs = b / (ms * 1e-3) / 1e9
            line = {"workload": f"{name} M={M} N={N} K={K}", "us_per_call": round(ms * 1e3, 3),
                    "GB/s": round(gbs, 1), "frac_hbm": round(gbs / hbm_peak, 4),
                    "path": "decode GEMV" if M <= 32 else "block-scaled GEMM",
                    "l2": f"{ncopies} weight copies, {ncopies * per_copy / 1e6:.0f} MB"}
            if M > 32:
                tf = 2.0 * M * N * K / (ms * 1e-3) / 1e12
                line["TFLOP/s"] = round(tf, 1)
            lines.append(line)
        del packed, work

    linear_lines("MXFP8 GEMV, 1x32 row codes 120..130", inputs.gemv_small(), (1,), False)
    linear_lines("MXFP8 decode linear, 32x32 codes, K padded to 2176",
                 inputs.decode_linear(K=2080, Ms=(1, 32)), (1, 32), True)
    linear_lines("MXFP8 sweep linear, 32x32 codes", inputs.decode_linear(K=1536, Ms=(1, 32, 256), N=24576),
                 (1, 32, 256), True)
    linear_lines("MXFP8 sweep linear, 32x32 codes", inputs.decode_linear(K=8192, Ms=(1, 32, 256), N=7168),
                 (1, 32, 256), True)

    lines += bench_sweep_experts(mx, inputs, dev, stream, hbm_peak, (1, 8, 64, 256))
    torch.cuda.empty_cache()
    return lines


def bench_sweep_experts(mx, inputs, dev, stream, hbm_peak, Ts):
    """The sweep experts E=256 N=4096 K=7168 top-8 (A16W4) at the token counts
    Ts, each timed as a graph of 32 back-to-back calls whose top-k ids rotate
    over 16 draws, so consecutive calls touch different experts."""
    lines = []
    E, N, K, topk = 256, 4096, 7168, 8
    m = inputs.moe_gate_up(E=E, N=N, K=K, T=max(Ts), topk=topk, device=dev)
    torch.cuda.synchronize()  # drawn on the default stream; packed and used on `stream`
    with torch.cuda.stream(stream):
        p = mx.mx_pack_weights(m["w"], m["codes"], "e2m1")
    del m["w"], m["codes"]
    g = inputs.generator(77, dev)
    nsets = 16
    id_sets = [inputs.topk_ids(max(Ts), E, topk, g) for _ in range(nsets)]
    torch.cuda.synchronize()
    for T in Ts:
        x = m["x"][:T].contiguous()
        ids = [s_[:T].contiguous() for s_ in id_sets]
        out = torch.empty((T, topk, N), dtype=torch.bfloat16, device=dev)
        work = torch.empty(mx.mxfp4_moe_workspace_size(T, topk, E, N, K), dtype=torch.uint8, device=dev)
        fns = [lambda i=i: mx.mxfp4_moe_linear(x, ids[i % nsets], p, out=out, workspace=work)
               for i in range(2 * nsets)]
        ms = graph_ms(stream, fns)
        D = statistics.mean(int(torch.unique(i_).numel()) for i_ in ids)
        b = moe_bytes(D, N, K, T, topk)
        gbs = b / (ms * 1e-3) / 1e9
        lines.append({"workload": f"MXFP4 A16W4 sweep experts E={E} N={N} K={K} T={T} top-{topk}",
                      "us_per_call": round(ms * 1e3, 3), "GB/s": round(gbs, 1),
                      "frac_hbm": round(gbs / hbm_peak, 4), "experts_touched": round(D, 2),
                      "l2": f"top-k ids rotate over {nsets} draws"})
    del p
    return lines


def bench_e2e(mx, packed, dev, stream, args):
    """The step through the public API: pinned host x -> device, the 4 calls, out ->
    pinned host, one stream synchronize a step.  ``value``: plain eager calls; ``graph``: the same
    step (copies included) captured once in a CUDA graph and replayed each step, the
    way a decode loop drives it, with each call's output copied back on a side
    stream while the later calls run (largest output first)."""
    # one pinned buffer holds the 4 inputs (and one the 4 outputs): a step moves
    # them with one host->device and one device->host copy
    rows = sum(MS)
    in_host = torch.randn((rows, K_DEC), generator=torch.Generator().manual_seed(1)).to(torch.bfloat16).pin_memory()
    out_host = torch.empty((rows, N_DEC), dtype=torch.bfloat16).pin_memory()
    in_dev = torch.empty((rows, K_DEC), dtype=torch.bfloat16, device=dev)
    out_dev = torch.empty((rows, N_DEC), dtype=torch.bfloat16, device=dev)
    offs = [sum(MS[:i]) for i in range(len(MS))]
    x_dev = {M: in_dev[o:o + M] for o, M in zip(offs, MS)}
    o_dev = {M: out_dev[o:o + M] for o, M in zip(offs, MS)}
    work = torch.empty(max(mx.mxfp8_linear_workspace_size(M, packed[0]) for M in MS) + 256, dtype=torch.uint8,
                       device=dev)
    n = max(20, min(args.steps, 500))
    h2d = in_host.numel() * 2
    d2h = out_host.numel() * 2
    nslots = len(packed) // len(MS)

    # each call's output goes back on a side stream as soon as it is ready,
    # the largest first, so only the last (smallest) copy follows the last kernel
    copy_stream = torch.cuda.Stream(dev)
    order = sorted(range(len(MS)), key=lambda i: -MS[i])
    o_host = {M: out_host[o:o + M] for o, M in zip(offs, MS)}
    done = [torch.cuda.Event() for _ in MS]

    def enqueue(s):
        # eager: one copy in, the 4 calls, one copy out (per-call stream and event
        # bookkeeping in Python would cost more than the overlap gains)
        in_dev.copy_(in_host, non_blocking=True)
        for i, M in enumerate(MS):
            mx.mxfp8_linear(x_dev[M], packed[(s % nslots) * len(MS) + i], out=o_dev[M], workspace=work)
        out_host.copy_(out_dev, non_blocking=True)

    def enqueue_overlapped(s):
        # captured once in a graph: each output goes back while the later calls run
        in_dev.copy_(in_host, non_blocking=True)
        for i in order:
            M = MS[i]
            mx.mxfp8_linear(x_dev[M], packed[(s % nslots) * len(MS) + i], out=o_dev[M], workspace=work)
            done[i].record(stream)
            copy_stream.wait_event(done[i])
            with torch.cuda.stream(copy_stream):
                o_host[M].copy_(o_dev[M], non_blocking=True)
        stream.wait_stream(copy_stream)  # the step ends when every output is on the host

    with torch.cuda.stream(stream):
        for s in range(5):
            enqueue(s)
            stream.synchronize()
        t0 = time.perf_counter()
        for s in range(n):
            enqueue(s)
            stream.synchronize()
        t1 = time.perf_counter()
        graphs = []
        for s in range(nslots):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                enqueue_overlapped(s)
            graphs.append(g)
        for s in range(5):
            graphs[s % nslots].replay()
            stream.synchronize()
        t2 = time.perf_counter()
        for s in range(n):
            graphs[s % nslots].replay()
            stream.synchronize()
        t3 = time.perf_counter()
    del graphs
    step_bytes = sum(linear_bytes(M, N_DEC, K_DEC, True) for M in MS)
    sec, sec_g = (t1 - t0) / n, (t3 - t2) / n
    return {"value": round(step_bytes / sec / 1e9, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": round(sec * 1e3, 4), "steps": n,
            "graph": {"value": round(step_bytes / sec_g / 1e9, 1), "unit": "GB/s",
                      "ms_per_step": round(sec_g * 1e3, 4)}}


def bench_sweep(mx, inputs, dev, stream, hbm_peak, bf16_peak):
    """The shape sweep: MXFP8 linears N=24576 K=1536 and N=7168 K=8192 at M = 1..256
    (M <= 32 on the decode GEMV, larger M on the block-scaled GEMM), and the MXFP4 MoE
    E=256 N=4096 K=7168 top-8 at T = 1..256.  Weights rotate over > 4x L2 of copies
    (one 3.8 GB expert tensor already is); per-call time = graph time / calls."""
    Ms = (1, 2, 4, 8, 16, 32, 64, 128, 256)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    lines = []

    def timed(fn, calls):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            fn()
            torch.cuda.synchronize()
            with torch.cuda.graph(g, stream=stream):
                for i in range(calls):
                    fn(i)
            g.replay()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            times = []
            for _ in range(5):
                torch.cuda._sleep(int(1e6))
                e0.record(stream)
                g.replay()
                e1.record(stream)
                torch.cuda.synchronize()
                times.append(e0.elapsed_time(e1) / calls)
        return statistics.median(times)

    for (N, K) in ((24576, 1536), (7168, 8192)):
        c = inputs.decode_linear(K=K, Ms=Ms, N=N)
        wd, cd = c["w"].to(dev), c["codes"].to(dev)
        per_copy = mx.mx_pack_size("e4m3", 1, N, K)
        ncopies = max(4, -(-4 * l2 // per_copy))
        with torch.cuda.stream(stream):
            packed = [mx.mx_pack_weights(wd, cd, "e4m3") for _ in range(ncopies)]
        work = torch.empty(max(256, mx.mxfp8_linear_workspace_size(max(Ms), packed[0])), dtype=torch.uint8,
                           device=dev)
        for M in Ms:
            x = c["xs"][M].to(dev)
            out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            ms = timed(lambda i=0: mx.mxfp8_linear(x, packed[i % ncopies], out=out, workspace=work), 2 * ncopies)
            b = linear_bytes(M, N, K, True)
            fl = 2.0 * M * N * K
            lines.append({"sweep": "mxfp8_linear", "N": N, "K": K, "M": M, "us": round(ms * 1e3, 3),
                          "GB/s": round(b / (ms * 1e-3) / 1e9, 1), "frac_hbm": round(b / (ms * 1e-3) / 1e9 / hbm_peak, 4),
                          "TFLOP/s": round(fl / (ms * 1e-3) / 1e12, 1)})
        del packed, work
    E, N, K, topk = 256, 4096, 7168, 8
    m = inputs.moe_gate_up(E=E, N=N, K=K, T=max(Ms), topk=topk, device=dev)
    torch.cuda.synchronize()  # drawn on the default stream; packed and used on `stream`
    with torch.cuda.stream(stream):
        p = mx.mx_pack_weights(m["w"], m["codes"], "e2m1")
    del m["w"], m["codes"]
    for T in Ms:
        x = m["x"][:T].contiguous()
        ids = m["ids"][:T].contiguous()
        out = torch.empty((T, topk, N), dtype=torch.bfloat16, device=dev)
        work = torch.empty(mx.mxfp4_moe_workspace_size(T, topk, E, N, K), dtype=torch.uint8, device=dev)
        ms = timed(lambda i=0: mx.mxfp4_moe_linear(x, ids, p, out=out, workspace=work), 4)
        D = int(torch.unique(ids).numel())
        b = moe_bytes(D, N, K, T, topk)
        lines.append({"sweep": "mxfp4_moe_linear", "E": E, "N": N, "K": K, "T": T, "topk": topk,
                      "experts_touched": D, "us": round(ms * 1e3, 3), "GB/s": round(b / (ms * 1e-3) / 1e9, 1),
                      "frac_hbm": round(b / (ms * 1e-3) / 1e9 / hbm_peak, 4)})
    return lines


# ------------------------------------------------------------- oracle (CPU)

def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return len(os.sched_getaffinity(0))


def oracle_step(c, rows=None):
    """One step of the workload on the oracle: the four calls, fp64 (on the
    first ``rows`` weight rows only, a multiple of 32, when given)."""
    from oracle.linear import mxfp8_linear as ref_linear
    w = c["w"].numpy()
    codes = c["codes"].numpy()
    if rows is not None:
        w, codes = w[:rows], codes[:rows // 32]
    for M in MS:
        x = c["xs"][M].float().numpy().astype(np.float64)
        ref_linear(x, w, codes)


def reference_rows(N, sec_full, steps, warmup, budget_s=150.0):
    """Weight rows a reference-arm step samples so that warmup + steps of them
    take about budget_s at most: all N when that fits, else the largest
    multiple of 32 that does (at least 32)."""
    total = max(1, steps + warmup) * sec_full
    if total <= budget_s:
        return N
    return max(32, int(N * budget_s / total) // 32 * 32)


def cpu_baseline(steps=1):
    from mxfp4_quantized_linear_gb300 import inputs
    c = inputs.decode_linear(K=K_DEC, Ms=MS, N=N_DEC)
    oracle_step(c)  # warm caches / imports
    t0 = time.perf_counter()
    for _ in range(steps):
        oracle_step(c)
    sec = (time.perf_counter() - t0) / steps
    step_bytes = sum(linear_bytes(M, N_DEC, K_DEC, True) for M in MS)
    return {"value": round(step_bytes / sec / 1e9, 4), "unit": "GB/s", "cores": blas_threads(),
            "kind": "oracle", "sample": f"{steps} full step(s) of the workload (M=1,4,16,32), "
                                        f"{sec:.3f} s per step, numpy fp64 decode + matmul"}


def run_reference(args, ws, rank):
    if rank != 0:
        return None
    from mxfp4_quantized_linear_gb300 import inputs
    c = inputs.decode_linear(K=K_DEC, Ms=MS, N=N_DEC)
    # one full step (the first warm-up) sizes the sample of every later step
    t0 = time.perf_counter()
    oracle_step(c)
    rows = reference_rows(N_DEC, time.perf_counter() - t0, args.steps, args.warmup)
    for _ in range(args.warmup - 1):
        oracle_step(c, rows)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(c, rows)
    sec = (time.perf_counter() - t0) / args.steps
    step_bytes = sum(linear_bytes(M, rows, K_DEC, True) for M in MS)
    v = step_bytes / sec / 1e9
    return {"impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": "GB/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(sec * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": WORKLOAD, "N": N_DEC, "K": K_DEC, "Ms": list(MS)},
            "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": blas_threads(), "kind": "oracle",
                             "sample": f"{args.steps} steps of the workload on the CPU oracle, each on "
                                       f"{rows} of the {N_DEC} weight rows"},
            "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-extras", action="store_true", help="skip the GEMM / MoE / e2e / CPU figures")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sweep", action="store_true",
                    help="print one JSON line per shape of the linear / MoE sweep instead of the step")
    ap.add_argument("--case", default=None,
                    choices=["mxf8_peak", "gemm_m4096", "moe_gate_up", "moe_expert", "moe_w4a8_prefill", "configs",
                             "moe_decode", "linear_n7168_k8192_m64"],
                    help="run only this secondary workload and print its JSON (e.g. to profile one kernel)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    ws, rank, local = dist_env()
    if ws > 1 and args.impl == "ours":
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    if args.impl == "reference":
        res = run_reference(args, ws, rank)
        if res is not None:
            print(json.dumps(res), flush=True)
        return
    if args.case:
        if rank == 0:
            import mxfp4_quantized_linear_gb300 as mx
            from mxfp4_quantized_linear_gb300 import inputs
            dev = torch.device("cuda", local)
            torch.cuda.set_device(dev)
            hbm_peak, bf16_peak, peak_kind = peaks()
            stream = torch.cuda.Stream(dev)
            fns = {"mxf8_peak": lambda: mx_peak(mx, stream),
                   "gemm_m4096": lambda: bench_prefill(mx, inputs, dev, stream, bf16_peak, peak_kind),
                   "moe_gate_up": lambda: bench_moe(mx, inputs, dev, stream, hbm_peak),
                   "moe_expert": lambda: bench_expert(mx, inputs, dev, stream, hbm_peak),
                   "moe_w4a8_prefill": lambda: bench_w4a8(mx, inputs, dev, stream, bf16_peak, peak_kind),
                   "configs": lambda: bench_configs(mx, inputs, dev, stream, hbm_peak, bf16_peak, peak_kind),
                   "moe_decode": lambda: bench_sweep_experts(mx, inputs, dev, stream, hbm_peak, (1,)),
                   "linear_n7168_k8192_m64": lambda: bench_linear_shape(mx, inputs, dev, stream, hbm_peak, 7168,
                                                                        8192, 64)}
            print(json.dumps({args.case: fns[args.case]()}), flush=True)
        return
    if args.sweep:
        if rank == 0:
            import mxfp4_quantized_linear_gb300 as mx
            from mxfp4_quantized_linear_gb300 import inputs
            dev = torch.device("cuda", local)
            torch.cuda.set_device(dev)
            hbm_peak, bf16_peak, _ = peaks()
            for line in bench_sweep(mx, inputs, dev, torch.cuda.Stream(dev), hbm_peak, bf16_peak):
                print(json.dumps(line), flush=True)
        return
    res = run_ours(args, ws, rank, local)
    if rank == 0:
        if not args.no_cpu_baseline and not args.no_extras:
            res["cpu_baseline"] = cpu_baseline()
        print(json.dumps(res), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
