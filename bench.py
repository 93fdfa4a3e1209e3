"""Benchmark of the MoE grouped-matmul hot path on GB300.

One step = one pass of the whole path over the production-shape MoE expert
layer ("GEMM Kernel 性能优化十问", Q6: G=256 experts, M = 2 x 4096 x top-8 =
65536 rows, K = 2048, N = 512):
    1. dynamic 1x128 FP8 quantization of X              (gmm_quantize_lhs)
    2. wi: FP8 blockwise GMM, fused silu(gate)*up -> h, with the 1x128 FP8
       quantization of h fused into its epilogue         (gmm_fp8_fwd_swiglu_quant)
    3. wo: FP8 blockwise GMM on the quantized h -> y     (gmm_fp8_fwd)
    4. wo weight gradient  dW_wo[g] = h_g^T dY_g         (tgmm_bf16)
    5. wi weight gradient  dW_wi[g] = X_g^T dH_g         (tgmm_bf16)
with one device metadata pass per step (group offsets and row tiles) that the
four grouped calls share (they get group_sizes = NULL).  The metric is
TFLOP/s counted as 2*M*K*N per GMM (FLOPs do not depend on precision, Q7),
summed over the four GMMs.  Weights are quantized once, offline, before
timing (128x128 blocks, as the method prescribes for static weights).

Beside the step (not in it) the same FP8 forward launches run with 4-bit E2M1
weights (packed two codes per byte, 128x128 fp32 scales), the bf16 forward of
both layers and the layer's bf16 dgrad.

Inputs are synthetic and seeded: routing from Zipf(1.1) expert popularity
with 8 dead experts, X ~ N(0,1) with 1% x50 outliers, W ~ N(0, 1/K), upstream
gradients ~ N(0,1).  Inputs are resident in HBM before the timed region;
L2 is flushed (a 256 MB write) between timed steps, outside the events.

--impl reference times the CPU oracle instead (a bounded row sample of the
same workload, on the host cores).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "FP8 GMM fwd & bf16 tgmm TFLOPS (2MKN)"
UNIT = "TFLOP/s"
WORKLOAD = ("production MoE expert layer, G=256 M=65536 (8192 tokens x top-8, Zipf(1.1) routing, "
            "8 empty experts): quantize X, FP8 wi K=2048 N=2x512 fused silu*up + FP8 cast of h, "
            "FP8 wo K=512 N=2048, bf16 tgmm dW_wo and dW_wi")
G, M, K, N = 256, 65536, 2048, 512
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_BF16_SUSTAINED = 1700.0


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            hbm = float(d.get("hbm_gbs"))
            bf = float(d.get("bf16_tflops"))
            bfs = float(d.get("bf16_tflops_sustained", bf))
            return dict(hbm_gbs=hbm, bf16=bf, bf16_sustained=bfs, source="measured")
        except Exception:
            pass
    return dict(hbm_gbs=FALLBACK_HBM_GBS, bf16=FALLBACK_BF16_TFLOPS,
                bf16_sustained=FALLBACK_BF16_SUSTAINED, source="fallback")


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}", "--format=csv,noheader",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [c.strip() for c in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1].split()[0]))
                smax.append(float(f[2].split()[0]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        os.unlink(self.path)
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": float(max(smax)) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


def max_over_ranks(value: float, device=None) -> float:
    """Largest value over all ranks (the slowest rank sets the job's time).
    Works on any torch.distributed backend (NCCL with a CUDA device, gloo on
    the CPU); a single process returns the value unchanged."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, flops_per_step: float, steps: int, total_ms_max: float) -> float:
    """Whole-job TFLOP/s: every rank ran `steps` steps of the same (replicated)
    workload; the job took as long as its slowest rank."""
    return world * flops_per_step * steps / (total_ms_max * 1e-3) / 1e12


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# ---------------------------------------------------------------------------
# FLOP and byte accounting (algorithmic: every operand once, output once)
# ---------------------------------------------------------------------------

def accounting(sizes: np.ndarray):
    live = int(np.count_nonzero(sizes))
    Mr = int(sizes.sum())
    f = {}
    b = {}
    # quantize X: read bf16, write e4m3 + fp32 scale per 128
    b["quantize_x"] = M * K * 2 + M * K + M * K // 128 * 4
    f["quantize_x"] = 0
    # wi fused: Xq, xs, live experts' Wq/ws in; h (bf16), hq (e4m3), hs (fp32) out
    f["gmm_fp8_wi"] = 2 * Mr * K * 2 * N
    b["gmm_fp8_wi"] = M * K + M * (K // 128) * 4 + live * K * 2 * N + live * (K // 128) * (2 * N // 128) * 4 \
        + M * N * 2 + M * N + M * (N // 128) * 4 + 4 * G
    f["gmm_fp8_wo"] = 2 * Mr * N * K
    b["gmm_fp8_wo"] = M * N + M * (N // 128) * 4 + live * N * K + live * (N // 128) * (K // 128) * 4 \
        + M * K * 2 + 4 * G
    f["tgmm_wo"] = 2 * Mr * N * K
    b["tgmm_wo"] = M * N * 2 + M * K * 2 + G * N * K * 2 + 4 * G
    f["tgmm_wi"] = 2 * Mr * K * 2 * N
    b["tgmm_wi"] = M * K * 2 + M * 2 * N * 2 + G * K * 2 * N * 2 + 4 * G
    return f, b


# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) from the
# committed ncu captures (profiles/), each valid only for the kernel source it
# was taken on: the SHA-256 of that .cu file is checked at run time and the
# traffic is reported as null once the kernel has changed.
MEASURED_TRAFFIC = {
    "tgmm_wi": {"bytes": 446344704 + 1012759552, "source": "tgmm.cu",
                "sha256": "da199b4f150f06595484317abf091437ea27ac6dcb9d3ab057ed4f5b74758ff0"},
}


def _traffic(kernel):
    import hashlib
    t = MEASURED_TRAFFIC.get(kernel)
    if not t:
        return None
    path = os.path.join(ROOT, "fp8_blockwise_quantized_gb300", "csrc", t["source"])
    try:
        h = hashlib.sha256(open(path, "rb").read()).hexdigest()
    except OSError:
        return None
    return t["bytes"] if h == t["sha256"] else None


KERNEL_KIND = {"quantize_x": "hbm", "gmm_fp8_wi": "fp8", "gmm_fp8_wo": "fp8",
               "tgmm_wo": "bf16", "tgmm_wi": "bf16"}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def run_gpu(args):
    import torch

    ws_, rank, local = _dist()
    if ws_ > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if ws_ > 1 else 0)
    torch.cuda.set_device(dev)

    import fp8_blockwise_quantized_gb300 as gmm
    from fp8_blockwise_quantized_gb300.build import build
    from fp8_blockwise_quantized_gb300.workloads import routing_sizes
    build()
    gmm.load()

    sizes_np = routing_sizes("prod_fp8")
    assert int(sizes_np.sum()) == M
    flops, nbytes = accounting(sizes_np)

    gen = torch.Generator(device=dev)
    gen.manual_seed(1004 + rank)

    def normal(shape, std=1.0, outlier=0.0):
        v = torch.randn(shape, generator=gen, device=dev, dtype=torch.float32)
        if std != 1.0:
            v.mul_(std)
        if outlier:
            m = torch.rand(shape, generator=gen, device=dev) < outlier
            v[m] *= 50.0
        return v.to(torch.bfloat16)

    x = normal((M, K), outlier=0.01)
    w_wi = normal((G, K, 2 * N), 1.0 / math.sqrt(K))
    w_wo = normal((G, N, K), 1.0 / math.sqrt(N))
    dy = normal((M, K))
    dh = normal((M, 2 * N))
    sizes = torch.from_numpy(sizes_np).to(dev)
    stream = torch.cuda.current_stream(dev)

    # offline weight quantization (untimed)
    wq_wi, ws_wi = gmm.quantize_rhs(w_wi)
    wq_wo, ws_wo = gmm.quantize_rhs(w_wo)

    xq = torch.empty((M, K), dtype=torch.uint8, device=dev)
    xs = torch.empty((K // 128, M), dtype=torch.float32, device=dev)
    h = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    hq = torch.empty((M, N), dtype=torch.uint8, device=dev)
    hs = torch.empty((N // 128, M), dtype=torch.float32, device=dev)
    y = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
    dw_wo = torch.empty((G, N, K), dtype=torch.bfloat16, device=dev)
    dw_wi = torch.empty((G, K, 2 * N), dtype=torch.bfloat16, device=dev)
    work = gmm.Workspace(G, M, dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    chk = gmm.binding._check

    names = ["quantize_x", "gmm_fp8_wi", "gmm_fp8_wo", "tgmm_wo", "tgmm_wi"]

    def step(ev=None):
        def mark(i):
            if ev is not None:
                ev[i].record(stream)
        mark(0)
        chk(gmm.gmm_quantize_lhs(x, M, K, xq, xs, stream), "quantize X")
        mark(1)
        # one metadata pass per step (the four grouped calls share the routing;
        # they get group_sizes = NULL and read it from the workspace)
        chk(gmm.gmm_group_metadata(sizes, G, M, work.buf, work.nbytes, stream), "metadata")
        chk(gmm.gmm_fp8_fwd_swiglu_quant(xq, xs, wq_wi, ws_wi, None, G, M, K, N, h, hq, hs, work.buf,
                                         work.nbytes, stream), "wi")
        mark(2)
        chk(gmm.gmm_fp8_fwd(hq, hs, wq_wo, ws_wo, None, G, M, N, K, 0, y, work.buf, work.nbytes,
                            stream), "wo")
        mark(3)
        chk(gmm.tgmm_bf16(h, dy, None, G, M, N, K, dw_wo, work.buf, work.nbytes, stream), "tgmm wo")
        mark(4)
        chk(gmm.tgmm_bf16(x, dh, None, G, M, K, 2 * N, dw_wi, work.buf, work.nbytes, stream),
            "tgmm wi")
        mark(5)

    n_marks = len(names) + 1
    launches_per_step = 6  # 1 quantize + 1 metadata + 2 fp8 GMM + 2 tgmm

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    st = work.status(stream)
    if st != 0:
        raise RuntimeError(f"device status {gmm.STATUS_NAMES.get(st, st)} after warm-up")

    # The timed steps carry events only at their boundaries: an event between
    # two kernels would stop the next one from starting its CTAs while the
    # previous finishes (programmatic dependent launch).  The per-kernel split
    # comes from a second pass below with an event between every call.
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    clocks = Clocks(dev.index if dev.index is not None else 0)
    clocks.start()
    # keep the GPU busy while the sampler starts (its first sample takes ~0.1 s)
    t_pre = time.perf_counter()
    while time.perf_counter() - t_pre < 0.4:
        step()
        torch.cuda.synchronize(dev)
    if ws_ > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for i in range(args.steps):
        flush.zero_()
        events[i][0].record(stream)
        step()
        events[i][1].record(stream)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - t0
    clk = clocks.stop()
    # per-kernel split: a second pass with an event between every call
    n_split = max(10, min(args.steps, 100))
    split_events = [[torch.cuda.Event(enable_timing=True) for _ in range(n_marks)] for _ in range(n_split)]
    for i in range(n_split):
        flush.zero_()
        step(split_events[i])
    torch.cuda.synchronize(dev)
    if ws_ > 1:
        torch.distributed.barrier()
    st = work.status(stream)
    if st != 0:
        raise RuntimeError(f"device status {gmm.STATUS_NAMES.get(st, st)} after timing")

    per_kernel = {n: [] for n in names}
    step_ms = [ev[0].elapsed_time(ev[1]) for ev in events]
    for ev in split_events:
        for j, n in enumerate(names):
            per_kernel[n].append(ev[j].elapsed_time(ev[j + 1]))
    ms = float(np.mean(step_ms))
    total_ms = float(np.sum(step_ms))
    step_dist = {"median": round(float(np.median(step_ms)), 4), "p10": round(float(np.percentile(step_ms, 10)), 4),
                 "p90": round(float(np.percentile(step_ms, 90)), 4)}
    if ws_ > 1:
        total_ms = max_over_ranks(total_ms, dev)
        ms = total_ms / args.steps
    step_flops = sum(flops.values())
    value = job_throughput(ws_, step_flops, args.steps, total_ms)

    peaks = _peaks()
    fp8_peak = 2.0 * peaks["bf16"]
    kern = {}
    for n in names:
        kms = float(np.mean(per_kernel[n]))
        gbs = nbytes[n] / (kms * 1e-3) / 1e9
        entry = {"ms": round(kms, 4), "GB/s": round(gbs, 1), "bytes": nbytes[n],
                 "frac_hbm": round(gbs / peaks["hbm_gbs"], 3)}
        if flops[n]:
            tf = flops[n] / (kms * 1e-3) / 1e12
            pk = fp8_peak if KERNEL_KIND[n] == "fp8" else peaks["bf16"]
            entry.update({"TFLOP/s": round(tf, 1), "flops": flops[n], "frac_tensor_peak": round(tf / pk, 3),
                          "AI": round(flops[n] / nbytes[n], 1)})
        kern[n] = entry
    dom = max(names, key=lambda n: kern[n]["ms"])
    dk = kern[dom]
    if KERNEL_KIND[dom] == "hbm" or dk.get("AI", 0) < (fp8_peak if KERNEL_KIND[dom] == "fp8" else peaks["bf16"]) \
            * 1e12 / (peaks["hbm_gbs"] * 1e9):
        roof = {"bound": "hbm", "achieved": dk["GB/s"], "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(dk["GB/s"] / peaks["hbm_gbs"], 3)}
    else:
        pk = fp8_peak if KERNEL_KIND[dom] == "fp8" else peaks["bf16"]
        roof = {"bound": "tensor", "achieved": dk["TFLOP/s"], "peak": pk, "unit": "TFLOP/s",
                "frac": round(dk["TFLOP/s"] / pk, 3)}
    roof.update({"kernel": dom, "traffic": args.traffic if args.traffic is not None else _traffic(dom),
                 "peak_source": f"of {peaks['source']}",
                 "per_launch_algorithmic_bytes": nbytes[dom]})

    # ---------------- bf16 forward baseline, timed beside the step (not in it)
    bf = {}
    dgrad = None
    if not args.no_bf16_baseline:
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        tb = []
        for i in range(max(3, args.steps)):
            flush.zero_()
            ev[0].record(stream)
            chk(gmm.gmm_bf16_fwd(x, w_wi, sizes, G, M, K, N, 1, h, work.buf, work.nbytes, stream), "bf16 wi")
            ev[1].record(stream)
            chk(gmm.gmm_bf16_fwd(h, w_wo, sizes, G, M, N, K, 0, y, work.buf, work.nbytes, stream), "bf16 wo")
            ev[2].record(stream)
            torch.cuda.synchronize(dev)
            if i >= 1:
                tb.append((ev[0].elapsed_time(ev[1]), ev[1].elapsed_time(ev[2])))
        wi_ms = float(np.mean([a for a, _ in tb]))
        wo_ms = float(np.mean([b for _, b in tb]))
        fp8_ms = kern["gmm_fp8_wi"]["ms"] + kern["gmm_fp8_wo"]["ms"]
        q_ms = kern["quantize_x"]["ms"]
        bf = {"wi_ms": round(wi_ms, 4), "wo_ms": round(wo_ms, 4),
              "wi_TFLOP/s": round(flops["gmm_fp8_wi"] / (wi_ms * 1e-3) / 1e12, 1),
              "wo_TFLOP/s": round(flops["gmm_fp8_wo"] / (wo_ms * 1e-3) / 1e12, 1),
              "fp8_over_bf16_gmm_only": round((wi_ms + wo_ms) / fp8_ms, 3),
              "fp8_over_bf16_with_quantize": round((wi_ms + wo_ms) / (fp8_ms + q_ms), 3)}

        # the layer's bf16 data gradients beside the step (not in it):
        # dH = dY . W_wo[g]^T and dX = d(gate|up) . W_wi[g]^T
        tdg = []
        for i in range(max(3, args.steps)):
            flush.zero_()
            ev[0].record(stream)
            chk(gmm.gmm_bf16_dgrad(dy, w_wo, sizes, G, M, N, K, h, work.buf, work.nbytes, stream), "dgrad dH")
            ev[1].record(stream)
            chk(gmm.gmm_bf16_dgrad(dh, w_wi, sizes, G, M, K, 2 * N, y, work.buf, work.nbytes, stream), "dgrad dX")
            ev[2].record(stream)
            torch.cuda.synchronize(dev)
            if i >= 1:
                tdg.append((ev[0].elapsed_time(ev[1]), ev[1].elapsed_time(ev[2])))
        dh_ms = float(np.mean([a for a, _ in tdg]))
        dx_ms = float(np.mean([b for _, b in tdg]))
        bf_peak = peaks["bf16"]
        dgrad = {"dH_ms": round(dh_ms, 4), "dX_ms": round(dx_ms, 4),
                 "dH_TFLOP/s": round(flops["gmm_fp8_wo"] / (dh_ms * 1e-3) / 1e12, 1),
                 "dX_TFLOP/s": round(flops["gmm_fp8_wi"] / (dx_ms * 1e-3) / 1e12, 1),
                 "frac_bf16_peak": round((flops["gmm_fp8_wo"] + flops["gmm_fp8_wi"]) /
                                         ((dh_ms + dx_ms) * 1e-3) / 1e12 / bf_peak, 3),
                 "note": "bf16 dgrad of the layer (dY . W_wo^T, d(gate|up) . W_wi^T), timed beside the step"}

    # ---------------- 4-bit (E2M1) weights, timed beside the step (not in it):
    # the same fused wi (writing h and its FP8 cast) and wo with the weights
    # packed two codes per byte, against the e4m3 launches of the step
    w4 = None
    if not args.no_w4:
        wq4_wi, ws4_wi = gmm.quantize_rhs_w4(w_wi)   # offline, untimed
        wq4_wo, ws4_wo = gmm.quantize_rhs_w4(w_wo)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        chk(gmm.gmm_group_metadata(sizes, G, M, work.buf, work.nbytes, stream), "metadata")
        t4 = []
        for i in range(max(3, min(args.steps, 100))):
            flush.zero_()
            ev[0].record(stream)
            chk(gmm.gmm_fp8_w4_fwd_swiglu_quant(xq, xs, wq4_wi, ws4_wi, None, G, M, K, N, h, hq, hs, work.buf,
                                                work.nbytes, stream), "w4 wi")
            ev[1].record(stream)
            chk(gmm.gmm_fp8_w4_fwd(hq, hs, wq4_wo, ws4_wo, None, G, M, N, K, 0, y, work.buf, work.nbytes, stream),
                "w4 wo")
            ev[2].record(stream)
            torch.cuda.synchronize(dev)
            if i >= 1:
                t4.append((ev[0].elapsed_time(ev[1]), ev[1].elapsed_time(ev[2])))
        st4 = work.status(stream)
        if st4 != 0:
            raise RuntimeError(f"device status {gmm.STATUS_NAMES.get(st4, st4)} after the 4-bit weight runs")
        live = int(np.count_nonzero(sizes_np))
        w4_bytes = {"wi": nbytes["gmm_fp8_wi"] - live * K * 2 * N // 2,
                    "wo": nbytes["gmm_fp8_wo"] - live * N * K // 2}
        w4 = {}
        for j, nm in enumerate(("wi", "wo")):
            ms4 = float(np.mean([t[j] for t in t4]))
            ref = kern[f"gmm_fp8_{nm}"]
            w4[nm] = {"ms": round(ms4, 4), "bytes": w4_bytes[nm],
                      "GB/s": round(w4_bytes[nm] / (ms4 * 1e-3) / 1e9, 1),
                      "TFLOP/s": round(flops[f"gmm_fp8_{nm}"] / (ms4 * 1e-3) / 1e12, 1),
                      "e4m3_ms": ref["ms"], "e4m3_bytes": ref["bytes"],
                      "speedup_over_e4m3": round(ref["ms"] / ms4, 3)}
        w4["note"] = ("E2M1 weights, 128x128 fp32 scales, packed two codes per byte in HBM; the live experts' "
                      "weight read halves; timed beside the step (the step itself uses e4m3 weights)")

    # ---------------- end to end through the public API, host buffers
    e2e = None
    if not args.no_e2e:
        x_h = x.cpu().pin_memory()
        dy_h = dy.cpu().pin_memory()
        dh_h = dh.cpu().pin_memory()
        s_h = sizes.cpu().pin_memory()
        y_h = torch.empty((M, K), dtype=torch.bfloat16).pin_memory()
        # Every step's inputs (X, group sizes, dY, dH) go in on a copy stream
        # while the previous step computes, and its y comes back on another
        # while the next one computes: two device copies of the inputs and of y
        # alternate between steps.  The host link is the bound (one direction
        # ~210 GB/s measured, more concurrent copy streams do not add to it).
        bufs = [{"x": torch.empty_like(x), "dy": torch.empty_like(dy), "dh": torch.empty_like(dh),
                 "s": torch.empty_like(sizes), "y": torch.empty((M, K), dtype=torch.bfloat16, device=dev)}
                for _ in range(2)]
        h2d_stream = torch.cuda.Stream(dev)
        d2h_stream = torch.cuda.Stream(dev)
        ev_in = [None, None]
        ev_done = [torch.cuda.Event(), torch.cuda.Event()]  # the step that used set b has finished with it
        ev_out = [torch.cuda.Event(), torch.cuda.Event()]   # and its y is on the host

        def issue_inputs(b):
            B = bufs[b]
            with torch.cuda.stream(h2d_stream):
                h2d_stream.wait_event(ev_done[b])
                h2d_stream.wait_event(ev_out[b])
                B["x"].copy_(x_h, non_blocking=True)
                B["s"].copy_(s_h, non_blocking=True)
                B["dy"].copy_(dy_h, non_blocking=True)
                B["dh"].copy_(dh_h, non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(h2d_stream)
                ev_in[b] = ev

        def compute(b):
            B = bufs[b]
            stream.wait_event(ev_in[b])
            chk(gmm.gmm_quantize_lhs(B["x"], M, K, xq, xs, stream), "e2e quantize X")
            chk(gmm.gmm_group_metadata(B["s"], G, M, work.buf, work.nbytes, stream), "e2e metadata")
            chk(gmm.gmm_fp8_fwd_swiglu_quant(xq, xs, wq_wi, ws_wi, None, G, M, K, N, h, hq, hs, work.buf,
                                             work.nbytes, stream), "e2e wi")
            chk(gmm.gmm_fp8_fwd(hq, hs, wq_wo, ws_wo, None, G, M, N, K, 0, B["y"], work.buf, work.nbytes, stream),
                "e2e wo")
            ev_y = torch.cuda.Event()
            ev_y.record(stream)
            with torch.cuda.stream(d2h_stream):
                d2h_stream.wait_event(ev_y)
                y_h.copy_(B["y"], non_blocking=True)
                ev_out[b].record(d2h_stream)
            chk(gmm.tgmm_bf16(h, B["dy"], None, G, M, N, K, dw_wo, work.buf, work.nbytes, stream), "e2e tgmm wo")
            chk(gmm.tgmm_bf16(B["x"], B["dh"], None, G, M, K, 2 * N, dw_wi, work.buf, work.nbytes, stream),
                "e2e tgmm wi")
            ev_done[b].record(stream)

        def e2e_steps(n):
            """n steps, pipelined; the stream ends with the last y on the host."""
            for b in range(2):  # both sets free from here on (after e0, when timing)
                ev_done[b].record(stream)
                ev_out[b].record(stream)
            issue_inputs(0)
            for i in range(n):
                if i + 1 < n:
                    issue_inputs((i + 1) % 2)
                compute(i % 2)
            stream.wait_event(ev_out[(n - 1) % 2])

        e2e_steps(2)
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n_e2e = max(3, min(args.steps, 20))
        e0.record(stream)
        e2e_steps(n_e2e)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        e_ms = e0.elapsed_time(e1) / n_e2e
        if ws_ > 1:
            e_ms = max_over_ranks(e_ms, dev)
        h2d = x.numel() * 2 + dy.numel() * 2 + dh.numel() * 2 + sizes.numel() * 4
        d2h = y.numel() * 2
        e2e = {"value": round(ws_ * step_flops / (e_ms * 1e-3) / 1e12, 2), "unit": UNIT,
               "ms_per_step": round(e_ms, 3), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "note": "pinned host X, group_sizes, dY, dH in; y out; weights resident and pre-quantized; "
                       "each step's inputs copied in while the previous step computes and its y copied "
                       "out while the next one computes (two device buffer sets); the first step's "
                       "copy-in and the last step's copy-out are inside the timed region"}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args.cpu_seconds)

    if ws_ > 1:
        torch.distributed.barrier()
    if rank != 0:
        return None
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": ws_, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 4), "step_ms": step_dist, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3 MMA + bf16 MMA, fp32 accumulate",
        "data": "synthetic (seeded; routing Zipf(1.1) top-8; X N(0,1) with 1% x50 outliers)",
        "config": {"workload": WORKLOAD, "G": G, "M": M, "K": K, "N": N, "step_gflop": round(step_flops / 1e9, 2),
                   "parallelism": f"replicas x{ws_}" if ws_ > 1 else "single GPU",
                   "l2": "flushed between steps (256 MB write, outside the events); per-step working set > 4 GB"},
        "roofline": roof, "kernels": kern,
        "kernels_note": f"per-kernel times from a second pass of {n_split} steps with an event between every "
                        "call (the timed steps carry boundary events only)",
        "bf16_fwd_baseline": bf or None, "bf16_dgrad": dgrad, "w4_weights": w4, "e2e": e2e,
        "cpu_baseline": cpu, "gpu_launches": launches_per_step * args.steps, "clocks": clk,
        "wall_s_timed_region": round(wall, 4),
    }
    return line


# ---------------------------------------------------------------------------
# CPU oracle arm
# ---------------------------------------------------------------------------

def _sample_problem(n_groups: int, rows_per_group: int, seed: int = 77):
    """A bounded sample of the production workload, as its own small GMM:
    n_groups experts (the largest, the smallest non-empty, the rest random),
    up to rows_per_group rows each, with that many rows' worth of inputs."""
    from fp8_blockwise_quantized_gb300.workloads import normal_bf16, routing_sizes
    rng = np.random.default_rng(seed)
    sizes = routing_sizes("prod_fp8")
    live = np.flatnonzero(sizes)
    pick = {int(live[np.argmax(sizes[live])]), int(live[np.argmin(sizes[live])])}
    rest = [g for g in live if g not in pick]
    pick.update(int(g) for g in rng.choice(rest, n_groups - len(pick), replace=False))
    groups = sorted(pick)
    sub = np.array([min(int(sizes[g]), rows_per_group) for g in groups], np.int32)
    m = int(sub.sum())
    x = normal_bf16((m, K), 1.0, rng, outlier_p=0.01)
    w_wi = normal_bf16((len(groups), K, 2 * N), 1.0 / math.sqrt(K), rng)
    w_wo = normal_bf16((len(groups), N, K), 1.0 / math.sqrt(N), rng)
    dy = normal_bf16((m, K), 1.0, rng)
    dh = normal_bf16((m, 2 * N), 1.0, rng)
    return sub, x, w_wi, w_wo, dy, dh


def oracle_step(sample):
    """One pass of the path on the sample, by the oracle; returns its FLOPs."""
    import oracle
    sub, x, w_wi, w_wo, dy, dh, wq_wi, ws_wi, wq_wo, ws_wo = sample
    m = int(sub.sum())
    xq, xs = oracle.quantize_lhs(x)
    h = oracle.round_to_bf16(oracle.gmm_fp8(xq, xs, wq_wi, ws_wi, sub, fuse=True))
    hq, hs = oracle.quantize_lhs(h)
    oracle.round_to_bf16(oracle.gmm_fp8(hq, hs, wq_wo, ws_wo, sub))
    oracle.tgmm_bf16(h, dy, sub)
    oracle.tgmm_bf16(x, dh, sub)
    return 2 * m * K * 2 * N * 2 + 2 * m * N * K * 2


def _prepare_sample(n_groups, rows):
    import oracle
    oracle.build()
    sub, x, w_wi, w_wo, dy, dh = _sample_problem(n_groups, rows)
    wq_wi, ws_wi = oracle.quantize_rhs(w_wi)   # offline, untimed (as on the GPU)
    wq_wo, ws_wo = oracle.quantize_rhs(w_wo)
    return (sub, x, w_wi, w_wo, dy, dh, wq_wi, ws_wi, wq_wo, ws_wo)


def cpu_baseline(seconds: float):
    import oracle
    sample = _prepare_sample(8, 32)
    t0 = time.perf_counter()
    fl = 0
    reps = 0
    while True:
        fl += oracle_step(sample)
        reps += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    return {"value": round(fl / dt / 1e12, 6), "unit": UNIT, "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": (f"{reps} pass(es) of the full path (quantize X, fused wi, quantize h, wo, both tgmm) "
                       f"over 8 experts x <=32 rows = {int(sample[0].sum())} rows of the production "
                       f"shapes (K=2048, N=2x512 / 2048), {dt:.1f} s"),
            "seconds": round(dt, 2)}


def run_reference(args):
    ws_, rank, _ = _dist()
    if rank != 0:
        return None
    import oracle
    sample = _prepare_sample(8, 32)
    for _ in range(args.warmup):
        oracle_step(sample)
    t0 = time.perf_counter()
    fl = 0
    for _ in range(args.steps):
        fl += oracle_step(sample)
    dt = time.perf_counter() - t0
    value = fl / dt / 1e12
    rows = int(sample[0].sum())
    cpu = {"value": round(value, 6), "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
           "sample": f"per step: the full path over 8 experts x <=32 rows = {rows} rows of the production shapes"}
    return {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": ws_,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)",
            "data": "synthetic (seeded)", "config": {"workload": WORKLOAD, "sample_rows": rows},
            "cpu_baseline": cpu,
            "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ---------------------------------------------------------------------------
# the oracle on the four small configurations, whole (not sampled): all host
# cores, and one core in a child process (OpenMP reads its thread count once)
# ---------------------------------------------------------------------------

ORACLE_CONFIGS = ["tiny_fp8", "wi_dev_fp8", "wo_dev_fp8", "tgmm_dev_bf16"]


def _oracle_config_pass(name: str):
    """One whole pass of the oracle on a configuration (weights quantized
    outside the timing, as on the GPU); returns (seconds, GFLOP)."""
    import oracle
    from fp8_blockwise_quantized_gb300.workloads import make_case
    oracle.build()
    c = make_case(name)
    if name == "tgmm_dev_bf16":
        t0 = time.perf_counter()
        oracle.tgmm_bf16(c.x, c.dy, c.group_sizes)
        dt = time.perf_counter() - t0
        return dt, 2.0 * c.M * c.K * c.N / 1e9
    wq, ws = oracle.quantize_rhs(c.w)
    t0 = time.perf_counter()
    xq, xs = oracle.quantize_lhs(c.x)
    oracle.round_to_bf16(oracle.gmm_fp8(xq, xs, wq, ws, c.group_sizes))
    dt = time.perf_counter() - t0
    return dt, 2.0 * c.M * c.K * c.N / 1e9


def run_oracle_configs():
    import oracle
    oracle.build()
    rows = []
    for name in ORACLE_CONFIGS:
        dt_all, gf = _oracle_config_pass(name)
        env = dict(os.environ, OMP_NUM_THREADS="1")
        out = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-config-one", name],
                             env=env, capture_output=True, text=True, check=True)
        one = json.loads(out.stdout.strip().splitlines()[-1])
        rows.append({"config": name, "gflop": round(gf, 3), "all_cores_s": round(dt_all, 3),
                     "cores": oracle.num_threads(), "one_core_s": round(one["seconds"], 3),
                     "all_cores_gflops": round(gf / dt_all, 3), "one_core_gflops": round(gf / one["seconds"], 3)})
    print(json.dumps({"oracle_configs": rows, "what": "quantize X + FP8 GMM (weights quantized beforehand) "
                                                      "or bf16 tgmm, whole configuration, one pass"}))


# ---------------------------------------------------------------------------
# single-kernel mode for profilers: production shapes, only what one kernel needs
# ---------------------------------------------------------------------------

def run_profile_case(args):
    import torch
    import fp8_blockwise_quantized_gb300 as gmm
    from fp8_blockwise_quantized_gb300.build import build
    from fp8_blockwise_quantized_gb300.workloads import routing_sizes
    build()
    dev = torch.device("cuda", 0)
    gen = torch.Generator(device=dev)
    gen.manual_seed(2024)
    sizes = torch.from_numpy(routing_sizes("prod_fp8")).to(dev)
    work = gmm.Workspace(G, M, dev)
    chk = gmm.binding._check
    case = args.profile_case

    def bf16(shape, std=1.0):
        return (torch.randn(shape, generator=gen, device=dev) * std).to(torch.bfloat16)

    if case == "fp8_w4_wi_quant":
        x = bf16((M, K))
        xq, xs = gmm.quantize_lhs(x)
        w = bf16((G, K, 2 * N), 1.0 / math.sqrt(K))
        wq, ws = gmm.quantize_rhs_w4(w)
        del x, w
        out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        hq = torch.empty((M, N), dtype=torch.uint8, device=dev)
        hs = torch.empty((N // 128, M), dtype=torch.float32, device=dev)
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        run = lambda: chk(gmm.gmm_fp8_w4_fwd_swiglu_quant(xq, xs, wq, ws, sizes, G, M, K, N, out, hq, hs, work.buf,
                                                          work.nbytes, None), case)
    elif case in ("fp8_wi", "fp8_wo", "fp8_wi_quant"):
        k, n, fuse = (K, N, 1) if case != "fp8_wo" else (N, K, 0)
        x = bf16((M, k))
        xq, xs = gmm.quantize_lhs(x)
        w = bf16((G, k, 2 * n if fuse else n), 1.0 / math.sqrt(k))
        wq, ws = gmm.quantize_rhs(w)
        del x, w
        out = torch.empty((M, n), dtype=torch.bfloat16, device=dev)
        hq = torch.empty((M, n), dtype=torch.uint8, device=dev)
        hs = torch.empty((n // 128, M), dtype=torch.float32, device=dev)
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        if case == "fp8_wi_quant":
            run = lambda: chk(gmm.gmm_fp8_fwd_swiglu_quant(xq, xs, wq, ws, sizes, G, M, k, n, out, hq, hs,
                                                           work.buf, work.nbytes, None), case)
        else:
            run = lambda: chk(gmm.gmm_fp8_fwd(xq, xs, wq, ws, sizes, G, M, k, n, fuse, out, work.buf,
                                              work.nbytes, None), case)
    elif case in ("tgmm_wi", "tgmm_wo"):
        k, n = (K, 2 * N) if case == "tgmm_wi" else (N, K)
        x = bf16((M, k))
        dy = bf16((M, n))
        dw = torch.empty((G, k, n), dtype=torch.bfloat16, device=dev)
        run = lambda: chk(gmm.tgmm_bf16(x, dy, sizes, G, M, k, n, dw, work.buf, work.nbytes, None), case)
    elif case == "quantize_x":
        x = bf16((M, K))
        xq = torch.empty((M, K), dtype=torch.uint8, device=dev)
        xs = torch.empty((K // 128, M), dtype=torch.float32, device=dev)
        run = lambda: chk(gmm.gmm_quantize_lhs(x, M, K, xq, xs, None), case)
    else:
        raise SystemExit(f"unknown profile case {case}")
    for _ in range(args.warmup + args.steps):
        run()
    torch.cuda.synchronize()
    st = work.status()
    print(json.dumps({"profile_case": case, "launches": args.warmup + args.steps, "status": st}))
    if st != 0:
        raise SystemExit(1)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-bf16-baseline", action="store_true")
    ap.add_argument("--no-w4", action="store_true", help="skip the 4-bit weight forward timed beside the step")
    ap.add_argument("--profile-case", default=None,
                    choices=["fp8_wi", "fp8_wi_quant", "fp8_w4_wi_quant", "fp8_wo", "tgmm_wi", "tgmm_wo",
                             "quantize_x"],
                    help="run one kernel at the production shape (for ncu) and exit")
    ap.add_argument("--oracle-configs", action="store_true",
                    help="time the CPU oracle on the four small configurations (all cores and one core) and exit")
    ap.add_argument("--oracle-config-one", default=None, help=argparse.SUPPRESS)
    ap.add_argument("--traffic", type=float, default=None,
                    help="ncu dram bytes per launch of the dominant kernel, if captured on the current kernel source")
    args = ap.parse_args()
    if args.oracle_config_one:
        dt, gf = _oracle_config_pass(args.oracle_config_one)
        print(json.dumps({"seconds": dt, "gflop": gf}))
        return
    if args.oracle_configs:
        run_oracle_configs()
        return
    if args.warmup < 3 and not args.profile_case:
        ap.error("--warmup must be >= 3")
    if args.profile_case:
        run_profile_case(args)
        return
    line = run_reference(args) if args.impl == "reference" else run_gpu(args)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
