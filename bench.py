#!/usr/bin/env python3
"""Throughput of the grouped MoE low-precision hot path on GB300.

One step = one NVFP4 mixture-of-experts up-projection over a batch of
synthetic tokens already resident in HBM:
    padded scale offsets -> per-expert amax -> NVFP4 tensor scales ->
    grouped NVFP4 activation quantize -> fused grouped NVFP4 GEMM + SwiGLU +
    NVFP4 requant
on 128 experts, 16384 tokens routed top-8 uniformly (131072 rows), hidden
K = 4096, I = 1536 (N = 2 x 1536 gate/up interleaved).  ``value`` is GEMM
TFLOP/s of the whole step (2 * rows * N * K per step).  The line also carries
the per-kernel figures of the other workloads (grouped quantize GB/s, FP8
rowwise TFLOP/s, decode-shaped GB/s, the chained GEMM -> SwiGLU path), the
dominant kernel's roofline, the sampled SM clocks, an end-to-end figure
through the same calls from pinned host buffers, and the CPU oracle timed on
a bounded sample.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

For N > 1 launch with torch.distributed.run: every rank runs the same step on
its own batch (weak scaling, no collective on the data path); the time is the
maximum over ranks.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "grouped MoE GEMM TFLOPS (FP8/NVFP4) % of peak; quantize GB/s % of HBM"
WORKLOAD = ("NVFP4 MoE up-projection: 128 experts, 16384 tokens top-8 uniform -> 131072 rows, "
            "K=4096, N=2x1536 gate/up interleaved; amax -> NVFP4 quantize -> fused "
            "GEMM+SwiGLU+NVFP4 requant")
E4, TOK4, TOPK4, K4, I4 = 128, 16384, 8, 4096, 1536
FP4_OVER_BF16 = 13.5 / 2.25      # nominal dense ratios
FP8_OVER_BF16 = 4.5 / 2.25
# nominal figures of the part (dense tensor rates, HBM3e bandwidth)
NOMINAL = {"hbm_gbs": 7900.0, "fp8_tflops": 4500.0, "fp4_tflops": 13500.0}
# Measured tcgen05 MMA ceiling of this part: one M128 x N256 instruction per
# 128 SM cycles for every kind, so FP4 (K = 64) does 2 * 128 * 256 * 64 / 128
# = 32768 flop per SM cycle (FP8 half, bf16 a quarter).
FP4_FLOP_PER_SM_CYCLE = 32768
# The NVFP4 GEMMs run 256-row x 256-column tiles over CTA pairs: each
# expert's rows are padded to whole 256-row pair tiles, the persistent pairs
# take tiles t, t + pairs, ...; every tile issues K / 64 pair MMAs of 128
# cycles.
FP4_PAIR_TILE_M, FP4_PAIR_TILE_N, FP4_MMA_K, FP4_MMA_CYCLES = 256, 256, 64, 128


def fp4_schedule_floor(counts, N, K, sms, sm_mhz):
    """MMA time (ms) of the fused GEMM's own schedule at the measured MMA
    rate, with the pair tiles it runs in all and on its busiest pair."""
    tiles = sum(-(-int(c) // FP4_PAIR_TILE_M) for c in counts if c) * -(-N // FP4_PAIR_TILE_N)
    pairs = sms // 2
    per_pair = -(-tiles // pairs)
    cycles = per_pair * (K // FP4_MMA_K) * FP4_MMA_CYCLES
    return cycles / (sm_mhz * 1e3), tiles, per_pair
# The fused GEMM's DRAM traffic comes from a committed ncu summary that names
# the sha256 of the kernel sources it was captured with; a changed kernel
# makes the figure stale and the bench reports null.
TRAFFIC_PROFILE = os.path.join(ROOT, "profiles", "launches_moe_up_projection_nvfp4_128experts.md")
KERNEL_SOURCES = ("fp4_fp8_quantization_gb300/csrc/gemm.cu",
                  "fp4_fp8_quantization_gb300/csrc/common.cuh")


def kernel_source_hash():
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def fused_traffic_bytes():
    """(bytes per launch, note): the DRAM read + write bytes of one full-size
    fused launch from the committed ncu summary, or None when the summary was
    captured with other kernel sources (or is missing)."""
    try:
        text = open(TRAFFIC_PROFILE).read()
    except OSError:
        return None, "no ncu summary"
    src = traf = None
    for line in text.splitlines():
        if line.startswith("kernel-sources-sha256:"):
            src = line.split(":", 1)[1].strip()
        if line.startswith("fused-gemm-dram-bytes-per-launch:"):
            traf = float(line.split(":", 1)[1].strip())
    cur = kernel_source_hash()
    if traf is None or src != cur:
        return None, f"ncu summary captured with kernel sources {src}, current {cur}: not re-captured"
    return traf, f"ncu dram__bytes_read.sum + dram__bytes_write.sum, kernel sources {cur}"


def emit(line, args):
    """Prints the result line; appends it to the metrics log when one is named."""
    text = json.dumps(line)
    print(text, flush=True)
    if args.log:
        with open(args.log, "a") as f:
            f.write(text + "\n")


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="moeq", choices=["moeq", "reference"])
    p.add_argument("--no-parts", action="store_true")
    p.add_argument("--no-cpu", action="store_true")
    p.add_argument("--log", default=os.environ.get("MOEQ_METRICS_LOG"),
                   help="also append the JSON line to this file (default: $MOEQ_METRICS_LOG)")
    p.add_argument("--profile", choices=["fused", "fused_mx", "quantize", "fp8", "decode_fp8",
                                          "chained", "swiglu", "dispatch"],
                   help="run only --warmup + --steps launches of one kernel on a small case "
                        "(inputs larger than L2, under 1 GB) for a profiler; no JSON line")
    return p.parse_args()


# ------------------------------------------------------------------ setup

def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    return rank, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return {"hbm_gbs": d["hbm_gbs"], "bf16": d["bf16_tflops"],
                "bf16_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16": 1900.0, "bf16_sustained": 1700.0, "source": "fallback"}


class Clocks:
    """nvidia-smi sampled every 100 ms while the GPU works."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,"
         "utilization.gpu")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = []
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 10:
                continue
            try:
                rows.append({"sm": float(f[1]), "max": float(f[2]), "hw": f[5], "hwt": f[6],
                             "swt": f[7], "pcap": f[8], "util": float(f[9])})
            except ValueError:
                continue
        busy = [r for r in rows if r["util"] > 0] or rows
        if not busy:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        reasons = []
        for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                          ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
            if any(r[key].lower() == "active" for r in busy):
                reasons.append(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in busy),
                "sm_max_mhz": max(r["max"] for r in busy), "reasons": reasons,
                "samples": len(busy)}


# --------------------------------------------------------------- workload

def nvfp4_expert_weights(num_experts, rows, K, std, seed, device="cuda"):
    """(packed [E, rows, K/2], tiled scales, tensor scales [E]): expert
    weights drawn as bf16 N(0, std) and quantized to NVFP4 by the library's
    own grouped quantizer, one group per expert (each expert's tensor scale
    from its amax)."""
    from fp4_fp8_quantization_gb300 import moeq, synth
    w = synth.bf16_normal((num_experts * rows, K), std, seed=seed, device=device)
    offs = torch.arange(num_experts + 1, dtype=torch.int32, device=device) * rows
    ids = torch.arange(num_experts, dtype=torch.int32, device=device)
    ts = torch.empty(num_experts, device=device)
    moeq.grouped_amax_scale(w, offs, ids, ts, num_experts)
    b = torch.empty((num_experts * rows, K // 2), dtype=torch.uint8, device=device)
    bsf = torch.empty(moeq.sf_bytes(num_experts * rows, K // 16), dtype=torch.uint8,
                      device=device)
    moeq.grouped_quantize("nvfp4", w, b, bsf, offs, offs, ids, ts, num_experts,
                          num_experts * rows, rows)
    del w
    return b.view(num_experts, rows, K // 2), bsf, ts


def swiglu_output_scales(y, ro, ids, num_experts):
    """Calibration of the SwiGLU output's NVFP4 tensor scale on the chained
    path's bf16 y: amax over each expert group of silu(gate) * up in fp32,
    / 2688 (1 for an empty or all-zero group).  PyTorch's fp32 SiLU stands in
    for the library's here: the result is an input scale, valid at any
    positive value."""
    dev = y.device
    h = torch.nn.functional.silu(y[:, 0::2].float()).mul_(y[:, 1::2].float()).abs_()
    rowmax = h.amax(dim=1)
    del h
    counts = torch.from_numpy(np.diff(ro.astype(np.int64))).to(dev)
    expert_of_row = torch.repeat_interleave(torch.from_numpy(ids.astype(np.int64)).to(dev), counts)
    emax = torch.zeros(num_experts, dtype=torch.float32, device=dev)
    emax.scatter_reduce_(0, expert_of_row, rowmax, reduce="amax")
    scale = (emax / torch.tensor(2688.0, dtype=torch.float32, device=dev))
    return torch.where(emax > 0, scale, torch.ones_like(scale))


def up_projection_inputs(seed, device="cuda"):
    """The 128-expert up-projection as configured: activations bf16 N(0, 1)
    (quantized in the timed step), gate/up weights NVFP4 from bf16 N(0, 0.02)
    with per-expert tensor scales, expert scales U[0.5, 2], and the SwiGLU
    output scales from a calibration run of the chained path on these
    inputs."""
    from fp4_fp8_quantization_gb300 import moeq, synth
    counts = synth.routing_counts(TOK4, TOPK4, E4, seed=seed)
    ro, ids = synth.ragged_groups(counts)
    T = int(ro[-1])
    rows = int(sum((int(c) + 127) // 128 * 128 for c in counts if c))
    N = 2 * I4
    b, bsf, ts_w = nvfp4_expert_weights(E4, N, K4, 0.02, seed + 2, device)
    d = {
        "counts": counts, "ro_h": ro, "ids_h": ids, "T": T, "rows": rows, "N": N,
        "ro": torch.from_numpy(ro.view(np.int32)).to(device),
        "ids": torch.from_numpy(ids).to(device),
        "so": torch.empty(len(ids) + 1, dtype=torch.int32, device=device),
        "x": synth.bf16_normal((T, K4), 1.0, seed=seed + 1, device=device),
        "b": b, "bsf": bsf, "ts_w": ts_w,
        "es": synth.uniform((E4,), 0.5, 2.0, seed=seed + 4, device=device),
        "ts": torch.empty(E4, device=device),
        "a": torch.empty((T, K4 // 2), dtype=torch.uint8, device=device),
        "asf": torch.empty(moeq.sf_bytes(rows, K4 // 16), dtype=torch.uint8, device=device),
        "c": torch.empty((T, I4 // 2), dtype=torch.uint8, device=device),
        "csf": torch.empty(moeq.sf_bytes(rows, I4 // 16), dtype=torch.uint8, device=device),
    }
    d["mt"] = int(counts.max())
    # calibration: quantize the activations, chained GEMM -> bf16 y, amax of h
    moeq.padded_scale_offsets(d["ro"], d["so"])
    moeq.grouped_amax_scale(d["x"], d["ro"], d["ids"], d["ts"], E4)
    moeq.grouped_quantize("nvfp4", d["x"], d["a"], d["asf"], d["ro"], d["so"], d["ids"], d["ts"],
                          E4, rows, d["mt"])
    y = torch.empty((T, N), dtype=torch.bfloat16, device=device)
    moeq.grouped_matmul_blockscaled("nvfp4", y, d["a"], d["asf"], b, bsf, d["es"], d["ro"],
                                    d["so"], d["ids"], N, K4, rows, d["mt"])
    d["ots"] = swiglu_output_scales(y, ro, ids, E4)
    del y
    return d


def up_projection_step(d, events=None):
    """The hot path; `events` (list of 5 CUDA events) brackets each kernel."""
    from fp4_fp8_quantization_gb300 import moeq
    rec = (lambda i: events[i].record()) if events else (lambda i: None)
    rec(0)
    moeq.padded_scale_offsets(d["ro"], d["so"])
    moeq.grouped_amax_scale(d["x"], d["ro"], d["ids"], d["ts"], E4)
    rec(1)
    moeq.grouped_quantize("nvfp4", d["x"], d["a"], d["asf"], d["ro"], d["so"], d["ids"], d["ts"],
                          E4, d["rows"], d["mt"])
    rec(2)
    moeq.grouped_matmul_swiglu(d["c"], d["csf"], d["a"], d["asf"], d["b"], d["bsf"], d["es"],
                               d["ots"], d["ro"], d["so"], d["ids"], I4, K4, d["rows"], d["mt"])
    rec(3)


KERNELS_PER_STEP = 6   # padded offsets, amax zeroing, amax, amax finalize, quantize, fused GEMM


def flops_up(d):
    return 2.0 * d["T"] * d["N"] * K4


# ------------------------------------------------------------ sub-parts

def time_kernel(fn, iters, flush=None, warmup=3, batch=1):
    """Device time (ms) of one call.  `fn` is a callable or a list of
    callables used in rotation (input sets whose total exceeds L2, so every
    call reads from HBM); an L2 flush (write of a buffer larger than L2)
    precedes every timed call when `flush` is given.  With batch > 1 the
    events bracket `batch` back-to-back calls (the launch of one overlaps
    the end of the previous) and the median over `iters` batches of the
    per-call time is returned; otherwise the mean over `iters` single
    calls."""
    fns = fn if isinstance(fn, (list, tuple)) else [fn]
    for i in range(max(warmup, 2 * batch)):
        fns[i % len(fns)]()
    ts = []
    k = 0
    for i in range(iters):
        if flush is not None:
            flush.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(batch):
            fns[k % len(fns)]()
            k += 1
        e1.record()
        ts.append((e0, e1))
    torch.cuda.synchronize()
    per = [a.elapsed_time(b) / batch for a, b in ts]
    return statistics.median(per) if batch > 1 else statistics.mean(per)


GRAPH_TIMING_NOTE = ("ms: device time per launch, 32 calls over the 4 input sets in one CUDA "
                     "graph, replay time / 32 (mean of 20 replays); binding_ms: median over 20 "
                     "batches of 8 back-to-back calls through the Python binding")


def graph_time_per_call(fns, reps=8):
    """Device time (ms) per call of `fns` (callables used in rotation): reps
    rounds of them captured in one CUDA graph on a side stream, replayed."""
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for f in fns:
            f()
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=side):
            for _ in range(reps):
                for f in fns:
                    f()
    torch.cuda.current_stream().wait_stream(side)
    return time_kernel(g.replay, 20) / (reps * len(fns))


def parts(pk, flush):
    from fp4_fp8_quantization_gb300 import moeq, synth
    hbm = pk["hbm_gbs"]
    fp8_peak = pk["bf16"] * FP8_OVER_BF16
    out = {}
    dev = "cuda"
    u32 = lambda a: torch.from_numpy(np.asarray(a, np.uint32).view(np.int32)).to(dev)

    # grouped activation quantize: 8 experts, 4096 tokens top-2, hidden 4096
    counts = synth.routing_counts(4096, 2, 8, seed=0)
    ro, ids = synth.ragged_groups(counts)
    T = int(ro[-1])
    rows = int(sum((int(c) + 127) // 128 * 128 for c in counts if c))
    # 4 input / output sets used in rotation: 4 x 67 MB of activations exceed
    # L2, so every timed call streams its input from HBM (no flush needed)
    NSET = 4
    xs = [synth.bf16_normal((T, 4096), 1.0, seed=1 + i, device=dev, outlier_p=0.001,
                            outlier_scale=50.0) for i in range(NSET)]
    ro_d, ids_d = u32(ro), torch.from_numpy(ids).to(dev)
    so_d = torch.empty(len(ids) + 1, dtype=torch.int32, device=dev)
    moeq.padded_scale_offsets(ro_d, so_d)
    ts = torch.empty(8, device=dev)
    # device time per launch: 32 calls over the rotating sets captured in one
    # CUDA graph, replayed (each kernel still waits for the previous one's
    # completion through its programmatic-launch edge); beside it the time per
    # call through the Python binding, batches of 8 back-to-back calls (host
    # issue included: ctypes marshalling, argument checks, launch)
    amax_fns = [lambda x=x: moeq.grouped_amax_scale(x, ro_d, ids_d, ts, 8) for x in xs]
    t_amax = graph_time_per_call(amax_fns)
    t_amax_b = time_kernel(amax_fns, 20, batch=8)
    for fmt, ob, v in (("nvfp4", 2048, 16), ("mxfp8", 4096, 32)):
        qs = [torch.empty((T, ob), dtype=torch.uint8, device=dev) for _ in range(NSET)]
        sfs = [torch.empty(moeq.sf_bytes(rows, 4096 // v), dtype=torch.uint8, device=dev)
               for _ in range(NSET)]
        fns = [lambda x=x, q=q, sf=sf, fmt=fmt: moeq.grouped_quantize(
            fmt, x, q, sf, ro_d, so_d, ids_d, ts, 8, rows) for x, q, sf in zip(xs, qs, sfs)]
        ms = graph_time_per_call(fns)
        ms_b = time_kernel(fns, 20, batch=8)
        nbytes = T * 4096 * 2 + qs[0].numel() + sfs[0].numel()
        out[f"quantize_{fmt}_8192x4096"] = {
            "ms": round(ms, 5), "GB/s": round(nbytes / ms / 1e6, 1),
            "frac_hbm": round(nbytes / ms / 1e6 / hbm, 4),
            "frac_hbm_nominal": round(nbytes / ms / 1e6 / NOMINAL["hbm_gbs"], 4), "bytes": nbytes,
            "binding_ms": round(ms_b, 5), "frac_hbm_binding": round(nbytes / ms_b / 1e6 / hbm, 4),
            "l2": "4 rotating input sets (268 MB > L2)",
            "timing": GRAPH_TIMING_NOTE}
    out["amax_8192x4096"] = {"ms": round(t_amax, 5),
                             "GB/s": round(T * 4096 * 2 / t_amax / 1e6, 1),
                             "frac_hbm": round(T * 4096 * 2 / t_amax / 1e6 / hbm, 4),
                             "binding_ms": round(t_amax_b, 5), "timing": GRAPH_TIMING_NOTE}
    del xs

    # tiny FP8 rowwise: E 4, groups of 7 / 16 / 9 rows on experts 2 / 0 / 3,
    # K 128, N 64 (a latency figure: one launch, back to back)
    ro_t = np.array([0, 7, 23, 32], np.uint32)
    ids_t = np.array([2, 0, 3], np.int32)
    a_t = synth.e4m3_normal((32, 128), 1.0, seed=40, device=dev)
    b_t = synth.e4m3_normal((4, 64, 128), 0.5, seed=41, device=dev)
    sa_t = synth.uniform((32,), 0.01, 0.1, seed=42, device=dev)
    sb_t = synth.uniform((4, 64), 0.005, 0.05, seed=43, device=dev)
    c_t = torch.empty((32, 64), dtype=torch.bfloat16, device=dev)
    ro_td, ids_td = u32(ro_t), torch.from_numpy(ids_t).to(dev)
    tiny = lambda: moeq.grouped_matmul_rowwise_fp8(c_t, a_t, b_t, sa_t, sb_t, ro_td, ids_td, 16)
    ms = time_kernel(tiny, 20, batch=8)
    # device-only: 64 launches captured in one CUDA graph, replayed; the
    # per-launch time excludes the host's issue cost (ctypes marshalling,
    # argument checks, cudaLaunchKernelEx)
    ms_graph = graph_time_per_call([tiny], reps=64)
    out["fp8_rowwise_tiny_32x64x128"] = {
        "us_per_call_binding": round(ms * 1e3, 2),
        "us_device_per_launch": round(ms_graph * 1e3, 2),
        "timing": "binding: median over 20 batches of 8 back-to-back calls through the Python "
                  "binding; device: 64 launches in one CUDA graph, replay time / 64 "
                  "(mean of 20 replays)"}

    # FP8 rowwise at MoE scale: 64 experts, 8192 tokens top-8 Zipf(1.1), K 7168, N 4096
    counts = synth.routing_counts(8192, 8, 64, seed=0, zipf_s=1.1)
    ro, ids = synth.ragged_groups(counts)
    T, N, K = int(ro[-1]), 4096, 7168
    a, sa = synth.fp8_rowwise((T, K), 1.0, seed=10, device=dev)
    b, sb = synth.fp8_rowwise((64, N, K), 0.02, seed=11, device=dev)
    c = torch.empty((T, N), dtype=torch.bfloat16, device=dev)
    ro_d, ids_d = u32(ro), torch.from_numpy(ids).to(dev)
    ms = time_kernel(lambda: moeq.grouped_matmul_rowwise_fp8(
        c, a, b, sa, sb.reshape(64, N), ro_d, ids_d, int(counts.max())), 10)
    fl = 2.0 * T * N * K
    out["fp8_rowwise_65536x4096x7168"] = {
        "ms": round(ms, 4), "TFLOP/s": round(fl / ms / 1e9, 1),
        "frac_fp8_peak": round(fl / ms / 1e9 / fp8_peak, 4),
        "frac_fp8_nominal": round(fl / ms / 1e9 / NOMINAL["fp8_tflops"], 4)}
    del a, b, c

    # decode-shaped: 256 experts, 64 tokens top-8 -> 512 rows, K 7168, N 4096
    counts = synth.routing_counts(64, 8, 256, seed=0)
    ro, ids = synth.ragged_groups(counts)
    T = int(ro[-1])
    active_bytes = len(ids) * N * K
    a, sa = synth.fp8_rowwise((T, K), 1.0, seed=20, device=dev)
    b, sb = synth.fp8_rowwise((256, N, K), 0.02, seed=21, device=dev)
    c = torch.empty((T, N), dtype=torch.bfloat16, device=dev)
    ro_d, ids_d = u32(ro), torch.from_numpy(ids).to(dev)
    ms = time_kernel(lambda: moeq.grouped_matmul_rowwise_fp8(
        c, a, b, sa, sb.reshape(256, N), ro_d, ids_d, int(counts.max())), 10)
    out["decode_fp8_rowwise_512rows_224experts"] = {
        "ms": round(ms, 4), "GB/s_active_weights": round(active_bytes / ms / 1e6, 1),
        "frac_hbm": round(active_bytes / ms / 1e6 / hbm, 4),
        "frac_hbm_nominal": round(active_bytes / ms / 1e6 / NOMINAL["hbm_gbs"], 4),
        "active_experts": len(ids)}
    del b
    rows = int(sum((int(cc) + 127) // 128 * 128 for cc in counts if cc))
    so_d = torch.empty(len(ids) + 1, dtype=torch.int32, device=dev)
    moeq.padded_scale_offsets(ro_d, so_d)
    b8 = synth.e4m3_normal((256, N, K), 1.0, seed=22, device=dev).view(torch.uint8)
    bsf = synth.random_bytes(256 * moeq.sf_bytes(N, K // 32), 116, 126, seed=23, device=dev)
    asf = synth.random_bytes(moeq.sf_bytes(rows, K // 32), 118, 130, seed=24, device=dev)
    ms = time_kernel(lambda: moeq.grouped_matmul_blockscaled(
        "mxfp8", c, a.view(torch.uint8), asf, b8, bsf, None, ro_d, so_d, ids_d, N, K, rows,
        int(counts.max())), 10)
    wbytes = active_bytes + len(ids) * moeq.sf_bytes(N, K // 32)
    out["decode_mxfp8_512rows_224experts"] = {
        "ms": round(ms, 4), "GB/s_active_weights": round(wbytes / ms / 1e6, 1),
        "frac_hbm": round(wbytes / ms / 1e6 / hbm, 4),
        "frac_hbm_nominal": round(wbytes / ms / 1e6 / NOMINAL["hbm_gbs"], 4)}
    del a, b8, c
    # single-rank expert dispatch: 16384 tokens routed top-8 over 128
    # experts, hidden 4096 -> 131072 MXFP4 rows (routing + gather-quantize)
    tok = synth.bf16_normal((TOK4, K4), 1.0, seed=70, device=dev)
    tk = torch.from_numpy(synth.topk_ids(TOK4, TOPK4, E4, seed=0)).to(dev)
    n_rows = TOK4 * TOPK4
    rows_d = moeq.dispatch_scale_rows(TOK4, TOPK4, E4)
    q_d = torch.empty((n_rows, K4 // 2), dtype=torch.uint8, device=dev)
    sf_d = torch.empty(moeq.sf_bytes(rows_d, K4 // 32), dtype=torch.uint8, device=dev)
    ro_dd = torch.empty(E4 + 1, dtype=torch.int32, device=dev)
    eid_d = torch.empty(E4, dtype=torch.int32, device=dev)
    src_d = torch.empty(n_rows, dtype=torch.int32, device=dev)
    so_dd = torch.empty(E4 + 1, dtype=torch.int32, device=dev)
    t_route = time_kernel(lambda: moeq.route_topk(tk, ro_dd, eid_d, src_d, so_dd), 20, batch=8)
    dst_d = torch.empty(n_rows, dtype=torch.int32, device=dev)
    t_disp = time_kernel(lambda: moeq.dispatch_mxfp4(tok, tk, q_d, sf_d, ro_dd, eid_d, src_d,
                                                     so_dd, dst_info=dst_d), 10)
    used_sf = int(so_dd[-1].item()) // 128 * (K4 // 32 // 4) * 512
    nbytes = tok.numel() * 2 + q_d.numel() + used_sf + tk.numel() * 4
    out["dispatch_mxfp4_16384tok_top8_128experts"] = {
        "route_us": round(t_route * 1e3, 2), "ms": round(t_disp, 4),
        "GB/s": round(nbytes / t_disp / 1e6, 1), "bytes": nbytes,
        "bytes_note": "tokens read once (token-major quantization) + MXFP4 rows + used "
                      "scale rows + top-k ids",
        "timing": "route: median of 20 batches of 8 calls; dispatch: mean of 10 calls"}
    del tok
    return out


def mx_part(d, pk):
    """The up-projection in MXFP4 throughout on the same workload: MXFP4
    quantize of the activations, then the fused MXFP4 GEMM + SwiGLU + MXFP4
    requant (E8M0 block-32 scales; random weights and weight scales)."""
    from fp4_fp8_quantization_gb300 import moeq, synth
    T, N, rows = d["T"], d["N"], d["rows"]
    a = torch.empty_like(d["a"])
    asf = torch.empty(moeq.sf_bytes(rows, K4 // 32), dtype=torch.uint8, device="cuda")
    # weights: bf16 N(0, 0.02) quantized to MXFP4 by the library, one group per expert
    w = synth.bf16_normal((E4 * N, K4), 0.02, seed=501, device="cuda")
    offs = torch.arange(E4 + 1, dtype=torch.int32, device="cuda") * N
    eids = torch.arange(E4, dtype=torch.int32, device="cuda")
    b = torch.empty((E4 * N, K4 // 2), dtype=torch.uint8, device="cuda")
    bsf = torch.empty(moeq.sf_bytes(E4 * N, K4 // 32), dtype=torch.uint8, device="cuda")
    moeq.grouped_quantize("mxfp4", w, b, bsf, offs, offs, eids, None, E4, E4 * N, N)
    del w
    b = b.view(E4, N, K4 // 2)
    c = torch.empty((T, I4 // 2), dtype=torch.uint8, device="cuda")
    csf = torch.empty(moeq.sf_bytes(rows, I4 // 32), dtype=torch.uint8, device="cuda")

    def quant():
        moeq.grouped_quantize("mxfp4", d["x"], a, asf, d["ro"], d["so"], d["ids"], None, E4, rows)

    def fused():
        moeq.grouped_matmul_swiglu_mx("mxfp4", c, csf, a, asf, b, bsf, d["es"], d["ro"], d["so"],
                                      d["ids"], I4, K4, rows, d["mt"])

    y = torch.empty((T, N), dtype=torch.bfloat16, device="cuda")
    c2, csf2 = torch.empty_like(c), torch.empty_like(csf)

    def gemm():
        moeq.grouped_matmul_blockscaled("mxfp4", y, a, asf, b, bsf, d["es"], d["ro"], d["so"],
                                        d["ids"], N, K4, rows, d["mt"])

    def sw():
        moeq.swiglu_quantize_mx("mxfp4", c2, csf2, y, d["ro"], d["so"], d["ids"], E4, rows,
                                d["mt"])

    t_q = time_kernel(quant, 10)
    t_f = time_kernel(fused, 10)
    t_g = time_kernel(gemm, 10)
    t_s = time_kernel(sw, 10)
    fl = flops_up(d)
    sw_bytes = y.numel() * 2 + c2.numel() + csf2.numel()
    return {"quantize_mxfp4_ms": round(t_q, 4), "fused_gemm_swiglu_mxfp4_ms": round(t_f, 4),
            "fused_TFLOP/s": round(fl / t_f / 1e9, 1),
            "fused_frac_fp4_peak": round(fl / t_f / 1e9 / (pk["bf16"] * FP4_OVER_BF16), 4),
            "chained_gemm_bf16_ms": round(t_g, 4),
            "chained_swiglu_quantize_mxfp4_ms": round(t_s, 4),
            "chained_swiglu_quantize_mxfp4_GB/s": round(sw_bytes / t_s / 1e6, 1),
            "chained_swiglu_frac_hbm": round(sw_bytes / t_s / 1e6 / pk["hbm_gbs"], 4),
            "fused_bytes_equal_chained": bool(torch.equal(c, c2) and torch.equal(csf, csf2)),
            "weights": "bf16 N(0, 0.02) quantized to MXFP4 by the library's grouped quantizer"}


def chained_part(d, pk):
    from fp4_fp8_quantization_gb300 import moeq
    y = torch.empty((d["T"], d["N"]), dtype=torch.bfloat16, device="cuda")
    c = torch.empty_like(d["c"])
    csf = torch.empty_like(d["csf"])

    def gemm():
        moeq.grouped_matmul_blockscaled("nvfp4", y, d["a"], d["asf"], d["b"], d["bsf"], d["es"],
                                        d["ro"], d["so"], d["ids"], d["N"], K4, d["rows"], d["mt"])

    def sw():
        moeq.swiglu_quantize(c, csf, y, d["ots"], d["ro"], d["so"], d["ids"], E4, d["rows"],
                             d["mt"])

    t_g = time_kernel(gemm, 10)
    t_s = time_kernel(sw, 10)
    same = bool(torch.equal(c, d["c"]) and torch.equal(csf, d["csf"]))
    fl = flops_up(d)
    return {"gemm_bf16_ms": round(t_g, 4), "gemm_TFLOP/s": round(fl / t_g / 1e9, 1),
            "swiglu_quantize_ms": round(t_s, 4),
            "swiglu_quantize_GB/s": round((y.numel() * 2 + c.numel() + csf.numel()) / t_s / 1e6, 1),
            "swiglu_quantize_frac_hbm": round((y.numel() * 2 + c.numel() + csf.numel()) / t_s / 1e6
                                              / pk["hbm_gbs"], 4),
            "chained_total_ms": round(t_g + t_s, 4), "fused_bytes_equal_chained": same}


def layer_part(d):
    """Whole MoE FFN expert layer on the same batch: the up-projection step
    followed by the NVFP4 down-projection GEMM (K = I = 1536, N = 4096) on the
    fused kernel's packed output and its padded scales."""
    from fp4_fp8_quantization_gb300 import moeq, synth
    H = K4
    bd, bdsf, _ = nvfp4_expert_weights(E4, H, I4, 0.02, 90)
    esd = synth.uniform((E4,), 0.5, 2.0, seed=92, device="cuda")
    out = torch.empty((d["T"], H), dtype=torch.bfloat16, device="cuda")

    def down():
        moeq.grouped_matmul_blockscaled("nvfp4", out, d["c"], d["csf"], bd, bdsf, esd, d["ro"],
                                        d["so"], d["ids"], H, I4, d["rows"], d["mt"])

    def layer():
        up_projection_step(d)
        down()

    t_down = time_kernel(down, 10)
    t_layer = time_kernel(layer, 10)
    fl = flops_up(d) + 2.0 * d["T"] * H * I4
    return {"down_proj_ms": round(t_down, 4),
            "down_proj_TFLOP/s": round(2.0 * d["T"] * H * I4 / t_down / 1e9, 1),
            "layer_ms": round(t_layer, 4), "layer_TFLOP/s": round(fl / t_layer / 1e9, 1),
            "layer": "amax -> NVFP4 quantize -> fused gate/up GEMM + SwiGLU + requant -> "
                     "NVFP4 down-projection GEMM (bf16 out)"}


# --------------------------------------------------------- CPU baseline

def cpu_oracle_sample(d, groups, max_rows=None):
    """Times the CPU oracle on the chosen groups of the up-projection
    workload (amax -> NVFP4 quantize -> float64 GEMM -> SwiGLU -> requant).
    Returns (seconds, flops, rows)."""
    from oracle import formats as F
    from oracle import gemm as OG
    from oracle import quantize as Q
    from oracle import swiglu as S
    ro, ids = d["ro_h"], d["ids_h"]
    rows_list, eids = [], []
    for g in groups:
        r0, r1 = int(ro[g]), int(ro[g + 1])
        if max_rows:
            r1 = min(r1, r0 + max_rows)
        rows_list.append((r0, r1))
        eids.append(int(ids[g]))
    counts = [r1 - r0 for r0, r1 in rows_list]
    sro = np.concatenate([[0], np.cumsum(counts)]).astype(np.uint32)
    sids = np.arange(len(groups), dtype=np.int32)
    idx = np.concatenate([np.arange(r0, r1) for r0, r1 in rows_list])
    x = d["x"][torch.from_numpy(idx).cuda()].float().cpu().numpy()
    N = d["N"]
    per = (N + 127) // 128 * (K4 // 64) * 512
    eid_t = torch.tensor(eids, device="cuda")
    b = d["b"][eid_t].cpu().numpy()
    bsf = d["bsf"].view(E4, per)[eid_t].cpu().numpy().reshape(-1)
    es = d["es"][eid_t].cpu().numpy()
    ots = d["ots"][eid_t].cpu().numpy()
    t0 = time.perf_counter()
    so = Q.padded_scale_offsets(sro)
    ts = Q.tensor_scale_from_amax(Q.group_amax(x, sro, sids, len(groups)))
    qa, qsf = Q.grouped_quantize("nvfp4", x, sro, so, sids, ts)
    ybits = OG.grouped_matmul_blockscaled("nvfp4", qa, qsf, b, bsf, es, sro, so, sids, N=N, K=K4,
                                          scale_rows_total=int(so[-1]))
    S.swiglu_quantize(F.decode_bf16(ybits), ots, sro, so, sids)
    dt = time.perf_counter() - t0
    return dt, 2.0 * len(idx) * N * K4, len(idx)


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


# ------------------------------------------------------------------ arms

def run_reference(args, rank, world):
    if rank != 0:
        return
    d = up_projection_inputs(seed=0)
    g = int(np.argmax(np.diff(d["ro_h"].astype(np.int64))))
    rows_per_step = 256
    for _ in range(args.warmup):
        cpu_oracle_sample(d, [g], rows_per_step)
    tot, fl = 0.0, 0.0
    for _ in range(args.steps):
        dt, f, _ = cpu_oracle_sample(d, [g], rows_per_step)
        tot += dt
        fl += f
    value = fl / tot / 1e12
    sample = (f"{rows_per_step} rows of one expert group per step through the CPU oracle "
              "(amax, NVFP4 quantize, float64 GEMM, SwiGLU, NVFP4 requant)")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": tot / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "parallelism": f"replicas{args.gpus}"},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cpu_cores(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    emit(line, args)


def token_step(B, d):
    """The up-projection from tokens and their top-k ids: per-expert amax and
    NVFP4 quantization token-major (each token read once), routing, fused
    GEMM + SwiGLU + requant (the same GEMM work as up_projection_step)."""
    from fp4_fp8_quantization_gb300 import moeq
    moeq.grouped_amax_scale_topk(B["tok"], B["tk"], B["ts"], E4)   # each token read once
    moeq.route_topk(B["tk"], B["ro"], B["ids"], B["src"], B["so"], dst_info=B["dst"])
    moeq.quantize_topk("nvfp4", B["tok"], B["tk"], B["dst"], B["a"], B["asf"], B["ro"], B["so"],
                       B["ts"], E4)                                 # each token read once
    moeq.grouped_matmul_swiglu(B["c"], B["csf"], B["a"], B["asf"], d["b"], d["bsf"], d["es"],
                               d["ots"], B["ro"], B["so"], B["ids"], I4, K4, B["rows"])


def run_e2e(d, args, world, fl, form):
    """Pipelined steps from pinned host buffers through the public calls: the
    host->device copy of step i+1 (on MOEQ_E2E_COPY_STREAMS copy streams,
    one by default) overlaps the compute of step i, the device->host copy of
    the packed output and its scales runs on its own stream, two device
    buffer sets alternate; K steps are timed, as in the device-timed region.
    form "tokens": H2D of the 16384 bf16 tokens + top-8 ids, token_step;
    form "rows": H2D of the 131072 gathered rows + group offsets,
    up_projection_step."""
    from fp4_fp8_quantization_gb300 import moeq, synth
    # host-to-device copy streams (one: 0.972 against 0.990 ms per step with
    # the copy split over four)
    n_copy = int(os.environ.get("MOEQ_E2E_COPY_STREAMS", "1"))
    if form == "tokens":
        host = {"tok": synth.bf16_normal((TOK4, K4), 1.0, seed=80).pin_memory(),
                "tk": torch.from_numpy(synth.topk_ids(TOK4, TOPK4, E4, seed=0)).pin_memory()}
        split = "tok"
        rows = moeq.dispatch_scale_rows(TOK4, TOPK4, E4)
        n = TOK4 * TOPK4

        def buffers():
            return {"tok": torch.empty((TOK4, K4), dtype=torch.bfloat16, device="cuda"),
                    "tk": torch.empty((TOK4, TOPK4), dtype=torch.int32, device="cuda"),
                    "ro": torch.empty(E4 + 1, dtype=torch.int32, device="cuda"),
                    "ids": torch.empty(E4, dtype=torch.int32, device="cuda"),
                    "src": torch.empty(n, dtype=torch.int32, device="cuda"),
                    "dst": torch.empty(n, dtype=torch.int32, device="cuda"),
                    "so": torch.empty(E4 + 1, dtype=torch.int32, device="cuda"),
                    "ts": torch.empty(E4, device="cuda"),
                    "a": torch.empty((n, K4 // 2), dtype=torch.uint8, device="cuda"),
                    "asf": torch.empty(moeq.sf_bytes(rows, K4 // 16), dtype=torch.uint8,
                                       device="cuda"),
                    "c": torch.empty((n, I4 // 2), dtype=torch.uint8, device="cuda"),
                    "csf": torch.empty(moeq.sf_bytes(rows, I4 // 16), dtype=torch.uint8,
                                       device="cuda"),
                    "rows": rows}

        def compute(B):
            token_step(B, d)
    else:
        host = {"x": d["x"].cpu().pin_memory(), "ro": d["ro"].cpu().pin_memory(),
                "ids": d["ids"].cpu().pin_memory()}
        split = "x"

        def buffers():
            B = dict(d)
            for k in ("x", "ro", "ids", "so", "ts", "a", "asf", "c", "csf"):
                B[k] = torch.empty_like(d[k])
            return B

        def compute(B):
            up_projection_step(B)
    bufs = [buffers(), buffers()]
    chs = [torch.empty(bufs[0]["c"].shape, dtype=torch.uint8).pin_memory() for _ in range(2)]
    sfhs = [torch.empty(bufs[0]["csf"].shape, dtype=torch.uint8).pin_memory() for _ in range(2)]
    h2d_streams = [torch.cuda.Stream() for _ in range(n_copy)]
    d2h_stream = torch.cuda.Stream()
    comp = torch.cuda.current_stream()
    comp_done, d2h_done = [None, None], [None, None]
    steps = max(3, args.steps)  # the same K as the device-timed region

    def issue(i):
        b = i % 2
        B = bufs[b]
        total = host[split].shape[0]
        chunk = (total + n_copy - 1) // n_copy
        ready = []
        for j, st in enumerate(h2d_streams):
            if comp_done[b] is not None:       # step i-2 has finished reading buffer b
                st.wait_event(comp_done[b])
            with torch.cuda.stream(st):
                r0, r1 = j * chunk, min(total, (j + 1) * chunk)
                B[split][r0:r1].copy_(host[split][r0:r1], non_blocking=True)
                if j == 0:
                    for k, t in host.items():
                        if k != split:
                            B[k].copy_(t, non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(st)
                ready.append(ev)
        for ev in ready:
            comp.wait_event(ev)
        if d2h_done[b] is not None:             # outputs of step i-2 are on the host
            comp.wait_event(d2h_done[b])
        compute(B)
        cd = torch.cuda.Event()
        cd.record(comp)
        comp_done[b] = cd
        d2h_stream.wait_event(cd)
        with torch.cuda.stream(d2h_stream):
            chs[b].copy_(B["c"], non_blocking=True)
            sfhs[b].copy_(B["csf"], non_blocking=True)
            dd = torch.cuda.Event()
            dd.record(d2h_stream)
            d2h_done[b] = dd

    for i in range(2):
        issue(i)
    torch.cuda.synchronize()
    barrier(world)
    t0 = time.perf_counter()
    for i in range(steps):
        issue(i)
    torch.cuda.synchronize()
    e2e_s = max_over_ranks((time.perf_counter() - t0) / steps, world)
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = chs[0].numel() + sfhs[0].numel()
    # plain host->device bandwidth of the largest input, for context
    h0, h1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    h0.record()
    bufs[0][split].copy_(host[split], non_blocking=True)
    h1.record()
    torch.cuda.synchronize()
    big = host[split].numel() * host[split].element_size()
    out = {"value": round(world * fl / e2e_s / 1e12, 2), "unit": "TFLOP/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "ms_per_step": round(e2e_s * 1e3, 3),
           "input": ("16384 bf16 tokens x 4096 + top-8 expert ids (int32); per-expert amax, "
                     "routing and NVFP4 quantization of the routed rows on the GPU"
                     if form == "tokens" else
                     "131072 pre-gathered bf16 rows x 4096 + group offsets"),
           "pipelining": (f"H2D of step i+1 on {n_copy} copy stream(s) and D2H of step i-1 "
                          f"overlap the compute of step i"),
           "single_copy_h2d_GB/s": round(big / h0.elapsed_time(h1) / 1e6, 1)}
    # the same compute without the copies, device time (CUDA events)
    dev_ms = time_kernel(lambda: compute(bufs[0]), steps)
    out["device_step_ms"] = round(dev_ms, 4)
    out["device_step_note"] = ("the compute of one step alone, inputs resident; the row-level "
                               "step of `value` quantizes through the group lookup, the token "
                               "form reads each token once")
    del bufs
    return out


def run_moeq(args, rank, world):
    from fp4_fp8_quantization_gb300 import moeq
    moeq.lib()
    pk = peaks()
    d = up_projection_inputs(seed=1000 * rank)
    torch.cuda.synchronize()
    for _ in range(args.warmup):
        up_projection_step(d)
    torch.cuda.synchronize()
    clocks = Clocks(torch.cuda.current_device())
    clocks.start()
    time.sleep(0.3)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_push("moeq timed steps")   # one range around the timed region
    start.record()
    for i in range(args.steps):
        up_projection_step(d, evs[i])
    end.record()
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    barrier(world)
    ms_total = start.elapsed_time(end)
    clk = clocks.stop()
    ms_total = max_over_ranks(ms_total, world)
    ms_step = ms_total / args.steps
    fl = flops_up(d)
    value = world * fl / (ms_step * 1e-3) / 1e12

    t_pre = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    t_q = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
    t_f = statistics.mean(e[2].elapsed_time(e[3]) for e in evs)
    fp4_peak = pk["bf16"] * FP4_OVER_BF16
    achieved = fl / (t_f * 1e-3) / 1e12
    traffic, traffic_note = fused_traffic_bytes()
    sm_mhz = clk.get("sm_mhz") or 2070.0
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    mma_ceiling = FP4_FLOP_PER_SM_CYCLE * sms * sm_mhz * 1e6 / 1e12
    floor_ms, floor_tiles, floor_per_pair = fp4_schedule_floor(d["counts"], d["N"], K4, sms, sm_mhz)
    roof = {"kernel": "grouped_gemm_kernel<NVFP4, fused SwiGLU>", "bound": "tensor",
            "achieved": round(achieved, 1), "peak": round(fp4_peak, 1), "unit": "TFLOP/s",
            "frac": round(achieved / fp4_peak, 4), "traffic": traffic,
            "traffic_note": traffic_note,
            "peak_note": f"{pk['source']} bf16 burst x {FP4_OVER_BF16:g} nominal fp4/bf16 ratio",
            "frac_nominal": round(achieved / NOMINAL["fp4_tflops"], 4),
            "mma_ceiling": round(mma_ceiling, 1),
            "frac_mma_ceiling": round(achieved / mma_ceiling, 4),
            "mma_ceiling_note": "measured tcgen05 FP4 rate of this part (32768 flop per SM cycle: "
                                "one M128xN256xK64 MMA per 128 cycles, 2x FP8, 4x bf16) x SMs x the "
                                "run's median SM clock",
            "mma_schedule_floor_ms": round(floor_ms, 4),
            "frac_mma_schedule_floor": round(floor_ms / t_f, 4),
            "mma_schedule_floor_note": (
                f"MMA time of the kernel's own schedule at that rate: expert rows padded to "
                f"256-row CTA-pair tiles, {floor_tiles} pair tiles of 256x256 "
                f"({fl / (2 * FP4_PAIR_TILE_M * FP4_PAIR_TILE_N * K4):.0f} without padding), "
                f"{floor_per_pair} on the busiest of {sms // 2} pairs, K/64 MMAs of 128 cycles "
                f"each"),
            "algorithmic_flops_per_launch": fl}
    breakdown = {"offsets_amax_ms": round(t_pre, 4), "quantize_nvfp4_ms": round(t_q, 4),
                 "fused_gemm_swiglu_ms": round(t_f, 4)}

    # end to end from pinned host memory: the layer's real input, the
    # tokens and their top-k expert ids (routing and row gather on the GPU);
    # and, for comparison, the 131072 pre-gathered rows of the timed step
    e2e = run_e2e(d, args, world, fl, "tokens")
    e2e["pregathered_rows_input"] = run_e2e(d, args, world, fl, "rows")

    extra = {}
    if rank == 0 and not args.no_parts:
        extra["chained_same_workload"] = chained_part(d, pk)
        extra["mxfp4_same_workload"] = mx_part(d, pk)
        extra["moe_layer_same_workload"] = layer_part(d)
        extra.update(parts(pk, None))
    err = moeq.get_device_error()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        lens = np.diff(d["ro_h"].astype(np.int64))
        groups = list(np.argsort(-lens)[:4])
        dt, f, n = cpu_oracle_sample(d, groups)
        cpu = {"value": round(f / dt / 1e12, 6), "unit": "TFLOP/s", "cores": cpu_cores(),
               "kind": "oracle", "seconds": round(dt, 2),
               "sample": f"{n} rows (the 4 largest of 128 expert groups) through the CPU oracle: "
                         "amax, NVFP4 quantize, float64 GEMM, SwiGLU, NVFP4 requant"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "nvfp4",
            "data": "synthetic",
            "config": {"workload": WORKLOAD, "experts": E4, "tokens": TOK4, "top_k": TOPK4,
                       "rows": d["T"], "K": K4, "N": d["N"], "global_batch": world * TOK4,
                       "parallelism": f"replicas{world}",
                       "l2": "inputs larger than L2 (1.07 GB bf16 activations, 0.81 GB FP4 weights)"},
            "gpu_launches": KERNELS_PER_STEP * args.steps,
            "clocks": clk, "roofline": roof, "breakdown": breakdown, "e2e": e2e,
            "cpu_baseline": cpu, "parts": extra, "device_error": err,
        }
        emit(line, args)


def run_profile_case(args):
    """Small cases for profiler captures: same kernels and launch shapes as
    the bench, fewer experts / rows (inputs still larger than L2)."""
    from fp4_fp8_quantization_gb300 import moeq, synth
    dev = "cuda"
    u32 = lambda a: torch.from_numpy(np.asarray(a, np.uint32).view(np.int32)).to(dev)
    if args.profile == "dispatch":
        # single-rank MXFP4 dispatch: 16384 tokens x 4096, top-8 of 128 experts
        tok = synth.bf16_normal((TOK4, K4), 1.0, seed=70, device=dev)
        tk = torch.from_numpy(synth.topk_ids(TOK4, TOPK4, E4, seed=0)).to(dev)
        n = TOK4 * TOPK4
        rows = moeq.dispatch_scale_rows(TOK4, TOPK4, E4)
        q = torch.empty((n, K4 // 2), dtype=torch.uint8, device=dev)
        sf = torch.empty(moeq.sf_bytes(rows, K4 // 32), dtype=torch.uint8, device=dev)
        i32 = dict(dtype=torch.int32, device=dev)
        ro, eids, src, so = (torch.empty(E4 + 1, **i32), torch.empty(E4, **i32),
                             torch.empty(n, **i32), torch.empty(E4 + 1, **i32))
        dst = torch.empty(n, **i32)
        fn = lambda: moeq.dispatch_mxfp4(tok, tk, q, sf, ro, eids, src, so, dst_info=dst)
    elif args.profile in ("fused", "fused_mx", "chained", "quantize", "swiglu"):
        # 32 experts, 4096 tokens top-8 -> 32768 rows, K 4096, I 1536
        counts = synth.routing_counts(4096, 8, 32, seed=0)
        ro, ids = synth.ragged_groups(counts)
        T, N, rows = int(ro[-1]), 2 * I4, int(sum((int(c) + 127) // 128 * 128 for c in counts))
        ro_d, ids_d = u32(ro), torch.from_numpy(ids).to(dev)
        so_d = torch.empty(len(ids) + 1, dtype=torch.int32, device=dev)
        moeq.padded_scale_offsets(ro_d, so_d)
        if args.profile == "quantize":
            # the grouped-quantize workload itself: 8 experts, 4096 tokens
            # top-2 -> 8192 rows, hidden 4096 (ncu flushes caches per pass)
            counts = synth.routing_counts(4096, 2, 8, seed=0)
            ro, ids = synth.ragged_groups(counts)
            T, rows = int(ro[-1]), int(sum((int(c) + 127) // 128 * 128 for c in counts if c))
            ro_d, ids_d = u32(ro), torch.from_numpy(ids).to(dev)
            so_d = torch.empty(len(ids) + 1, dtype=torch.int32, device=dev)
            moeq.padded_scale_offsets(ro_d, so_d)
            x = synth.bf16_normal((T, K4), 1.0, seed=1, device=dev)
            ts = synth.uniform((8,), 0.001, 0.002, seed=2, device=dev)
            q = torch.empty((T, K4 // 2), dtype=torch.uint8, device=dev)
            sf = torch.empty(moeq.sf_bytes(rows, K4 // 16), dtype=torch.uint8, device=dev)
            fn = lambda: moeq.grouped_quantize("nvfp4", x, q, sf, ro_d, so_d, ids_d, ts, 8, rows)
        elif args.profile == "fused_mx":
            # the fused MXFP4 GEMM + SwiGLU + MXFP4 requant on the same shapes
            a = synth.random_fp4_packed((T, K4 // 2), seed=1, device=dev)
            asf = synth.random_bytes(moeq.sf_bytes(rows, K4 // 32), 118, 130, seed=2, device=dev)
            b = synth.random_fp4_packed((32, N, K4 // 2), seed=3, device=dev)
            bsf = synth.random_bytes(32 * moeq.sf_bytes(N, K4 // 32), 116, 126, seed=4,
                                     device=dev)
            es = synth.uniform((32,), 0.5, 2.0, seed=5, device=dev)
            c = torch.empty((T, I4 // 2), dtype=torch.uint8, device=dev)
            csf = torch.empty(moeq.sf_bytes(rows, I4 // 32), dtype=torch.uint8, device=dev)
            fn = lambda: moeq.grouped_matmul_swiglu_mx("mxfp4", c, csf, a, asf, b, bsf, es, ro_d,
                                                       so_d, ids_d, I4, K4, rows)
        else:
            a = synth.random_fp4_packed((T, K4 // 2), seed=1, device=dev)
            asf = synth.random_bytes(moeq.sf_bytes(rows, K4 // 16), 0x20, 0x30, seed=2, device=dev)
            b = synth.random_fp4_packed((32, N, K4 // 2), seed=3, device=dev)
            bsf = synth.random_bytes(32 * moeq.sf_bytes(N, K4 // 16), 0x18, 0x28, seed=4,
                                     device=dev)
            es = synth.uniform((32,), 0.5, 2.0, seed=5, device=dev)
            ots = synth.uniform((32,), 1.0, 4.0, seed=6, device=dev)
            c = torch.empty((T, I4 // 2), dtype=torch.uint8, device=dev)
            csf = torch.empty(moeq.sf_bytes(rows, I4 // 16), dtype=torch.uint8, device=dev)
            if args.profile == "fused":
                fn = lambda: moeq.grouped_matmul_swiglu(c, csf, a, asf, b, bsf, es, ots, ro_d,
                                                        so_d, ids_d, I4, K4, rows)
            elif args.profile == "swiglu":
                # the chained SwiGLU + NVFP4 requant on a 201 MB bf16 gate/up matrix
                y = synth.bf16_normal((T, N), 1.0, seed=7, device=dev)
                fn = lambda: moeq.swiglu_quantize(c, csf, y, ots, ro_d, so_d, ids_d, 32, rows)
            else:
                y = torch.empty((T, N), dtype=torch.bfloat16, device=dev)
                fn = lambda: moeq.grouped_matmul_blockscaled("nvfp4", y, a, asf, b, bsf, es, ro_d,
                                                             so_d, ids_d, N, K4, rows)
    else:
        # FP8 rowwise: 16 experts, 2048 tokens top-8 Zipf -> 16384 rows (fp8) or
        # decode-shaped 64 experts, 16 tokens top-8 -> 128 rows; K 7168, N 4096
        if args.profile == "fp8":
            counts = synth.routing_counts(2048, 8, 16, seed=0, zipf_s=1.1)
            E = 16
        else:
            counts = synth.routing_counts(16, 8, 64, seed=0)
            E = 64
        ro, ids = synth.ragged_groups(counts)
        T, N, K = int(ro[-1]), 4096, 7168
        a, sa = synth.fp8_rowwise((T, K), 1.0, seed=1, device=dev)
        b, sb = synth.fp8_rowwise((E, N, K), 0.02, seed=2, device=dev)
        c = torch.empty((T, N), dtype=torch.bfloat16, device=dev)
        ro_d, ids_d = u32(ro), torch.from_numpy(ids).to(dev)
        fn = lambda: moeq.grouped_matmul_rowwise_fp8(c, a, b, sa, sb.reshape(E, N), ro_d, ids_d,
                                                     int(counts.max()))
    torch.cuda.synchronize()
    for _ in range(args.warmup + args.steps):
        fn()
    torch.cuda.synchronize()
    assert moeq.get_device_error() == 0
    print(f"profile case {args.profile}: {args.warmup} + {args.steps} launches ok")


def main():
    args = parse_args()
    if args.profile:
        torch.cuda.set_device(0)
        run_profile_case(args)
        return
    rank, world = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_moeq(args, rank, world)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
