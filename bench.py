#!/usr/bin/env python3
"""Benchmark of the MXFP4 dense linear on GB300.

Headline workload (the decode sweep): M in {1, 4, 16, 32, 64} x (N, K) in
{(14336, 5120), (5120, 14336), (34816, 5120)}: bf16 activations ~N(0,1) with
1% outlier channels (x20), FP4 weights with E8M0 scales 2^U{-8..2}, bf16 out.
One step runs the whole path once per case: per-1x32 activation quantization
then the W4A4 GEMM (weights repacked once at load time, off the clock).

Metric: weight-stream GB/s = algorithmic bytes (packed weights + bf16
activations + bf16 outputs) / time.  Every case of a step reads its own
copy of the packed weights (15 distinct buffers, 0.87 GB), so no weight is
re-read from L2 between uses.

The timed region is the replay of CUDA graphs holding the steps; the
roofline's achieved bandwidth is a step's algorithmic bytes over the average
step time there.  `e2e` repeats the step through the public API with eager
calls, every step copying its activations from pinned host memory and its
outputs back, the copies of neighbouring steps overlapping the calls on
copy streams.  Secondary lines: prefill TFLOPS (M in {2048, 8192}, with bias),
the A16WFP4 BMM, the fused RMSNorm producer and the MXFP4-output GEMM.
`--impl reference` times the CPU oracle on the same workload.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

DECODE_MS = (1, 4, 16, 32, 64)
DECODE_NK = ((14336, 5120), (5120, 14336), (34816, 5120))
PREFILL_MS = (2048, 8192)
W_SCALE_DECODE = (-8, 2)
W_SCALE_PREFILL = (-6, 0)
FP4_OVER_BF16 = 6.0            # nominal dense FP4 / BF16 tensor throughput on GB300 (13.5 / 2.25 PF)
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
METRIC = "MXFP4 GEMM TFLOPS (prefill) & weight-stream GB/s (decode M<=64), 1xGB300"


def ceil_div(a, b):
    return -(-a // b)


def linear_bytes(M, N, K):
    """Algorithmic bytes of one dense-linear call fed bf16 activations."""
    return N * K // 2 + N * ceil_div(K, 32) + M * K * 2 + M * N * 2


def gemm_kernel_bytes(M, N, K):
    """Algorithmic bytes of the GEMM kernel alone (activations already quantized)."""
    return N * K // 2 + N * ceil_div(K, 32) + M * K // 2 + M * ceil_div(K, 32) + M * N * 2


def launches_per_call(M, N, K):
    """Kernels one mxfp4_gemm call with a bf16 input launches.  M <= 8: one
    (quantization, GEMM and split-tile sums in one kernel); 8 < M <= 64: the
    quantizer, then the decode GEMM.  Larger M: quantizer, GEMM, and the fix-up
    when a CTA boundary cuts a tile (none when the GEMM takes whole tiles per
    CTA, as it does when that leaves under 8% of the last wave idle)."""
    import torch
    kt = ceil_div(K, 256)
    if M <= 64:
        return 1 if M <= 8 else 2
    grid = min(torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count, 256)
    tiles = ceil_div(M, 128) * ceil_div(N, 256)
    total = tiles * kt
    grid = min(grid, total)
    waves = tiles / grid
    if tiles >= grid and (ceil_div(tiles, grid) - waves) / waves < 0.08:
        return 2                                   # whole tiles per CTA: no fix-up
    split = any(((c * total) // grid) % kt for c in range(1, grid))
    return 2 + (1 if split else 0)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


def kernel_source_hash():
    """sha256 (first 16 hex digits) of the decode kernel's sources, with //
    comments and blank lines dropped: a comment edit does not change the kernel."""
    h = hashlib.sha256()
    for f in ("decode.cu", "gemm_common.cuh", "quant_math.cuh", "ptx.cuh", "internal.h"):
        for line in open(os.path.join(ROOT, "mxfp4_quantized_gemm_gb300", "csrc", f), encoding="utf-8"):
            code = line.split("//", 1)[0].rstrip()
            if code:
                h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def recorded_traffic(cases):
    """DRAM bytes per decode launch, averaged over `cases`: the DRAM/algorithmic
    ratio ncu measured for each (N,K) (profiles/decode_gemm_traffic.txt) times
    each case's algorithmic bytes.  None unless the ratios were taken on this
    kernel source."""
    p = os.path.join(ROOT, "profiles", "decode_gemm_traffic.txt")
    try:
        fields = {}
        for line in open(p):
            if "=" in line and not line.startswith("#"):
                k, v = line.split("=", 1)
                fields[k.strip()] = v.strip()
        if fields.get("source_hash") != kernel_source_hash():
            return None
        tot = sum(float(fields[f"ratio_{N}_{K}"]) * linear_bytes(M, N, K) for (M, N, K) in cases)
        return round(tot / len(cases))
    except Exception:
        return None


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None
        # raw samples: $BENCH_CLOCK_DIR/clocks_<pid>.csv if set, else a temporary file
        d = os.environ.get("BENCH_CLOCK_DIR") or tempfile.gettempdir()
        self.path = os.path.join(d, f"clocks_{os.getpid()}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        self.proc.wait()
        self.fh.close()
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        loaded = [v for v in sm if v > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ dist
def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def dist_max(value: float, world: int) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def throughput_gbs(bytes_per_step: float, steps: int, world: int, ms_max: float) -> float:
    """Whole-job GB/s: every rank runs `steps` steps of `bytes_per_step`; `ms_max` is
    the slowest rank's time for them (weak scaling: work per rank is fixed)."""
    return bytes_per_step * steps * world / (ms_max * 1e-3) / 1e9


def dist_barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------ ours
def make_event(torch, external):
    try:
        return torch.cuda.Event(enable_timing=True, external=external)
    except TypeError:
        return torch.cuda.Event(enable_timing=True)


def run_ours(args, world, rank, local):
    import numpy as np
    import torch

    import __graft_entry__
    __graft_entry__.build()
    from mxfp4_quantized_gemm_gb300 import capi, synth

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    hbm_peak, bf16_peak, bf16_sust, peak_src = load_peaks()

    def to_dev(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    # ---- packed weights: one distinct copy per case (15 buffers)
    cases = []
    for M in DECODE_MS:
        for (N, K) in DECODE_NK:
            cases.append((M, N, K))
    packed_master = {}
    for (N, K) in DECODE_NK:
        wc = synth.weight_codes(N, K, seed=0, tensor_id=2)
        ws = synth.weight_scales(N, K, *W_SCALE_DECODE, seed=0, tensor_id=3)
        buf = torch.empty(capi.mxfp4_packed_weight_bytes(1, N, K), dtype=torch.uint8, device=dev)
        capi.mxfp4_pack_weights(to_dev(wc), to_dev(ws), 1, N, K, buf)
        packed_master[(N, K)] = buf
    torch.cuda.synchronize()

    # every case's activations and outputs live in one device buffer each (and
    # one pinned host buffer each, for the end-to-end step)
    x_sizes = [M * K for (M, N, K) in cases]
    o_sizes = [M * N for (M, N, K) in cases]
    x_all = torch.empty(sum(x_sizes), dtype=torch.bfloat16, device=dev)
    o_all = torch.empty(sum(o_sizes), dtype=torch.bfloat16, device=dev)
    x_all_host = torch.empty(sum(x_sizes), dtype=torch.bfloat16).pin_memory()
    o_all_host = torch.empty(sum(o_sizes), dtype=torch.bfloat16).pin_memory()
    state = []
    xo = oo = 0
    for i, (M, N, K) in enumerate(cases):
        x_bits = synth.activations(M, K, seed=1 + i, tensor_id=1, outlier_frac=0.01)
        ws_bytes = capi.mxfp4_gemm_workspace_bytes(M, N, K)
        x_all_host[xo:xo + M * K].copy_(synth.bf16_tensor(x_bits).reshape(-1))
        state.append({
            "M": M, "N": N, "K": K,
            "packed": packed_master[(N, K)].clone(),
            "x": x_all[xo:xo + M * K],
            "out": o_all[oo:oo + M * N],
            "ws": torch.zeros(ws_bytes, dtype=torch.uint8, device=dev),
            "ws_bytes": ws_bytes,
        })
        xo += M * K
        oo += M * N
    x_all.copy_(x_all_host)
    del packed_master
    torch.cuda.synchronize()

    stream = torch.cuda.Stream(device=dev)
    sptr = stream.cuda_stream

    def step(events=None):
        for j, c in enumerate(state):
            if events is not None:
                events[j][0].record(stream)
            # the user's call: bf16 activations in, quantization inside the call
            capi.mxfp4_gemm(c["x"], c["K"], None, None, 0, c["packed"], None, c["out"], c["N"], c["M"], c["N"],
                            c["K"], c["ws"], c["ws_bytes"], sptr)
            if events is not None:
                events[j][1].record(stream)

    # eager warm-up (sets kernel attributes, checks for device errors)
    with torch.cuda.stream(stream):
        for _ in range(3):
            step()
    stream.synchronize()
    assert capi.mxfp4_get_device_error(sptr) == capi.OK

    # graph of G steps; the last one carries timing events at case boundaries
    # (each case is one decode kernel launch)
    K_steps, W_steps = args.steps, args.warmup
    G = max(g for g in range(1, min(K_steps, 50) + 1) if K_steps % g == 0)
    ev = [[make_event(torch, True), make_event(torch, True)] for _ in state]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            for g in range(G):
                step(ev if g == G - 1 else None)
    stream.synchronize()
    replays = K_steps // G
    warm_replays = max(1, ceil_div(W_steps, G))
    with torch.cuda.stream(stream):
        for _ in range(warm_replays):
            graph.replay()
    stream.synchronize()

    clocks = ClockSampler(local)
    clocks.start()
    t0, t1 = make_event(torch, False), make_event(torch, False)
    dist_barrier(world)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        t0.record(stream)
        for _ in range(replays):
            graph.replay()
        t1.record(stream)
    torch.cuda.synchronize()
    dist_barrier(world)
    clk = clocks.stop()
    assert capi.mxfp4_get_device_error(sptr) == capi.OK
    ms_total = t0.elapsed_time(t1)
    ms_total = dist_max(ms_total, world)

    bytes_step = sum(linear_bytes(c["M"], c["N"], c["K"]) for c in state)
    value = throughput_gbs(bytes_step, K_steps, world, ms_total)

    # spread: the same K steps timed four more times right after the timed
    # region (reported beside `value`, which is the first measurement only)
    repeat_gbs = []
    for _ in range(4):
        r0, r1 = make_event(torch, False), make_event(torch, False)
        dist_barrier(world)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            r0.record(stream)
            for _ in range(replays):
                graph.replay()
            r1.record(stream)
        torch.cuda.synchronize()
        repeat_gbs.append(round(throughput_gbs(bytes_step, K_steps, world, dist_max(r0.elapsed_time(r1), world)), 2))
    assert capi.mxfp4_get_device_error(sptr) == capi.OK

    # per-case durations: events of the last step of the last replay (inside
    # the timed region); the events stop consecutive calls from overlapping, so
    # these are isolated-call times, a diagnostic
    per_case_ms = [ev[j][0].elapsed_time(ev[j][1]) for j in range(len(state))]
    # roofline: algorithmic bytes of a step over this GPU's average step time
    # in the timed region (every launch there belongs to the decode path)
    achieved = bytes_step / (ms_total / K_steps * 1e-3) / 1e9
    traffic = recorded_traffic([(c['M'], c['N'], c['K']) for c in state])

    # ---- e2e through the public API, pipelined as a serving loop runs it:
    # every step copies its activations host -> device (pinned, one copy),
    # makes the 15 calls (quantization inside) and copies all outputs back
    # (one copy).  Two device buffer sets and one stream per copy direction
    # let the H2D copy of step i + 1 and the D2H copy of step i - 1 run while
    # step i computes; events keep each buffer from being overwritten before
    # it is consumed.
    e2e_steps = max(3, min(args.e2e_steps, K_steps))
    h2d = x_all.numel() * 2
    d2h = o_all.numel() * 2
    xb = [x_all, torch.empty_like(x_all)]
    ob = [o_all, torch.empty_like(o_all)]
    o_host = [o_all_host, torch.empty_like(o_all_host).pin_memory()]
    views = []
    for b in range(2):
        vs, xo, oo = [], 0, 0
        for c in state:
            vs.append((xb[b][xo:xo + c["M"] * c["K"]], ob[b][oo:oo + c["M"] * c["N"]]))
            xo += c["M"] * c["K"]
            oo += c["M"] * c["N"]
        views.append(vs)
    h2d_stream = torch.cuda.Stream(device=dev)
    d2h_stream = torch.cuda.Stream(device=dev)
    ev_h2d = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_d2h = [torch.cuda.Event() for _ in range(2)]

    def e2e_run(n):
        for b in range(2):                       # all buffers free
            ev_comp[b].record(stream)
            ev_d2h[b].record(d2h_stream)
        for i in range(n):
            b = i & 1
            with torch.cuda.stream(h2d_stream):
                h2d_stream.wait_event(ev_comp[b])           # step i - 2 no longer reads xb[b]
                xb[b].copy_(x_all_host, non_blocking=True)
                ev_h2d[b].record(h2d_stream)
            stream.wait_event(ev_h2d[b])
            stream.wait_event(ev_d2h[b])                    # ob[b] of step i - 2 is on the host
            for c, (xv, ov) in zip(state, views[b]):
                capi.mxfp4_gemm(xv, c["K"], None, None, 0, c["packed"], None, ov, c["N"], c["M"], c["N"],
                                c["K"], c["ws"], c["ws_bytes"], sptr)
            ev_comp[b].record(stream)
            with torch.cuda.stream(d2h_stream):
                d2h_stream.wait_event(ev_comp[b])
                o_host[b].copy_(ob[b], non_blocking=True)
                ev_d2h[b].record(d2h_stream)
        stream.wait_event(ev_d2h[(n - 1) & 1])             # the last results are on the host
        stream.wait_event(ev_d2h[n & 1])

    e2e_run(3)
    torch.cuda.synchronize()
    e0, e1 = make_event(torch, False), make_event(torch, False)
    e0.record(stream)
    e2e_run(e2e_steps)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = dist_max(e0.elapsed_time(e1), world)
    e2e_value = throughput_gbs(bytes_step, e2e_steps, world, e2e_ms)

    extra = {}
    if not args.no_secondary:
        extra["prefill"] = run_prefill(args, torch, np, capi, synth, dev, stream, bf16_peak, peak_src)
        extra["bmm"] = run_bmm(args, torch, np, capi, synth, dev, stream, hbm_peak, bf16_sust)
        extra["rmsnorm_quant"] = run_norm_quant(args, torch, np, capi, synth, dev, stream, hbm_peak)
        extra["gemm_mxfp4_out"] = run_mxfp4_out(args, torch, np, capi, synth, dev, stream, hbm_peak)

    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K_steps,
        "warmup": W_steps,
        "ms_per_step": round(ms_total / K_steps, 5),
        "value_spread": {"repeats_after_timed_region": repeat_gbs,
                         "min": min([round(value, 2)] + repeat_gbs), "max": max([round(value, 2)] + repeat_gbs),
                         "note": "the same K steps timed four more times, back to back after the timed region"},
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e2m1xe2m1->f32 (bf16 out)",
        "data": "synthetic",
        "config": {
            "workload": "decode W4A4 sweep: M in {1,4,16,32,64} x (N,K) in {(14336,5120),(5120,14336),(34816,5120)}; "
                        "bf16 activations N(0,1) with 1% outlier channels x20, quantized per call; FP4 weights, "
                        "E8M0 scales 2^U{-8..2}; bf16 out, no bias",
            "cases_per_step": len(state),
            "l2": "inputs larger than L2: each case reads its own packed-weight copy (15 buffers, "
                  f"{sum(c['packed'].numel() for c in state) / 1e9:.2f} GB per step)",
            "timing": f"CUDA graph of {G} steps replayed {replays}x, CUDA events around the replays; each case "
                      "is one mxfp4_gemm call: one decode_kernel launch for M <= 8 (quantization, GEMM and "
                      "split-K sums inside), quant_kernel then decode_kernel for 8 < M <= 64; consecutive "
                      "launches overlap by programmatic dependent launch",
            "parallelism": f"replicas x{world}",
        },
        "roofline": {
            "bound": "hbm",
            "kernel": "decode_kernel (with quant_kernel before it for 8 < M <= 64): activation quantization, "
                      "GEMM, split-K sums, bias, bf16 store",
            "duration": "average time per step of the timed region (all 15 calls), CUDA events on the launching "
                        "stream",
            "bytes_per_launch": "N*K/2 + N*K/32 (packed W) + 2*M*K (bf16 A) + 2*M*N (bf16 out)",
            "achieved": round(achieved, 1),
            "peak": hbm_peak,
            "peak_source": f"{peak_src} hbm_gbs",
            "unit": "GB/s",
            "frac": round(achieved / hbm_peak, 4),
            "traffic": traffic,
            "per_case_us_isolated": {f"M{c['M']}_N{c['N']}_K{c['K']}": round(ms * 1e3, 2)
                                     for c, ms in zip(state, per_case_ms)},
        },
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": e2e_steps,
                "note": "eager public-API calls; each step's H2D (pinned) and D2H copies run on their own "
                        "streams, overlapping the neighbouring steps' calls (two buffer sets)"},
        "gpu_launches": sum(launches_per_call(c["M"], c["N"], c["K"]) for c in state) * K_steps,
        "clocks": clk,
    }
    line.update(extra)
    if rank == 0 and not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    return line, rank


def measured_mxf4_peak(torch, capi, dev):
    """Dense kind::mxf4 rate of this GPU (TFLOP/s): 128x256x64 block-scaled MMAs issued back to back
    on every SM (mxfp4_diag_tensor_rate, 16 per step, depth 32), median of three launches."""
    var = next(v for v in range(capi.mxfp4_diag_tensor_rate_variants())
               if capi.mxfp4_diag_tensor_rate_info(v) == {"pair": 0, "kind": 0, "mmas": 16, "copies": 0, "form": 0,
                                                           "issuers": 1, "split": 0})
    ns = torch.zeros(capi.mxfp4_diag_max_units(), dtype=torch.int64, device=dev)
    steps, meds = 2000, []
    for _ in range(3):
        ns.zero_()
        units = capi.mxfp4_diag_tensor_rate(var, 256, steps, 32, ns)
        torch.cuda.synchronize()
        v = [x for x in ns[:units].cpu().tolist() if x > 0]
        meds.append(statistics.median(v))
    return units * 16 * 2.0 * 128 * 256 * 64 * steps / (statistics.median(meds) * 1e-9) / 1e12


def run_prefill(args, torch, np, capi, synth, dev, stream, bf16_peak, peak_src):
    sptr = stream.cuda_stream
    fp4_nominal = bf16_peak * FP4_OVER_BF16
    fp4_peak = measured_mxf4_peak(torch, capi, dev)
    results = {}
    tot_flop, tot_ms = 0.0, 0.0
    for (N, K) in DECODE_NK:
        wc = synth.weight_codes(N, K, seed=0, tensor_id=2)
        ws = synth.weight_scales(N, K, *W_SCALE_PREFILL, seed=0, tensor_id=3)
        packed = torch.empty(capi.mxfp4_packed_weight_bytes(1, N, K), dtype=torch.uint8, device=dev)
        capi.mxfp4_pack_weights(torch.from_numpy(wc).to(dev), torch.from_numpy(ws).to(dev), 1, N, K, packed)
        bias = synth.bf16_tensor(synth.bias(N, seed=0)).to(dev)
        for M in PREFILL_MS:
            x = synth.bf16_tensor(synth.activations(M, K, seed=M, tensor_id=1)).to(dev)
            out = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
            wsb = capi.mxfp4_gemm_workspace_bytes(M, N, K)
            work = torch.zeros(wsb, dtype=torch.uint8, device=dev)

            def call():
                capi.mxfp4_gemm(x, K, None, None, 0, packed, bias, out, N, M, N, K, work, wsb, sptr)

            with torch.cuda.stream(stream):
                for _ in range(3):
                    call()
            stream.synchronize()
            reps = 20
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                a.record(stream)
                for _ in range(reps):
                    call()
                b.record(stream)
            stream.synchronize()
            ms = a.elapsed_time(b) / reps
            flop = 2.0 * M * N * K
            results[f"M{M}_N{N}_K{K}"] = {"us": round(ms * 1e3, 1), "tflops": round(flop / (ms * 1e-3) / 1e12, 1)}
            tot_flop += flop
            tot_ms += ms
        del packed
    tflops = tot_flop / (tot_ms * 1e-3) / 1e12
    return {"metric": "prefill W4A4 TFLOPS (quant + GEMM + bias), M in {2048, 8192}", "value": round(tflops, 1),
            "unit": "TFLOP/s", "peak": round(fp4_peak, 1),
            "peak_source": "measured in this run: dense kind::mxf4 128x256x64 MMAs back to back on every SM "
                           "(mxfp4_diag_tensor_rate)",
            "frac": round(tflops / fp4_peak, 4),
            "peak_bf16_x6": round(fp4_nominal, 1),
            "frac_of_bf16_x6": round(tflops / fp4_nominal, 4),
            "peak_bf16_x6_source": f"{peak_src} bf16_tflops x {FP4_OVER_BF16} (nominal dense FP4/BF16)",
            "cases": results,
            "l2": "back-to-back calls on one weight copy (compute-bound)"}


def run_bmm(args, torch, np, capi, synth, dev, stream, hbm_peak, bf16_sust):
    sptr = stream.cuda_stream
    B = 64
    res = {}
    tot_bytes, tot_ms = 0.0, 0.0
    for name, N, K, layout in (("kup", 512, 192, capi.OUT_BMN), ("vup", 256, 512, capi.OUT_MBN)):
        wc = synth.weight_codes(N, K, seed=1, batch=B)
        ws = synth.weight_scales(N, K, -6, 0, seed=1, batch=B)
        packed = torch.empty(capi.mxfp4_packed_weight_bytes(B, N, K), dtype=torch.uint8, device=dev)
        capi.mxfp4_pack_weights(torch.from_numpy(wc).to(dev), torch.from_numpy(ws).to(dev), B, N, K, packed)
        for M in (16, 4096):
            x = synth.bf16_tensor(synth.bmm_activations(B, M, K, seed=M)).to(dev)
            out = torch.empty(B * M * N, dtype=torch.bfloat16, device=dev)

            def call():
                capi.a16wfp4_bmm(x, packed, out, B, M, N, K, layout, sptr)

            with torch.cuda.stream(stream):
                for _ in range(3):
                    call()
            stream.synchronize()
            reps = 20
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                a.record(stream)
                for _ in range(reps):
                    call()
                b.record(stream)
            stream.synchronize()
            ms = a.elapsed_time(b) / reps
            nbytes = B * M * K * 2 + B * N * K * (0.5 + 1 / 32) + B * M * N * 2
            res[f"{name}_M{M}"] = {"us": round(ms * 1e3, 1), "gbs": round(nbytes / (ms * 1e-3) / 1e9, 1),
                                   "tflops": round(2.0 * B * M * N * K / (ms * 1e-3) / 1e12, 1)}
            tot_bytes += nbytes
            tot_ms += ms
    gbs = tot_bytes / (tot_ms * 1e-3) / 1e9
    return {"metric": "A16WFP4 MLA absorbed BMM GB/s, B=64, M in {16, 4096}", "value": round(gbs, 1),
            "unit": "GB/s", "peak": hbm_peak, "frac": round(gbs / hbm_peak, 4), "cases": res,
            "l2": "back-to-back calls; x and out exceed L2 at M=4096"}


def run_mxfp4_out(args, torch, np, capi, synth, dev, stream, hbm_peak):
    """mxfp4_gemm_mxfp4_out against mxfp4_gemm (bf16 out) on decode and prefill
    shapes (bf16 activations, N = 14336, K = 5120, no bias); 4 weight copies
    rotate so that every call reads its weights from HBM; 20 calls replay from
    a CUDA graph."""
    sptr = stream.cuda_stream
    N, K, copies, reps = 14336, 5120, 4, 20
    wc = synth.weight_codes(N, K, seed=0)
    ws = synth.weight_scales(N, K, *W_SCALE_DECODE, seed=0)
    pk0 = torch.empty(capi.mxfp4_packed_weight_bytes(1, N, K), dtype=torch.uint8, device=dev)
    capi.mxfp4_pack_weights(torch.from_numpy(wc).to(dev), torch.from_numpy(ws).to(dev), 1, N, K, pk0)
    pks = [pk0] + [pk0.clone() for _ in range(copies - 1)]
    res = {}
    for M in (1, 16, 64, 8192):
        x = synth.bf16_tensor(synth.activations(M, K, seed=M, outlier_frac=0.01)).to(dev)
        wsb = capi.mxfp4_gemm_workspace_bytes(M, N, K)
        work = torch.zeros(max(wsb, 1), dtype=torch.uint8, device=dev)
        out = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        codes = torch.empty(M, N // 2, dtype=torch.uint8, device=dev)
        scales = torch.empty(M, N // 32, dtype=torch.uint8, device=dev)
        times = {}
        for mode in ("bf16", "mxfp4"):
            def call(i):
                if mode == "bf16":
                    capi.mxfp4_gemm(x, K, None, None, 0, pks[i % copies], None, out, N, M, N, K, work, wsb, sptr)
                else:
                    capi.mxfp4_gemm_mxfp4_out(x, K, None, None, 0, pks[i % copies], None, codes, scales, M, N, K,
                                              work, wsb, sptr)
            with torch.cuda.stream(stream):
                for i in range(3):
                    call(i)
            stream.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.stream(stream):
                with torch.cuda.graph(graph, stream=stream):
                    for i in range(reps):
                        call(i)
            stream.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                graph.replay()
                a.record(stream)
                graph.replay()
                b.record(stream)
            stream.synchronize()
            assert capi.mxfp4_get_device_error(sptr) == capi.OK
            times[mode] = a.elapsed_time(b) / reps
            del graph
        out_bytes = M * N // 2 + M * N // 32
        nbytes = N * K / 2 + N * K / 32 + 2 * M * K + out_bytes
        res[f"M{M}"] = {"us_bf16_out": round(times["bf16"] * 1e3, 2), "us_mxfp4_out": round(times["mxfp4"] * 1e3, 2),
                        "gbs_mxfp4_out": round(nbytes / (times["mxfp4"] * 1e-3) / 1e9, 1),
                        "tflops_mxfp4_out": round(2.0 * M * N * K / (times["mxfp4"] * 1e-3) / 1e12, 1)}
    return {"metric": "W4A4 GEMM with MXFP4 output epilogue vs bf16 output, N = 14336, K = 5120",
            "unit": "us per call", "cases": res,
            "bytes_per_launch": "N*K/2 + N*K/32 (packed W) + 2*M*K (bf16 A) + M*N/2 + M*N/32 (MXFP4 out)",
            "l2": "4 rotating weight copies; 20 calls replayed from a CUDA graph"}


def run_norm_quant(args, torch, np, capi, synth, dev, stream, hbm_peak):
    """The fused RMSNorm -> MXFP4 producer (TILED output, K = 5120), with and
    without the fused residual add; 4 rotating input copies per case so that
    the M = 8192 inputs come from HBM."""
    sptr = stream.cuda_stream
    K, copies, reps = 5120, 4, 20
    res = {}
    big_bytes, big_ms = 0.0, 0.0
    for M in (1, 16, 64, 8192):
        for with_res in (False, True):
            xs = [synth.bf16_tensor(synth.activations(M, K, seed=M + i)).to(dev) for i in range(copies)]
            rs = [synth.bf16_tensor(synth.residual(M, K, seed=M + i)).to(dev) if with_res else None
                  for i in range(copies)]
            g = synth.bf16_tensor(synth.norm_gamma(K, seed=M)).to(dev)
            nc, ns = capi.mxfp4_act_code_bytes(M, K, 1), capi.mxfp4_act_scale_bytes(M, K, 1)
            codes = torch.empty(nc, dtype=torch.uint8, device=dev)
            scales = torch.empty(ns, dtype=torch.uint8, device=dev)

            def call(i):
                capi.mxfp4_rmsnorm_quant_act(xs[i % copies], K, rs[i % copies], K, g, 1e-6, M, K, codes, scales,
                                             1, None, 0, sptr)

            with torch.cuda.stream(stream):
                for i in range(3):
                    call(i)
            stream.synchronize()
            # the calls replay from a CUDA graph: device time, not host launch cost
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.stream(stream):
                with torch.cuda.graph(graph, stream=stream):
                    for i in range(reps):
                        call(i)
            stream.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                graph.replay()
                a.record(stream)
                graph.replay()
                b.record(stream)
            stream.synchronize()
            assert capi.mxfp4_get_device_error(sptr) == capi.OK
            ms = a.elapsed_time(b) / reps
            nbytes = M * K * 2 * (3 if with_res else 1) + K * 2 + nc + ns
            res[f"M{M}{'_res' if with_res else ''}"] = {"us": round(ms * 1e3, 2),
                                                        "gbs": round(nbytes / (ms * 1e-3) / 1e9, 1)}
            if M == 8192:
                big_bytes += nbytes
                big_ms += ms
            del xs, rs, graph
    gbs = big_bytes / (big_ms * 1e-3) / 1e9
    return {"metric": "fused RMSNorm -> MXFP4 producer GB/s (M = 8192, K = 5120, TILED out, with and without "
                      "the residual add)", "value": round(gbs, 1), "unit": "GB/s", "peak": hbm_peak,
            "frac": round(gbs / hbm_peak, 4),
            "bytes_per_launch": "2*M*K (x) [+ 4*M*K residual read+write] + 2*K (gamma) + TILED codes + scales",
            "cases": res, "l2": "4 rotating input copies per case; 20 back-to-back calls replayed from a CUDA graph"}


# ------------------------------------------------------------------ oracle timing
def oracle_sample_step(ref, synth, np, M, N, K, rows_w):
    """The oracle's dense linear on M activation rows against a `rows_w`-row slice of the weights."""
    x = ref.bf16_bits_to_f64(synth.activations(M, K, seed=5, outlier_frac=0.01))
    wc = synth.weight_codes(rows_w, K, seed=N)
    ws = synth.weight_scales(rows_w, K, *W_SCALE_DECODE, seed=N)
    t = time.perf_counter()
    ref.quant_then_gemm(x, wc, ws, K)
    return time.perf_counter() - t, linear_bytes(M, rows_w, K)


def cpu_baseline(seconds: float):
    import numpy as np

    from mxfp4_quantized_gemm_gb300 import synth
    from oracle import mxfp4_ref as ref
    rows_w = 2048
    tot_t, tot_b, n = 0.0, 0, 0
    deadline = time.perf_counter() + seconds
    while time.perf_counter() < deadline or n < 3:
        M = DECODE_MS[n % len(DECODE_MS)]
        N, K = DECODE_NK[(n // len(DECODE_MS)) % len(DECODE_NK)]
        t, b = oracle_sample_step(ref, synth, np, M, N, K, rows_w)
        tot_t += t
        tot_b += b
        n += 1
    return {"value": round(tot_b / tot_t / 1e9, 4), "unit": "GB/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{n} decode-sweep cases, each the oracle's quantize + dequantized fp64 matmul of all "
                      f"M rows against a {rows_w}-row slice of the weights (numpy/BLAS, default threads)"}


def run_reference(args, world, rank):
    if rank != 0:
        return None, rank
    import numpy as np

    from mxfp4_quantized_gemm_gb300 import synth
    from oracle import mxfp4_ref as ref
    rows_w = 64
    cases = [(M, N, K) for M in DECODE_MS for (N, K) in DECODE_NK]
    for i in range(args.warmup):
        M, N, K = cases[i % len(cases)]
        oracle_sample_step(ref, synth, np, M, N, K, rows_w)
    tot_t, tot_b = 0.0, 0
    for i in range(args.steps):
        M, N, K = cases[i % len(cases)]
        t, b = oracle_sample_step(ref, synth, np, M, N, K, rows_w)
        tot_t += t
        tot_b += b
    value = tot_b / tot_t / 1e9
    sample = (f"each step: one decode-sweep case (cycling the 15), the oracle's quantize + dequantized fp64 "
              f"matmul against a {rows_w}-row slice of the weights")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 5), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(tot_t / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "decode W4A4 sweep (sampled weight rows), CPU oracle"},
        "cpu_baseline": {"value": round(value, 5), "unit": "GB/s", "cores": os.cpu_count(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 5), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    return line, rank


def run_single_bmm(args):
    """Run one MLA absorbed BMM (`kup` or `vup`, B = 64) `calls` times (for ncu captures)."""
    import torch

    import __graft_entry__
    __graft_entry__.build()
    from mxfp4_quantized_gemm_gb300 import capi, synth
    kind, M = args.single_bmm.split(",")
    M = int(M)
    B, N, K, layout = (64, 512, 192, capi.OUT_BMN) if kind == "kup" else (64, 256, 512, capi.OUT_MBN)
    wc = synth.weight_codes(N, K, seed=N, batch=B)
    ws = synth.weight_scales(N, K, -6, 0, seed=N, batch=B)
    pk = torch.empty(capi.mxfp4_packed_weight_bytes(B, N, K), dtype=torch.uint8, device="cuda")
    capi.mxfp4_pack_weights(torch.from_numpy(wc).cuda(), torch.from_numpy(ws).cuda(), B, N, K, pk)
    x = synth.bf16_tensor(synth.bmm_activations(B, M, K, seed=M)).cuda()
    out = torch.empty(B * M * N, dtype=torch.bfloat16, device="cuda")
    for _ in range(args.calls):
        capi.a16wfp4_bmm(x, pk, out, B, M, N, K, layout)
    torch.cuda.synchronize()
    assert capi.mxfp4_get_device_error() == capi.OK
    print(f"single bmm {kind} M={M}: {args.calls} calls ok")


def run_single_norm(args):
    """Run the fused RMSNorm -> MXFP4 producer on M rows of K = 5120 `calls` times (for ncu captures)."""
    import torch

    import __graft_entry__
    __graft_entry__.build()
    from mxfp4_quantized_gemm_gb300 import capi, synth
    M, with_res = int(args.single_norm.split(",")[0]), args.single_norm.endswith(",res")
    K = 5120
    x = synth.bf16_tensor(synth.activations(M, K, seed=M)).cuda()
    r = synth.bf16_tensor(synth.residual(M, K, seed=M)).cuda() if with_res else None
    g = synth.bf16_tensor(synth.norm_gamma(K, seed=M)).cuda()
    codes = torch.empty(capi.mxfp4_act_code_bytes(M, K, 1), dtype=torch.uint8, device="cuda")
    scales = torch.empty(capi.mxfp4_act_scale_bytes(M, K, 1), dtype=torch.uint8, device="cuda")
    for _ in range(args.calls):
        capi.mxfp4_rmsnorm_quant_act(x, K, r, K, g, 1e-6, M, K, codes, scales, 1)
    torch.cuda.synchronize()
    assert capi.mxfp4_get_device_error() == capi.OK
    print(f"single rmsnorm_quant M={M} K={K} residual={with_res}: {args.calls} calls ok")


def run_single(args):
    """Run one dense-linear shape `calls` times over `copies` weight copies (for ncu captures)."""
    import torch

    import __graft_entry__
    __graft_entry__.build()
    from mxfp4_quantized_gemm_gb300 import capi, synth
    M, N, K = (int(v) for v in args.single.split(","))
    wc = synth.weight_codes(N, K, seed=0)
    ws = synth.weight_scales(N, K, *W_SCALE_DECODE, seed=0)
    pk = torch.empty(capi.mxfp4_packed_weight_bytes(1, N, K), dtype=torch.uint8, device="cuda")
    capi.mxfp4_pack_weights(torch.from_numpy(wc).cuda(), torch.from_numpy(ws).cuda(), 1, N, K, pk)
    pks = [pk] + [pk.clone() for _ in range(args.copies - 1)]
    x = synth.bf16_tensor(synth.activations(M, K, seed=1, outlier_frac=0.01)).cuda()
    out = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    codes = torch.empty(M * (N // 2), dtype=torch.uint8, device="cuda")
    scales = torch.empty(M * ceil_div(N, 32), dtype=torch.uint8, device="cuda")
    wsb = capi.mxfp4_gemm_workspace_bytes(M, N, K)
    work = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
    for i in range(args.calls):
        if args.mxfp4_out:
            capi.mxfp4_gemm_mxfp4_out(x, K, None, None, 0, pks[i % len(pks)], None, codes, scales, M, N, K, work, wsb)
        elif args.pairs:
            capi.mxfp4_diag_gemm_pair(x, K, None, None, 0, pks[i % len(pks)], None, out, N, M, N, K, work, wsb)
        else:
            capi.mxfp4_gemm(x, K, None, None, 0, pks[i % len(pks)], None, out, N, M, N, K, work, wsb)
    torch.cuda.synchronize()
    assert capi.mxfp4_get_device_error() == capi.OK
    form = " (MXFP4 out)" if args.mxfp4_out else (" (CTA pairs)" if args.pairs else "")
    print(f"single {M},{N},{K}{form}: {args.calls} calls ok")


def run_prefill_pairs(args):
    """The prefill sweep's calls timed on the library's GEMM path and on the CTA-pair kernel
    (mxfp4_diag_gemm_pair) where that applies: one JSON line of per-call microseconds."""
    import numpy as np
    import torch

    import __graft_entry__
    __graft_entry__.build()
    from mxfp4_quantized_gemm_gb300 import capi, synth
    dev = torch.device("cuda", 0)
    stream = torch.cuda.Stream(device=dev)
    sptr = stream.cuda_stream
    cases = {}
    for (N, K) in DECODE_NK:
        wc = synth.weight_codes(N, K, seed=0, tensor_id=2)
        ws = synth.weight_scales(N, K, *W_SCALE_PREFILL, seed=0, tensor_id=3)
        packed = torch.empty(capi.mxfp4_packed_weight_bytes(1, N, K), dtype=torch.uint8, device=dev)
        capi.mxfp4_pack_weights(torch.from_numpy(wc).to(dev), torch.from_numpy(ws).to(dev), 1, N, K, packed)
        bias = synth.bf16_tensor(synth.bias(N, seed=0)).to(dev)
        for M in PREFILL_MS:
            x = synth.bf16_tensor(synth.activations(M, K, seed=M, tensor_id=1)).to(dev)
            out = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
            wsb = capi.mxfp4_gemm_workspace_bytes(M, N, K)
            work = torch.zeros(wsb, dtype=torch.uint8, device=dev)
            row = {}
            for name, fn in (("library_us", capi.mxfp4_gemm), ("pair_us", capi.mxfp4_diag_gemm_pair)):
                def call():
                    fn(x, K, None, None, 0, packed, bias, out, N, M, N, K, work, wsb, sptr)
                try:
                    with torch.cuda.stream(stream):
                        for _ in range(3):
                            call()
                except capi.Mxfp4Error as e:
                    if e.status != capi.ERR_UNSUPPORTED_SHAPE:
                        raise
                    row[name] = None
                    continue
                stream.synchronize()
                reps = 20
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                with torch.cuda.stream(stream):
                    a.record(stream)
                    for _ in range(reps):
                        call()
                    b.record(stream)
                stream.synchronize()
                row[name] = round(a.elapsed_time(b) / reps * 1e3, 1)
            cases[f"M{M}_N{N}_K{K}"] = row
        del packed
    assert capi.mxfp4_get_device_error() == capi.OK
    print(json.dumps({"prefill_pairs": cases,
                      "note": "quantizer + GEMM (+ fix-up) per call, back-to-back calls on one weight copy; "
                              "pair_us null where the CTA-pair kernel does not apply"}), flush=True)


# (N of each MMA, depth) pairs measured for every instruction mix of mxfp4_diag_tensor_rate: a
# k-step of the 1-CTA GEMM kernels is "mxf4 1cta 4 mma + 6 cp" at N = 256; depth 4 is the round trip
# of a 4-stage ring, depth 32 leaves the tensor pipe's throughput.
TC_RATE_POINTS = ((256, 4), (256, 32), (128, 32), (64, 32))


def run_tc_rates(args):
    """Tensor-pipe issue rates of the library's instruction mixes on every SM at once
    (mxfp4_diag_tensor_rate), and the dense FP4 / bf16 rates they imply; one JSON line."""
    import torch

    import __graft_entry__
    __graft_entry__.build()
    from mxfp4_quantized_gemm_gb300 import capi
    dev = torch.device("cuda", 0)
    props = torch.cuda.get_device_properties(dev)
    ns = torch.zeros(capi.mxfp4_diag_max_units(), dtype=torch.int64, device=dev)
    addr = torch.zeros(2, dtype=torch.int32, device=dev)
    capi.mxfp4_diag_pair_alloc_probe(addr)
    torch.cuda.synchronize()
    a = [int(v) & 0xFFFFFFFF for v in addr.cpu().tolist()]
    cols = [v & 0x3FFFFFFF for v in a]
    ranks = sorted(v >> 30 for v in a)
    pair_ok = cols[0] == cols[1] and ranks == [0, 1]
    steps = args.tc_steps
    clocks = ClockSampler(0)
    clocks.start()
    rows = []
    only = None if args.tc_only is None else {int(v) for v in args.tc_only.split(",")}
    for var in range(capi.mxfp4_diag_tensor_rate_variants()):
        if only is not None and var not in only:
            continue
        info = capi.mxfp4_diag_tensor_rate_info(var)
        pair, kind, mmas, copies, form, issuers, split = (info[k] for k in ("pair", "kind", "mmas", "copies", "form",
                                                                           "issuers", "split"))
        name = (f"{('mxf4', 'bf16', 'mxf4nvf4')[kind]} {'2cta' if pair else '1cta'} {mmas} mma"
                + (f" + {copies} cp{'128x256b' if form else ''}" if copies else "")
                + (f" x{issuers} issuers" if issuers > 1 else "")
                + ({1: ", copies first, a commit per 4 mma", 2: ", commit after the next copies"}.get(split, "")))
        for n, depth in TC_RATE_POINTS:
            if (pair and n < 64) or (issuers > 1 and n > 128) or (mmas == 0 and n != 256):
                continue
            if pair and not pair_ok:
                rows.append({"name": name, "skipped": "cta_group::2 allocation is not collective"})
                break
            m = 256 if pair else 128
            k = 16 if kind == 1 else 64
            meds = []
            for _ in range(3):
                ns.zero_()
                units = capi.mxfp4_diag_tensor_rate(var, n, steps, depth, ns)
                torch.cuda.synchronize()
                v = [x for x in ns[:units].cpu().tolist() if x > 0]
                if len(v) != units:
                    raise RuntimeError(f"{name}: {units - len(v)} units timed out")
                meds.append(statistics.median(v))
            med = statistics.median(meds)
            ns_step = med / steps
            flop = units * issuers * mmas * 2.0 * m * n * k * steps
            rows.append({"name": name, "n": n, "depth": depth, "units": units, "ns_per_step": round(ns_step, 1),
                         "ns_per_mma": round(ns_step / mmas, 1) if mmas else None,
                         "tflops": round(flop / (med * 1e-9) / 1e12, 1)})
    clk = clocks.stop()
    fp4 = [r["tflops"] for r in rows if r["name"].startswith("mxf4 ") and "cp" not in r["name"] and "tflops" in r]
    nvf4 = [r["tflops"] for r in rows if r["name"].startswith("mxf4nvf4") and "cp" not in r["name"] and "tflops" in r]
    bf16 = [r["tflops"] for r in rows if r["name"].startswith("bf16") and "tflops" in r]
    print(json.dumps({"tc_rates": rows, "pair_alloc": {"cols": cols, "collective": pair_ok},
                      "mxf4_dense_peak_tflops": max(fp4) if fp4 else None,
                      "mxf4nvf4_2x_dense_peak_tflops": max(nvf4) if nvf4 else None,
                      "bf16_dense_peak_tflops": max(bf16) if bf16 else None,
                      "sms": props.multi_processor_count, "steps": steps, "clocks": clk}), flush=True)


TIMELINE_POINTS = ("start", "w_req", "wait", "first_mma", "last_mma", "acc_done", "cluster", "done")


def run_timeline(args):
    """Per-call timeline of the decode sweep from the library's timeline build: the 15 calls of one
    step replayed from a CUDA graph (steps back to back, as in the timed region), each decode
    launch's CTAs stamping %globaltimer at fixed points.  Prints one table row per call: the
    median over CTAs of each point, in microseconds from the call's earliest CTA start, and the
    call's span from its dependency wait opening to its last CTA finishing."""
    import numpy as np
    import torch

    from mxfp4_quantized_gemm_gb300 import build
    build.build()
    os.environ["MXFP4_GB300_LIB"] = build.build(variant="timeline")
    from mxfp4_quantized_gemm_gb300 import capi, synth
    dev = torch.device("cuda", 0)
    cases = [(M, N, K) for M in DECODE_MS for (N, K) in DECODE_NK]
    st = []
    for i, (M, N, K) in enumerate(cases):
        wc = synth.weight_codes(N, K, seed=0, tensor_id=2)
        ws = synth.weight_scales(N, K, *W_SCALE_DECODE, seed=0, tensor_id=3)
        pk = torch.empty(capi.mxfp4_packed_weight_bytes(1, N, K), dtype=torch.uint8, device=dev)
        capi.mxfp4_pack_weights(torch.from_numpy(wc).to(dev), torch.from_numpy(ws).to(dev), 1, N, K, pk)
        x = synth.bf16_tensor(synth.activations(M, K, seed=1 + i, tensor_id=1, outlier_frac=0.01)).to(dev)
        wsb = capi.mxfp4_gemm_workspace_bytes(M, N, K)
        st.append((M, N, K, pk, x, torch.empty(M, N, dtype=torch.bfloat16, device=dev),
                   torch.zeros(wsb, dtype=torch.uint8, device=dev), wsb))
    stream = torch.cuda.Stream(device=dev)
    sptr = stream.cuda_stream

    def step():
        for (M, N, K, pk, x, out, work, wsb) in st:
            capi.mxfp4_gemm(x, K, None, None, 0, pk, None, out, N, M, N, K, work, wsb, sptr)

    with torch.cuda.stream(stream):
        step()
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            for _ in range(4):
                step()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    assert capi.mxfp4_get_device_error(sptr) == capi.OK
    stamps, nxt = capi.mxfp4_diag_decode_timeline()
    n = len(cases)
    rows = []
    raw = {}
    prev_end = None
    for j in range(n):
        seq = nxt - n + j
        a = stamps[seq % 64].astype(np.uint64)
        live = (a[:, 0] >> np.uint64(48)) == np.uint64(seq & 0xFFFF)
        a = a[live].copy()
        # point 0 keeps only the timer's low 48 bits: take the high bits from
        # point 1 (stamped by every CTA shortly after), one 2^48 period back
        # if the low bits wrapped in between
        low = a[:, 0] & np.uint64(0xFFFFFFFFFFFF)
        p0 = (a[:, 1] & ~np.uint64(0xFFFFFFFFFFFF)) | low
        a[:, 0] = np.where(p0 > a[:, 1], p0 - np.uint64(1 << 48), p0)
        a = a.astype(np.int64)
        raw[cases[j]] = a
        t0 = a[:, 0].min()
        rel = (a - t0) / 1e3
        med = {TIMELINE_POINTS[p]: round(float(np.median(rel[:, p][a[:, p] > 0])), 2) if (a[:, p] > 0).any()
               else None for p in range(8)}
        wait_open = a[:, 2].min()
        end = a[:, 7].max()
        M, N, K = cases[j][:3]
        rows.append({"case": f"M{M}_N{N}_K{K}", "ctas": int(live.sum()), "median_us": med,
                     "last_done_us": round((end - t0) / 1e3, 2),
                     "wait_open_us": round((wait_open - t0) / 1e3, 2),
                     "span_wait_to_done_us": round((end - wait_open) / 1e3, 2),
                     "gap_prev_done_to_wait_us": None if prev_end is None else round((wait_open - prev_end) / 1e3, 2)})
        prev_end = end
    if args.timeline_raw:
        np.savez(args.timeline_raw, **{f"M{M}_N{N}_K{K}": a for (M, N, K), a in raw.items()})
    print(json.dumps({"timeline": rows, "points": TIMELINE_POINTS}), flush=True)
    hdr = "case".ljust(20) + "".join(p.rjust(10) for p in TIMELINE_POINTS) + "   gap  span(wait->done)"
    print(hdr, file=sys.stderr)
    for r in rows:
        print(r["case"].ljust(20) + "".join(str(r["median_us"][p]).rjust(10) for p in TIMELINE_POINTS)
              + f"  {r['gap_prev_done_to_wait_us']}  {r['span_wait_to_done_us']}", file=sys.stderr)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=100)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--single", type=str, default=None,
                    help="profiling mode: M,N,K of one dense-linear call (bf16 input), no JSON line")
    ap.add_argument("--single-bmm", type=str, default=None,
                    help="profiling mode: kup,M or vup,M of one A16WFP4 BMM call, no JSON line")
    ap.add_argument("--single-norm", type=str, default=None,
                    help="profiling mode: M or M,res of one fused RMSNorm -> MXFP4 call (K = 5120), no JSON line")
    ap.add_argument("--mxfp4-out", action="store_true",
                    help="with --single: the MXFP4 output form (mxfp4_gemm_mxfp4_out)")
    ap.add_argument("--tc-rates", action="store_true",
                    help="measure tensor-pipe issue rates (scale copies, MMAs, CTA pairs) and print one JSON line")
    ap.add_argument("--tc-steps", type=int, default=4000)
    ap.add_argument("--tc-only", type=str, default=None,
                    help="with --tc-rates: comma-separated variant indexes to measure (default all)")
    ap.add_argument("--timeline-raw", type=str, default=None,
                    help="with --timeline: also save every CTA's stamps (ns) to this .npz file")
    ap.add_argument("--timeline", action="store_true",
                    help="per-call timeline of the decode sweep from the library's timeline build (one JSON line)")
    ap.add_argument("--pairs", action="store_true",
                    help="with --single: run the shape on the CTA-pair kernel (mxfp4_diag_gemm_pair)")
    ap.add_argument("--prefill-pairs", action="store_true",
                    help="time the prefill sweep's calls on the library path and on the CTA-pair kernel")
    ap.add_argument("--calls", type=int, default=6)
    ap.add_argument("--copies", type=int, default=4)
    args = ap.parse_args()
    if args.tc_rates:
        run_tc_rates(args)
        return
    if args.prefill_pairs:
        run_prefill_pairs(args)
        return
    if args.timeline:
        run_timeline(args)
        return
    if args.single:
        run_single(args)
        return
    if args.single_bmm:
        run_single_bmm(args)
        return
    if args.single_norm:
        run_single_norm(args)
        return
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        # rank 0 alone times the oracle on the host cores; other ranks exit at once
        world, rank = int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0"))
        line, rank = run_reference(args, world, rank)
        if rank == 0 and line is not None:
            print(json.dumps(line), flush=True)
        return
    world, rank, local = dist_init()
    if True:
        line, rank = run_ours(args, world, rank, local)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
