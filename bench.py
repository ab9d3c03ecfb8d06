#!/usr/bin/env python3
"""Benchmark of the quantized linear layer on GB300.

Default workload (one "step"): the four linear layers of a Llama-3-8B block
(qkv K=4096 N=6144, o_proj 4096x4096, gate_up K=4096 N=28672, down K=14336
N=4096) as W4A16 (G=128 asymmetric INT4, FP16 scale, 4-bit zero-point) at
decode batches M = 1, 4 and 16: 12 GEMM calls per step, weights resident in
HBM.  The metric is quantized-linear weight GB/s: packed weight bytes
(codes + scales + zeros) read per step / step time.

Timing: CUDA graphs of one step each over 5 rotating copies of the packed
weights (pass p of the step sequence reads copy p % 5, so 4 passes = 452 MB of
other weights, > 3x L2, stream between two reads of one copy), CUDA events on
the launching stream, W warm-up steps, K timed steps.  The same line carries
``prefill`` (W8A8 FP8 at M = 2048 / 8192 on the four layers, TFLOP/s and
fraction of the FP8 peak) and ``crossover`` (W4A16 vs W8A8 on the two
crossover shapes at M = 1 ... 512: measured crossover M beside the roofline
prediction), each with operands rotated past L2 the same way.  Under torchrun every rank runs the same workload on
its own GPU (replicas, weak scaling) and the slowest rank's time is used.

    python bench.py [--steps K] [--warmup W] [--gpus N] [--impl reference]
    python bench.py --sweep crossover|prefill|70b|decode|blocks|epilogue   (tables, not the bench line)
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

LAYERS_8B = [("qkv", 4096, 6144), ("o_proj", 4096, 4096), ("gate_up", 4096, 28672), ("down", 14336, 4096)]
MS_DECODE = (1, 4, 16)
ROTATE = 5
NOMINAL_HBM_GBS = 8000.0  # the part's nominal HBM3e rate (~8 TB/s), reported beside the measured peak
WORKLOAD = "llama3-8b W4A16 decode layers (qkv/o/gate_up/down) at M=1,4,16"


def w4_weight_bytes(N, K):
    return N * K // 2 + 2 * N * (K // 128) + N * (K // 128) // 2


def w4_alg_bytes(M, N, K):
    return w4_weight_bytes(N, K) + 2 * M * K + 2 * M * N


def w8_alg_bytes(M, N, K):
    return N * K + M * K + 4 * M + 4 + 2 * M * N


# DRAM traffic of the small-M W4A16 kernel from one ncu capture (profiles/
# w4a16_decode_llama8b_launch_list.md): dram__bytes_read.sum + dram__bytes_write.sum
# for M = 1, K = 4096, N = 28672, against that launch's algorithmic bytes.  The
# traffic of a bench launch is scaled from it by its algorithmic bytes (traffic grows
# in proportion: the weights are streamed once).
TRAFFIC_CAPTURE = {"kernel": "w4a16_mma_splitk", "dram_bytes": 61064448 + 8448,
                   "alg_bytes": 28672 * 4096 // 2 + 2 * 28672 * 32 + 28672 * 32 // 2 + 2 * 4096 + 2 * 28672}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.t:
            self.t.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------- helpers

def dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    return world, rank, local


def dist_max(x: float, world: int, device: str = "cuda") -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def make_event(external: bool):
    import torch
    if external:
        try:
            return torch.cuda.Event(enable_timing=True, external=True)
        except TypeError:
            return None
    return torch.cuda.Event(enable_timing=True)


# ---------------------------------------------------------------------------- our arm

def build_workload(rank: int):
    import torch

    import precision_quantized_linear_gb300 as q
    from precision_quantized_linear_gb300 import synthetic as syn
    from precision_quantized_linear_gb300.layers import W4A16Linear

    layers = []
    for i, (name, K, N) in enumerate(LAYERS_8B):
        W = syn.make_weight(N, K, seed=1000 * (rank + 1) + i)
        lin = W4A16Linear(torch.from_numpy(W.view(np.int16)).cuda())
        sets = [(lin.codes, lin.scales, lin.zeros)]
        for r in range(1, ROTATE):
            sets.append((lin.codes.clone(), lin.scales.clone(), lin.zeros.clone()))
        layers.append({"name": name, "K": K, "N": N, "lin": lin, "sets": sets})
    # every activation of a step in one device buffer and every output in
    # another (16-byte-aligned views), so that the end-to-end step moves its
    # inputs and results with one copy each way
    xkeys = [(M, K) for M in MS_DECODE for K in sorted({K for _, K, _ in LAYERS_8B})]
    ykeys = [(M, L["name"], L["N"]) for M in MS_DECODE for L in layers]
    xlen = sum((M * K + 7) // 8 * 8 for M, K in xkeys)
    ylen = sum((M * N + 7) // 8 * 8 for M, _, N in ykeys)

    def views(xbuf, ybuf):
        xs, ys, o = {}, {}, 0
        for M, K in xkeys:
            xs[(M, K)] = xbuf[o:o + M * K].view(M, K)
            o += (M * K + 7) // 8 * 8
        o = 0
        for M, name, N in ykeys:
            ys[(M, name)] = ybuf[o:o + M * N].view(M, N)
            o += (M * N + 7) // 8 * 8
        return xs, ys
    # two buffer sets: the end-to-end step double-buffers its inputs and outputs
    flat = []
    for b in range(2):
        xbuf = torch.empty(xlen, dtype=torch.int16, device="cuda")
        ybuf = torch.empty(ylen, dtype=torch.int16, device="cuda")
        xs_b, ys_b = views(xbuf, ybuf)
        for M, K in xkeys:
            xs_b[(M, K)].copy_(torch.from_numpy(syn.make_act(M, K, seed=77 + M + K).view(np.int16)))
        flat.append({"x": xbuf, "y": ybuf, "xs": xs_b, "ys": ys_b})
    ws_bytes = max(q.qlin_workspace_size(q.OP_W4A16_GEMM, M, L["N"], L["K"]) for M in MS_DECODE for L in layers)
    ws = torch.zeros(max(ws_bytes, 256), dtype=torch.uint8, device="cuda")
    return layers, flat[0]["xs"], flat[0]["ys"], ws, flat


def pass_calls(M, layers, copy):
    """One pass over the four layers at batch M, all on weight copy `copy`."""
    return [(M, L, copy) for L in layers]


def step_calls(step, layers):
    """The calls of step `step`: passes M = 1, 4, 16; pass p (counted over all
    steps) reads weight copy p % ROTATE, so between two reads of one copy of a
    layer ROTATE - 1 whole passes (>= 3 x L2 of other weights) are streamed."""
    out = []
    for i, M in enumerate(MS_DECODE):
        out += pass_calls(M, layers, (step * len(MS_DECODE) + i) % ROTATE)
    return out


def kernel_of(M):
    import precision_quantized_linear_gb300 as q
    return "w4a16_mma_splitk" if M <= q.qlin_gemv_max_m(q.OP_W4A16_GEMM) else "w4a16_tc"


def run_ours(args):
    import torch

    import precision_quantized_linear_gb300 as q

    world, rank, local = dist_setup(args)
    q.build()
    q.load()
    layers, xs, ys, ws, flat = build_workload(rank)
    stream = torch.cuda.Stream()
    peaks = load_peaks()
    l2 = l2_bytes()
    pass_bytes = sum(w4_weight_bytes(L["N"], L["K"]) for L in layers)
    assert (ROTATE - 1) * pass_bytes >= 3 * l2, "weight rotation too short to defeat L2"

    def issue(calls):
        for M, L, r in calls:
            c, s, z = L["sets"][r]
            q.qlin_w4a16_gemm(xs[(M, L["K"])], c, s, z, ys[(M, L["name"])], M, L["N"], L["K"], 128, ws,
                              ws.numel(), stream)

    # correctness of the launch configuration before timing
    with torch.cuda.stream(stream):
        issue(step_calls(0, layers))
    torch.cuda.synchronize()
    err = q.qlin_get_device_error(stream)
    if err:
        raise RuntimeError("device error %d before timing" % err)

    # one CUDA graph per step of the rotation (the copy pattern repeats every
    # ROTATE steps), holding only the kernels (programmatic launches of
    # consecutive kernels may overlap)
    graphs = []
    for st in range(ROTATE):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            issue(step_calls(st, layers))
        graphs.append(g)
    torch.cuda.synchronize()

    for i in range(args.warmup):
        graphs[i % ROTATE].replay()
    torch.cuda.synchronize()

    clocks = ClockSampler(local)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = make_event(False), make_event(False)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for i in range(args.steps):
            graphs[(args.warmup + i) % ROTATE].replay()
        e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    step_ms_local = e0.elapsed_time(e1) / args.steps
    step_ms = dist_max(step_ms_local, world)

    calls = step_calls(0, layers)
    weight_bytes = sum(w4_weight_bytes(L["N"], L["K"]) for M, L, _ in calls)
    alg_bytes = sum(w4_alg_bytes(M, L["N"], L["K"]) for M, L, _ in calls)
    value = world * weight_bytes / (step_ms * 1e-3) / 1e9
    # every launch of the step is the small-M W4A16 kernel: its average launch
    # duration is the timed region over the launches in it (consecutive
    # launches overlap through programmatic dependent launch, as in serving)
    kernels = {kernel_of(M) for M, _, _ in calls}
    assert len(kernels) == 1
    dom = kernels.pop()
    launch_ms = step_ms / len(calls)
    achieved = alg_bytes / len(calls) / (launch_ms * 1e-3) / 1e9

    # per batch size: a graph of ROTATE passes at that M over the rotating copies
    per_m_gbs = {}
    for M in MS_DECODE:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for r in range(ROTATE):
                issue(pass_calls(M, layers, r))
        g.replay()
        torch.cuda.synchronize()
        a, b = make_event(False), make_event(False)
        with torch.cuda.stream(stream):
            a.record(stream)
            for _ in range(5):
                g.replay()
            b.record(stream)
        torch.cuda.synchronize()
        t = a.elapsed_time(b) / (5 * ROTATE)
        per_m_gbs[str(M)] = round(pass_bytes / (t * 1e-3) / 1e9, 1)

    # single-launch latency: one call outside any graph (launch amortisation is
    # what the graphs above measure without): an event, one call through the
    # C ABI on an idle stream, an event; median of 50, per layer at M = 1
    latency_us = {}
    for L in layers:
        samples = []
        for i in range(50):
            a, b = make_event(False), make_event(False)
            torch.cuda.synchronize()
            with torch.cuda.stream(stream):
                a.record(stream)
                issue([(1, L, i % ROTATE)])
                b.record(stream)
            torch.cuda.synchronize()
            samples.append(a.elapsed_time(b) * 1e3)
        latency_us[L["name"]] = round(float(np.median(samples)), 2)

    e2e = run_e2e(args, layers, xs, ys, ws, flat, stream, world)
    extra = {}
    if not args.no_sweeps and world == 1:
        clk2 = ClockSampler(local)
        clk2.start()
        p8_probe = fp8_peak_probe()
        extra["prefill"] = measure_prefill(peaks, l2)
        extra["crossover"] = measure_crossover(peaks, l2)
        extra["prefill"]["fp8_probe_tflops"] = round(p8_probe, 1) if p8_probe else None
        extra["sweep_clocks"] = clk2.stop()
    traffic_per_launch = round(TRAFFIC_CAPTURE["dram_bytes"] / TRAFFIC_CAPTURE["alg_bytes"] * alg_bytes / len(calls))

    out = {
        "metric": "quantized-linear weight GB/s (decode) & TFLOPS (prefill) vs batch M, % of roofline",
        "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(step_ms, 5), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int4 weights x bf16 activations, fp32 accumulate", "data": "synthetic (seeded N(0,0.02) weights with 1% x20 outlier channels, N(0,1) activations)",
        "config": {"workload": WORKLOAD, "layers_KxN": [[K, N] for _, K, N in LAYERS_8B], "M": list(MS_DECODE),
                   "G": 128, "calls_per_step": len(calls), "weight_bytes_per_step": weight_bytes,
                   "alg_bytes_per_step": alg_bytes,
                   "l2": "inputs larger than L2: %d rotating weight copies; pass p reads copy p %% %d, so %.0f MB "
                         "of other weights (%.1f x L2) stream between two reads of one copy" %
                         (ROTATE, ROTATE, (ROTATE - 1) * pass_bytes / 1e6, (ROTATE - 1) * pass_bytes / l2),
                   "timing": "CUDA graph per step, CUDA events on the launching stream around the timed steps"},
        "per_M_weight_gbs": per_m_gbs,
        "single_launch_us_m1": latency_us,
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                     "traffic": traffic_per_launch,
                     "traffic_note": "bytes per launch, scaled from one ncu capture (M=1, 4096x28672) by "
                                     "algorithmic bytes",
                     "peak_source": peaks["source"],
                     "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
                     "nominal_peak": NOMINAL_HBM_GBS, "launches_timed": len(calls) * args.steps,
                     "ms_per_launch": round(launch_ms, 5), "share_of_step": 1.0},
        "gpu_launches": len(calls) * args.steps,
        "clocks": clk,
        "e2e": e2e,
    }
    out.update(extra)
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            out["cpu_baseline"] = cpu_baseline(seconds=args.cpu_seconds)
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def l2_bytes():
    import torch
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    return int(getattr(props, "L2_cache_size", 126 * 2 ** 20))


def rotation(bytes_per_copy, l2):
    """Copies of an operand so that one copy is read again only after >= 3 x L2 of others."""
    return max(2, int(np.ceil(3 * l2 / bytes_per_copy)) + 1)


def measure_prefill(peaks, l2):
    """W8A8 FP8 prefill (M = 2048 and 8192 on the four Llama-3-8B shapes, 0.1 % of
    tokens x50): TFLOP/s of the GEMM and of activation quantisation + GEMM,
    against the FP8 dense peak (the measured BF16 peak x 2, the nominal ratio)."""
    import torch

    import precision_quantized_linear_gb300 as q
    from precision_quantized_linear_gb300 import synthetic as syn
    from precision_quantized_linear_gb300.layers import MXFP4Linear, MXFP8Linear, NVFP4Linear, W8A8Linear

    p8 = 2.0 * peaks["bf16_tflops_sustained"]
    p4 = 6.0 * peaks["bf16_tflops_sustained"]   # nominal dense FP4 / BF16 = 13.5 / 2.25
    rows, mx_rows = [], []
    f4_rows = {"mxfp4": [], "nvfp4": []}
    for K, N in [(4096, 6144), (4096, 4096), (4096, 28672), (14336, 4096)]:
        Wd = torch.from_numpy(syn.make_weight(N, K, seed=K + N).view(np.int16)).cuda()
        lin = W8A8Linear(Wd)
        linmx = MXFP8Linear(Wd)
        lin4 = {"mxfp4": MXFP4Linear(Wd), "nvfp4": NVFP4Linear(Wd)}
        del Wd
        nrot = rotation(N * K, l2)
        sets = [lin.Wq] + [lin.Wq.clone() for _ in range(nrot - 1)]
        mxsets = [(linmx.Wq, linmx.ws_sf)] + [(linmx.Wq.clone(), linmx.ws_sf.clone()) for _ in range(nrot - 1)]
        for M in (2048, 8192):
            X = torch.from_numpy(syn.make_act(M, K, seed=M + 7, token_outlier_frac=0.001).view(np.int16)).cuda()
            Y = torch.empty((M, N), dtype=torch.int16, device="cuda")
            Xq = torch.empty((M, K), dtype=torch.uint8, device="cuda")
            sx = torch.empty(M, dtype=torch.float32, device="cuda")
            nb = q.qlin_workspace_size(q.OP_W8A8_GEMM, M, N, K)
            ws = torch.zeros(max(nb, 256), dtype=torch.uint8, device="cuda")
            q.qlin_quant_act_fp8(X, M, K, Xq, sx)
            us = time_launches([lambda st, wq=wq: q.qlin_w8a8_fp8_gemm(Xq, sx, wq, lin.sw, Y, M, N, K, ws, ws.numel(),
                                                                      st) for wq in sets])
            qus = time_launches([lambda st: q.qlin_quant_act_fp8(X, M, K, Xq, sx, st)])
            flops = 2 * M * N * K
            t_roof = max(flops / (p8 * 1e12), w8_alg_bytes(M, N, K) / (peaks["hbm_gbs"] * 1e9)) * 1e6
            rows.append({"K": K, "N": N, "M": M, "us": round(us, 2), "TFLOPS": round(flops / (us * 1e-6) / 1e12, 1),
                         "frac": round(t_roof / us, 3), "quant_us": round(qus, 2),
                         "TFLOPS_with_quant": round(flops / ((us + qus) * 1e-6) / 1e12, 1)})
            # MXFP8 (E8M0 scales per 32 columns applied by the tensor cores) on the same operands
            Xmq, xms = linmx.quant_act(X)
            nbm = q.qlin_workspace_size(q.OP_MXFP8_GEMM, M, N, K)
            wsm = torch.zeros(max(nbm, 256), dtype=torch.uint8, device="cuda")
            usm = time_launches([lambda st, wq=wq, wsf=wsf: q.qlin_mxfp8_gemm(Xmq, xms, wq, wsf, Y, M, N, K, wsm,
                                                                             wsm.numel(), st) for (wq, wsf) in mxsets])
            qusm = time_launches([lambda st: q.qlin_quant_mxfp8(X, M, K, Xmq, xms, st)])
            alg_mx = w8_alg_bytes(M, N, K) + (M + N) * K // 32
            t_roof = max(flops / (p8 * 1e12), alg_mx / (peaks["hbm_gbs"] * 1e9)) * 1e6
            mx_rows.append({"K": K, "N": N, "M": M, "us": round(usm, 2),
                            "TFLOPS": round(flops / (usm * 1e-6) / 1e12, 1), "frac": round(t_roof / usm, 3),
                            "quant_us": round(qusm, 2)})
            # FP4 (E2M1 with hardware block scaling): MXFP4 (kind::mxf4), NVFP4 (kind::mxf4nvf4)
            for fmt, l4 in lin4.items():
                ops = l4.quant_act(X)
                op = q.OP_MXFP4_GEMM if fmt == "mxfp4" else q.OP_NVFP4_GEMM
                nb4 = q.qlin_workspace_size(op, M, N, K)
                ws4 = torch.zeros(max(nb4, 256), dtype=torch.uint8, device="cuda")
                wsets = [(l4.Wq, l4.ws_sf)] + [(l4.Wq.clone(), l4.ws_sf.clone()) for _ in range(nrot - 1)]
                if fmt == "mxfp4":
                    calls = [lambda st, wq=wq, wsf=wsf: q.qlin_mxfp4_gemm(ops[0], ops[1], wq, wsf, Y, M, N, K, ws4,
                                                                         ws4.numel(), st) for (wq, wsf) in wsets]
                    qcall = [lambda st: q.qlin_quant_mxfp4(X, M, K, ops[0], ops[1], st)]
                    sf_bytes = (M + N) * K // 32
                else:
                    calls = [lambda st, wq=wq, wsf=wsf: q.qlin_nvfp4_gemm(ops[0], ops[1], ops[2], wq, wsf, l4.sgw, Y, M,
                                                                         N, K, ws4, ws4.numel(), st)
                             for (wq, wsf) in wsets]
                    qcall = [lambda st: (q.qlin_nvfp4_tensor_scale(X, M * K, ops[2], st),
                                         q.qlin_quant_nvfp4(X, M, K, ops[2], ops[0], ops[1], st))]
                    sf_bytes = (M + N) * K // 16
                us4 = time_launches(calls)
                qus4 = time_launches(qcall)
                alg4 = (M + N) * K // 2 + sf_bytes + 2 * M * N
                t_roof = max(flops / (p4 * 1e12), alg4 / (peaks["hbm_gbs"] * 1e9)) * 1e6
                f4_rows[fmt].append({"K": K, "N": N, "M": M, "us": round(us4, 2),
                                     "TFLOPS": round(flops / (us4 * 1e-6) / 1e12, 1), "frac": round(t_roof / us4, 3),
                                     "quant_us": round(qus4, 2)})
                del ops, ws4, wsets, calls, qcall
            assert q.qlin_get_device_error() == 0
            del X, Y, Xq, sx, ws, Xmq, xms, wsm
        del lin, sets, linmx, mxsets, lin4
        torch.cuda.empty_cache()

    def total(rs):
        f = sum(2 * r["M"] * r["N"] * r["K"] for r in rs)
        t = sum(r["us"] for r in rs)
        return round(f / (t * 1e-6) / 1e12, 1), round(f / (t * 1e-6) / 1e12 / p8, 3)
    tf, fr = total(rows)
    tfm, frm = total(mx_rows)
    f4 = {}
    for fmt, rs in f4_rows.items():
        f = sum(2 * r["M"] * r["N"] * r["K"] for r in rs)
        t = sum(r["us"] for r in rs)
        f4[fmt] = {"TFLOPS": round(f / (t * 1e-6) / 1e12, 1), "frac": round(f / (t * 1e-6) / 1e12 / p4, 3),
                   "cases": rs}
    f4["mxfp4"]["workload"] = ("MXFP4 (E2M1, E8M0 scale per 32 columns, hardware block scaling, tcgen05 kind::mxf4) "
                               "on the same shapes and M")
    f4["nvfp4"]["workload"] = ("NVFP4 (E2M1, E4M3 scale per 16 columns + FP32 tensor scales, tcgen05 "
                               "kind::mxf4nvf4) on the same shapes and M; quant_us includes the tensor-scale reduction")
    for v in f4.values():
        v["peak_tflops"] = round(p4, 1)
        v["peak_source"] = "measured bf16 sustained x 6 (nominal dense FP4/BF16 ratio)"
    return {"workload": "W8A8 FP8 prefill M=2048/8192 on the Llama-3-8B shapes (tcgen05 kind::f8f6f4)",
            "peak_tflops": round(p8, 1), "peak_source": "measured bf16 sustained x 2 (nominal FP8/BF16 ratio)",
            "TFLOPS": tf, "frac": fr, "cases": rows,
            "mxfp8": {"workload": "MXFP8 (E8M0 scale per 32 columns, hardware block scaling, tcgen05 "
                                  "kind::mxf8f6f4) on the same shapes and M", "TFLOPS": tfm, "frac": frm,
                      "cases": mx_rows},
            "mxfp4": f4["mxfp4"], "nvfp4": f4["nvfp4"]}


def measure_crossover(peaks, l2):
    """W4A16 vs W8A8 (activation quantisation + GEMM) on K=4096 N=14336 and
    K=14336 N=4096 at M = 1 ... 512, both through the default dispatch: the
    measured crossover M beside the roofline prediction."""
    import torch

    import precision_quantized_linear_gb300 as q
    from precision_quantized_linear_gb300 import synthetic as syn
    from precision_quantized_linear_gb300.layers import W4A16Linear, W8A8Linear

    rows = []
    for K, N in [(4096, 14336), (14336, 4096)]:
        W = torch.from_numpy(syn.make_weight(N, K, seed=K + N).view(np.int16)).cuda()
        lin4, lin8 = W4A16Linear(W), W8A8Linear(W)
        del W
        sets4 = [(lin4.codes, lin4.scales, lin4.zeros)] + [
            (lin4.codes.clone(), lin4.scales.clone(), lin4.zeros.clone())
            for _ in range(rotation(w4_weight_bytes(N, K), l2) - 1)]
        sets8 = [lin8.Wq] + [lin8.Wq.clone() for _ in range(rotation(N * K, l2) - 1)]
        for M in (1, 2, 4, 8, 16, 32, 64, 128, 256, 512):
            X = torch.from_numpy(syn.make_act(M, K, seed=M + 7).view(np.int16)).cuda()
            Y = torch.empty((M, N), dtype=torch.int16, device="cuda")
            Xq = torch.empty((M, K), dtype=torch.uint8, device="cuda")
            sx = torch.empty(M, dtype=torch.float32, device="cuda")
            nb = max(q.qlin_workspace_size(q.OP_W4A16_GEMM, M, N, K), q.qlin_workspace_size(q.OP_W8A8_GEMM, M, N, K))
            ws = torch.zeros(max(nb, 256), dtype=torch.uint8, device="cuda")
            us4 = time_launches([lambda st, c=c, s=s, z=z: q.qlin_w4a16_gemm(X, c, s, z, Y, M, N, K, 128, ws,
                                                                            ws.numel(), st) for (c, s, z) in sets4])

            def w8(st, wq):
                q.qlin_quant_act_fp8(X, M, K, Xq, sx, st)
                q.qlin_w8a8_fp8_gemm(Xq, sx, wq, lin8.sw, Y, M, N, K, ws, ws.numel(), st)
            us8 = time_launches([lambda st, wq=wq: w8(st, wq) for wq in sets8])
            nb48 = q.qlin_workspace_size(q.OP_W4A8_GEMM, M, N, K)
            ws48 = torch.zeros(max(nb48, 256), dtype=torch.uint8, device="cuda")

            def w48(st, c, s, z):
                q.qlin_quant_act_fp8(X, M, K, Xq, sx, st)
                q.qlin_w4a8_gemm(Xq, sx, c, s, z, Y, M, N, K, 128, ws48, ws48.numel(), st)
            us48 = time_launches([lambda st, c=c, s=s, z=z: w48(st, c, s, z) for (c, s, z) in sets4])
            rows.append({"K": K, "N": N, "M": M, "variant": "w4", "us": us4})
            rows.append({"K": K, "N": N, "M": M, "variant": "w8", "us": us8})
            rows.append({"K": K, "N": N, "M": M, "variant": "w4a8", "us": us48})
            assert q.qlin_get_device_error() == 0
        del lin4, lin8, sets4, sets8
        torch.cuda.empty_cache()
    summary = crossover_summary(rows, peaks["bf16_tflops"], 2.0 * peaks["bf16_tflops"], peaks["hbm_gbs"],
                                quant_in_w8=True)
    summary["how"] = ("W8A8 time = qlin_quant_act_fp8 + qlin_w8a8_fp8_gemm; both through the default dispatch; "
                      "roofline with the measured HBM and BF16 peaks, FP8 = 2 x BF16")
    summary["w4a8_us"] = {"%dx%d" % (K, N): {str(r["M"]): round(r["us"], 2) for r in rows
                                              if (r["K"], r["N"]) == (K, N) and r["variant"] == "w4a8"}
                          for K, N in [(4096, 14336), (14336, 4096)]}
    summary["w4a8_how"] = "W4A8 time = qlin_quant_act_fp8 + qlin_w4a8_gemm (INT4 weights, E4M3 tokens)"
    return summary


def run_e2e(args, layers, xs, ys, ws, flat, stream, world):
    """Same metric through the C ABI, host buffers in and out every step. Each
    step's activations arrive in one copy from pinned host memory and its
    outputs return in one copy to pinned host memory, on two copy streams and
    double-buffered the way a serving loop overlaps them: step i + 1's inputs
    arrive while step i computes, step i's outputs return while step i + 1
    computes.  The twelve qlin_w4a16_gemm calls of a step go straight to the C
    entry point with their arguments prepared once (pointers of the
    pre-allocated buffers).  The timed region ends when the last step's outputs
    are on the host."""
    import torch

    import precision_quantized_linear_gb300 as q
    lib = q.load()
    gemm = lib.qlin_w4a16_gemm
    hx = torch.empty(flat[0]["x"].shape, dtype=flat[0]["x"].dtype, pin_memory=True).copy_(flat[0]["x"].cpu())
    hy = [torch.empty(flat[0]["y"].shape, dtype=flat[0]["y"].dtype, pin_memory=True) for _ in range(2)]
    h2d = hx.numel() * 2
    d2h = hy[0].numel() * 2
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    sh = stream.cuda_stream
    # the calls of step i depend on i % ROTATE (the weight copy of each pass) and i % 2 (the buffer set)
    plans = {}
    for ph in range(ROTATE):
        for b in range(2):
            fb = flat[b]
            plans[(ph, b)] = [(fb["xs"][(M, L["K"])].data_ptr(), L["sets"][r][0].data_ptr(), L["sets"][r][1].data_ptr(),
                               L["sets"][r][2].data_ptr(), fb["ys"][(M, L["name"])].data_ptr(), M, L["N"], L["K"], 128,
                               ws.data_ptr(), ws.numel(), sh) for M, L, r in step_calls(ph, layers)]
    ready = [torch.cuda.Event(), torch.cuda.Event()]
    done = [torch.cuda.Event(), torch.cuda.Event()]     # buffer set b: its GEMMs are done (its X is free)
    out_ev = [torch.cuda.Event(), torch.cuda.Event()]   # buffer set b: its outputs are on the host (its Y is free)
    used = [False, False]

    def step(i):
        b = i % 2
        if used[b]:
            s_in.wait_event(done[b])
            stream.wait_event(out_ev[b])
        with torch.cuda.stream(s_in):
            flat[b]["x"].copy_(hx, non_blocking=True)
        ready[b].record(s_in)
        stream.wait_event(ready[b])
        for a in plans[(i % ROTATE, b)]:
            st = gemm(*a)
            if st != 0:
                raise q.QlinError(st, "qlin_w4a16_gemm")
        done[b].record(stream)
        s_out.wait_event(done[b])
        with torch.cuda.stream(s_out):
            hy[b].copy_(flat[b]["y"], non_blocking=True)
        out_ev[b].record(s_out)
        used[b] = True

    for i in range(max(1, args.warmup)):
        step(i)
    torch.cuda.synchronize()
    barrier(world)
    n = max(1, args.steps)
    e0, e1 = make_event(False), make_event(False)
    e0.record(stream)
    s_in.wait_stream(stream)
    for i in range(n):
        step(i)
    stream.wait_event(out_ev[(n - 1) % 2])
    e1.record(stream)
    torch.cuda.synchronize()
    ms = dist_max(e0.elapsed_time(e1) / n, world)
    wbytes = sum(w4_weight_bytes(L["N"], L["K"]) for M, L, _ in step_calls(0, layers))
    return {"value": round(world * wbytes / (ms * 1e-3) / 1e9, 1), "unit": "GB/s", "ms_per_step": round(ms, 5),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "how": "per step: one copy of all X from pinned host memory, 12 qlin_w4a16_gemm calls through the C ABI "
                   "(no graph), one copy of all Y to pinned host memory; copies on two streams, double-buffered with "
                   "the compute"}


# ---------------------------------------------------------------------------- oracle (CPU) arms

def _oracle_sample():
    """The decode workload for the oracle: the four Llama-3-8B layers (quantised
    once) and the activations at M = 1, 4, 16, as the GPU arm draws them."""
    import oracle
    from precision_quantized_linear_gb300 import synthetic as syn
    wqs = {}
    for i, (name, K, N) in enumerate(LAYERS_8B):
        wqs[name] = oracle.quantize_w4(syn.make_weight(N, K, seed=1000 + i))
    xs = {(M, K): syn.make_act(M, K, seed=77 + M + K) for M in MS_DECODE for K in {K for _, K, _ in LAYERS_8B}}
    calls = [(M, name, K, N) for M in MS_DECODE for name, K, N in LAYERS_8B]
    return oracle, wqs, xs, calls


def cpu_baseline(seconds: float = 10.0):
    """The oracle as it stands, on the host cores, over a bounded sample of the
    decode step (its twelve calls in step order, as many as fit in `seconds`),
    plus the tiny configuration (M=1, K=N=512) on one core."""
    from precision_quantized_linear_gb300 import synthetic as syn
    oracle, wqs, xs, calls = _oracle_sample()
    t0 = time.perf_counter()
    done, wbytes = 0, 0
    while True:
        M, name, K, N = calls[done % len(calls)]
        oracle.w4a16_full(xs[(M, K)], wqs[name])
        done += 1
        wbytes += w4_weight_bytes(N, K)
        if time.perf_counter() - t0 >= seconds and done >= len(calls):
            break
    dt = time.perf_counter() - t0
    cores = oracle.num_threads()
    # the tiny configuration single-threaded: quantise + pack, then the GEMM
    oracle.set_num_threads(1)
    W1 = syn.make_weight(512, 512, seed=0, outlier_frac=0.0)
    X1 = syn.make_act(1, 512, seed=0)
    t1 = time.perf_counter()
    reps = 0
    while time.perf_counter() - t1 < 1.0:
        wq1 = oracle.quantize_w4(W1)
        oracle.pack_tile(wq1)
        reps += 1
    t_pack = (time.perf_counter() - t1) / reps
    t2 = time.perf_counter()
    reps2 = 0
    while time.perf_counter() - t2 < 1.0:
        oracle.w4a16_full(X1, wq1)
        reps2 += 1
    t_gemm = (time.perf_counter() - t2) / reps2
    oracle.set_num_threads(cores)
    return {"value": round(wbytes / dt / 1e9, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": "oracle W4A16 GEMM (dequantise + fp64 GEMM) over the decode step's calls in order "
                      "(4 Llama-3-8B layers x M=1,4,16): %d calls in %.1f s" % (done, dt),
            "tiny_single_thread": {"config": "M=1 K=N=512 G=128", "cores": 1,
                                   "quantise_pack_ms": round(t_pack * 1e3, 3), "gemm_ms": round(t_gemm * 1e3, 3),
                                   "gemm_GFLOPS": round(2 * 512 * 512 / t_gemm / 1e9, 3)}}


def run_reference(args):
    """The oracle as the reference arm: step i runs call i of the decode step
    (cycling over its twelve calls), a bounded sample of the workload."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    oracle, wqs, xs, calls = _oracle_sample()
    for i in range(args.warmup):
        M, name, K, N = calls[i % len(calls)]
        oracle.w4a16_full(xs[(M, K)], wqs[name])
    t0 = time.perf_counter()
    wbytes = 0
    for i in range(args.steps):
        M, name, K, N = calls[(args.warmup + i) % len(calls)]
        oracle.w4a16_full(xs[(M, K)], wqs[name])
        wbytes += w4_weight_bytes(N, K)
    dt = time.perf_counter() - t0
    value = wbytes / dt / 1e9
    ms = dt * 1e3 / args.steps
    sample = ("step i: oracle W4A16 GEMM (dequantise + fp64 GEMM) of call i of the decode step "
              "(4 Llama-3-8B layers x M=1,4,16, cycled)")
    out = {"impl": "reference", "metric": "quantized-linear weight GB/s (decode) & TFLOPS (prefill) vs batch M, % of roofline",
           "value": round(value, 4), "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
           "dtype": "f64", "data": "synthetic", "config": {"workload": WORKLOAD},
           "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
                            "sample": sample},
           "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


# ---------------------------------------------------------------------------- sweeps

def fp8_peak_probe():
    """Dense E4M3 GEMM throughput of the vendor library (torch._scaled_mm), TFLOP/s."""
    import torch
    try:
        n = 8192
        a = torch.randn(n, n, device="cuda").to(torch.float8_e4m3fn)
        b = torch.randn(n, n, device="cuda").to(torch.float8_e4m3fn).t()
        one = torch.ones((), device="cuda")
        for _ in range(3):
            torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
        torch.cuda.synchronize()
        e0, e1 = make_event(False), make_event(False)
        e0.record()
        for _ in range(20):
            torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
        e1.record()
        torch.cuda.synchronize()
        return 2 * n ** 3 * 20 / (e0.elapsed_time(e1) * 1e-3) / 1e12
    except Exception as ex:  # noqa: BLE001
        print("fp8 probe failed:", ex, file=sys.stderr)
        return None


def time_launches(launches, reps=10, warm=3):
    """Average device time of one launch: a CUDA graph holding the given
    launch closures (one per rotating weight copy), replayed `reps` times."""
    import torch
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        for f in launches:
            f(st)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        for f in launches:
            f(st)
    for _ in range(warm):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = make_event(False), make_event(False)
    with torch.cuda.stream(st):
        e0.record(st)
        for _ in range(reps):
            g.replay()
        e1.record(st)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / (reps * len(launches)) * 1e3   # microseconds


def crossover_summary(rows, p16_tf, p8_tf, bw_gbs, quant_in_w8=False):
    """Measured W4A16-vs-W8A8 crossover M (W8A8 counted as activation quantisation + GEMM)
    beside the roofline predictions of the arithmetic-intensity argument."""
    out = {"crossover": []}
    for (K, N) in sorted({(r["K"], r["N"]) for r in rows}):
        w4 = {r["M"]: r["us"] for r in rows if (r["K"], r["N"]) == (K, N) and r["variant"] == "w4"}
        w8 = {r["M"]: r["us"] + (0.0 if quant_in_w8 else r.get("quant_us", 0.0))
              for r in rows if (r["K"], r["N"]) == (K, N) and r["variant"] == "w8"}
        ms = sorted(set(w4) & set(w8))
        measured = next((m for m in ms if w8[m] <= w4[m] and all(w8[x] <= w4[x] for x in ms if x >= m)), None)

        def t4(m):
            return max(2 * m * N * K / (p16_tf * 1e12), w4_alg_bytes(m, N, K) / (bw_gbs * 1e9))

        def t8(m, with_quant):
            t = max(2 * m * N * K / (p8_tf * 1e12), w8_alg_bytes(m, N, K) / (bw_gbs * 1e9))
            return t + (3 * m * K + 4 * m) / (bw_gbs * 1e9) if with_quant else t
        pred_gemm = next((m for m in range(1, 8193) if t8(m, False) <= t4(m)), None)
        pred_quant = next((m for m in range(1, 8193) if t8(m, True) <= t4(m)), None)
        out["crossover"].append({
            "K": K, "N": N, "measured_M": measured,
            "measured_us": {str(m): [round(w4[m], 2), round(w8[m], 2)] for m in ms},
            "roofline_M_gemm_only": pred_gemm, "roofline_M_with_act_quant": pred_quant,
            "simplified_P16_over_2BW": round(p16_tf * 1e12 / (2 * bw_gbs * 1e9), 1),
            "w4a16_transition_M": round((p16_tf * 1e12 / (bw_gbs * 1e9)) * 0.51953125 / 2, 1)})
    return out


def run_sweep(args):
    import torch

    import precision_quantized_linear_gb300 as q
    from precision_quantized_linear_gb300 import synthetic as syn
    from precision_quantized_linear_gb300.layers import W4A8Linear, W4A16Linear, W8A8BlockLinear, W8A8Linear

    torch.cuda.set_device(0)
    q.build()
    q.load()
    peaks = load_peaks()
    p8 = fp8_peak_probe()
    p16 = peaks["bf16_tflops"]
    bw = peaks["hbm_gbs"]
    l2 = torch.cuda.get_device_properties(0).L2_cache_size if hasattr(torch.cuda.get_device_properties(0), "L2_cache_size") else 126 * 2 ** 20
    print(json.dumps({"peaks": peaks, "fp8_probe_tflops": p8, "l2_bytes": l2}), flush=True)
    p8_use = p8 if p8 else 2 * p16

    results = []
    if args.sweep == "crossover":
        shapes = [(4096, 14336), (14336, 4096)]
        plan = [("w4", M) for M in (1, 2, 4, 8, 16, 32, 64, 128, 256, 512)] + \
               [("w8", M) for M in (1, 2, 4, 8, 16, 32, 64, 128, 256, 512)] + \
               [("w4a8", M) for M in (1, 2, 4, 8, 16, 32, 64, 128, 256, 512)]
    elif args.sweep == "prefill":
        shapes = [(4096, 6144), (4096, 4096), (4096, 28672), (14336, 4096)]
        plan = [("w8", M) for M in (2048, 8192)] + [("w4", M) for M in (2048, 8192)]
    elif args.sweep == "70b":
        shapes = [(8192, 10240), (8192, 8192), (8192, 57344), (28672, 8192)]
        plan = [("w4", M) for M in (1, 64, 256)] + [("w8", M) for M in (256, 4096)] + \
               [("w4a8", M) for M in (1, 64, 256)]
    elif args.sweep == "epilogue":  # fused bias + SiLU / GELU beside the plain calls
        shapes = [(4096, 4096), (4096, 28672)]
        plan = [(v, M) for M in (1, 16, 256, 2048) for v in ("w4", "w4:silu", "w4:gelu", "w8", "w8:silu")]
    elif args.sweep == "blocks":  # FP8 block scaling beside per-tensor FP8, decode to prefill
        shapes = [(4096, 6144), (4096, 4096), (4096, 28672), (14336, 4096)]
        plan = [(v, M) for M in (1, 16, 2048, 8192) for v in ("w8", "w8b")]
    else:  # decode: GEMV vs tensor-core path per M, for the dispatch threshold
        shapes = [(4096, 6144), (4096, 4096), (4096, 28672), (14336, 4096)]
        plan = [(v, M) for M in (1, 2, 3, 4, 5, 8, 16) for v in ("w4gemv", "w4tc", "w8gemv", "w8tc")]

    for (K, N) in shapes:
        W = torch.from_numpy(syn.make_weight(N, K, seed=K + N).view(np.int16)).cuda()
        lin4 = W4A16Linear(W)
        lin8 = W8A8Linear(W)
        lin8b = W8A8BlockLinear(W) if args.sweep == "blocks" else None
        del W
        w4b, w8b = w4_weight_bytes(N, K), N * K
        r4 = max(1, int(np.ceil(3 * l2 / w4b)))
        r8 = max(1, int(np.ceil(3 * l2 / w8b)))
        sets4 = [(lin4.codes, lin4.scales, lin4.zeros)] + [
            (lin4.codes.clone(), lin4.scales.clone(), lin4.zeros.clone()) for _ in range(r4 - 1)]
        sets8 = [lin8.Wq] + [lin8.Wq.clone() for _ in range(r8 - 1)]
        sets8b = ([(lin8b.Wq, lin8b.sw)] + [(lin8b.Wq.clone(), lin8b.sw.clone()) for _ in range(r8 - 1)]
                  if lin8b is not None else [])
        bias = torch.from_numpy(syn.make_act(1, N, seed=N)[0].view(np.int16)).cuda()
        for (v, M) in plan:
            v, _, actname = v.partition(":")
            act = {"": q.ACT_NONE, "silu": q.ACT_SILU, "gelu": q.ACT_GELU}[actname]
            X = torch.from_numpy(syn.make_act(M, K, seed=M + 7, token_outlier_frac=0.001).view(np.int16)).cuda()
            Y = torch.empty((M, N), dtype=torch.int16, device="cuda")
            Xq = torch.empty((M, K), dtype=torch.uint8, device="cuda")
            sx = torch.empty(M, dtype=torch.float32, device="cuda")
            row = {"K": K, "N": N, "M": M, "variant": v + (":bias+" + actname if actname else "")}
            flops = 2 * M * N * K
            if v in ("w4", "w4gemv", "w4tc"):
                path = {"w4": q.PATH_AUTO, "w4gemv": q.PATH_GEMV, "w4tc": q.PATH_TC}[v]
                nb = q.qlin_workspace_size(q.OP_W4A16_GEMM, M, N, K)
                ws = torch.zeros(max(nb, 256), dtype=torch.uint8, device="cuda")
                if act == q.ACT_NONE:
                    fns = [lambda st, c=c, s=s, z=z: q.qlin_w4a16_gemm_ex(X, c, s, z, Y, M, N, K, 128, ws, ws.numel(),
                                                                         path, st) for (c, s, z) in sets4]
                else:
                    fns = [lambda st, c=c, s=s, z=z: q.qlin_w4a16_gemm_fused(X, c, s, z, Y, M, N, K, 128, bias, act, ws,
                                                                            ws.numel(), path, st) for (c, s, z) in sets4]
                us = time_launches(fns)
                alg = w4_alg_bytes(M, N, K)
                t_roof = max(flops / (p16 * 1e12), alg / (bw * 1e9)) * 1e6
                row.update(us=round(us, 2), weight_GBps=round(w4b / (us * 1e-6) / 1e9, 1),
                           TFLOPS=round(flops / (us * 1e-6) / 1e12, 2), roof_us=round(t_roof, 2),
                           roof_frac=round(t_roof / us, 3),
                           bound="hbm" if alg / (bw * 1e9) > flops / (p16 * 1e12) else "tensor")
            elif v == "w4a8":
                lin48 = W4A8Linear.__new__(W4A8Linear)
                lin48.N, lin48.K, lin48.G = N, K, 128
                nb = q.qlin_workspace_size(q.OP_W4A8_GEMM, M, N, K)
                ws = torch.zeros(max(nb, 256), dtype=torch.uint8, device="cuda")
                q.qlin_quant_act_fp8(X, M, K, Xq, sx)
                fns = [lambda st, c=c, s=s, z=z: q.qlin_w4a8_gemm(Xq, sx, c, s, z, Y, M, N, K, 128, ws, ws.numel(), st)
                       for (c, s, z) in sets4]
                us = time_launches(fns)
                qus = time_launches([lambda st: q.qlin_quant_act_fp8(X, M, K, Xq, sx, st)])
                alg = w4_alg_bytes(M, N, K) - M * K
                t_roof = max(flops / (p8_use * 1e12), alg / (bw * 1e9)) * 1e6
                row.update(us=round(us, 2), quant_us=round(qus, 2), weight_GBps=round(w4b / (us * 1e-6) / 1e9, 1),
                           TFLOPS=round(flops / (us * 1e-6) / 1e12, 2), roof_us=round(t_roof, 2),
                           roof_frac=round(t_roof / us, 3),
                           bound="hbm" if alg / (bw * 1e9) > flops / (p8_use * 1e12) else "tensor")
            elif v == "w8b":
                nb = q.qlin_workspace_size(q.OP_W8A8_BLOCK_GEMM, M, N, K)
                ws = torch.zeros(max(nb, 256), dtype=torch.uint8, device="cuda")
                sxb = torch.empty((K // 128, M), dtype=torch.float32, device="cuda")
                q.qlin_quant_act_fp8_blocks(X, M, K, Xq, sxb)
                fns = [lambda st, wq=wq, sw=sw: q.qlin_w8a8_fp8_block_gemm(Xq, sxb, wq, sw, Y, M, N, K, ws, ws.numel(),
                                                                          st) for (wq, sw) in sets8b]
                us = time_launches(fns)
                qus = time_launches([lambda st: q.qlin_quant_act_fp8_blocks(X, M, K, Xq, sxb, st)])
                alg = w8_alg_bytes(M, N, K) + 4 * M * (K // 128) + 4 * (N // 128) * (K // 128)
                t_roof = max(flops / (p8_use * 1e12), alg / (bw * 1e9)) * 1e6
                row.update(us=round(us, 2), quant_us=round(qus, 2), weight_GBps=round(w8b / (us * 1e-6) / 1e9, 1),
                           TFLOPS=round(flops / (us * 1e-6) / 1e12, 2), roof_us=round(t_roof, 2),
                           roof_frac=round(t_roof / us, 3),
                           bound="hbm" if alg / (bw * 1e9) > flops / (p8_use * 1e12) else "tensor",
                           fp8_peak="probe" if p8 else "2x bf16 (assumed)")
            else:
                path = {"w8": q.PATH_AUTO, "w8gemv": q.PATH_GEMV, "w8tc": q.PATH_TC}[v]
                nb = q.qlin_workspace_size(q.OP_W8A8_GEMM, M, N, K)
                ws = torch.zeros(max(nb, 256), dtype=torch.uint8, device="cuda")
                q.qlin_quant_act_fp8(X, M, K, Xq, sx)
                if act == q.ACT_NONE:
                    fns = [lambda st, wq=wq: q.qlin_w8a8_fp8_gemm_ex(Xq, sx, wq, lin8.sw, Y, M, N, K, ws, ws.numel(),
                                                                     path, st) for wq in sets8]
                else:
                    fns = [lambda st, wq=wq: q.qlin_w8a8_fp8_gemm_fused(Xq, sx, wq, lin8.sw, Y, M, N, K, bias, act, ws,
                                                                        ws.numel(), path, st) for wq in sets8]
                us = time_launches(fns)
                qus = time_launches([lambda st: q.qlin_quant_act_fp8(X, M, K, Xq, sx, st)])
                alg = w8_alg_bytes(M, N, K)
                t_roof = max(flops / (p8_use * 1e12), alg / (bw * 1e9)) * 1e6
                row.update(us=round(us, 2), quant_us=round(qus, 2), weight_GBps=round(w8b / (us * 1e-6) / 1e9, 1),
                           TFLOPS=round(flops / (us * 1e-6) / 1e12, 2), roof_us=round(t_roof, 2),
                           roof_frac=round(t_roof / us, 3),
                           bound="hbm" if alg / (bw * 1e9) > flops / (p8_use * 1e12) else "tensor",
                           fp8_peak="probe" if p8 else "2x bf16 (assumed)")
            assert q.qlin_get_device_error() == 0
            print(json.dumps(row), flush=True)
            results.append(row)
        del lin4, lin8, lin8b, sets4, sets8, sets8b
        torch.cuda.empty_cache()
    if args.sweep == "crossover":
        print(json.dumps(crossover_summary(results, p16, p8_use, bw)), flush=True)
    if args.sweep == "epilogue":
        sweep_epilogue_blocks(l2)


def sweep_epilogue_blocks(l2):
    """The fused bias + SiLU epilogue of the block formats, W4A8 and block-scaled
    FP8 against their plain GEMMs (activations quantised once, outside the timing;
    weight copies rotated past L2)."""
    import torch

    import precision_quantized_linear_gb300 as q
    from precision_quantized_linear_gb300 import synthetic as syn
    from precision_quantized_linear_gb300.layers import (MXFP4Linear, MXFP8Linear, NVFP4Linear, W4A8Linear,
                                                          W8A8BlockLinear)
    K, N = 4096, 28672
    W = torch.from_numpy(syn.make_weight(N, K, seed=K + N).view(np.int16)).cuda().view(torch.bfloat16)
    bias = torch.from_numpy(syn.make_act(1, N, seed=N)[0].view(np.int16)).cuda().view(torch.bfloat16)
    kinds = {"mxfp8": (MXFP8Linear, 1.0), "mxfp4": (MXFP4Linear, 0.5), "nvfp4": (NVFP4Linear, 0.5),
             "w4a8": (W4A8Linear, 0.51953125), "w8a8b": (W8A8BlockLinear, 1.0)}
    for name, (cls, bpw) in kinds.items():
        copies = max(1, int(np.ceil(3 * l2 / (bpw * N * K))))
        lins = [cls(W, bias=bias) for _ in range(copies)]
        for M in (16, 256, 2048):
            X = torch.from_numpy(syn.make_act(M, K, seed=M + 7).view(np.int16)).cuda().view(torch.bfloat16)
            ops = lins[0].quant_act(X)
            Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
            row = {"K": K, "N": N, "M": M, "variant": name}
            for act, key in ((q.ACT_NONE, "us_bias"), (q.ACT_SILU, "us_bias_silu")):
                row[key] = round(time_launches([lambda st, l=l: l.gemm(*ops, Y=Y, stream=st, act=act) for l in lins]), 2)
            saved = [l.bias for l in lins]
            for l in lins:
                l.bias = None
            row["us_plain"] = round(time_launches([lambda st, l=l: l.gemm(*ops, Y=Y, stream=st) for l in lins]), 2)
            for l, b in zip(lins, saved):
                l.bias = b
            row["cost_silu"] = "%+.0f %%" % (100.0 * (row["us_bias_silu"] / row["us_plain"] - 1.0))
            assert q.qlin_get_device_error() == 0
            print(json.dumps(row), flush=True)
        del lins
        torch.cuda.empty_cache()


def run_case(args):
    """A few launches of one GEMM configuration (small ncu captures)."""
    import torch

    import precision_quantized_linear_gb300 as q
    from precision_quantized_linear_gb300 import synthetic as syn
    from precision_quantized_linear_gb300.layers import (MXFP4Linear, MXFP8Linear, NVFP4Linear, W4A8Linear, W4A16Linear,
                                                          W8A8BlockLinear, W8A8Linear)

    torch.cuda.set_device(0)
    q.build()
    q.load()
    M, N, K = args.M, args.N, args.K
    path = {"auto": q.PATH_AUTO, "gemv": q.PATH_GEMV, "tc": q.PATH_TC}[args.path]
    W = torch.from_numpy(syn.make_weight(N, K, seed=5).view(np.int16)).cuda()
    X = torch.from_numpy(syn.make_act(M, K, seed=6).view(np.int16)).cuda()
    if args.case == "w4a16":
        lin = W4A16Linear(W)
        fn = lambda: lin(X, path=path)  # noqa: E731
    elif args.case == "w4a8":
        lin = W4A8Linear(W)
        Xq, sx = lin.quant_act(X)
        fn = lambda: lin.gemm(Xq, sx)  # noqa: E731
    elif args.case == "mxfp8":
        lin = MXFP8Linear(W)
        Xq, xs = lin.quant_act(X)
        fn = lambda: lin.gemm(Xq, xs)  # noqa: E731
    elif args.case == "mxfp4":
        lin = MXFP4Linear(W)
        Xq, xs = lin.quant_act(X)
        fn = lambda: lin.gemm(Xq, xs)  # noqa: E731
    elif args.case == "nvfp4":
        lin = NVFP4Linear(W)
        Xq, xs, sgx = lin.quant_act(X)
        fn = lambda: lin.gemm(Xq, xs, sgx)  # noqa: E731
    elif args.case == "w8a8b":
        lin = W8A8BlockLinear(W)
        Xq, sx = lin.quant_act(X)
        fn = lambda: lin.gemm(Xq, sx)  # noqa: E731
    else:
        lin = W8A8Linear(W)
        Xq, sx = lin.quant_act(X)
        fn = lambda: lin.gemm(Xq, sx, path=path)  # noqa: E731
    del W
    fn()
    torch.cuda.synchronize()
    e0, e1 = make_event(False), make_event(False)
    e0.record()
    for _ in range(args.reps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    assert q.qlin_get_device_error() == 0
    print(json.dumps({"case": args.case, "M": M, "N": N, "K": K, "path": args.path,
                      "us_per_call": round(e0.elapsed_time(e1) * 1e3 / args.reps, 2)}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--sweep", default=None, choices=["crossover", "prefill", "70b", "decode", "blocks", "epilogue"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sweeps", action="store_true", help="decode line only (no prefill / crossover objects)")
    ap.add_argument("--case", default=None, choices=["w4a16", "w8a8", "w8a8b", "w4a8", "mxfp8", "mxfp4",
                                                          "nvfp4"])
    ap.add_argument("--M", type=int, default=16)
    ap.add_argument("--N", type=int, default=28672)
    ap.add_argument("--K", type=int, default=4096)
    ap.add_argument("--path", default="auto", choices=["auto", "gemv", "tc"])
    ap.add_argument("--reps", type=int, default=3)
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
        return
    if args.sweep:
        run_sweep(args)
        return
    if args.case:
        run_case(args)
        return
    run_ours(args)


if __name__ == "__main__":
    main()
