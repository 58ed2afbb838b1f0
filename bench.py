"""Benchmark: W4 group-128 weight-only linear on one GB300.

Workload (one step): one decode token (M = 1) through the seven Llama-3.1-8B projections
(q/o 4096x4096, k/v 1024x4096, gate/up 14336x4096, down 4096x14336) of 32 layers, each
layer with its own seeded synthetic weights (W ~ N(0, 0.02) with 0.1 % outliers x20,
asymmetric round-to-nearest quantization, group 128): 224 launches of the decode GEMV
reading 3.77 GB of packed weights + scales + zeros a step, far more than the 129 MB L2,
so every step streams from HBM.  The launches of each projection kind are captured in a
CUDA graph; CUDA events between the graphs time each kind.

Reported: value = algorithmic HBM GB/s of the whole step (bytes of packed weights, f32
scales, u8 zeros, bf16 x and y), roofline of the dominant kernel against the measured
copy bandwidth, an end-to-end figure through the public API with host buffers, and the
CPU oracle's throughput on a bounded sample of the same work.  Beside it, the second half
of the metric: the seven projections at M = 2048 on the tensor-core GEMM (TFLOP/s and the
dominant kernel against the measured bf16 peak), an M sweep of the gate projection
(M = 1 .. 2048) across both regimes, and the per-row int8 / int4 and MXFP4-experts
variants at their configurations (GB/s against the HBM peak).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "W4 g128 linear: HBM GB/s & % of peak at M=1; TFLOP/s & % of peak at M=2048"
UNIT = "GB/s"
LAYERS = 32
GROUP = 128
WORKLOAD = "llama-3.1-8b decode, 7 projections x 32 layers, W4A16 group 128, M=1"


def proj_bytes(n: int, k: int, m: int = 1) -> int:
    """Algorithmic bytes of one projection: packed codes + f32 scale + u8 zero + x + y."""
    return n * k // 2 + n * (k // GROUP) * 5 + 2 * m * k + 2 * m * n


def load_traffic(key: str):
    """DRAM bytes a launch measured by ncu for this kernel and shape (profiles/traffic.json),
    or None when not captured for the kernel as it stands."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            return json.load(f).get(key)
    except (OSError, ValueError):
        return None


def load_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ---------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clock / throttle samples during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.file = None

    def start(self):
        self.file = tempfile.TemporaryFile(mode="w+")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        self.proc.wait()
        self.file.seek(0)
        rows = [r.split(",") for r in self.file.read().strip().splitlines() if r.strip()]
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for r in rows:
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except (ValueError, IndexError):
                continue
            for name, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        busy = [s for s in sm if s > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------- oracle leg
def cpu_oracle_sample(target_s: float = 10.0, threads: int | None = None):
    """Oracle throughput (GB/s of algorithmic bytes) on a bounded sample of the step:
    leading rows of each of the seven projections, M = 1, on `threads` host threads (all
    host cores by default)."""
    import numpy as np

    import oracle
    from weight_only_quantized_linear_gb300 import synth

    threads = oracle.max_threads() if threads is None else int(threads)
    oracle.set_threads(threads)
    rng = np.random.default_rng(0)
    rows = 64
    done_bytes = 0
    elapsed = 0.0
    sampled = []
    while elapsed < target_s:
        for name in synth.LLAMA_ORDER:
            n, k = synth.LLAMA_PROJ[name]
            packed = rng.integers(0, 256, (rows, k // 2)).astype(np.uint8)
            scale = (rng.random((rows, k // GROUP)) * 0.01 + 1e-3).astype(np.float32)
            zero = rng.integers(0, 16, (rows, k // GROUP)).astype(np.uint8)
            x = synth.normal_bf16((1, k), seed=1).view(__import__("torch").int16).numpy().view(np.uint16)
            t0 = time.perf_counter()
            oracle.linear_int4_groups(x, packed, scale, zero, None, rows, GROUP)
            elapsed += time.perf_counter() - t0
            done_bytes += rows * k // 2 + rows * (k // GROUP) * 5 + 2 * k + 2 * rows
            sampled.append(name)
        rows *= 2
    return done_bytes / elapsed / 1e9, threads, (
        f"oracle linear_int4_groups (f64 sums, {threads} threads) on the leading rows of the 7 "
        f"Llama projections, doubling rows until {target_s:.0f} s: {done_bytes / 1e6:.1f} MB in {elapsed:.1f} s")


def run_reference(args):
    """--impl reference: the CPU oracle as it stands, on the host cores, same metric."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    per_step = []
    step_s = []
    info = None
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        v, threads, sample = cpu_oracle_sample(target_s=2.0)
        if i >= args.warmup:
            per_step.append(v)
            step_s.append(time.perf_counter() - t0)
        info = (threads, sample)
    value = statistics.median(per_step)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * statistics.mean(step_s), 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD + " (bounded CPU sample per step)"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": info[0], "kind": "oracle", "sample": info[1]},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------------------- GPU leg
PREFILL_M = 2048
SWEEP_M = (1, 4, 16, 64, 128, 512, 2048)


def time_rotating(fn, reps: int, stream) -> float:
    """Mean device time (us) of fn(i) for i = 0..reps-1 after two warm-up calls; callers
    rotate through per-layer weights and inputs, more bytes than L2 holds."""
    import torch

    with torch.cuda.stream(stream):
        fn(0)
        fn(1)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(reps):
            fn(i)
        e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e3 / reps


def run_prefill(dev, weights, layers, peaks, stream):
    """Tensor-core regime: the seven projections at M = 2048 (one launch each, per-layer
    weights and activations in rotation), and an M sweep on the gate projection."""
    import torch

    import weight_only_quantized_linear_gb300 as wq
    from weight_only_quantized_linear_gb300 import synth

    names = synth.LLAMA_ORDER
    reps = max(4, layers)
    xs = {k: [synth.normal_bf16((PREFILL_M, k), seed=50 + i, device="cpu").to(dev) for i in range(min(layers, 8))]
          for k in (4096, 14336)}
    per = {}
    tot_flops = 0.0
    tot_us = 0.0
    for n in names:
        N, K = synth.LLAMA_PROJ[n]
        y = torch.empty((PREFILL_M, N), dtype=torch.bfloat16, device=dev)
        # split-K scratch for the shapes with fewer output tiles than SMs (k, v)
        ws = wq.alloc_workspace(wq.wq_linear_int4_groups_workspace(PREFILL_M, N, K, GROUP), dev)

        def call(i, n=n, K=K, y=y, ws=ws):
            p_, s_, z_ = weights[i % layers][n]
            wq.wq_linear_int4_groups(xs[K][i % len(xs[K])], p_, s_, z_, None, GROUP, y=y, workspace=ws,
                                     stream=stream)

        us = time_rotating(call, reps, stream)
        fl = 2.0 * PREFILL_M * N * K
        per[n] = {"us_per_launch": round(us, 2), "tflops": round(fl / us / 1e6, 1), "kernel": wq.wq_last_launch()}
        tot_flops += fl
        tot_us += us
    dom = max(names, key=lambda n: per[n]["us_per_launch"])
    dN, dK = synth.LLAMA_PROJ[dom]
    dom_tf = 2.0 * PREFILL_M * dN * dK / per[dom]["us_per_launch"] / 1e6
    peak = peaks["bf16_tflops"]
    prefill = {
        "M": PREFILL_M, "tflops": round(tot_flops / tot_us / 1e6, 1),
        "frac_of_bf16_peak": round(tot_flops / tot_us / 1e6 / peak, 4),
        "us_per_layer": round(tot_us, 2), "per_projection": per,
        "roofline": {"bound": "tensor", "achieved": round(dom_tf, 1), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(dom_tf / peak, 4), "traffic": load_traffic(f"prefill {dN}x{dK} M={PREFILL_M}"),
                     "kernel": f"{per[dom]['kernel']} on {dom} {dN}x{dK}, M={PREFILL_M}",
                     "flops_per_launch": 2 * PREFILL_M * dN * dK,
                     "peak_source": peaks["source"] + " (bf16_tflops, burst: each launch timed alone)"},
        "how": "CUDA events over launches rotating through 32 layers' weights (and 8 activation sets)",
    }
    # M sweep on the gate projection (decode GEMV below M = 32, tensor-core GEMM from 32 on)
    N, K = synth.LLAMA_PROJ["gate"]
    sweep = {}
    for M in SWEEP_M:
        xm = [x[:M].contiguous() for x in xs[K]]
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        wsb = wq.wq_linear_int4_groups_workspace(M, N, K, GROUP)
        ws = [wq.alloc_workspace(wsb, dev) for _ in range(layers)] if wsb else [None] * layers

        def call(i, M=M, xm=xm, y=y, ws=ws):
            p_, s_, z_ = weights[i % layers]["gate"]
            wq.wq_linear_int4_groups(xm[i % len(xm)], p_, s_, z_, None, GROUP, y=y, workspace=ws[i % layers],
                                     stream=stream)

        us = time_rotating(call, reps, stream)
        sweep[str(M)] = {"us": round(us, 2), "gbs": round(proj_bytes(N, K, M) / (us * 1e-6) / 1e9, 1),
                         "tflops": round(2.0 * M * N * K / us / 1e6, 2), "kernel": wq.wq_last_launch()}
    # the regime crossover: the decode kernels and the tensor-core GEMM at M = 17 .. 128
    cross = {}
    for M in (17, 24, 32, 48, 64, 96, 128):
        xm = [x[:M].contiguous() for x in xs[K]]
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        row = {}
        for regime, min_m in (("decode", 100000), ("tcgen05", 1)):
            wq.wq_set_tuning(wq.WQ_TUNE_GEMM_MIN_M, min_m)
            try:
                wsb = wq.wq_linear_int4_groups_workspace(M, N, K, GROUP)
                ws = [wq.alloc_workspace(wsb, dev) for _ in range(layers)] if wsb else [None] * layers

                def call(i, M=M, xm=xm, y=y, ws=ws):
                    p_, s_, z_ = weights[i % layers]["gate"]
                    wq.wq_linear_int4_groups(xm[i % len(xm)], p_, s_, z_, None, GROUP, y=y, workspace=ws[i % layers],
                                             stream=stream)

                us = time_rotating(call, reps, stream)
                row[regime] = {"us": round(us, 2), "kernel": wq.wq_last_launch()}
            finally:
                wq.wq_set_tuning(wq.WQ_TUNE_GEMM_MIN_M, 0)
        row["faster"] = min(("decode", "tcgen05"), key=lambda r: row[r]["us"])
        cross[str(M)] = row
    sweep["crossover_gate_14336x4096"] = cross
    return prefill, sweep


def run_variants(dev, peaks, stream):
    """The format variants at their configurations: per-row int8 and int4 (M = 1, 8, 16 on
    14336 x 4096 and 4096 x 14336) and MXFP4 experts in the shared-input form (E = 32,
    K = 2880, N = 5760 and 2880, top-4 of 32, R = 1, 8, 64).  Weight copies and routing
    tables rotate so that every launch reads its bytes from HBM."""
    import torch

    import weight_only_quantized_linear_gb300 as wq
    from weight_only_quantized_linear_gb300 import synth

    hbm = peaks["hbm_gbs"]
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    rows = {}
    for (N, K) in ((14336, 4096), (4096, 14336)):
        i8, i4 = [], []
        for c in range(8):
            w = synth.weight_f32(N, K, seed=700 + c, device=dev)
            if c < 4:
                q, sc, _ = wq.wq_quantize_groups(w, K, 8, wq.WQ_SYM, dev_status=st)
                i8.append((q, sc[:, 0].contiguous()))
            q4, sc4, _ = wq.wq_quantize_groups(w, K, 4, wq.WQ_SYM, dev_status=st)
            i4.append((wq.wq_pack_int4(q4, False, dev_status=st).view(torch.int8), sc4[:, 0].contiguous()))
            del w
        for M in (1, 8, 16):
            x = synth.normal_bf16((M, K), seed=9, device="cpu").to(dev)
            y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            for bits, mats in ((8, i8), (4, i4)):
                wsb = wq.wq_linear_rows_workspace(M, N, K, bits)
                ws = [wq.alloc_workspace(wsb, dev) for _ in range(len(mats))] if wsb else [None] * len(mats)
                fn = wq.wq_linear_int8_rows if bits == 8 else wq.wq_linear_int4_rows

                def call(i, fn=fn, mats=mats, ws=ws, x=x, y=y):
                    qq, ss = mats[i % len(mats)]
                    fn(x, qq, ss, None, y=y, workspace=ws[i % len(mats)], stream=stream)

                us = time_rotating(call, 32, stream)
                nbytes = (N * K if bits == 8 else N * K // 2) + 4 * N + 2 * M * K + 2 * M * N
                gbs = nbytes / (us * 1e-6) / 1e9
                rows[f"int{bits} {N}x{K} M={M}"] = {"us": round(us, 2), "gbs": round(gbs, 1),
                                                    "frac_of_hbm_peak": round(gbs / hbm, 4)}
    mx = {}
    E, K, S = 32, 2880, 4
    for N in (5760, 2880):
        copies = [synth.mxfp4_experts(E, N, K, seed=800 + c, device=dev) for c in range(2)]
        for R in (1, 8, 64):
            routes = [synth.routing_topk(R, E, S, seed=900 + R + j, device=dev)[0] for j in range(8)]
            touched = sum(len(set(r.flatten().tolist())) for r in routes) / len(routes)
            x = synth.normal_bf16((R, 1, K), seed=11, device="cpu").to(dev)
            y = torch.empty((R, S, N), dtype=torch.bfloat16, device=dev)
            wsb = wq.wq_mxfp4_experts_shared_workspace(R, S, E, N, K)
            ws = wq.alloc_workspace(wsb, dev) if wsb else None

            def call(i, copies=copies, routes=routes, x=x, y=y, ws=ws):
                b_, s_ = copies[i % 2]
                wq.wq_mxfp4_experts_shared(x, b_, s_, routes[i % 8], y=y, workspace=ws, stream=stream)

            us = time_rotating(call, 32, stream)
            nbytes = touched * N * K * (0.5 + 1 / 32) + 2 * R * K + 2 * R * S * N
            gbs = nbytes / (us * 1e-6) / 1e9
            mx[f"N={N} R={R}"] = {"us": round(us, 2), "experts_touched": round(touched, 2), "gbs": round(gbs, 1),
                                  "frac_of_hbm_peak": round(gbs / hbm, 4), "kernel": wq.wq_last_launch()}
            # the combine form (softmax weights over the four slots, y [R, N]) and the per-slot
            # form (x [R, S, K]): the same weight bytes
            weights = [torch.softmax(synth.routing_topk(R, E, S, seed=900 + R + j)[1], -1).to(dev) for j in range(8)]
            yc = torch.empty((R, N), dtype=torch.bfloat16, device=dev)
            wsc = torch.empty(wq.wq_mxfp4_combine_experts_workspace(R, S, E, N, K), dtype=torch.uint8, device=dev)

            def call_c(i, copies=copies, routes=routes, weights=weights, x=x, yc=yc, wsc=wsc):
                b_, s_ = copies[i % 2]
                wq.wq_mxfp4_combine_experts(x, b_, s_, routes[i % 8], weights[i % 8], y=yc, workspace=wsc,
                                            stream=stream)

            us_c = time_rotating(call_c, 32, stream)
            gbs_c = (nbytes - 2 * R * S * N + 2 * R * N) / (us_c * 1e-6) / 1e9
            mx[f"combine N={N} R={R}"] = {"us": round(us_c, 2), "gbs": round(gbs_c, 1),
                                          "frac_of_hbm_peak": round(gbs_c / hbm, 4)}
            xs_ = synth.normal_bf16((R, S, K), seed=12, device="cpu").to(dev)

            def call_s(i, copies=copies, routes=routes, xs_=xs_, y=y):
                b_, s_ = copies[i % 2]
                wq.wq_mxfp4_experts(xs_, b_, s_, routes[i % 8], y=y, stream=stream)

            us_s = time_rotating(call_s, 32, stream)
            gbs_s = (nbytes + 2 * R * (S - 1) * K) / (us_s * 1e-6) / 1e9
            mx[f"per-slot N={N} R={R}"] = {"us": round(us_s, 2), "gbs": round(gbs_s, 1),
                                           "frac_of_hbm_peak": round(gbs_s / hbm, 4)}
        # many routed rows (prefill / serving batches): the grouped tensor-core GEMM, its
        # four launches (routing tables, gather, GEMM) timed together; dense-equivalent
        # FLOPs 2 * R * S * N * K against the bf16 tensor peak
        for R in (512, 2048):
            routes = [synth.routing_topk(R, E, S, seed=950 + R + j, device=dev)[0] for j in range(4)]
            x = synth.normal_bf16((R, K), seed=13, device="cpu").to(dev)
            y = torch.empty((R, S, N), dtype=torch.bfloat16, device=dev)
            ws = wq.alloc_workspace(wq.wq_mxfp4_experts_shared_workspace(R, S, E, N, K), dev)

            def call_g(i, copies=copies, routes=routes, x=x, y=y, ws=ws):
                b_, s_ = copies[i % 2]
                wq.wq_mxfp4_linear_experts_shared(x, b_, s_, routes[i % 4], y=y, workspace=ws, stream=stream)

            us_g = time_rotating(call_g, 8, stream)
            tf = 2.0 * R * S * N * K / (us_g * 1e-6) / 1e12
            mx[f"grouped N={N} R={R}"] = {"us": round(us_g, 2), "tflops": round(tf, 1),
                                          "frac_of_bf16_peak": round(tf / peaks["bf16_tflops"], 4),
                                          "kernel": wq.wq_last_launch()}
    torch.cuda.synchronize()
    if int(st.item()) != 0:
        raise RuntimeError(f"quantize/pack device status {int(st.item())}")
    return rows, mx


def run_fused_decode(dev, weights, layers, xs, stream, steps, warmup):
    """The decode step with the projections that share an input stored concatenated along
    N, as serving engines store them: qkv [6144, K] and gate_up [28672, K], one launch
    each, so 4 launches a layer (qkv, o, gate_up, down) instead of 7.  Same weights, same
    bytes, same outputs (rows of y in projection order)."""
    import torch

    import weight_only_quantized_linear_gb300 as wq
    from weight_only_quantized_linear_gb300 import synth

    groups = (("qkv", ("q", "k", "v")), ("o", ("o",)), ("gate_up", ("gate", "up")), ("down", ("down",)))
    fused = []
    for l in range(layers):
        lw = {}
        for gname, parts in groups:
            if len(parts) == 1:
                lw[gname] = weights[l][parts[0]]
            else:
                lw[gname] = tuple(torch.cat([weights[l][p][i] for p in parts], dim=0) for i in range(3))
        fused.append(lw)
    shapes = {g: (sum(synth.LLAMA_PROJ[p][0] for p in parts), synth.LLAMA_PROJ[parts[0]][1])
              for g, parts in groups}
    ys = {(l, g): torch.empty((1, shapes[g][0]), dtype=torch.bfloat16, device=dev)
          for l in range(layers) for g, _ in groups}
    ws = {g: [wq.alloc_workspace(wq.wq_linear_int4_groups_workspace(1, *shapes[g], GROUP), dev)
              for _ in range(layers)] for g, _ in groups}

    def launch_kind(g):
        K = shapes[g][1]
        for l in range(layers):
            p_, s_, z_ = fused[l][g]
            wq.wq_linear_int4_groups(xs[K], p_, s_, z_, None, GROUP, y=ys[(l, g)], workspace=ws[g][l],
                                     stream=stream)

    with torch.cuda.stream(stream):
        for g, _ in groups:
            launch_kind(g)
    torch.cuda.synchronize()
    graphs = {}
    for g, _ in groups:
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            launch_kind(g)
        graphs[g] = gr
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(groups) + 1)] for _ in range(steps)]
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            for g, _ in groups:
                graphs[g].replay()
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for st in range(steps):
            for i, (g, _) in enumerate(groups):
                evs[st][i].record(stream)
                graphs[g].replay()
            evs[st][len(groups)].record(stream)
        t1.record(stream)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / steps
    step_bytes = sum(proj_bytes(*synth.LLAMA_PROJ[n]) for n in synth.LLAMA_ORDER) * layers
    per = {}
    for i, (g, _) in enumerate(groups):
        us = sum(e[i].elapsed_time(e[i + 1]) for e in evs) / (steps * layers) * 1e3
        per[g] = {"shape": f"{shapes[g][0]}x{shapes[g][1]}", "us_per_launch": round(us, 3),
                  "gbs": round(proj_bytes(*shapes[g]) / (us * 1e-6) / 1e9, 1)}
    del fused
    return {"value": round(step_bytes / (ms * 1e-3) / 1e9, 1), "unit": UNIT, "ms_per_step": round(ms, 4),
            "us_per_layer": round(ms * 1e3 / layers, 3), "launches_per_step": 4 * layers,
            "per_launch": per,
            "how": "q/k/v and gate/up weights concatenated along N (one launch each), 4 launches a layer; "
                   "same bytes and outputs as the 7-launch step"}


def run_stream_ceiling(dev, peaks, stream, reps: int = 20):
    """The per-launch read ceiling: a kernel that only reads (wq_bench_stream_read), 32
    launches back to back in a CUDA graph, each over its own buffer (1 GB in all at the
    largest size, far above L2), at the byte counts of the decode launches (down/gate/up
    31.69 MB, q/o 9.06 MB, k/v 2.27 MB).  variant 0: plain 16-byte loads; variant 1: a
    bulk-copy ring per SM that fills before the dependency wait (programmatic dependent
    launch), as a decode kernel with immutable weights may."""
    import torch

    import weight_only_quantized_linear_gb300 as wq
    from weight_only_quantized_linear_gb300 import synth

    sizes = {"31.69 MB (gate/up/down)": proj_bytes(*synth.LLAMA_PROJ["down"]),
             "9.06 MB (q/o)": proj_bytes(*synth.LLAMA_PROJ["q"]),
             "2.27 MB (k/v)": proj_bytes(*synth.LLAMA_PROJ["k"])}
    nbuf = 32
    big = max(sizes.values())
    stride = (big + 4095) // 4096 * 4096
    pool = torch.empty(nbuf * stride, dtype=torch.uint8, device=dev)
    pool.random_(0, 256)
    sink = torch.zeros(1, dtype=torch.int32, device=dev)
    out = {}
    for label, nbytes in sizes.items():
        nb = nbytes // 16 * 16
        row = {}
        for variant in (0, 1):
            def launch_all():
                for i in range(nbuf):
                    wq.wq_bench_stream_read(pool[i * stride:], variant, sink, stream=stream, nbytes=nb)
            with torch.cuda.stream(stream):
                launch_all()
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                launch_all()
            with torch.cuda.stream(stream):
                g.replay()
                torch.cuda.synchronize()
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for _ in range(reps):
                    g.replay()
                e1.record(stream)
            torch.cuda.synchronize()
            us = e0.elapsed_time(e1) * 1e3 / (reps * nbuf)
            gbs = nb / (us * 1e-6) / 1e9
            row["plain_loads" if variant == 0 else "bulk_ring_pdl"] = {
                "us_per_launch": round(us, 3), "gbs": round(gbs, 1),
                "frac_of_hbm_peak": round(gbs / peaks["hbm_gbs"], 4)}
        out[label] = row
    if int(sink.item()) != 0:
        raise RuntimeError("stream probe wrote its sink")
    del pool
    return out


def run_prepared_decode(dev, weights, layers, xs, stream, steps, warmup, row_major_per_kind):
    """The decode step on the prepared layout (wq_prepare_int4_groups at load time, outside
    the timed region; wq_linear_int4_groups_prepared in the step): the same 7 projections
    x 32 layers, the same algorithmic bytes, against the row-major layout's step."""
    import torch

    import weight_only_quantized_linear_gb300 as wq
    from weight_only_quantized_linear_gb300 import synth

    names = synth.LLAMA_ORDER
    prep = [{n: wq.wq_prepare_int4_groups(*weights[l][n], GROUP) for n in names} for l in range(layers)]
    torch.cuda.synchronize()
    ys = {(l, n): torch.empty((1, synth.LLAMA_PROJ[n][0]), dtype=torch.bfloat16, device=dev)
          for l in range(layers) for n in names}
    ws = {n: [wq.alloc_workspace(wq.wq_linear_int4_groups_prepared_workspace(1, *synth.LLAMA_PROJ[n], GROUP), dev)
              for _ in range(layers)] for n in names}
    launched = {}

    def launch_kind(n):
        N, K = synth.LLAMA_PROJ[n]
        for l in range(layers):
            wq.wq_linear_int4_groups_prepared(xs[K], prep[l][n], N, None, GROUP, y=ys[(l, n)], workspace=ws[n][l],
                                              stream=stream)

    with torch.cuda.stream(stream):
        for n in names:
            launch_kind(n)
            launched[n] = wq.wq_last_launch()
    torch.cuda.synchronize()
    graphs = {}
    for n in names:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            launch_kind(n)
        graphs[n] = g
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)] for _ in range(steps)]
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            for n in names:
                graphs[n].replay()
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for st in range(steps):
            for i, n in enumerate(names):
                evs[st][i].record(stream)
                graphs[n].replay()
            evs[st][len(names)].record(stream)
        t1.record(stream)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / steps
    step_bytes = sum(proj_bytes(*synth.LLAMA_PROJ[n]) for n in names) * layers
    per = {}
    for i, n in enumerate(names):
        us = sum(e[i].elapsed_time(e[i + 1]) for e in evs) / (steps * layers) * 1e3
        per[n] = {"us_per_launch": round(us, 3), "gbs": round(proj_bytes(*synth.LLAMA_PROJ[n]) / (us * 1e-6) / 1e9, 1),
                  "row_major_us": row_major_per_kind[n]["us_per_launch"], "kernel": launched[n]}
    del prep, graphs
    return {"value": round(step_bytes / (ms * 1e-3) / 1e9, 1), "unit": UNIT, "ms_per_step": round(ms, 4),
            "per_projection": per,
            "how": "weights repacked once at load (wq_prepare_int4_groups, not timed); same bytes, same step"}


def build_weights(dev, layers: int, seed0: int = 1000):
    """Per layer and projection: packed u8 [N, K/2], scale f32 [N, K/G], zero u8 [N, K/G]."""
    import torch

    import weight_only_quantized_linear_gb300 as wq
    from weight_only_quantized_linear_gb300 import synth

    weights = []
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    for layer in range(layers):
        lw = {}
        for j, name in enumerate(synth.LLAMA_ORDER):
            n, k = synth.LLAMA_PROJ[name]
            w = synth.weight_f32(n, k, seed=seed0 + layer * 7 + j, outlier_frac=0.001, device=dev)
            codes, scale, zero = wq.wq_quantize_groups(w, GROUP, 4, wq.WQ_ASYM, dev_status=st)
            del w
            packed = wq.wq_pack_int4(codes, True, dev_status=st)
            del codes
            lw[name] = (packed, scale, zero)
        weights.append(lw)
    torch.cuda.synchronize()
    if int(st.item()) != 0:
        raise RuntimeError(f"quantize/pack device status {int(st.item())}")
    return weights


def run_gpu(args):
    import torch
    import torch.distributed as dist

    import weight_only_quantized_linear_gb300 as wq
    from weight_only_quantized_linear_gb300 import synth

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    wq.build()
    # decode serving: weights are written once at load time and never during a step, so
    # each launch may start streaming its weights while the previous one finishes
    wq.wq_set_static_weights(True)
    peaks = load_peaks()

    layers = args.layers
    weights = build_weights(dev, layers, seed0=1000 + 97 * rank)
    names = synth.LLAMA_ORDER
    xs = {k: synth.normal_bf16((1, k), seed=5 + k, device="cpu").to(dev) for k in (4096, 14336)}
    ys = {(l, n): torch.empty((1, synth.LLAMA_PROJ[n][0]), dtype=torch.bfloat16, device=dev)
          for l in range(layers) for n in names}
    ws = {}
    for n in names:
        N, K = synth.LLAMA_PROJ[n]
        b = wq.wq_linear_int4_groups_workspace(1, N, K, GROUP)
        # one workspace per layer and projection: launches never share counters
        ws[n] = [wq.alloc_workspace(b, dev) for _ in range(layers)]
    stream = torch.cuda.Stream(device=dev)

    def launch_kind(n):
        N, K = synth.LLAMA_PROJ[n]
        for l in range(layers):
            p, s, z = weights[l][n]
            wq.wq_linear_int4_groups(xs[K], p, s, z, None, GROUP, y=ys[(l, n)], workspace=ws[n][l], stream=stream)

    # warm the kernels once outside capture (attributes, descriptors), then capture; note
    # the kernel instance the library picks for each projection
    launched = {}
    with torch.cuda.stream(stream):
        for n in names:
            launch_kind(n)
            launched[n] = wq.wq_last_launch()
    torch.cuda.synchronize()
    graphs = {}
    for n in names:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            launch_kind(n)
        graphs[n] = g
    torch.cuda.synchronize()

    step_bytes = sum(proj_bytes(*synth.LLAMA_PROJ[n]) for n in names) * layers
    launches_per_step = len(names) * layers

    def one_step(evs=None):
        for i, n in enumerate(names):
            if evs is not None:
                evs[i].record(stream)
            graphs[n].replay()
        if evs is not None:
            evs[len(names)].record(stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            one_step()
    torch.cuda.synchronize()

    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    clocks.start()
    step_events = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)] for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t_start.record(stream)
        for s in range(args.steps):
            one_step(step_events[s])
        t_end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    per_kind_pre = {}
    for i, n in enumerate(names):
        us = sum(evs[i].elapsed_time(evs[i + 1]) for evs in step_events) / (args.steps * layers) * 1e3
        per_kind_pre[n] = {"us_per_launch": round(us, 3)}

    # ---------------- the other legs: fused decode step, M = 2048, M sweep, variants ----------------
    prefill = sweep = rows_leg = mxfp4_leg = None
    clocks_p = ClockSampler(dev.index if dev.index is not None else 0)
    clocks_p.start()
    ceiling = run_stream_ceiling(dev, peaks, stream)
    fused_leg = run_fused_decode(dev, weights, layers, xs, stream, max(10, min(args.steps, 500)), args.warmup)
    prepared_leg = run_prepared_decode(dev, weights, layers, xs, stream, max(10, min(args.steps, 500)), args.warmup,
                                       per_kind_pre)
    if not args.no_prefill:
        prefill, sweep = run_prefill(dev, weights, layers, peaks, stream)
        rows_leg, mxfp4_leg = run_variants(dev, peaks, stream)
    clk_other = clocks_p.stop()
    total_ms = t_start.elapsed_time(t_end)
    if world > 1:
        t = torch.tensor([total_ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms = float(t.item())
    ms_per_step = total_ms / args.steps
    value = step_bytes * world / (ms_per_step * 1e-3) / 1e9

    per_kind_ms = {n: 0.0 for n in names}
    for evs in step_events:
        for i, n in enumerate(names):
            per_kind_ms[n] += evs[i].elapsed_time(evs[i + 1])
    per_kind = {}
    for n in names:
        N, K = synth.LLAMA_PROJ[n]
        us = per_kind_ms[n] / (args.steps * layers) * 1e3
        per_kind[n] = {"us_per_launch": round(us, 3), "gbs": round(proj_bytes(N, K) / (us * 1e-6) / 1e9, 1),
                       "kernel": launched[n]}
    dom = max(names, key=lambda n: per_kind_ms[n])
    dN, dK = synth.LLAMA_PROJ[dom]
    dom_us = per_kind[dom]["us_per_launch"]
    achieved = proj_bytes(dN, dK) / (dom_us * 1e-6) / 1e9
    traffic = load_traffic(f"decode {dN}x{dK}")

    # ---------------- end to end through the public API, host buffers ----------------
    x_host = {k: v.cpu().pin_memory() for k, v in xs.items()}
    last = [(layers - 1, n) for n in names]
    y_host = {key: torch.empty(ys[key].shape, dtype=torch.bfloat16).pin_memory() for key in last}
    h2d = sum(v.numel() * 2 for v in x_host.values())
    d2h = sum(v.numel() * 2 for v in y_host.values())
    e2e_steps = max(3, min(args.steps, 500))
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(e2e_steps):
            for k in xs:
                xs[k].copy_(x_host[k], non_blocking=True)
            one_step()
            for key in last:
                y_host[key].copy_(ys[key], non_blocking=True)
        e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    e2e_value = step_bytes * world / (e2e_ms * 1e-3) / 1e9

    # the same, with every public API call made eagerly each step (no graph): the host
    # side of the C ABI (validation, tensor maps, launch through ctypes) is inside the
    # timed region, 224 calls a step
    eager_steps = max(3, min(args.steps, 200))
    with torch.cuda.stream(stream):
        for _ in range(2):
            for n in names:
                launch_kind(n)
    torch.cuda.synchronize()
    h0 = time.perf_counter()
    e0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(eager_steps):
            for k in xs:
                xs[k].copy_(x_host[k], non_blocking=True)
            for n in names:
                launch_kind(n)
            for key in last:
                y_host[key].copy_(ys[key], non_blocking=True)
        e1.record(stream)
    torch.cuda.synchronize()
    eager_host_ms = (time.perf_counter() - h0) * 1e3 / eager_steps
    eager_ms = e0.elapsed_time(e1) / eager_steps
    eager_value = step_bytes * world / (eager_ms * 1e-3) / 1e9

    cpu = None
    if rank == 0 and not args.no_cpu:
        v, threads, sample = cpu_oracle_sample(target_s=args.cpu_seconds)
        v1, _, sample1 = cpu_oracle_sample(target_s=max(2.0, args.cpu_seconds / 2), threads=1)
        cpu = {"value": round(v, 4), "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample,
               "single_thread": {"value": round(v1, 4), "unit": UNIT, "cores": 1, "sample": sample1}}

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16 activations, u4 weights, f32 accumulate",
            "data": "synthetic",
            "config": {"workload": WORKLOAD, "M": 1, "group": GROUP, "layers": layers,
                       "bytes_per_step": step_bytes, "l2": "inputs larger than L2 (3.77 GB of weights a step)",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       "static_weights": "wq_set_static_weights(1): weights are load-time constants"},
            "frac_of_hbm_peak": round(value / world / peaks["hbm_gbs"], 4),
            "us_per_layer": round(ms_per_step * 1e3 / layers, 3),
            "per_projection": per_kind,
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": traffic,
                         "kernel": f"{launched[dom]} on {dom} {dN}x{dK}",
                         "bytes_per_launch": proj_bytes(dN, dK), "peak_source": peaks["source"] + " (hbm_gbs)"},
            "e2e": {"value": round(e2e_value, 1), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "how": "public API calls captured in CUDA graphs; pinned x copied in and the last layer's "
                           "outputs copied out inside the timed region"},
            "e2e_eager": {"value": round(eager_value, 1), "unit": UNIT, "ms_per_step": round(eager_ms, 4),
                          "host_ms_per_step": round(eager_host_ms, 4), "calls_per_step": launches_per_step,
                          "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                          "how": "every wq_linear_int4_groups call made through ctypes each step (no graph): "
                                 "host validation, tensor-map encoding and launch inside the timed region"},
            "stream_ceiling": ceiling,
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clk,
            "cpu_baseline": cpu,
            "prefill_m2048": prefill,
            "decode_fused_qkv_gateup": fused_leg,
            "decode_prepared_layout": prepared_leg,
            "m_sweep_gate": sweep,
            "rows_int8_int4": rows_leg,
            "mxfp4_experts_shared": mxfp4_leg,
            "clocks_other_legs": clk_other,
        }
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_profile_case(args):
    """A few launches of one kernel on one projection, for profiler captures: decode_gate /
    decode_down / decode_k (M = 1, workspace on, as timed above), prepared_down (M = 1 on the
    repacked layout), prefill_gate / prefill_down / prefill_k (M = 2048) or mxfp4_gateup (MXFP4
    experts, one row routed to 4 of 32)."""
    import torch

    import weight_only_quantized_linear_gb300 as wq
    from weight_only_quantized_linear_gb300 import synth

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    wq.build()
    if args.profile_case == "mxfp4_gateup":
        # MXFP4 experts, shared input: E = 32, gate/up N = 5760, K = 2880, one row, top-4
        E, N, K, S, R = 32, 5760, 2880, 4, args.profile_rows
        blocks, scales = synth.mxfp4_experts(E, N, K, seed=800, device=dev)
        route = synth.routing_topk(R, E, S, seed=900 + R + 1, device=dev)[0]
        x = synth.normal_bf16((R, 1, K), seed=11, device="cpu").to(dev)
        y = torch.empty((R, S, N), dtype=torch.bfloat16, device=dev)
        wsb = wq.wq_mxfp4_experts_shared_workspace(R, S, E, N, K)
        ws = wq.alloc_workspace(wsb, dev) if wsb else None
        for _ in range(3):
            wq.wq_mxfp4_experts_shared(x, blocks, scales, route, y=y, workspace=ws)
        torch.cuda.synchronize()
        print(f"profile case {args.profile_case}: R={R} S={S} E={E} N={N} K={K}, 3 launches")
        return 0
    kind, proj = args.profile_case.split("_")
    N, K = synth.LLAMA_PROJ[proj]
    M = PREFILL_M if kind == "prefill" else 1
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    w = synth.weight_f32(N, K, seed=1000, outlier_frac=0.001, device=dev)
    codes, scale, zero = wq.wq_quantize_groups(w, GROUP, 4, wq.WQ_ASYM, dev_status=st)
    packed = wq.wq_pack_int4(codes, True, dev_status=st)
    del w, codes
    x = synth.normal_bf16((M, K), seed=5, device="cpu").to(dev)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    if kind == "prepared":
        # the decode step on the load-time repacked layout (the repack itself is not timed)
        prep = wq.wq_prepare_int4_groups(packed, scale, zero, GROUP)
        ws = wq.alloc_workspace(wq.wq_linear_int4_groups_prepared_workspace(M, N, K, GROUP), dev)
        for _ in range(3):
            wq.wq_linear_int4_groups_prepared(x, prep, N, None, GROUP, y=y, workspace=ws, dev_status=st)
    else:
        ws = wq.alloc_workspace(wq.wq_linear_int4_groups_workspace(M, N, K, GROUP), dev)
        for _ in range(3):
            wq.wq_linear_int4_groups(x, packed, scale, zero, None, GROUP, y=y, workspace=ws, dev_status=st)
    torch.cuda.synchronize()
    if int(st.item()) != 0:
        raise RuntimeError(f"device status {int(st.item())}")
    print(f"profile case {args.profile_case}: M={M} N={N} K={K}, 3 launches")
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--layers", type=int, default=LAYERS)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--profile-rows", type=int, default=1, help="routed rows R of the mxfp4_gateup profile case")
    ap.add_argument("--profile-case", choices=["decode_gate", "decode_down", "decode_k", "prefill_gate", "prefill_down",
                                               "prefill_k", "prepared_down", "mxfp4_gateup"],
                    help="run three launches of one kernel (for profiler captures) and exit")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.profile_case:
        return run_profile_case(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
