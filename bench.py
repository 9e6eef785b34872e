"""Benchmark of the Q4_K decode hot path on GB300.

Headline (the JSON line's `value`): weight-streaming throughput in GB/s of one
decode step of a Qwen2.5-7B-shaped model -- 28 layers x 7 Q4_K GEMVs (q, k, v,
o, gate, up, down), batch 1 -- with all inputs resident in HBM, the step's
launches (q/k/v fused into one, gate/up into one: 4 per layer) replayed from a
CUDA graph.  Algorithmic bytes per step = the Q4_K
weights (4.5 bits/weight) + fp32 activations read + fp32 outputs written.

The same line carries the batch-2/5/9 VerifyBatch sweep, the fused LM-head +
argmax latency (152064 x 3584, batch 1 and 5), the prefill tiles, the roofline
of the dominant kernel, an end-to-end figure through the public API with host
buffers, clocks sampled during the timed regions, and the CPU oracle timed on
the host cores.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

`--impl reference` times the CPU oracle (the reference arm) on a
bounded sample of the same workload and prints the same kind of line.
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

METRIC = "Q4_K GEMV weight GB/s & % of HBM peak (batch 1/5); LM-head+argmax µs"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
LAYERS = 28
SPEC_HBM_GBS = 8000.0   # nominal GB300 HBM3e bandwidth, the figure the 80 % target is stated against


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            return {"hbm_gbs": float(d.get("hbm_gbs", FALLBACK_HBM_GBS)),
                    "bf16_tflops": float(d.get("bf16_tflops", FALLBACK_BF16_TFLOPS)),
                    "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d.get("bf16_tflops", FALLBACK_BF16_TFLOPS))),
                    "source": "measured"}
        except Exception:
            pass
    return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
            "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def max_over_ranks(value: float, device=None) -> float:
    """Largest value over all ranks of the default process group (itself when
    there is none).  Timing is reported as the slowest rank's."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world: int, slowest_seconds: float) -> float:
    """Units processed by all ranks (weak scaling: each rank does the same
    work) divided by the slowest rank's time."""
    return units_per_rank * world / slowest_seconds


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled while timed work runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
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
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        busy = [s for s in sm if s > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- CPU oracle (reference arm / baseline)
def oracle_sample(seconds_target: float = 8.0):
    """Time the CPU oracle on layer 0's seven matrices (batch 1); returns GB/s of weight bytes."""
    import oracle
    import synth
    oracle.build()
    layer = synth.qwen_layer_weights(0)
    xs = {K: synth.normal_f32((1, K), (0, 9, K)) for K in {k for _, _, k, _ in layer}}
    threads = oracle.max_threads()
    wbytes = sum(W.nbytes for *_, W in layer)
    reps, t0 = 0, time.perf_counter()
    while True:
        for name, N, K, W in layer:
            oracle.gemv(W, xs[K], N, K, threads=threads)
        reps += 1
        if time.perf_counter() - t0 > seconds_target:
            break
    dt = time.perf_counter() - t0
    # the same code on one thread (the correctness reference's own speed), one pass
    t1 = time.perf_counter()
    for name, N, K, W in layer:
        oracle.gemv(W, xs[K], N, K, threads=1)
    dt1 = time.perf_counter() - t1
    return {"value": wbytes * reps / dt / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "single_thread_value": wbytes / dt1 / 1e9,
            "sample": f"layer 0 of the Qwen2.5-7B-shaped decode (7 Q4_K GEMVs, {wbytes} weight bytes), batch 1, "
                      f"{reps} passes in {dt:.1f} s, fp64 accumulation, OpenMP over rows; "
                      f"single_thread_value: one pass on one thread ({dt1:.1f} s)"}


def _best_and_cv(fn, min_reps=3, max_s=3.0):
    """Best-of-N wall time of fn() with its coefficient of variation (the
    dotLLM README's benchmark method: best of several runs, CV reported)."""
    import numpy as np
    ts, t_all = [], time.perf_counter()
    while len(ts) < min_reps or (time.perf_counter() - t_all < max_s and len(ts) < 50):
        t0 = time.perf_counter()
        fn()
        ts.append(time.perf_counter() - t0)
        if time.perf_counter() - t_all > 4 * max_s:
            break
    return min(ts), float(np.std(ts) / np.mean(ts)), len(ts)


def oracle_configs():
    """The CPU oracle (fp64, OpenMP over rows on all host cores) on the other
    configurations: the single 4096 x 4096 GEMV and the LM head + argmax in
    full, the batch-5 VerifyBatch pass over layer 0 (the 28-layer step time
    extrapolated from it), and the four Llama-3-8B prefill shapes at T = 32
    and T = 512 in full."""
    import oracle
    import synth
    oracle.build()
    th = oracle.max_threads()
    out = {"cores": th}
    W0 = synth.q4k_weights(4096, 4096, (0, 0))
    x0 = synth.normal_f32((1, 4096), (0, 1))
    best, cv, n = _best_and_cv(lambda: oracle.gemv(W0, x0, 4096, 4096, threads=th))
    b0 = 4096 * 16 * 144 + 4 * 4096 * 2
    out["single_gemv_4096x4096_b1"] = {"ms_best": best * 1e3, "cv": cv, "reps": n, "gbs": b0 / best / 1e9}
    layer = synth.qwen_layer_weights(0)
    xs5 = {K: synth.normal_f32((5, K), (0, 9, K, 5)) for K in {k for _, _, k, _ in layer}}
    best, cv, n = _best_and_cv(lambda: [oracle.gemv(W, xs5[K], N, K, threads=th) for _, N, K, W in layer])
    b5 = sum(N * (K // 256) * 144 + 4 * 5 * K + 4 * 5 * N for _, N, K, _ in layer)
    out["verify_batch5_layer0"] = {"ms_best": best * 1e3, "cv": cv, "reps": n, "gbs": b5 / best / 1e9,
                                   "ms_per_step_28_layers_extrapolated": best * 1e3 * LAYERS}
    del layer, xs5
    Nv, Kv = 152064, 3584
    Wl = synth.q4k_weights(Nv, Kv, (3, 0))
    xl = synth.normal_f32((1, Kv), (3, 2))
    best, cv, n = _best_and_cv(lambda: oracle.argmax(oracle.gemv(Wl, xl, Nv, Kv, threads=th)[0]))
    out["lm_head_argmax_b1"] = {"ms_best": best * 1e3, "cv": cv, "reps": n,
                                "gbs": (Nv * (Kv // 256) * 144 + 4 * Kv + 4) / best / 1e9}
    del Wl
    pf = {}
    for name, N, K in synth.llama3_8b_prefill_shapes():
        Wp = synth.q4k_weights(N, K, (4, N, K))
        for T in (32, 512):
            X = synth.normal_bf16_bits((T, K), (4, T, K))
            best, cv, n = _best_and_cv(lambda: oracle.prefill(Wp, X, N, K, threads=th),
                                       min_reps=1 if T == 512 else 3, max_s=0.5 if T == 512 else 2.0)
            pf[f"{name}_{N}x{K}_T{T}"] = {"ms_best": best * 1e3, "cv": cv, "reps": n,
                                          "gflops": 2.0 * N * K * T / best / 1e9}
    out["prefill"] = pf
    return out


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    import synth
    oracle.build()
    layer = synth.qwen_layer_weights(0)
    xs = {K: synth.normal_f32((1, K), (0, 9, K)) for K in {k for _, _, k, _ in layer}}
    threads = oracle.max_threads()
    step_bytes = sum(W.nbytes + 4 * K + 4 * N for _, N, K, W in layer)

    def step():
        for name, N, K, W in layer:
            oracle.gemv(W, xs[K], N, K, threads=threads)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    value = step_bytes * args.steps / dt / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": "qwen2.5-7b-shaped decode GEMVs, batch 1 (sample: layer 0's 7 matrices per step)",
                       "batch": 1},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": "each step = layer 0's 7 Q4_K GEMVs (q,k,v,o,gate,up,down), batch 1"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- GPU arm
def kernel_source_hash():
    """Hash of the GEMV kernel's code with comments and whitespace removed, so
    that the recorded DRAM traffic stays valid across comment-only edits and is
    dropped as soon as any code changes."""
    import re
    h = hashlib.sha256()
    for f in ("q4k_gemv.cu", "q4k_dev.cuh", "ptx.cuh"):
        src = open(os.path.join(ROOT, "q4_dequant_gemv_gb300", "csrc", f)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        h.update(re.sub(r"\s+", "", src).encode())
    return h.hexdigest()[:16]


def recorded_traffic():
    """DRAM bytes per algorithmic byte of the batch-1 GEMV kernel, from the
    committed ncu summary, if it was captured from the current kernel source."""
    p = os.path.join(ROOT, "profiles", "gemv_traffic.txt")
    if not os.path.exists(p):
        return None
    d = {}
    for line in open(p):
        if ":" in line and not line.startswith("#"):
            k, v = line.split(":", 1)
            d[k.strip()] = v.strip()
    if d.get("source_hash") != kernel_source_hash():
        return None
    try:
        return {"dram_bytes_per_weight_byte": float(d["dram_bytes_per_algorithmic_byte"])}
    except (KeyError, ValueError):
        return None


def run_ours(args):
    import numpy as np
    import torch

    import __graft_entry__
    import q4_dequant_gemv_gb300 as q4k
    import synth

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    __graft_entry__.build()
    pk = peaks()

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    # ---- weights of 28 Qwen2.5-7B-shaped layers, resident in HBM
    shapes = synth.qwen25_7b_shapes()
    Ws = []
    for layer in range(LAYERS):
        lw = synth.qwen_layer_weights(layer)
        Ws.append([torch.from_numpy(W).to(dev) for _, _, _, W in lw])
    # Activations: q/k/v share one input, gate/up share one (as in a decoder
    # layer); o and down have their own.  All live in one flat buffer per batch
    # size, layer-major, so that the end-to-end run moves each layer's inputs
    # and outputs as one contiguous range.
    kinds = (("attn", 3584, 50), ("o", 3584, 51), ("mlp", 3584, 52), ("down", 18944, 53))
    x_per_layer = sum(K for _, K, _ in kinds)
    y_per_layer = sum(N for _, N, _ in shapes)
    x_elems_per_row = LAYERS * x_per_layer
    y_elems_per_row = LAYERS * y_per_layer
    x_flat = torch.empty(16 * x_elems_per_row, dtype=torch.float32, device=dev)
    y_flat = torch.empty(16 * y_elems_per_row, dtype=torch.float32, device=dev)

    kind_off = {}
    acc = 0
    for kname, K, _ in kinds:
        kind_off[kname] = (acc, K)
        acc += K

    def x_view(B, layer, kind):
        """[B, K] activations of one (layer, consumer); contiguous, batch-major."""
        off, K = kind_off[kind]
        start = B * (layer * x_per_layer + off)
        return x_flat[start:start + B * K].view(B, K)

    def y_view(B, layer, mi):
        off = sum(N for _, N, _ in shapes[:mi])
        N = shapes[mi][1]
        start = B * (layer * y_per_layer + off)
        return y_flat[start:start + B * N].view(B, N)

    g_x = synth.rng(7, 7)
    x_flat.copy_(torch.from_numpy(g_x.standard_normal(x_flat.numel(), dtype=np.float32)))
    src = {"q": "attn", "k": "attn", "v": "attn", "o": "o", "gate": "mlp", "up": "mlp", "down": "down"}
    stream = torch.cuda.Stream(device=dev)

    def step_bytes(B):
        return LAYERS * sum(N * (K // 256) * 144 + 4 * B * K + 4 * B * N for _, N, K in shapes)

    def decode_step(B, pdl=True, fused=True, tc=False, q8=False, hook=None):
        """One decode step: 28 layers x 7 GEMVs.  fused: q/k/v share one launch
        and gate/up share one (4 launches per layer); otherwise 7 launches.
        tc: batch 1 on the tensor-core inner product instead of the integer one.
        q8: batch 1 with x quantized Q8_K style (its own error bound).
        hook(layer, when) runs before ("pre") and after ("post") each layer's
        launches (the end-to-end step issues its copies there)."""
        for layer in range(LAYERS):
            if hook is not None:
                hook(layer, "pre")
            W, y = Ws[layer], (lambda mi: y_view(B, layer, mi))
            if fused:
                q4k.gemv_grouped(W[0:3], x_view(B, layer, "attn"), [y(0), y(1), y(2)], stream=stream, pdl=pdl,
                                 tensor_core=tc, q8k=q8)
                q4k.gemv(W[3], x_view(B, layer, "o"), y(3), stream=stream, pdl=pdl, tensor_core=tc, q8k=q8)
                q4k.gemv_grouped(W[4:6], x_view(B, layer, "mlp"), [y(4), y(5)], stream=stream, pdl=pdl,
                                 tensor_core=tc, q8k=q8)
                q4k.gemv(W[6], x_view(B, layer, "down"), y(6), stream=stream, pdl=pdl, tensor_core=tc, q8k=q8)
            else:
                for mi, (name, N, K) in enumerate(shapes):
                    q4k.gemv(W[mi], x_view(B, layer, src[name]), y(mi), stream=stream, pdl=pdl, tensor_core=tc)
            if hook is not None:
                hook(layer, "post")

    def capture(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            fn()   # eager warm-up (sets kernel attributes)
            stream.synchronize()
            with torch.cuda.graph(g, stream=stream):
                fn()
        stream.synchronize()
        return g

    def time_graph(g, steps, warmup):
        # graph replays go to the current stream: make it the timed stream
        with torch.cuda.stream(stream):
            for _ in range(warmup):
                g.replay()
            stream.synchronize()
            barrier()
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(steps):
                g.replay()
            e1.record(stream)
        e1.synchronize()
        torch.cuda.synchronize()
        barrier()
        ms = max_over_ranks(e0.elapsed_time(e1), device=dev)
        return ms / steps

    clocks = ClockSampler(local)
    clocks.start()

    # ---- headline: batch 1
    g1 = capture(lambda: decode_step(1))
    ms1 = time_graph(g1, args.steps, args.warmup)
    bytes1 = step_bytes(1)
    value = whole_job_rate(bytes1, world, ms1 * 1e-3) / 1e9

    # ---- time per kind of launch: the 28 launches of one kind (q/k/v, o,
    # gate/up, down) replayed alone in a graph with PDL, per launch, beside the
    # time its bytes take at the peak of record
    def kind_step(kind, B=1):
        for layer in range(LAYERS):
            W, y = Ws[layer], (lambda mi: y_view(B, layer, mi))
            if kind == "qkv":
                q4k.gemv_grouped(W[0:3], x_view(B, layer, "attn"), [y(0), y(1), y(2)], stream=stream, pdl=True)
            elif kind == "o":
                q4k.gemv(W[3], x_view(B, layer, "o"), y(3), stream=stream, pdl=True)
            elif kind == "gate_up":
                q4k.gemv_grouped(W[4:6], x_view(B, layer, "mlp"), [y(4), y(5)], stream=stream, pdl=True)
            else:
                q4k.gemv(W[6], x_view(B, layer, "down"), y(6), stream=stream, pdl=True)
    kind_mats = {"qkv": (0, 1, 2), "o": (3,), "gate_up": (4, 5), "down": (6,)}
    kinds_us = {}
    for kind, mats in kind_mats.items():
        gk = capture(lambda k=kind: kind_step(k))
        msk = time_graph(gk, max(20, args.steps // 4), args.warmup)
        del gk
        kb = sum(shapes[m][1] * (shapes[m][2] // 256) * 144 + 4 * shapes[m][2] + 4 * shapes[m][1] for m in mats)
        kinds_us[kind] = {"us_per_launch": msk * 1e3 / LAYERS, "bytes_per_launch": kb,
                          "us_at_peak": kb / (pk["hbm_gbs"] * 1e9) * 1e6}

    # ---- read-only streaming probe (the ceiling a weight stream can reach on
    # this GPU; a copy's read+write rate, the peak of record, is lower)
    probe_buf = torch.empty(2 << 30, dtype=torch.uint8, device=dev)
    with torch.cuda.stream(stream):
        pbest, pbytes = None, 0
        for _ in range(6):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            pbytes = q4k.stream_read(probe_buf, stream=stream)
            e1.record(stream)
            e1.synchronize()
            t = e0.elapsed_time(e1)
            pbest = t if pbest is None else min(pbest, t)
    del probe_buf
    read_probe = {"gbs": pbytes / (pbest * 1e-3) / 1e9, "bytes": pbytes, "best_of": 6,
                  "kernel": "q4k_stream_read (one CTA per SM, 32 KB bulk copies, 4-deep ring)"}

    # ---- the same step with one launch per matrix (196 launches), for contrast
    g1u = capture(lambda: decode_step(1, fused=False))
    ms1u = time_graph(g1u, max(20, args.steps // 4), args.warmup)
    del g1u
    unfused = {"gbs": bytes1 / (ms1u * 1e-3) / 1e9, "us_per_step": ms1u * 1e3, "launches_per_step": LAYERS * 7}

    # ---- the same step with batch 1 on the tensor-core inner product (fp16 x parts, mma.sync)
    g1t = capture(lambda: decode_step(1, tc=True))
    ms1t = time_graph(g1t, max(20, args.steps // 4), args.warmup)
    del g1t
    tensor_core_b1 = {"gbs": bytes1 / (ms1t * 1e-3) / 1e9, "us_per_step": ms1t * 1e3,
                      "kernel": "q4k_gemv_kernel<1,false,0> (mma.sync m16n8k16, x as fp16 hi+lo)"}

    # ---- the same step with x quantized Q8_K style (one int8 code per element; own error bound)
    g1q = capture(lambda: decode_step(1, q8=True))
    ms1q = time_graph(g1q, max(20, args.steps // 4), args.warmup)
    del g1q
    q8k_b1 = {"gbs": bytes1 / (ms1q * 1e-3) / 1e9, "us_per_step": ms1q * 1e3,
              "kernel": "q4k_gemv_kernel<1,false,2> (dp4a, x as Q8_K int8 codes per 256-block)",
              "numerics": "W times the Q8_K-quantized x: differs from W x by <= sum|w| d/2 per row"}

    # ---- VerifyBatch sweep (same weights)
    sweep = {}
    for B in (2, 5, 9):
        gB = capture(lambda B=B: decode_step(B))
        msB = time_graph(gB, max(10, args.steps // 4), args.warmup)
        sweep[f"batch{B}"] = {"gbs": step_bytes(B) / (msB * 1e-3) / 1e9, "us_per_step": msB * 1e3,
                              "us_per_layer": msB * 1e3 / LAYERS,
                              "frac_of_peak": step_bytes(B) / (msB * 1e-3) / 1e9 / pk["hbm_gbs"],
                              "frac_of_spec_8tbs": step_bytes(B) / (msB * 1e-3) / 1e9 / SPEC_HBM_GBS}
        del gB

    # ---- fused LM head + argmax, batch 1 and 5
    Nv, Kv = 152064, 3584
    Wlm = torch.from_numpy(synth.q4k_weights(Nv, Kv, (3, 0))).to(dev)
    xlm = torch.from_numpy(synth.normal_f32((5, Kv), (3, 2))).to(dev)
    idx = torch.empty(5, dtype=torch.int32, device=dev)
    lm = {}
    for B in (1, 5):
        g = capture(lambda B=B: q4k.gemv_argmax(Wlm, xlm[:B], idx[:B], stream=stream))
        ms = time_graph(g, max(20, args.steps // 2), args.warmup)
        b = Nv * (Kv // 256) * 144 + 4 * B * Kv + 4 * B
        lm[f"batch{B}"] = {"us": ms * 1e3, "gbs": b / (ms * 1e-3) / 1e9, "frac_of_peak": b / (ms * 1e-3) / 1e9 / pk["hbm_gbs"],
                           "frac_of_spec_8tbs": b / (ms * 1e-3) / 1e9 / SPEC_HBM_GBS}
        del g
        # contrast: the plain GEMV writes all logits, then a separate argmax pass (torch) reads them back
        ylog = torch.empty((B, Nv), dtype=torch.float32, device=dev)
        g = capture(lambda B=B: (q4k.gemv(Wlm, xlm[:B], ylog, stream=stream), torch.argmax(ylog, dim=1)))
        ms = time_graph(g, max(20, args.steps // 2), args.warmup)
        lm[f"batch{B}"]["gemv_then_separate_argmax_us"] = ms * 1e3
        del g, ylog
    del Wlm

    # ---- Q6_K GEMV at batch 1 (the LM-head and some down-projection matrices of
    # Q4_K_M files): a Qwen2.5-7B-shaped LM head and down projection; weights
    # under 4x L2 are cycled through byte copies
    q6 = {}
    l2b = torch.cuda.get_device_properties(dev).L2_cache_size
    for name6, N6, K6 in (("lm_head", 152064, 3584), ("down", 3584, 18944)):
        W6 = torch.from_numpy(synth.q6k_weights(N6, K6, (8, N6, K6))).to(dev)
        nc6 = max(1, -(-4 * l2b // W6.numel())) if W6.numel() < 4 * l2b else 1
        W6s = [W6] + [W6.clone() for _ in range(nc6 - 1)]
        x6 = torch.from_numpy(synth.normal_f32((1, K6), (8, 1, K6))).to(dev)
        y6 = torch.empty((1, N6), dtype=torch.float32, device=dev)
        g = capture(lambda: [q4k.q6k_gemv(Wq, x6, y6, stream=stream) for Wq in W6s])
        ms = time_graph(g, max(4, args.steps // (4 * nc6)), args.warmup) / nc6
        del g
        # the same matrix in planar form (repacked once, as at model load)
        W6ps = [q4k.q6k_repack_planar(Wq, K6, stream=stream) for Wq in W6s]
        stream.synchronize()
        g = capture(lambda: [q4k.q6k_gemv_planar(Wp, x6, N6, y6, stream=stream) for Wp in W6ps])
        msp = time_graph(g, max(4, args.steps // (4 * nc6)), args.warmup) / nc6
        del g, W6s, W6, W6ps
        b6 = N6 * (K6 // 256) * 210 + 4 * K6 + 4 * N6
        b6p = q4k.q6k_planar_bytes(N6, K6) + 4 * K6 + 4 * N6
        q6[f"{name6}_{N6}x{K6}"] = {
            "us": msp * 1e3, "gbs": b6p / (msp * 1e-3) / 1e9, "frac_of_peak": b6p / (msp * 1e-3) / 1e9 / pk["hbm_gbs"],
            "path": "q6k_gemv_planar (weights repacked once into 16-byte aligned planes)",
            "gguf_form": {"us": ms * 1e3, "gbs": b6 / (ms * 1e-3) / 1e9,
                          "frac_of_peak": b6 / (ms * 1e-3) / 1e9 / pk["hbm_gbs"], "path": "q6k_gemv"},
            "weight_copies": nc6}

    # ---- one 4096 x 4096 GEMV at batch 1.  Its 9.5 MB of weights fit in L2,
    # so the timed launches cycle through byte copies of W totalling 4x the L2
    # size (copy 0 is the seeded matrix the parity test checks); best of the
    # replays and their coefficient of variation.
    N0 = K0 = 4096
    W0 = torch.from_numpy(synth.q4k_weights(N0, K0, (0, 0))).to(dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    ncopy = -(-4 * l2 // W0.numel())
    Wc = [W0] + [W0.clone() for _ in range(ncopy - 1)]
    x0 = torch.from_numpy(synth.normal_f32((1, K0), (0, 1))).to(dev)
    y0 = torch.empty((1, N0), dtype=torch.float32, device=dev)
    g0 = capture(lambda: [q4k.gemv(W, x0, y0, stream=stream, pdl=True) for W in Wc])
    per = []
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            g0.replay()
        for _ in range(max(8, -(-200 // ncopy))):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g0.replay()
            e1.record(stream)
            e1.synchronize()
            per.append(e0.elapsed_time(e1) / ncopy)
    del g0, Wc, W0
    b0 = N0 * (K0 // 256) * 144 + 4 * K0 + 4 * N0
    best, mean = min(per), float(np.mean(per))
    single = {"shape": "4096x4096", "batch": 1, "us_best": best * 1e3, "us_mean": mean * 1e3,
              "cv": float(np.std(per) / mean), "gbs_best": b0 / (best * 1e-3) / 1e9,
              "frac_of_peak": b0 / (best * 1e-3) / 1e9 / pk["hbm_gbs"],
              "frac_of_spec_8tbs": b0 / (best * 1e-3) / 1e9 / SPEC_HBM_GBS,
              "weight_copies": ncopy, "launches_timed": len(per) * ncopy,
              "l2": f"{ncopy} distinct copies of W ({ncopy * N0 * (K0 // 256) * 144 / 1e6:.0f} MB) cycled, 4x L2"}

    # ---- end to end through the public API with host buffers (batch 1): every
    # step copies all of its activations in from pinned host memory and all of
    # its outputs back out.  The copies run on a second stream beside the
    # launches: layer 0's inputs first, the other layers' inputs while layer 0
    # runs, and each group of layers' outputs while later layers run; only the
    # last group's outputs follow the last launch.  Copies and launches are
    # one graph.
    # The host buffers are page-locked with cudaHostRegister rather than taken
    # from torch's pinned-memory cache, whose copy bookkeeping records events
    # that a graph capture cannot hold.
    nx1, ny1 = x_elems_per_row, y_elems_per_row
    host_arrays = [np.empty(nx1, dtype=np.float32), np.empty(ny1, dtype=np.float32)]
    h_x, h_y = (torch.from_numpy(a) for a in host_arrays)
    for t in (h_x, h_y):
        torch.cuda.check_error(torch.cuda.cudart().cudaHostRegister(t.data_ptr(), t.numel() * 4, 0))
    h_x.copy_(x_flat[:nx1].cpu())
    h2d, d2h = nx1 * 4, ny1 * 4
    copy_stream = torch.cuda.Stream(device=dev)
    out_groups = [(0, 4), (4, 8), (8, 12), (12, 16), (16, 20), (20, 24), (24, 27), (27, LAYERS)]

    def e2e_hook(layer, when):
        if when == "pre" and layer == 1:
            stream.wait_stream(copy_stream)          # inputs of layers 1.. are in
        if when != "post":
            return
        for lo, hi in out_groups:
            if layer + 1 != hi:
                continue
            a, b = lo * y_per_layer, hi * y_per_layer
            if hi == LAYERS:                          # the last group: in order
                h_y[a:b].copy_(y_flat[a:b], non_blocking=True)
            else:
                copy_stream.wait_stream(stream)
                with torch.cuda.stream(copy_stream):
                    h_y[a:b].copy_(y_flat[a:b], non_blocking=True)

    def e2e_step():
        copy_stream.wait_stream(stream)
        x_flat[:x_per_layer].copy_(h_x[:x_per_layer], non_blocking=True)
        with torch.cuda.stream(copy_stream):
            x_flat[x_per_layer:nx1].copy_(h_x[x_per_layer:], non_blocking=True)
        decode_step(1, hook=e2e_hook)
        stream.wait_stream(copy_stream)

    g_e2e = capture(e2e_step)
    y_flat[:ny1].fill_(float("nan"))
    h_y.fill_(float("nan"))
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            g_e2e.replay()
        stream.synchronize()
        e2e_copies_exact = bool(torch.equal(h_y, y_flat[:ny1].cpu()))
        barrier()
        t0 = time.perf_counter()
        e2e_steps = max(10, args.steps // 4)
        for _ in range(e2e_steps):
            g_e2e.replay()
        stream.synchronize()
        e2e_ms = max_over_ranks((time.perf_counter() - t0) * 1e3 / e2e_steps, device=dev)
    del g_e2e
    stream.synchronize()
    for t in (h_x, h_y):
        torch.cuda.check_error(torch.cuda.cudart().cudaHostUnregister(t.data_ptr()))
    if not e2e_copies_exact:
        raise RuntimeError("end-to-end step: the outputs copied to the host differ from the device outputs")
    e2e_val = whole_job_rate(bytes1, world, e2e_ms * 1e-3) / 1e9

    # ---- roofline of the dominant kernel (the batch-1 GEMV; the step is only its launches)
    launches_per_step = LAYERS * 4
    achieved = bytes1 / (ms1 * 1e-3) / 1e9
    tr = recorded_traffic()
    traffic = None
    if tr is not None:
        traffic = tr["dram_bytes_per_weight_byte"] * bytes1 / launches_per_step
    roof = {"kernel": "q4k_gemv_kernel<1,false,1> (batch 1, integer dp4a inner product)", "bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"],
            "unit": "GB/s", "frac": achieved / pk["hbm_gbs"], "traffic": traffic,
            "algorithmic_bytes_per_launch": bytes1 / launches_per_step,
            "avg_launch_us": ms1 * 1e3 / launches_per_step,
            "peak_source": pk["source"] + " (hbm copy bandwidth)"}

    # ---- prefill tiles (Llama-3-8B shapes)
    prefill = {}
    try:
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        for name, N, K in synth.llama3_8b_prefill_shapes():
            Wp = torch.from_numpy(synth.q4k_weights(N, K, (4, N, K))).to(dev)
            # weights smaller than 4x L2 are cycled through byte copies so that
            # every launch reads them from HBM
            ncopy = max(1, -(-4 * l2 // Wp.numel())) if Wp.numel() < l2 else 1
            Wps = [Wp] + [Wp.clone() for _ in range(ncopy - 1)]
            # (T = 32 also through q4k_gemm_prefill_exact, the no-weight-rounding entry point)
            for T, exact in ((32, False), (32, True), (512, False)):
                Xb = torch.from_numpy(synth.normal_bf16_bits((T, K), (4, T, K)).view(np.int16)).to(dev).view(torch.bfloat16)
                Yp = torch.empty((T, N), dtype=torch.float32, device=dev)
                g = capture(lambda: [q4k.gemm_prefill(Wq, Xb, Yp, stream=stream, exact=exact) for Wq in Wps])
                ms = time_graph(g, max(4, args.steps // (4 * ncopy)), args.warmup) / ncopy
                flops = 2.0 * N * K * T
                byts = N * (K // 256) * 144 + 2 * T * K + 4 * T * N
                ideal_s = max(byts / (pk["hbm_gbs"] * 1e9), flops / (pk["bf16_tflops"] * 1e12))
                prefill[f"{name}_{N}x{K}_T{T}" + ("_exact" if exact else "")] = {
                    "us": ms * 1e3, "tflops": flops / (ms * 1e-3) / 1e12, "gbs": byts / (ms * 1e-3) / 1e9,
                    "frac_tensor": flops / (ms * 1e-3) / 1e12 / pk["bf16_tflops"],
                    "frac_hbm": byts / (ms * 1e-3) / 1e9 / pk["hbm_gbs"],
                    "frac_roofline": ideal_s / (ms * 1e-3),
                    "weight_copies": ncopy}
                del g
            del Wp, Wps
    except Exception as e:  # prefill not available yet
        prefill = {"unavailable": str(e).splitlines()[0][:200]}

    ck = clocks.stop()

    out = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms1, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None,
        "dtype": "q4_k u4 weights x int8 hi+lo parts of x (dp4a, int32 per sub-block), fp32 scales and sums",
        "data": "synthetic",
        "arithmetic": "batch 1: x as two int8 parts per super-block, dp4a with the 4-bit weights into int32 "
                      "per sub-block, scales and accumulation in fp32; batch >= 2: fp16 hi+lo x and exact fp16 "
                      "weights on mma.sync, fp32 accumulation",
        "config": {"workload": "qwen2.5-7b-shaped decode: 28 layers x 7 Q4_K GEMVs (q,k,v,o 3584x3584/512x3584, "
                               "gate/up 18944x3584, down 3584x18944), batch 1",
                   "batch": 1, "layers": LAYERS, "weight_bytes_per_step": LAYERS * sum(N * (K // 256) * 144 for _, N, K in shapes),
                   "algorithmic_bytes_per_step": bytes1, "cuda_graph": True, "pdl": True,
                   "fused_dispatch": "q/k/v in one launch, gate/up in one launch (4 launches per layer)",
                   "l2": "inputs larger than L2 (3.67 GB of weights streamed per step)",
                   "parallelism": f"replicas x{world}"},
        "frac_of_peak": value / world / pk["hbm_gbs"],
        "frac_of_spec_8tbs": value / world / SPEC_HBM_GBS,
        "frac_of_read_probe": value / world / read_probe["gbs"],
        "read_probe": read_probe,
        "us_per_layer": ms1 * 1e3 / LAYERS,
        "tok_per_s_equiv": 1e3 / ms1,
        "per_kind_us": kinds_us,
        "unfused_one_launch_per_matrix": unfused,
        "batch1_tensor_core_path": tensor_core_b1,
        "batch1_q8k_activations": q8k_b1,
        "single_gemv_4096": single,
        "q6k_gemv_batch1": q6,
        "prefill": prefill,
        "roofline": roof,
        "e2e": {"value": e2e_val, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms, "path": "pinned H2D of all step activations and D2H of all outputs on a second stream overlapped with the 112 launches (layer 0 inputs first, outputs in 8 layer groups, the last one layer), one graph per step"},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": ck,
        "peaks": pk,
    }
    if rank == 0:
        cb = oracle_sample(args.cpu_seconds)
        if not args.skip_cpu_configs:
            cb["configs"] = oracle_configs()
        out["cpu_baseline"] = cb
        # the metric's three figures, last in the line: batch-1 and batch-5
        # decode GB/s with their fractions of the peak, and the LM head + argmax
        b5 = sweep["batch5"]
        out["verify_batch"] = sweep
        out["lm_head_argmax"] = lm
        out["metric_figures"] = {
            "batch1_gbs": value / world, "batch1_frac_of_peak": value / world / pk["hbm_gbs"],
            "batch1_ms_per_step": ms1,
            "batch5_gbs": b5["gbs"], "batch5_frac_of_peak": b5["frac_of_peak"], "batch5_ms_per_step": b5["us_per_step"] / 1e3,
            "lm_head_argmax_us_batch1": lm["batch1"]["us"], "lm_head_argmax_us_batch5": lm["batch5"]["us"]}
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_profile_case(spec: str, iters: int):
    """One op repeated `iters` times on seeded inputs, for ncu captures.
    spec = gemv:N:K:B | argmax:N:K:B | prefill:N:K:T | q6k:N:K:B | q6kp:N:K:B"""
    import numpy as np
    import torch

    import __graft_entry__
    import q4_dequant_gemv_gb300 as q4k
    import synth
    __graft_entry__.build()
    if spec.startswith("decode"):
        # decode:L:B -- L Qwen2.5-7B-shaped layers (7 GEMVs each), eager launches
        _, L, B = spec.split(":")
        L, B = int(L), int(B)
        layers = [[(N, K, torch.from_numpy(W).cuda()) for _, N, K, W in synth.qwen_layer_weights(l)] for l in range(L)]
        xs = {K: torch.from_numpy(synth.normal_f32((B, K), (9, K))).cuda() for K in (3584, 18944)}
        ys = [[torch.empty((B, N), device="cuda") for N, _, _ in lw] for lw in layers]
        for _ in range(iters):
            for lw, yl in zip(layers, ys):
                for (N, K, W), y in zip(lw, yl):
                    q4k.gemv(W, xs[K], y, pdl=True)
        torch.cuda.synchronize()
        print(f"profile case {spec} x{iters} done")
        return
    kind, N, K, B = spec.split(":")
    N, K, B = int(N), int(K), int(B)
    if kind == "q6k":
        # q6k:N:K:B -- the Q6_K GEMV
        W6 = torch.from_numpy(synth.q6k_weights(N, K, (9, N, K))).cuda()
        x = torch.from_numpy(synth.normal_f32((B, K), (9, B))).cuda()
        y = torch.empty((B, N), dtype=torch.float32, device="cuda")
        for _ in range(iters):
            q4k.q6k_gemv(W6, x, y)
        torch.cuda.synchronize()
        print(f"profile case {spec} x{iters} done")
        return
    if kind == "q6kp":
        # q6kp:N:K:B -- the Q6_K GEMV on the planar form
        W6 = torch.from_numpy(synth.q6k_weights(N, K, (9, N, K))).cuda()
        Wp = q4k.q6k_repack_planar(W6, K)
        del W6
        x = torch.from_numpy(synth.normal_f32((B, K), (9, B))).cuda()
        y = torch.empty((B, N), dtype=torch.float32, device="cuda")
        for _ in range(iters):
            q4k.q6k_gemv_planar(Wp, x, N, y)
        torch.cuda.synchronize()
        print(f"profile case {spec} x{iters} done")
        return
    W = torch.from_numpy(synth.q4k_weights(N, K, (9, N, K))).cuda()
    if kind == "prefill":
        X = torch.from_numpy(synth.normal_bf16_bits((B, K), (9, B)).view(np.int16)).cuda().view(torch.bfloat16)
        Y = torch.empty((B, N), dtype=torch.float32, device="cuda")
        for _ in range(iters):
            q4k.gemm_prefill(W, X, Y)
    else:
        x = torch.from_numpy(synth.normal_f32((B, K), (9, B))).cuda()
        if kind == "gemv":
            y = torch.empty((B, N), dtype=torch.float32, device="cuda")
            for _ in range(iters):
                q4k.gemv(W, x, y)
        else:
            idx = torch.empty(B, dtype=torch.int32, device="cuda")
            for _ in range(iters):
                q4k.gemv_argmax(W, x, idx)
    torch.cuda.synchronize()
    print(f"profile case {spec} x{iters} done")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=8.0)
    ap.add_argument("--skip-cpu-configs", action="store_true", help="time the oracle on the headline sample only")
    ap.add_argument("--profile-case", default=None, help="gemv:N:K:B | argmax:N:K:B | prefill:N:K:T | q6k:N:K:B | q6kp:N:K:B | decode:L:B (ncu helper)")
    ap.add_argument("--iters", type=int, default=3)
    args = ap.parse_args()
    if args.profile_case:
        run_profile_case(args.profile_case, args.iters)
        return
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
