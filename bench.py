"""Benchmark of the Q4_K decode hot path on GB300.

Headline (the JSON line's `value`): weight-streaming throughput in GB/s of one
decode step of a Qwen2.5-7B-shaped model -- 28 layers x 7 Q4_K GEMVs (q, k, v,
o, gate, up, down), batch 1 -- with all inputs resident in HBM, the 196
launches replayed from a CUDA graph.  Algorithmic bytes per step = the Q4_K
weights (4.5 bits/weight) + fp32 activations read + fp32 outputs written.

The same line carries the batch-2/5/9 VerifyBatch sweep, the fused LM-head +
argmax latency (152064 x 3584, batch 1 and 5), the prefill tiles, the roofline
of the dominant kernel, an end-to-end figure through the public API with host
buffers, clocks sampled during the timed regions, and the CPU oracle timed on
the host cores.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

`--impl reference` times the CPU oracle (the reference arm of this build) on a
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
    return {"value": wbytes * reps / dt / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"layer 0 of the Qwen2.5-7B-shaped decode (7 Q4_K GEMVs, {wbytes} weight bytes), batch 1, "
                      f"{reps} passes in {dt:.1f} s, fp64 accumulation, OpenMP over rows"}


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
    h = hashlib.sha256()
    for f in ("q4k_gemv.cu", "ptx.cuh"):
        h.update(open(os.path.join(ROOT, "q4_dequant_gemv_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic():
    """DRAM bytes per weight byte from a committed ncu capture of the current kernel source."""
    p = os.path.join(ROOT, "profiles", "gemv_traffic.json")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p))
    except Exception:
        return None
    if d.get("source_hash") != kernel_source_hash():
        return None
    return d


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
    xs_by_layer = []
    for layer in range(LAYERS):
        # distinct activations per consumer: q/k/v share one, gate/up share one (as in a decoder layer)
        xa = synth.normal_f32((16, 3584), (layer, 50))
        xo = synth.normal_f32((16, 3584), (layer, 51))
        xm = synth.normal_f32((16, 3584), (layer, 52))
        xd = synth.normal_f32((16, 18944), (layer, 53))
        xs_by_layer.append({"attn": torch.from_numpy(xa).to(dev), "o": torch.from_numpy(xo).to(dev),
                            "mlp": torch.from_numpy(xm).to(dev), "down": torch.from_numpy(xd).to(dev)})
    src = {"q": "attn", "k": "attn", "v": "attn", "o": "o", "gate": "mlp", "up": "mlp", "down": "down"}
    ys = [[torch.empty((16, N), dtype=torch.float32, device=dev) for _, N, _ in shapes] for _ in range(LAYERS)]
    stream = torch.cuda.Stream(device=dev)

    def step_bytes(B):
        return LAYERS * sum(N * (K // 256) * 144 + 4 * B * K + 4 * B * N for _, N, K in shapes)

    def decode_step(B, pdl=True):
        for layer in range(LAYERS):
            for mi, (name, N, K) in enumerate(shapes):
                x = xs_by_layer[layer][src[name]][:B]
                q4k.gemv(Ws[layer][mi], x, ys[layer][mi][:B], stream=stream, pdl=pdl)

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
        ms = e0.elapsed_time(e1)
        if world > 1:
            import torch.distributed as dist
            t = torch.tensor([ms], device=dev)
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            ms = float(t.item())
        return ms / steps

    clocks = ClockSampler(local)
    clocks.start()

    # ---- headline: batch 1
    g1 = capture(lambda: decode_step(1))
    ms1 = time_graph(g1, args.steps, args.warmup)
    bytes1 = step_bytes(1)
    value = bytes1 / (ms1 * 1e-3) / 1e9 * world

    # ---- VerifyBatch sweep (same weights)
    sweep = {}
    for B in (2, 5, 9):
        gB = capture(lambda B=B: decode_step(B))
        msB = time_graph(gB, max(10, args.steps // 4), args.warmup)
        sweep[f"batch{B}"] = {"gbs": step_bytes(B) / (msB * 1e-3) / 1e9, "us_per_step": msB * 1e3,
                              "us_per_layer": msB * 1e3 / LAYERS,
                              "frac_of_peak": step_bytes(B) / (msB * 1e-3) / 1e9 / pk["hbm_gbs"]}
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
        lm[f"batch{B}"] = {"us": ms * 1e3, "gbs": b / (ms * 1e-3) / 1e9, "frac_of_peak": b / (ms * 1e-3) / 1e9 / pk["hbm_gbs"]}
        del g
    del Wlm

    # ---- prefill tiles (Llama-3-8B shapes)
    prefill = {}
    try:
        for name, N, K in synth.llama3_8b_prefill_shapes():
            Wp = torch.from_numpy(synth.q4k_weights(N, K, (4, N, K))).to(dev)
            for T in (32, 512):
                Xb = torch.from_numpy(synth.normal_bf16_bits((T, K), (4, T, K)).view(np.int16)).to(dev).view(torch.bfloat16)
                Yp = torch.empty((T, N), dtype=torch.float32, device=dev)
                g = capture(lambda: q4k.gemm_prefill(Wp, Xb, Yp, stream=stream))
                ms = time_graph(g, max(20, args.steps // 4), args.warmup)
                flops = 2.0 * N * K * T
                byts = N * (K // 256) * 144 + 2 * T * K + 4 * T * N
                prefill[f"{name}_{N}x{K}_T{T}"] = {
                    "us": ms * 1e3, "tflops": flops / (ms * 1e-3) / 1e12, "gbs": byts / (ms * 1e-3) / 1e9,
                    "frac_tensor": flops / (ms * 1e-3) / 1e12 / pk["bf16_tflops"],
                    "frac_hbm": byts / (ms * 1e-3) / 1e9 / pk["hbm_gbs"]}
                del g
            del Wp
    except Exception as e:  # prefill not available yet
        prefill = {"unavailable": str(e).splitlines()[0][:200]}

    ck = clocks.stop()

    # ---- end to end through the public API with host buffers (batch 1)
    h_in = {k: [xs_by_layer[l][k][:1].cpu().pin_memory() for l in range(LAYERS)] for k in ("attn", "o", "mlp", "down")}
    h_out = [[torch.empty((1, N), dtype=torch.float32).pin_memory() for _, N, _ in shapes] for _ in range(LAYERS)]
    h2d = sum(t.numel() * 4 for v in h_in.values() for t in v)
    d2h = sum(t.numel() * 4 for row in h_out for t in row)

    def e2e_step():
        for k, lst in h_in.items():
            for l in range(LAYERS):
                xs_by_layer[l][k][:1].copy_(lst[l], non_blocking=True)
        g1.replay()
        for l in range(LAYERS):
            for mi in range(len(shapes)):
                h_out[l][mi].copy_(ys[l][mi][:1], non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            e2e_step()
        stream.synchronize()
        barrier()
        t0 = time.perf_counter()
        e2e_steps = max(10, args.steps // 4)
        for _ in range(e2e_steps):
            e2e_step()
        stream.synchronize()
        e2e_ms = (time.perf_counter() - t0) * 1e3 / e2e_steps
    e2e_val = bytes1 / (e2e_ms * 1e-3) / 1e9 * world

    # ---- roofline of the dominant kernel (the batch-1 GEMV; the step is only its launches)
    launches_per_step = LAYERS * len(shapes)
    achieved = bytes1 / (ms1 * 1e-3) / 1e9
    tr = recorded_traffic()
    traffic = None
    if tr is not None:
        traffic = tr["dram_bytes_per_weight_byte"] * bytes1 / launches_per_step
    roof = {"kernel": "q4k_gemv_kernel<1,false>", "bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"],
            "unit": "GB/s", "frac": achieved / pk["hbm_gbs"], "traffic": traffic,
            "algorithmic_bytes_per_launch": bytes1 / launches_per_step,
            "avg_launch_us": ms1 * 1e3 / launches_per_step,
            "peak_source": pk["source"] + " (hbm copy bandwidth)"}

    out = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms1, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": "qwen2.5-7b-shaped decode: 28 layers x 7 Q4_K GEMVs (q,k,v,o 3584x3584/512x3584, "
                               "gate/up 18944x3584, down 3584x18944), batch 1",
                   "batch": 1, "layers": LAYERS, "weight_bytes_per_step": LAYERS * sum(N * (K // 256) * 144 for _, N, K in shapes),
                   "algorithmic_bytes_per_step": bytes1, "cuda_graph": True, "pdl": True,
                   "l2": "inputs larger than L2 (3.67 GB of weights streamed per step)",
                   "parallelism": f"replicas x{world}"},
        "frac_of_peak": value / world / pk["hbm_gbs"],
        "us_per_layer": ms1 * 1e3 / LAYERS,
        "tok_per_s_equiv": 1e3 / ms1,
        "verify_batch": sweep,
        "lm_head_argmax": lm,
        "prefill": prefill,
        "roofline": roof,
        "e2e": {"value": e2e_val, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms, "path": "pinned host x -> H2D, graph of 196 q4k_gemv calls, D2H of all y"},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": ck,
        "peaks": pk,
    }
    if rank == 0:
        out["cpu_baseline"] = oracle_sample(args.cpu_seconds) if world == 1 or rank == 0 else None
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=8.0)
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
