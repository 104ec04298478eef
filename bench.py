"""Benchmark of the W4A16 MoE block on GB300 (one JSON line on stdout).

Default workload: the 40-layer stack of Qwen3.6-35B-A3B-shaped MoE layers
(H=2048, I=512, 256 routed experts, top-8, one shared expert, 4-bit weights
in groups of 64 with bf16 scale and bias) on a T=4096 prefill chunk with
Zipf-skewed routing; ~18.2 GB of packed weights resident in HBM. One step is
one pass of the whole stack: per layer, router + top-k, histogram/scan/block
map, scatter, gather, grouped gate/up GEMM with SwiGLU, grouped down GEMM,
combine, and the stack update x <- bf16(x + moe(rmsnorm(x))/sqrt(40)) (the
RMS-normalised stream is each layer's input).

value: tokens/s over the timed steps (inputs resident in HBM; the packed
weights, 18 GB, are far larger than L2, so every step streams them from HBM).
e2e: the same through the C ABI with x copied in from pinned host memory and
the result copied back, inside the timed region.
roofline: the dominant kernel (grouped gate/up GEMM) against the measured
dense bf16 peak (burst, or the sustained figure when the clock record of the
timed region shows the power cap); the down GEMM's figures beside it.
cpu_baseline: the fp64 oracle on a bounded sample.
decode: the same stack on decode-sized batches T = 1, 4, 8 (1000 graph-replayed
steps each by default), HBM roofline as for --workload decode_t*_l40.

--workload decode_t{1,4,8}_l40: the same 40-layer stack on a decode batch of
T tokens through the small-M path. Every step copies a fresh batch from a
pool of 64 pre-generated device batches and replays the 40-layer step from
a CUDA graph; the roofline is HBM bandwidth over the packed bytes of the
experts each layer's routing selects (counted from the routing itself).

--tokens N --chunk C: a prompt of N tokens through the stack in chunks of at
most C tokens (the plan's capacity; moe_forward_stack runs each chunk through
all layers), e.g. the long-prompt sweep of the chunked-prefill summary.

--impl reference times the oracle (the CPU reference of this build) on the
same workload, a bounded sample per step.
Multi-GPU: independent replicas (the block does not shard), one per rank.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-block prefill tokens/s (W4A16, 1 GB300) + % of tensor/HBM roofline"
METRIC_DECODE = "MoE-block decode tokens/s (W4A16, 1 GB300) + % of HBM roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
PROFILE_GATEUP = os.path.join(ROOT, "profiles", "w4_grouped_gemm_tc_gateup_t4096.txt")
GEMM_SRC = os.path.join(ROOT, "bit_grouped_gemm_gb300", "csrc", "gemm_tc.cu")


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="prefill_t4096_l40_zipf")
    ap.add_argument("--layers", type=int, default=0, help="override the layer count (profiling)")
    ap.add_argument("--tokens", type=int, default=0,
                    help="override the prompt length of a prefill workload")
    ap.add_argument("--chunk", type=int, default=0,
                    help="chunked prefill: plan capacity (tokens per chunk); default: the "
                         "whole prompt in one chunk")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-decode", action="store_true",
                    help="skip the decode-sized batches (T = 1, 4, 8) of the default line")
    ap.add_argument("--decode-steps", type=int, default=1000,
                    help="graph-replayed steps per decode batch size")
    return ap.parse_args(argv)


# ----------------------------------------------------------------- helpers


def dist_info():
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def cpu_model():
    """Host CPU model name (x86 /proc/cpuinfo 'model name', else lscpu's
    'Model name' as on Arm), or None."""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return None


def tensor_peak(peaks, src, clocks):
    """The dense bf16 peak a tensor-bound kernel of this run is measured
    against: the burst figure, unless the clock record of the timed region
    shows the power cap or SM clocks below 90% of their maximum, in which
    case the sustained (power-capped) figure."""
    burst = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    sustained = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    capped = False
    if clocks and clocks.get("sm_mhz") and clocks.get("sm_max_mhz"):
        capped = ("sw_power_cap" in clocks.get("reasons", [])
                  or clocks["sm_mhz"] < 0.9 * clocks["sm_max_mhz"])
    if capped:
        return sustained, f"{src} bf16_tflops_sustained (of {src}): power cap or low SM clock seen"
    return burst, f"{src} bf16_tflops, burst (of {src}): SM clock at maximum, no power cap seen"


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def source_hash(path):
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def profiled_traffic(profile_path, kernel_src):
    """DRAM bytes per launch from a committed ncu summary, or None when the
    kernel source changed since the capture (keys 'source_sha256_16' and
    'dram_bytes_per_launch' in the summary)."""
    try:
        kv = {}
        with open(profile_path) as f:
            for line in f:
                if ":" in line:
                    k, v = line.split(":", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("source_sha256_16") != source_hash(kernel_src):
            return None
        return float(kv["dram_bytes_per_launch"])
    except Exception:
        return None


def max_over_ranks(v, pg):
    """The largest of every rank's v (the job is as slow as its slowest
    replica); v itself on a single process."""
    if pg is None:
        return v
    import torch
    dev = "cuda" if pg.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(v)], device=dev)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def replica_value(world_size, tokens, steps, ms):
    """Whole-job tokens/s of `world_size` replicas, each pushing `tokens`
    tokens through `steps` steps, timed by the slowest rank (`ms`)."""
    return world_size * tokens * steps / (ms / 1e3)


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.4)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) >= 9:
                        rows.append(parts)
        except Exception:
            return None
        if not rows:
            return None

        def num(s):
            try:
                return float(s)
            except ValueError:
                return None
        sm = sorted(v for v in (num(r[1]) for r in rows) if v is not None)
        mx = [v for v in (num(r[2]) for r in rows) if v is not None]
        reasons = sorted({self.REASONS[i] for r in rows for i in range(4)
                          if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": sm[len(sm) // 2] if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ------------------------------------------------------------- the oracle


def oracle_sample_rate(w, layers_dev, threads, sample_tokens, sample_layers, min_seconds=0.0):
    """Oracle tokens/s of the whole stack, from `sample_tokens` rows through
    `sample_layers` layers (or, with min_seconds, through layers 0, 1, ...
    until that much CPU time has been spent, at most sample_layers), scaled by
    the layers done / layers. Returns (rate, seconds, layers done)."""
    import oracle
    from bit_grouped_gemm_gb300 import synth
    from tests import parity
    sh = w.shape
    xb = parity.bits(synth.tokens_x(w, "cpu")[:sample_tokens])
    orc = oracle.get()
    elapsed = 0.0
    done = 0
    for li in range(sample_layers):
        if min_seconds and done and elapsed >= min_seconds:
            break
        L = layers_dev[li]
        wr = parity.bits(L.router_w)
        rb = None if L.router_bias is None else L.router_bias.cpu().numpy()
        routed = parity.host_set(L.routed)
        shared = parity.host_set(L.shared) if L.shared is not None else None
        t0 = time.perf_counter()
        xn = orc.rmsnorm(xb)
        out = orc.moe_rows(xn, wr, rb, routed, shared, sh.top_k, sh.group_size,
                           nthreads=threads)
        xb = orc.residual(xb, out["y"], 1.0 / math.sqrt(w.layers))
        elapsed += time.perf_counter() - t0
        done += 1
    return sample_tokens * done / elapsed / w.layers, elapsed, done


def workload(args):
    from bit_grouped_gemm_gb300 import synth
    w = synth.standard_workloads()[args.workload]
    if args.layers:
        w = dataclasses.replace(w, layers=args.layers)
    if args.tokens and w.tokens > 16:
        w = dataclasses.replace(w, tokens=args.tokens,
                                name=w.name.replace(f"t{w.tokens}_", f"t{args.tokens}_"))
    return w


# ------------------------------------------------------------------- main


def main(argv=None):
    args = parse_args(argv)
    ws, rank, local = dist_info()
    if args.impl == "reference":
        return run_reference(args, ws, rank)
    import torch
    from bit_grouped_gemm_gb300 import binding as bg
    from bit_grouped_gemm_gb300 import build, stack

    torch.cuda.set_device(local)
    pg = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        pg = dist
    build.build()
    bg.load_library()

    w = workload(args)
    if w.tokens <= 16:
        return run_decode(args, w, ws, rank, local, pg)
    sh = w.shape
    T = w.tokens
    from bit_grouped_gemm_gb300 import synth
    layers = stack.make_layers(w, "cuda")
    weight_bytes = sum(L.nbytes() for L in layers)
    alpha = stack.residual_alpha(w.layers)
    chunk = min(T, args.chunk) if args.chunk > 0 else T
    plan = bg.moe_plan_create(bg.plan_desc(sh.hidden, sh.inter, sh.num_experts, sh.top_k,
                                           sh.group_size, int(sh.has_shared), chunk), local)
    stream = torch.cuda.current_stream()
    x0 = synth.tokens_x(w, "cuda")
    x = x0.clone()
    xn = torch.empty((chunk, sh.hidden), dtype=x.dtype, device="cuda")
    layer_arr = bg.moe_layers(layers)

    # one step: the whole stack through the native driver (chunks of `chunk`
    # tokens, each through all layers)
    def step():
        x.copy_(x0)
        bg.moe_forward_stack(plan, x, xn, T, layer_arr, alpha)

    for _ in range(max(args.warmup, 0)):
        step()
    torch.cuda.synchronize()
    assert bg.moe_get_error(plan) == 0

    # --- timed region: inputs resident in HBM, no instrumentation
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize()
    if pg:
        pg.barrier()
    ms = max_over_ranks(ev0.elapsed_time(ev1), pg)
    assert bg.moe_get_error(plan) == 0
    ms_per_step = ms / args.steps
    value = replica_value(ws, T, args.steps, ms)

    # --- the same steps again with CUDA events around every kernel launch
    # (library timing mode, events on the launching stream): the per-kernel
    # breakdown and the roofline of the dominant kernel come from here
    bg.moe_enable_timing(plan, True)
    bg.moe_read_timing(plan)
    torch.cuda.synchronize()
    for _ in range(args.steps):
        step()
    torch.cuda.synchronize()
    kt = bg.moe_read_timing(plan)
    bg.moe_enable_timing(plan, False)
    assert bg.moe_get_error(plan) == 0

    # --- end to end: pinned host x in, result out, through the public C ABI
    e2e = None
    if not args.no_e2e:
        xh = x0.cpu().pin_memory()
        out_h = torch.empty_like(xh).pin_memory()

        def e2e_step():
            x.copy_(xh, non_blocking=True)
            bg.moe_forward_stack(plan, x, xn, T, layer_arr, alpha)
            out_h.copy_(x, non_blocking=True)
        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        if pg:
            pg.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        ems = max_over_ranks(e0.elapsed_time(e1), pg)
        e2e = {"value": replica_value(ws, T, args.steps, ems), "unit": "tokens/s",
               "h2d_bytes_per_step": xh.numel() * xh.element_size(),
               "d2h_bytes_per_step": out_h.numel() * out_h.element_size()}

    # --- roofline of the dominant kernel (grouped gate/up GEMM + SwiGLU)
    peaks, peak_src = load_peaks()
    clocks = clk.summary()
    n_pairs = T * (sh.top_k + int(sh.has_shared))
    gu_ms, gu_n = kt["gate_up_gemm"]
    dn_ms, dn_n = kt["down_gemm"]
    # per launch: one layer of one chunk (the average over the step's launches)
    flops_gateup = 4.0 * sh.hidden * sh.inter * n_pairs * w.layers * args.steps / max(gu_n, 1)
    flops_down = 2.0 * sh.hidden * sh.inter * n_pairs * w.layers * args.steps / max(dn_n, 1)
    achieved = flops_gateup / (gu_ms / gu_n / 1e3) / 1e12 if gu_n else None
    achieved_dn = flops_down / (dn_ms / dn_n / 1e3) / 1e12 if dn_n else None
    peak, peak_note = tensor_peak(peaks, peak_src, clocks)
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": (achieved / peak) if achieved else None,
                "traffic": profiled_traffic(PROFILE_GATEUP, GEMM_SRC),
                "kernel": "w4_grouped_gemm_tc, gate/up + SwiGLU (one launch per layer)",
                "peak_source": peak_note,
                "algorithmic_flops_per_launch": flops_gateup,
                "down_gemm": {"achieved": achieved_dn,
                              "frac": (achieved_dn / peak) if achieved_dn else None,
                              "algorithmic_flops_per_launch": flops_down}}
    step_flops = w.layers * (n_pairs * 6.0 * sh.hidden * sh.inter +
                             T * 2.0 * sh.hidden * sh.num_experts)
    kernels = {k: {"ms_per_step": v[0] / args.steps, "launches_per_step": v[1] / args.steps}
               for k, v in kt.items()}
    gpu_launches = int(sum(v[1] for v in kt.values()))

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        threads = os.cpu_count() or 1
        # layer after layer until ~12 s of CPU work (the sample stays bounded:
        # 16 tokens per thread, at most the whole stack)
        st = min(T, 16 * threads)
        rate, el, sl = oracle_sample_rate(w, layers, threads, st, w.layers, min_seconds=12.0)
        cpu = {"value": rate, "unit": "tokens/s", "cores": threads, "kind": "oracle",
               "cpu_model": cpu_model(),
               "sample": f"{st} tokens x layers 0-{sl - 1} of the {T}-token {w.layers}-layer "
                         f"stack, fp64 oracle on {threads} threads, {el:.1f} s, "
                         f"scaled by {sl}/{w.layers}"}

    # --- decode-sized batches through the same 40-layer stack (same weights)
    decode = None
    if not args.no_decode and w.layers > 1:
        decode = {}
        for td in (1, 4, 8):
            wd = synth.standard_workloads()[f"decode_t{td}_l40"]
            if wd.layers != w.layers or wd.seed != w.seed:
                wd = dataclasses.replace(wd, layers=w.layers, seed=w.seed)
            r = measure_decode(wd, layers, local, pg, ws, steps=args.decode_steps,
                               warmup=max(args.warmup, 10))
            decode[f"t{td}"] = r

    out = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "precision": "bf16 inputs; fp16 MMA operands (activations converted, weights rebuilt "
                     "as fp16(q*scale+bias)); fp32 accumulation",
        "data": "synthetic",
        "config": {"workload": w.name, "tokens": T, "layers": w.layers, "hidden": sh.hidden,
                   "inter": sh.inter, "experts": sh.num_experts, "top_k": sh.top_k,
                   "shared_experts": int(sh.has_shared), "group_size": sh.group_size,
                   "routing": w.routing + (f"(s={w.zipf_s})" if w.routing == "zipf" else ""),
                   "chunk": chunk,
                   "weights_gb": round(weight_bytes / 1e9, 2),
                   "l2": "inputs larger than L2: every step streams the packed weights "
                         f"({weight_bytes / 1e9:.1f} GB) from HBM",
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"},
        "algorithmic_tflop_per_step": step_flops / 1e12,
        "achieved_tflops_stack": step_flops / (ms_per_step / 1e3) / 1e12,
        "roofline": roofline,
        "kernels": kernels,
        "gpu_launches": gpu_launches,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "clocks": clocks,
        "decode": decode,
    }
    if rank == 0:
        print(json.dumps(out), flush=True)
    bg.moe_plan_destroy(plan)
    if pg:
        pg.destroy_process_group()


def measure_decode(w, layers, local, pg, ws, steps, warmup):
    """Decode-sized batch through the stack: the whole step captured in one
    CUDA graph, replayed `steps` times with a fresh batch copied in from a
    device pool before each replay; HBM roofline over the packed bytes of the
    experts each layer's routing selects. Returns the summary dict."""
    import torch
    from bit_grouped_gemm_gb300 import binding as bg, stack, synth
    sh = w.shape
    T = w.tokens
    alpha = stack.residual_alpha(w.layers)
    plan = bg.moe_plan_create(bg.plan_desc(sh.hidden, sh.inter, sh.num_experts, sh.top_k,
                                           sh.group_size, int(sh.has_shared), T), local)
    try:
        pool = synth.decode_pool(w, 64, "cuda")
        x = torch.empty((T, sh.hidden), dtype=torch.bfloat16, device="cuda")
        xn = torch.empty_like(x)
        arr = bg.moe_layers(layers)
        for i in range(3):
            x.copy_(pool[i])
            bg.moe_forward_stack(plan, x, xn, T, arr, alpha)
        torch.cuda.synchronize()
        assert bg.moe_get_error(plan) == 0
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, capture_error_mode="thread_local"):
            bg.moe_forward_stack(plan, x, xn, T, arr, alpha)
        torch.cuda.synchronize()
        stream = torch.cuda.current_stream()
        for i in range(warmup):
            x.copy_(pool[i % pool.shape[0]], non_blocking=True)
            graph.replay()
        torch.cuda.synchronize()
        if pg:
            pg.barrier()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with ClockSampler(local) as clk:
            ev0.record(stream)
            for i in range(steps):
                x.copy_(pool[i % pool.shape[0]], non_blocking=True)
                graph.replay()
            ev1.record(stream)
            torch.cuda.synchronize()
        if pg:
            pg.barrier()
        ms = max_over_ranks(ev0.elapsed_time(ev1), pg)
        assert bg.moe_get_error(plan) == 0
        step_bytes, experts_per_layer = decode_step_bytes(w, layers, plan, pool)
        peaks, peak_src = load_peaks()
        peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
        ms_per_step = ms / steps
        achieved = step_bytes / (ms_per_step / 1e3) / 1e9
        del graph
        return {"tokens": T, "layers": w.layers, "steps": steps, "warmup": warmup,
                "ms_per_step": ms_per_step,
                "value": replica_value(ws, T, steps, ms), "unit": "tokens/s",
                "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                             "frac": achieved / peak,
                             "peak_source": f"{peak_src} hbm_gbs (of {peak_src})",
                             "algorithmic_bytes_per_step": step_bytes,
                             "distinct_routed_experts_per_layer": experts_per_layer},
                "graph": "whole step (moe_forward_stack) replayed from one CUDA graph; fresh "
                         "batch per step",
                "path": {1: "tensor-core", 2: "small-M", 3: "fused decode layer"}.get(
                    bg.moe_last_gemm_path(plan)),
                "clocks": clk.summary()}
    finally:
        bg.moe_plan_destroy(plan)


def decode_step_bytes(w, layers, plan, pool, samples=8):
    """Algorithmic HBM bytes of one decode step: for every layer, the packed
    weights, scales and biases of each distinct routed expert the layer's
    routing selects plus the shared expert's, and the router weight. Counted
    by running the timed call (moe_forward_stack) one layer at a time
    (untimed) on `samples` pool batches, reading each layer's routing from
    the plan, and averaging."""
    import numpy as np
    import torch
    from bit_grouped_gemm_gb300 import binding as bg, stack
    from tests import parity
    sh = w.shape
    T = w.tokens
    per_expert = 3 * (sh.hidden * sh.inter // 2 + 2 * 2 * sh.hidden * sh.inter // sh.group_size)
    router = sh.hidden * sh.num_experts * 2
    alpha = stack.residual_alpha(w.layers)
    x = torch.empty((T, sh.hidden), dtype=torch.bfloat16, device="cuda")
    xn = torch.empty_like(x)
    x.copy_(pool[0])
    r = bg.moe_route(plan, x, T, layers[0].router_w, layers[0].router_bias)   # array addresses
    idx_view = parity.device_view(r.topk_idx, T * sh.top_k, torch.int32)
    total, experts = 0.0, 0
    for i in range(samples):
        x.copy_(pool[i])
        for L in layers:
            bg.moe_forward_stack(plan, x, xn, T, bg.moe_layers([L]), alpha)
            active = len(np.unique(idx_view.cpu().numpy()))
            experts += active
            total += (active + int(sh.has_shared)) * per_expert + router
    torch.cuda.synchronize()
    return total / samples, experts / samples / w.layers


def run_decode(args, w, ws, rank, local, pg):
    """Decode: the 40-layer step on T <= 16 tokens, replayed from a CUDA graph
    with a fresh batch per step; roofline = HBM bandwidth over the selected
    experts' packed bytes."""
    import torch
    from bit_grouped_gemm_gb300 import binding as bg, stack, synth
    sh = w.shape
    T = w.tokens
    layers = stack.make_layers(w, "cuda")
    alpha = stack.residual_alpha(w.layers)
    plan = bg.moe_plan_create(bg.plan_desc(sh.hidden, sh.inter, sh.num_experts, sh.top_k,
                                           sh.group_size, int(sh.has_shared), T), local)
    pool = synth.decode_pool(w, 64, "cuda")
    x = torch.empty((T, sh.hidden), dtype=torch.bfloat16, device="cuda")
    xn = torch.empty_like(x)
    arr = bg.moe_layers(layers)
    for i in range(3):
        x.copy_(pool[i])
        bg.moe_forward_stack(plan, x, xn, T, arr, alpha)
    torch.cuda.synchronize()
    assert bg.moe_get_error(plan) == 0
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, capture_error_mode="thread_local"):
        bg.moe_forward_stack(plan, x, xn, T, arr, alpha)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()

    def step(i):
        x.copy_(pool[i % pool.shape[0]], non_blocking=True)
        graph.replay()

    for i in range(max(args.warmup, 0)):
        step(i)
    torch.cuda.synchronize()
    if pg:
        pg.barrier()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        ev0.record(stream)
        for i in range(args.steps):
            step(i)
        ev1.record(stream)
        torch.cuda.synchronize()
    if pg:
        pg.barrier()
    ms = max_over_ranks(ev0.elapsed_time(ev1), pg)
    assert bg.moe_get_error(plan) == 0
    ms_per_step = ms / args.steps

    # per-kernel breakdown: the same steps without the graph, library timing on
    bg.moe_enable_timing(plan, True)
    bg.moe_read_timing(plan)
    for i in range(min(args.steps, 50)):
        x.copy_(pool[i % pool.shape[0]])
        bg.moe_forward_stack(plan, x, xn, T, arr, alpha)
    torch.cuda.synchronize()
    kt = bg.moe_read_timing(plan)
    bg.moe_enable_timing(plan, False)
    nk = min(args.steps, 50)
    kernels = {k: {"ms_per_step": v[0] / nk, "launches_per_step": v[1] / nk} for k, v in kt.items()}
    gpu_launches = int(round(sum(v[1] for v in kt.values()) / nk)) * args.steps

    # end to end: x from pinned host memory, result back, around each replay
    e2e = None
    if not args.no_e2e:
        xh = pool[: min(64, pool.shape[0])].cpu().pin_memory()
        out_h = torch.empty((T, sh.hidden), dtype=torch.bfloat16).pin_memory()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(args.steps):
            x.copy_(xh[i % xh.shape[0]], non_blocking=True)
            graph.replay()
            out_h.copy_(x, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        ems = max_over_ranks(e0.elapsed_time(e1), pg)
        e2e = {"value": replica_value(ws, T, args.steps, ems), "unit": "tokens/s",
               "h2d_bytes_per_step": T * sh.hidden * 2, "d2h_bytes_per_step": T * sh.hidden * 2}

    step_bytes, experts_per_layer = decode_step_bytes(w, layers, plan, pool)
    peaks, peak_src = load_peaks()
    peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    achieved = step_bytes / (ms_per_step / 1e3) / 1e9
    out = {
        "metric": METRIC_DECODE, "value": replica_value(ws, T, args.steps, ms), "unit": "tokens/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "precision": "bf16 inputs; fp16 MMA operands; fp32 accumulation",
        "data": "synthetic",
        "config": {"workload": w.name, "tokens": T, "layers": w.layers, "hidden": sh.hidden,
                   "inter": sh.inter, "experts": sh.num_experts, "top_k": sh.top_k,
                   "shared_experts": int(sh.has_shared), "group_size": sh.group_size,
                   "routing": w.routing + (f"(s={w.zipf_s})" if w.routing == "zipf" else ""),
                   "graph": "40-layer step replayed from one CUDA graph",
                   "inputs": "fresh batch per step from a pool of 64 device batches",
                   "l2": "the selected experts' packed bytes per step "
                         f"({step_bytes / 1e9:.2f} GB) exceed L2; weights of 40 layers (18.2 GB) rotate",
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": None,
                     "kernel": "whole 40-layer decode step (one fused launch per layer for T <= 8, "
                               "else routing and small-M grouped GEMMs)",
                     "peak_source": f"{peak_src} hbm_gbs (of {peak_src})",
                     "algorithmic_bytes_per_step": step_bytes,
                     "distinct_routed_experts_per_layer": experts_per_layer},
        "kernels": kernels,
        "gpu_launches": gpu_launches,
        "cpu_baseline": None,
        "e2e": e2e,
        "clocks": clk.summary(),
    }
    if rank == 0:
        print(json.dumps(out), flush=True)
    bg.moe_plan_destroy(plan)
    if pg:
        pg.destroy_process_group()


def run_reference(args, ws, rank):
    """The oracle (this build's CPU reference) on the same workload: each step
    is a bounded sample of tokens through one layer, scaled to the stack."""
    if rank != 0:
        return
    import torch
    from bit_grouped_gemm_gb300 import stack
    w = workload(args)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    L0 = [stack.make_layer(w, 0, dev)]
    threads = os.cpu_count() or 1
    sample = min(w.tokens, 4 * threads)
    for _ in range(max(args.warmup, 0)):
        oracle_sample_rate(w, L0, threads, min(sample, threads), 1)
    tok, secs = 0, 0.0
    for _ in range(args.steps):
        _, el, _ = oracle_sample_rate(w, L0, threads, sample, 1)
        tok += sample
        secs += el
    value = tok / secs / w.layers
    cpu = {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
           "cpu_model": cpu_model(),
           "sample": f"{sample} tokens of layer 0 per step, fp64 oracle on {threads} "
                     f"threads, scaled by 1/{w.layers}"}
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * secs / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "tokens": w.tokens, "layers": w.layers},
        "cpu_baseline": cpu,
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


if __name__ == "__main__":
    main()
