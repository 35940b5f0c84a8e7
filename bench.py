#!/usr/bin/env python
"""Throughput of the DFlash KV-injection draft step on GB300.

A step is one draft round of the batched serving workload (32 sequences,
cached context U[256, 4096], block 16, 2 draft layers, d=4096, 32 query / 8
KV heads of 128, k=5 target layers): one context projection of the 16 new
context rows of every sequence, then per layer a KV inject and a block
attention, then a crop back to the step's starting lengths so that every
step sees the same cache (crop moves no data). The metric is draft blocks
per second per layer = batch * layers / step time.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Under torchrun (N > 1) every rank runs its own replica of the workload (the
path shards by sequence with no exchange) and rank 0 prints one JSON line.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

TRACED = ["attention", "gemm", "combine", "head_epilogue", "rmsnorm", "schedule"]
METRIC = "draft blocks/sec per layer at B=32, ctx≤4K, block 16; attn HBM GB/s vs roofline"
UNIT = "blocks/s/layer"
WORKLOAD = "serve_b32"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="launch every call eagerly")
    ap.add_argument("--paged", action="store_true", help="paged KV cache (128-row pages)")
    ap.add_argument("--kv", choices=["bf16", "fp8"], default="bf16",
                    help="cache element type: bf16, or fp8 (E4M3 codes, per-layer scales)")
    ap.add_argument("--round-only", action="store_true",
                    help="skip the extra measurements (prefill GEMMs, bookkeeping, layer output)")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f,
                stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not self.path:
            return None
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
                except ValueError:
                    continue
        os.unlink(self.path)
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r)
                          if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------
# algorithmic bytes and flops (per launch) for the roofline
# ---------------------------------------------------------------------------

def attention_bytes(w, starts, window=0):
    """K/V rows read + Q read + output written, per layer launch (bf16 Q and output;
    K/V bf16, or one byte per element for an fp8 cache, whose Q is two bytes per
    element as well: the codes and the remainder codes).

    Keys read per sequence: [max(0, start - W + 1), start + bs) with a sliding
    window W, else [0, start + bs).
    """
    e = 2
    ekv = 1 if w.kv == "fp8" else 2
    rows = 0
    for s in starts:
        lo = max(0, int(s) - window + 1) if window > 0 else 0
        rows += int(s) + w.bs - lo
    kv = rows * w.n_kv * w.d_h * 2 * ekv
    q = w.batch * w.n_h * w.bs * w.d_h * e
    out = w.batch * w.bs * w.n_h * w.d_h * e
    return int(kv + q + out)


def mean_attention_bytes(w, starts):
    """Average over the draft layers (their windows differ in hybrid workloads)."""
    return int(sum(attention_bytes(w, starts, win) for win in w.windows) / len(w.windows))


TRAFFIC_RUN = None  # workload / cache element type / layout of this run


def measured_traffic(kernel, run=None):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on this run's
    workload, cache element type and layout (or on `run`), and the kernel source is
    unchanged."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "traffic_serve_b32.json")) as f:
            t = json.load(f)["runs"][run or TRAFFIC_RUN][kernel]
        with open(os.path.join(ROOT, t["source"]), "rb") as f:
            if hashlib.sha256(f.read()).hexdigest()[:16] != t["sha256_16"]:
                return None
        return t["bytes_per_launch"]
    except Exception:
        return None


def gemm_cost(M, K, N):
    flops = 2.0 * M * K * N
    bytes_ = 2.0 * (M * K + N * K) + 4.0 * M * N
    return flops, bytes_


# ---------------------------------------------------------------------------
# reference arm / CPU baseline: the float64 oracle on a bounded sample
# ---------------------------------------------------------------------------

def oracle_sample_rate(w, budget_s=12.0, max_steps=None):
    """Times the oracle on whole-sequence rounds (all layers) until the budget is spent.

    Returns (blocks/s/layer, seconds, sequences done, per-step seconds).
    """
    from oracle import dflash_oracle as O
    from speculative_decoding_draft_dflash_gb300 import synth

    L0 = synth.prefill_lens(w)
    W_fc, g_h = synth.W_fc(w), synth.gamma_h(w)
    Wq = [synth.W_Q(w, l) for l in range(w.n_layers)]
    Wk = [synth.W_K(w, l) for l in range(w.n_layers)]
    Wv = [synth.W_V(w, l) for l in range(w.n_layers)]
    gq = [synth.gamma_q(w, l) for l in range(w.n_layers)]
    gk = [synth.gamma_k(w, l) for l in range(w.n_layers)]
    steps = []
    total = 0.0
    b = 0
    while (max_steps is None and total < budget_s) or (max_steps is not None and len(steps) < max_steps):
        cache = O.DraftKVCache(w.n_layers, 1, w.n_kv, w.d_h,
                               fp8_scales=synth.kv_scales(w) if w.kv == "fp8" else None)
        for l in range(w.n_layers):
            K, V = synth.cache_rows(w, l, b, int(L0[b]))
            cache.set_rows(l, 0, K, V)
        hid = synth.hidden_states_rows(w, 1, b, w.new_ctx)
        H = [synth.block_embeddings(w, 1, l, b)[None] for l in range(w.n_layers)]
        t0 = time.perf_counter()
        C = O.ctx_project(hid, W_fc, g_h, w.eps)
        for l in range(w.n_layers):
            O.kv_inject(cache, l, C, [0, w.new_ctx], Wk[l], Wv[l], gk[l], w.n_kv, w.d_h, w.eps,
                        w.theta)
            O.block_attn(cache, l, H[l], Wq[l], Wk[l], Wv[l], gq[l], gk[l], w.n_h, w.n_kv, w.d_h,
                         w.eps, w.theta, w.windows[l])
        O.cache_crop(cache, [int(L0[b]) + w.new_ctx])
        dt = time.perf_counter() - t0
        steps.append(dt)
        total += dt
        b = (b + 1) % w.batch
    rate = len(steps) * w.n_layers / total
    return rate, total, len(steps), steps


def run_reference(args, w):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    cores = os.cpu_count()
    _, _, _, warm = oracle_sample_rate(w, max_steps=max(1, args.warmup))
    rate, total, n, steps = oracle_sample_rate(w, max_steps=max(1, args.steps))
    ms = 1e3 * total / n
    sample = (f"{n} whole-sequence rounds (ctx_project of {w.new_ctx} rows + {w.n_layers} x "
              f"(kv_inject + block_attn) + crop) of {w.name}, one sequence per step")
    line = {"impl": "reference", "metric": METRIC, "value": rate, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_of(w),
            "cpu_baseline": {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": rate, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line, default=_json_default), flush=True)


def _json_default(o):
    if hasattr(o, "item"):
        return o.item()
    raise TypeError(f"not JSON serialisable: {type(o)}")


def step_bytes(w, starts):
    """Bytes one draft round touches at least once: KV cache rows read + weights."""
    e = 4 if w.dtype == "f32" else 2
    weights = (w.k * w.d * w.d + w.n_layers * w.d * (w.n_h + 2 * w.n_kv) * w.d_h) * e
    cache = sum(attention_bytes(w, starts, win) for win in w.windows)
    return weights + cache


def config_of(w):
    from speculative_decoding_draft_dflash_gb300 import synth
    starts = synth.prefill_lens(w) + w.new_ctx
    cfg = {"workload": w.name, "batch": w.batch, "context": f"U[{w.prefill_lo},{w.prefill_hi}]",
           "new_context_rows": w.new_ctx, "block_size": w.bs, "draft_layers": w.n_layers,
           "d": w.d, "n_h": w.n_h, "n_kv": w.n_kv, "d_h": w.d_h, "k_target_layers": w.k,
           "windows": list(w.windows)}
    if w.kv == "fp8":
        cfg["kv_cache"] = "fp8 E4M3 codes, one scale per layer for K and for V"
    mb = step_bytes(w, starts) / 1e6
    cfg["l2"] = (f"inputs larger than L2: every step reads the KV cache rows and the weights, "
                 f"{mb:.0f} MB in all, over the 129 MB L2" if mb > 129 else
                 f"step working set {mb:.0f} MB fits in the 129 MB L2: rates are L2-assisted")
    return cfg


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def max_over_ranks(x, world, device="cuda"):
    """The largest of every rank's value (the slowest replica sets the job's time)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world, w, ms_per_step):
    """Blocks per second per layer over all replicas: each rank drafts its own batch."""
    return world * w.batch * w.n_layers / (ms_per_step * 1e-3)


def run_ours(args, w):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev_index = torch.cuda.current_device()

    from speculative_decoding_draft_dflash_gb300 import build
    build.build()
    from speculative_decoding_draft_dflash_gb300 import dflash as D
    from speculative_decoding_draft_dflash_gb300 import synth
    from speculative_decoding_draft_dflash_gb300.runner import DeviceWorkload

    stream = torch.cuda.Stream()
    torch.cuda.set_stream(stream)
    dev = DeviceWorkload(w, paged=args.paged)
    L0 = synth.prefill_lens(w)
    counts = np.full(w.batch, w.new_ctx, dtype=np.int64)
    x = dev.round_inputs(1, L0, counts=counts, crop_to=L0)
    torch.cuda.synchronize()
    assert D.dflash_status_get(stream) == 0

    def step():
        dev.run_round(x, crop=True, stream=stream)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    # eager warm-up (first calls resolve symbols and encode tensor maps), then the
    # step captured in a CUDA graph: the timed region is one replay of K captured steps
    for _ in range(2):
        step()
    torch.cuda.synchronize()

    def capture(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(n):
                step()
        return g

    if args.no_graph:
        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize()
        launches0 = D.dflash_launch_count()
        run_timed = lambda: [step() for _ in range(args.steps)]  # noqa: E731
    else:
        g1 = capture(1)
        for _ in range(args.warmup):
            g1.replay()
        torch.cuda.synchronize()
        assert D.dflash_status_get(stream) == 0, "device status after warm-up"
        launches0 = D.dflash_launch_count()
        gK = capture(args.steps)
        run_timed = gK.replay
    launches = D.dflash_launch_count() - launches0 if not args.no_graph else None

    # ---- timed region: K steps, CUDA events on the launching stream ----
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev_index) as clk:
        barrier()
        ev0.record(stream)
        run_timed()
        ev1.record(stream)
        barrier()
    if args.no_graph:
        launches = D.dflash_launch_count() - launches0
    t_ms = max_over_ranks(ev0.elapsed_time(ev1), world)
    ms_per_step = t_ms / args.steps
    value = whole_job_rate(world, w, ms_per_step)
    assert D.dflash_status_get(stream) == 0, "device status after the timed region"

    # ---- per-kernel durations: the same K steps again, with CUDA event pairs that
    # the library records around each launch on its own stream (captured as event
    # nodes). Kept out of the timed region above: each event node costs microseconds.
    # a layer's projections: one grouped launch (context K/V + block Q/K/V) when
    # dflash_draft_layer groups them, else a K/V and a Q/K/V launch
    gemm_names = [["gemm_fc"] + ["gemm_layer"] * w.n_layers,
                  ["gemm_fc"] + [n for _ in range(w.n_layers) for n in ("gemm_kv", "gemm_qkv")]]
    kernels, t_traced = traced_kernels(args, D, stream, capture, run_timed, gemm_names)
    pk = peaks()
    starts = L0 + w.new_ctx
    attn_bytes = mean_attention_bytes(w, starts)
    M = w.batch * w.new_ctx
    costs = {"gemm_fc": gemm_cost(M, w.k * w.d, w.d),
             "gemm_kv": gemm_cost(M, w.d, 2 * w.n_kv * w.d_h),
             "gemm_qkv": gemm_cost(w.batch * w.bs, w.d, (w.n_h + 2 * w.n_kv) * w.d_h)}
    costs["gemm_layer"] = tuple(a + b for a, b in zip(costs["gemm_kv"], costs["gemm_qkv"]))
    rf = lambda name: roofline_for(name, kernels, costs, attn_bytes, pk)  # noqa: E731
    dominant = max(kernels, key=lambda k: kernels[k]["share_of_step"] * (k in costs or k == "attention"))
    roofline = rf(dominant)
    others = {k: rf(k) for k in kernels if k != dominant and (k in costs or k == "attention")}
    extras = not args.round_only
    prefill = run_prefill_gemms(args, w, dev, stream, D, pk) if w.prefill_inject and extras else None
    bookkeeping = time_accept(args, w, stream, D) if extras else None
    layer_rest = time_layer_out(args, w, stream, D, pk) if w.dtype == "bf16" and extras else None
    fp8 = (time_fp8_cache(args, w, stream, D, pk)
           if w.dtype == "bf16" and w.kv == "bf16" and extras and world == 1 else None)

    round2 = time_round2(args, w, dev, stream, D) if w.rounds > 1 and extras else None

    # ---- end to end: host inputs in, host results out, through the same calls ----
    e2e = run_e2e(args, w, dev, x, stream, D)
    config2 = (time_config2(args, stream, D, pk)
               if w.name == WORKLOAD and extras and world == 1 else None)

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {**config_of(w), **({"cache": "paged, 128-row pages"} if args.paged else {})},
            "clocks": clk.summary(), "e2e": e2e,
            "gpu_launches": int(launches), "roofline": roofline, "roofline_other": others,
            "kernels": kernels,
            "timing": ("value: one replay of a CUDA graph of the K steps, no tracing; kernel "
                       "durations (roofline.achieved, kernels): a second replay of the same K "
                       "steps with CUDA event pairs around each launch (%.3f ms/step with "
                       "the events)" % (t_traced / args.steps)) if not args.no_graph else
                      "eager launches; kernel durations from a second traced pass"}
    if prefill is not None:
        line["prefill_gemms"] = prefill
    if round2 is not None:
        line["round2"] = round2
    if config2 is not None:
        line["config2"] = config2
    if fp8 is not None:
        line["kv_fp8"] = fp8
    if bookkeeping is not None:
        line["bookkeeping"] = bookkeeping
    if layer_rest is not None:
        line["layer_output"] = layer_rest
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, total, n, _ = oracle_sample_rate(w, budget_s=12.0)
        line["cpu_baseline"] = {"value": rate, "unit": UNIT, "cores": os.cpu_count(),
                                "kind": "oracle",
                                "sample": f"{n} whole-sequence rounds of {w.name} "
                                          f"({total:.1f} s, float64 NumPy, default BLAS threads)"}
    if rank == 0:
        print(json.dumps(line, default=_json_default), flush=True)
    if world > 1:
        dist.destroy_process_group()


def traced_kernels(args, D, stream, capture, run_timed, gemm_names):
    """Per-kernel durations from one more pass of the K steps with CUDA event pairs."""
    import torch
    D.dflash_trace_start(TRACED, 64 * args.steps)
    t_ev0 = torch.cuda.Event(enable_timing=True)
    t_ev1 = torch.cuda.Event(enable_timing=True)
    if args.no_graph:
        t_ev0.record(stream)
        run_timed()
        t_ev1.record(stream)
    else:
        gT = capture(args.steps)
        t_ev0.record(stream)
        gT.replay()
        t_ev1.record(stream)
    torch.cuda.synchronize()
    trace = D.dflash_trace_stop()
    t_traced = t_ev0.elapsed_time(t_ev1)
    per = {}
    for name, ms in trace:
        per.setdefault(name, []).append(ms)
    # gemm launches in their order within a step; gemm_names is one list of names per
    # step, or several candidates told apart by the number of launches per step
    gemm_times = per.pop("gemm", [])
    if gemm_names and isinstance(gemm_names[0], (list, tuple)):
        per_step = len(gemm_times) // max(1, args.steps)
        gemm_names = next((g for g in gemm_names if len(g) == per_step), gemm_names[0])
    for i, ms in enumerate(gemm_times):
        per.setdefault(gemm_names[i % len(gemm_names)], []).append(ms)
    kernels = {k: {"launches": len(v), "avg_us": 1e3 * sum(v) / len(v),
                   "share_of_step": sum(v) / t_traced} for k, v in per.items() if v}
    return kernels, t_traced


def roofline_for(name, kernels, costs, attn_bytes, pk):
    k = kernels[name]
    dur = k["avg_us"] * 1e-6
    if name == "attention":
        ach = attn_bytes / dur / 1e9
        return {"kernel": name, "bound": "hbm", "achieved": ach, "peak": pk["hbm_gbs"],
                "unit": "GB/s", "frac": ach / pk["hbm_gbs"], "traffic": measured_traffic(name),
                "algorithmic_bytes_per_launch": attn_bytes,
                "frac_of_nominal_8TBs": ach / 8000.0, "peak_source": pk["source"]}
    if name in costs:
        fl, by = costs[name]
        ridge = pk["bf16_tflops"] * 1e12 / (pk["hbm_gbs"] * 1e9)
        if fl / by > ridge:
            # the GEMMs run for tens of microseconds inside a replay of a few milliseconds at
            # the maximum SM clock: the burst peak is their denominator
            ach = fl / dur / 1e12
            return {"kernel": name, "bound": "tensor", "achieved": ach,
                    "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                    "frac": ach / pk["bf16_tflops"],
                    "frac_of_sustained": ach / pk["bf16_tflops_sustained"],
                    "traffic": measured_traffic(name), "algorithmic_flops_per_launch": fl,
                    "peak_source": pk["source"] + " burst"}
        ach = by / dur / 1e9
        return {"kernel": name, "bound": "hbm", "achieved": ach, "peak": pk["hbm_gbs"],
                "unit": "GB/s", "frac": ach / pk["hbm_gbs"], "traffic": measured_traffic(name),
                "algorithmic_bytes_per_launch": by, "peak_source": pk["source"]}
    return None


def run_prefill_gemms(args, w, dev, stream, D, pk):
    """The prefill of a workload whose cache is filled by projection + inject: crop every
    layer to 0, then project and inject the sum(L0) prefill rows again (the same rows land
    in the same slots), so the fc and K/V GEMMs run at M = sum(L0). Returns their rooflines."""
    import torch
    from speculative_decoding_draft_dflash_gb300 import synth
    counts = dev.L0
    M = int(counts.sum())
    hid = [torch.from_numpy(np.ascontiguousarray(h)).to(device="cuda", dtype=dev.dt)
           for h in synth.hidden_states(w, 0, counts)]
    cu = torch.from_numpy(synth.cu_rows(counts).astype(np.int32)).cuda()
    zero = torch.zeros(w.batch, dtype=torch.int32, device="cuda")
    C = torch.empty((M, w.d), dtype=dev.dt, device="cuda")

    def pstep():
        D.dflash_cache_crop(dev.cache, zero, stream)
        D.dflash_ctx_project(dev.dims, hid, M, dev.W_fc, dev.g_h, C, dev.ws, stream)
        for l in range(w.n_layers):
            D.dflash_kv_inject(dev.dims, dev.cache, l, C, cu, M, dev.W_K[l], dev.W_V[l], dev.g_k[l],
                               dev.rope, dev.table_len, dev.ws, stream)

    def capture(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(n):
                pstep()
        return g

    steps = max(10, min(args.steps, 50))
    pstep()
    torch.cuda.synchronize()
    g1 = capture(1)
    for _ in range(3):
        g1.replay()
    torch.cuda.synchronize()
    assert D.dflash_status_get(stream) == 0, "device status after the prefill warm-up"
    pargs = argparse.Namespace(**{**vars(args), "steps": steps})
    kernels, _ = traced_kernels(pargs, D, stream, capture, lambda: [pstep() for _ in range(steps)],
                                ["gemm_fc"] + ["gemm_kv"] * w.n_layers)
    assert D.dflash_status_get(stream) == 0, "device status after the prefill pass"
    costs = {"gemm_fc": gemm_cost(M, w.k * w.d, w.d), "gemm_kv": gemm_cost(M, w.d, 2 * w.n_kv * w.d_h)}
    out = {"M": M, "steps": steps}
    for name in ("gemm_fc", "gemm_kv"):
        if name in kernels:
            out[name] = {**roofline_for(name, kernels, costs, 0, pk), "avg_us": kernels[name]["avg_us"]}
    # the rest of the prefill's launches: hidden_norm and (when the K/V projection splits K)
    # the per-head epilogue and the length update, per launch
    out["other_kernels_us"] = {k: v["avg_us"] for k, v in kernels.items() if k not in costs}
    if "gemm_kv" in kernels:
        # the whole context K/V projection of one layer: its GEMM and, when the GEMM splits K,
        # the per-head epilogue kernel (norm, RoPE, cache rows) that finishes it
        us = kernels["gemm_kv"]["avg_us"] + sum(kernels[k]["avg_us"] for k in ("head_epilogue",)
                                                if k in kernels)
        tf = costs["gemm_kv"][0] / (us * 1e-6) / 1e12
        out["kv_projection"] = {"avg_us": us, "achieved": tf, "unit": "TFLOP/s",
                                "frac": tf / pk["bf16_tflops"], "peak": pk["bf16_tflops"]}
    return out


def _graph_ms(stream, step, n):
    """Milliseconds per step over one replay of a CUDA graph of n steps (after a warm replay)."""
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(n):
            step()
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / n


def _traced_attention(stream, D, step, n, n_layers):
    """Average attention launch time (ms) over a traced graph replay of n steps."""
    import torch
    D.dflash_trace_start(["attention"], 4 * n * n_layers)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(n):
            step()
    g.replay()
    torch.cuda.synchronize()
    att = [t for k, t in D.dflash_trace_stop() if k == "attention"]
    return sum(att) / max(1, len(att))


def time_round2(args, w, dev, stream, D):
    """Round 2 of the two-round schedule: the cache holds L0 + 16 context rows (round 1's
    inject, cropped after its block), round 2 injects a_i ~ U{1..bs} rows per sequence
    (acceptance + 1, a ragged M), runs the block and crops back to L0 + 16. Timed like the
    main step (graph replay); the cache is left at L0 afterwards."""
    import torch
    from speculative_decoding_draft_dflash_gb300 import synth
    L0 = synth.prefill_lens(w)
    L1 = L0 + w.new_ctx
    x1 = dev.round_inputs(1, L0, counts=np.full(w.batch, w.new_ctx, dtype=np.int64), crop_to=L1)
    dev.run_round(x1, crop=True, stream=stream)          # lens: L0 -> L0 + 16
    counts = synth.accepted_plus_one(w, 2)
    x2 = dev.round_inputs(2, L1, counts=counts, crop_to=L1)
    step = lambda: dev.run_round(x2, crop=True, stream=stream)  # noqa: E731
    step()
    torch.cuda.synchronize()
    assert D.dflash_status_get(stream) == 0, "device status after round 2"
    n = max(10, min(args.steps, 50))
    ms = _graph_ms(stream, step, n)
    att = _traced_attention(stream, D, step, n, w.n_layers)
    assert D.dflash_status_get(stream) == 0, "device status after round 2"
    D.dflash_cache_crop(dev.cache, torch.from_numpy(L0.astype(np.int32)).to("cuda"), stream)
    torch.cuda.synchronize()
    return {"value": whole_job_rate(1, w, ms), "unit": UNIT, "ms_per_step": ms, "steps": n,
            "inject_rows": int(counts.sum()), "attention_avg_us": 1e3 * att,
            "schedule": "lens L0+16 -> inject a_i ~ U{1..16} -> block (+16) -> crop to L0+16"}


def time_config2(args, stream, D, pk):
    """The Qwen3-8B-shaped batch-1 layer: its prefill GEMMs at M = 1024 (fc and context K/V,
    the tensor-core measurement point) and its draft round (16 new context rows, block 16 at
    positions 1040-1055): rate, attention time and the attention's HBM fraction."""
    import torch
    from speculative_decoding_draft_dflash_gb300 import synth
    from speculative_decoding_draft_dflash_gb300.runner import DeviceWorkload
    w2 = synth.WORKLOADS["qwen3_8b_b1"]
    dev = DeviceWorkload(w2)
    prefill = run_prefill_gemms(args, w2, dev, stream, D, pk)
    L0 = synth.prefill_lens(w2)
    x = dev.round_inputs(1, L0, counts=np.full(1, w2.new_ctx, dtype=np.int64), crop_to=L0)
    step = lambda: dev.run_round(x, crop=True, stream=stream)  # noqa: E731
    step()
    torch.cuda.synchronize()
    n = max(20, min(args.steps, 100))
    ms = _graph_ms(stream, step, n)
    att = _traced_attention(stream, D, step, n, w2.n_layers)
    assert D.dflash_status_get(stream) == 0, "device status after the batch-1 round"
    by = mean_attention_bytes(w2, L0 + w2.new_ctx)
    ach = by / (att * 1e-3) / 1e9
    out = {"workload": w2.name, "prefill_gemms": prefill,
           "round": {"value": whole_job_rate(1, w2, ms), "unit": UNIT, "ms_per_step": ms,
                     "steps": n},
           "attention": {"avg_us": 1e3 * att, "algorithmic_bytes_per_launch": by,
                         "achieved": ach, "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": ach / pk["hbm_gbs"],
                         "note": "4.6 MB per launch, 8 (sequence, KV head) pairs: latency-bound "
                                 "at batch 1; the HBM target applies at the serving workload"}}
    del dev
    torch.cuda.empty_cache()
    return out


def time_fp8_cache(args, w, stream, D, pk):
    """The same draft round on an fp8 (E4M3) cache: step rate, and the attention's duration
    and HBM fraction with the cache read at one byte per element (a second device copy of
    the workload; the bf16 one above is left as it was)."""
    import torch
    from speculative_decoding_draft_dflash_gb300 import synth
    from speculative_decoding_draft_dflash_gb300.runner import DeviceWorkload
    w8 = w.replace(kv="fp8")
    dev = DeviceWorkload(w8, paged=args.paged)
    L0 = synth.prefill_lens(w8)
    x = dev.round_inputs(1, L0, counts=np.full(w8.batch, w8.new_ctx, dtype=np.int64), crop_to=L0)
    step = lambda: dev.run_round(x, crop=True, stream=stream)  # noqa: E731
    for _ in range(2):
        step()
    torch.cuda.synchronize()
    n = max(10, min(args.steps, 50))

    def capture(k):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(k):
                step()
        return g

    g = capture(n)
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / n
    D.dflash_trace_start(["attention"], 4 * n * w8.n_layers)
    gT = capture(n)
    gT.replay()
    torch.cuda.synchronize()
    att = [t for k, t in D.dflash_trace_stop() if k == "attention"]
    assert D.dflash_status_get(stream) == 0, "device status after the fp8 cache run"
    avg = sum(att) / max(1, len(att))
    by = mean_attention_bytes(w8, L0 + w8.new_ctx)
    ach = by / (avg * 1e-3) / 1e9
    out = {"value": whole_job_rate(1, w8, ms), "unit": UNIT, "ms_per_step": ms, "steps": n,
           "attention": {"avg_us": 1e3 * avg, "algorithmic_bytes_per_launch": by,
                         "achieved": ach, "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": ach / pk["hbm_gbs"],
                         "traffic": measured_traffic(
                             "attention",
                             f"{w8.name}/fp8/{'paged' if args.paged else 'contiguous'}")},
           "cache": "E4M3 codes, one scale per layer for K and for V"}
    del dev
    torch.cuda.empty_cache()
    return out


def time_accept(args, w, stream, D):
    """dflash_accept at this batch: one round's acceptance lengths, next inject offsets,
    next block starts and anchors from seeded draft / posterior tokens (launch-bound)."""
    import torch
    rng = np.random.Generator(np.random.PCG64(99))
    B, bs = w.batch, w.bs
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()  # noqa: E731
    block = dev(rng.integers(0, 1000, size=(B, bs)))
    post = dev(rng.integers(0, 1000, size=(B, bs)))
    ctx = dev(synth_lens(w))
    outs = [torch.empty(n, dtype=torch.int32, device="cuda") for n in (B, B + 1, B, B)]
    call = lambda: D.dflash_accept(block, post, ctx, *outs, stream=stream)  # noqa: E731

    def capture(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(n):
                call()
        return g

    call()
    torch.cuda.synchronize()
    n = max(10, min(args.steps, 100))
    D.dflash_trace_start(["accept"], n + 8)
    g = capture(n)
    g.replay()
    torch.cuda.synchronize()
    ms = [t for k, t in D.dflash_trace_stop() if k == "accept"]
    return {"kernel": "accept", "launches": len(ms), "avg_us": 1e3 * sum(ms) / max(1, len(ms)),
            "batch": B, "block": bs, "bound": "launch"}


def time_layer_out(args, w, stream, D, pk):
    """The rest of a draft layer on the block rows (o_proj + residual, post norm, SwiGLU MLP +
    residual) at this workload's width: time per call and the rooflines of its three GEMMs."""
    import torch
    from speculative_decoding_draft_dflash_gb300 import synth
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to("cuda", torch.bfloat16)  # noqa: E731
    M, d, a, f = w.batch * w.bs, w.d, w.n_h * w.d_h, w.ffn
    dims = D.make_dims(w.d, w.n_h, w.n_kv, w.d_h, w.k, w.bs, w.eps, w.dtype)
    Wt = [dev(g(w, 0)) for g in (synth.W_O, synth.gamma_post, synth.W_gate, synth.W_up, synth.W_down)]
    attn, x = dev(synth.attn_rows(w, 1, 0)), dev(synth.residual(w, 1, 0))
    out = torch.empty_like(x)
    ws = torch.empty(D.dflash_layer_out_workspace_bytes(dims, M, f), dtype=torch.uint8, device="cuda")
    call = lambda: D.dflash_layer_out(dims, M, attn, x, Wt[0], Wt[1], f, Wt[2], Wt[3], Wt[4],  # noqa: E731
                                      out, ws, stream)

    def capture(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(n):
                call()
        return g

    call()
    torch.cuda.synchronize()
    n = max(10, min(args.steps, 50))
    g = capture(n)
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    us = 1e3 * e0.elapsed_time(e1) / n
    assert D.dflash_status_get(stream) == 0, "device status after the layer output"
    pargs = argparse.Namespace(**{**vars(args), "steps": n})
    kernels, _ = traced_kernels(pargs, D, stream, capture, lambda: [call() for _ in range(n)],
                                ["gemm_o_proj", "gemm_gate_up", "gemm_down"])
    costs = {"gemm_o_proj": gemm_cost(M, a, d), "gemm_gate_up": gemm_cost(M, d, 2 * f),
             "gemm_down": gemm_cost(M, f, d)}
    total_flops = sum(c[0] for c in costs.values())
    return {"rows": M, "d": d, "d_ff": f, "us_per_call": us,
            "tflops_per_call": total_flops / (us * 1e-6) / 1e12,
            "gemms": {k: {**roofline_for(k, kernels, costs, 0, pk), "avg_us": kernels[k]["avg_us"]}
                      for k in costs if k in kernels},
            "timing": "one graph replay of the calls, no tracing; GEMM durations from a traced replay"}


def synth_lens(w):
    from speculative_decoding_draft_dflash_gb300 import synth
    return synth.prefill_lens(w) + w.new_ctx


def run_e2e(args, w, dev, x, stream, D):
    """The same steps through the same calls, with every step's inputs copied in from pinned
    host memory and its outputs copied back. Two buffer slots: step i+1's inputs upload and
    step i-1's outputs download on copy streams while step i computes (a step's compute
    waits for its upload; a slot is refilled only once the step that used it is done and
    its outputs are out)."""
    import torch
    from speculative_decoding_draft_dflash_gb300.runner import RoundInputs

    def clone(xx):
        return RoundInputs(xx.rnd, xx.counts, [t.clone() for t in xx.hidden], xx.cu_rows.clone(),
                           [t.clone() for t in xx.H], xx.crop_to.clone(), xx.M)

    slots = [x, clone(x)]
    outs = [dev.out, [torch.empty_like(o) for o in dev.out]]
    hid_h = [t.cpu().pin_memory() for t in x.hidden]
    H_h = [t.cpu().pin_memory() for t in x.H]
    cu_h = x.cu_rows.cpu().pin_memory()
    crop_h = x.crop_to.cpu().pin_memory()
    out_h = [[torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in dev.out] for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in hid_h + H_h + [cu_h, crop_h])
    d2h = sum(t.numel() * t.element_size() for t in out_h[0])
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    Ev = lambda: torch.cuda.Event()  # noqa: E731

    def steps(n):
        """n pipelined steps; every cross-stream dependency is an event of this sequence."""
        fork = Ev()
        fork.record(stream)
        s_in.wait_event(fork)
        s_out.wait_event(fork)
        ev_in, ev_done, ev_out = [None, None], [None, None], [None, None]
        for i in range(n):
            k = i % 2
            xi, oi = slots[k], outs[k]
            with torch.cuda.stream(s_in):
                if ev_done[k] is not None:
                    s_in.wait_event(ev_done[k])       # step i-2 is done with slot k
                for dst, src in zip(xi.hidden, hid_h):
                    dst.copy_(src, non_blocking=True)
                for dst, src in zip(xi.H, H_h):
                    dst.copy_(src, non_blocking=True)
                xi.cu_rows.copy_(cu_h, non_blocking=True)
                xi.crop_to.copy_(crop_h, non_blocking=True)
                ev_in[k] = Ev()
                ev_in[k].record(s_in)
            stream.wait_event(ev_in[k])
            if ev_out[k] is not None:
                stream.wait_event(ev_out[k])          # step i-2's outputs are copied out
            dev.run_round(xi, crop=True, stream=stream, out=oi)
            ev_done[k] = Ev()
            ev_done[k].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_done[k])
                for dst, src in zip(out_h[k], oi):
                    dst.copy_(src, non_blocking=True)
                ev_out[k] = Ev()
                ev_out[k].record(s_out)
        for e in ev_out + ev_in:                       # join the copy streams
            if e is not None:
                stream.wait_event(e)

    with torch.cuda.stream(stream):
        steps(2)
    torch.cuda.synchronize()
    if args.no_graph:
        with torch.cuda.stream(stream):
            steps(max(3, args.warmup))
    else:
        g1 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g1, stream=stream):
            steps(2)
        for _ in range(max(3, args.warmup)):
            g1.replay()
        gK = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gK, stream=stream):
            steps(args.steps)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    if args.no_graph:
        with torch.cuda.stream(stream):
            steps(args.steps)
    else:
        gK.replay()
    ev1.record(stream)
    torch.cuda.synchronize()
    assert D.dflash_status_get(stream) == 0
    ms = max_over_ranks(ev0.elapsed_time(ev1), world) / args.steps
    return {"value": whole_job_rate(world, w, ms), "unit": UNIT,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "ms_per_step": ms,
            "overlap": "two buffer slots: step i+1's inputs upload and step i-1's outputs "
                       "download on copy streams while step i computes"}


def main():
    args = parse()
    from speculative_decoding_draft_dflash_gb300 import synth
    w = synth.WORKLOADS[args.workload]
    if args.kv == "fp8":
        w = w.replace(kv="fp8")
    global TRAFFIC_RUN
    TRAFFIC_RUN = f"{w.name}/{w.kv}/{'paged' if args.paged else 'contiguous'}"
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
