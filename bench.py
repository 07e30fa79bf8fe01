"""Benchmark of the fused MoE layer forward pass on GB300.

One step = one moe_forward (gate, align/permute, gate_up+SwiGLU GEMM, down GEMM,
unpermute+reduce) over one batch of T synthetic tokens with the Mixtral-8x7B
layer shape (H=4096, I=14336, E=8, top_k=2, softmax renormalised, bf16
weights ~N(0, 0.02)); default T = 4096.  Inputs are resident in HBM; the expert
weights (2.8 GB) exceed L2, so no flush is needed between steps.

Prints ONE JSON line (rank 0).  `--impl reference` times the fp64 CPU oracle
instead, on a bounded token sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE layer tokens/s and achieved % of roofline (HBM or tensor) vs batch 1–4096"
UNIT = "tokens/s"
CONFIG_NAME = "mixtral"
WORKLOADS = {"mixtral_tp2": "mixtral_8x7b_moe_layer_tp2_slice", "qwen2_tp4": "qwen2_57b_a14b_moe_layer_fp8_tp4_slice",
             "dsv3_tp8": "deepseek_v3_moe_layer_int4_tp8_slice", "scout_tp8": "llama4_scout_moe_layer_tp8_slice",
             "mixtral": "mixtral_8x7b_moe_layer", "qwen2": "qwen2_57b_a14b_moe_layer_fp8",
             "dsv3": "deepseek_v3_moe_layer_int4", "dsv3_awq": "deepseek_v3_moe_layer_int4_zero_points",
             "qwen2_dyn": "qwen2_57b_a14b_moe_layer_fp8_dynamic_scales",
             "mixtral_w8": "mixtral_8x7b_moe_layer_int8", "scout": "llama4_scout_moe_layer", "tiny": "tiny_moe_layer",
             "dsv3_paired": "deepseek_v3_moe_layer_int4_paired_codes",
             "dsv3_awq_paired": "deepseek_v3_moe_layer_int4_zero_points_paired_codes",
             "dsv3_paired_tp8": "deepseek_v3_moe_layer_int4_paired_codes_tp8_slice"}


def lib_wdtype(shape):
    """The weight format the library is told: int4 shapes whose codes are
    prepared once by moe_repack_int4 run as MOE_W_INT4_G128_PAIRED."""
    return "int4_paired" if shape.int4_order == "paired" else shape.wdtype


def lib_codes(moe, shape, w):
    """w13 / w2 as the library reads them: the generated codes, or for the paired
    format a copy prepared by moe_repack_int4 (one-time weight preparation, not
    part of a step).  The oracle keeps reading the generated codes."""
    if shape.int4_order == "paired":
        return moe.repack_int4(w.w13), moe.repack_int4(w.w2)
    return w.w13, w.w2


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", 0)), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def init_replicas(backend="nccl"):
    """Process group of a torchrun launch (one rank per GPU, independent
    replicas: no collective touches the data path), or None for one process."""
    world = _env_int("WORLD_SIZE", 1)
    if world <= 1:
        return None
    import torch.distributed as dist
    if not dist.is_initialized():
        dist.init_process_group(backend)
    return dist


def max_over_ranks(dist, value, device):
    """The slowest rank's value (the job finishes when every replica has)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world, tokens_per_rank, ms_max):
    """Whole-job tokens/s: every replica's tokens over the slowest rank's time."""
    return world * tokens_per_rank / (ms_max / 1e3)


def _env_int(name, default):
    try:
        return int(os.environ.get(name, default))
    except ValueError:
        return default


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi clock / throttle samples every 50 ms; `mark()` brackets the
    timed region, whose samples the summary keeps (all samples if none fell
    inside, e.g. a region shorter than the interval, flagged in the summary).
    The raw samples go to MOE_CLOCK_LOG_DIR/clocks_rank<i>.csv when that variable
    names a directory, else to a temporary file removed after the summary."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,timestamp")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        log_dir = os.environ.get("MOE_CLOCK_LOG_DIR")
        self.keep = bool(log_dir)
        if self.keep:
            self.path = os.path.join(log_dir, f"clocks_rank{gpu_index}.csv")
        else:
            fd, self.path = tempfile.mkstemp(prefix=f"moe_clocks_rank{gpu_index}_", suffix=".csv")
            os.close(fd)
        self.t0 = self.t1 = None

    def mark(self, start: bool):
        if start:
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None:
            if not self.keep:
                try:
                    os.remove(self.path)
                except OSError:
                    pass
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        rows = []
        try:
            for line in open(self.path):
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    sm, smax = float(parts[1]), float(parts[2])
                except ValueError:
                    continue
                try:  # e.g. 2026/12/02 14:09:14.123 (host local time)
                    ts = time.mktime(time.strptime(parts[9].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                    ts += float("0." + parts[9].split(".")[1]) if "." in parts[9] else 0.0
                except (ValueError, IndexError):
                    ts = None
                rows.append((ts, sm, smax, [n for n, v in zip(names, parts[5:9]) if v.lower() == "active"]))
        except OSError:
            pass
        if not self.keep:
            try:
                os.remove(self.path)
            except OSError:
                pass
        inside = [r for r in rows if r[0] is not None and self.t0 is not None and self.t1 is not None
                  and self.t0 <= r[0] <= self.t1]
        use = inside or rows
        reasons = sorted({n for r in use for n in r[3]})
        return {"sm_mhz": statistics.median([r[1] for r in use]) if use else None,
                "sm_max_mhz": use[-1][2] if use else None, "reasons": reasons, "samples": len(use),
                "samples_in_timed_region": len(inside)}


# --------------------------------------------------------------- our arm

def layer_bytes_flops(shape, T, touched):
    """Algorithmic bytes / flops of one forward (weights of touched experts,
    x in, out, logits; 6*k*H*I flops per token)."""
    from synth import SHAPES  # noqa
    H, I, E, k = shape.H, shape.I, shape.E, shape.top_k
    if shape.wdtype == "bf16":
        wbytes = 3 * H * I * 2
    elif shape.wdtype == "fp8":
        wbytes = 3 * H * I + 8
    else:
        wbytes = 3 * H * I // (2 if shape.wdtype == "int4" else 1) + \
            3 * H * I // shape.group_size * (3 if shape.zero_point else 2)
    B = touched * wbytes + T * H * 2 * 2 + T * E * 4
    F = 6.0 * k * H * I * T
    return B, F


def run_ours(args):
    import torch
    import mixture_experts_layer_gate_gb300 as moe
    from synth import SHAPES, T_SWEEP, make_tokens, make_weights

    world = _env_int("WORLD_SIZE", 1)
    rank = _env_int("RANK", 0)
    local = _env_int("LOCAL_RANK", 0)
    dist = init_replicas("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    moe.load()
    if args.tuning:
        moe.set_tuning(**json.loads(args.tuning))
    shape = SHAPES[args.config]
    if args.E:
        # profiling aid: same layer shape with fewer experts (smaller device footprint)
        import dataclasses
        shape = dataclasses.replace(shape, E=args.E)
    T = args.T
    hbm, bf16_peak, bf16_sust, peak_src = _peaks()

    w = make_weights(shape, dev, seed=0)
    tok = make_tokens(shape, T, dev, seed=rank)
    p = moe.problem(T, shape.H, shape.I, shape.E, shape.top_k, scoring=shape.scoring,
                    renormalize=shape.renormalize, n_group=shape.n_group, topk_group=shape.topk_group,
                    routed_scaling_factor=shape.routed_scaling_factor, wdtype=lib_wdtype(shape),
                    act_scale=shape.act_scale)
    codes = lib_codes(moe, shape, w)
    wts = moe.Weights(codes[0], codes[1], w.w13_scale, w.w2_scale, tok.a1_scale, tok.a2_scale,
                       w.w13_zero, w.w2_zero)
    ws = moe.alloc_workspace(p, dev)
    out = torch.empty((T, shape.H), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.Stream(device=dev)
    plan = moe.get_plan(p)

    def fwd():
        moe.forward(p, wts, tok.x, tok.logits, tok.bias, out, ws, stream.cuda_stream)

    # capture one step in a CUDA graph (routing stays on the device)
    with torch.cuda.stream(stream):
        fwd()
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    n0 = moe.launch_count()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            fwd()
    launches_per_step = moe.launch_count() - n0  # kernels the library put into one step
    for _ in range(args.warmup):
        with torch.cuda.stream(stream):
            graph.replay()
    stream.synchronize()
    err = moe.get_device_error(ws, stream.cuda_stream)
    if err != 0:
        raise RuntimeError(f"device error {err}")

    # routing facts for the roofline
    ids = torch.empty((T, shape.top_k), dtype=torch.int32, device=dev)
    tw = torch.empty((T, shape.top_k), dtype=torch.float32, device=dev)
    moe.gate_topk(p, tok.logits, tok.bias, ids, tw, stream.cuda_stream)
    stream.synchronize()
    touched = int(torch.unique(ids).numel())
    B, F = layer_bytes_flops(shape, T, touched)

    # A step whose bytes could stay in L2 gets L2 flushed before it (outside its events)
    l2 = l2_bytes(torch, dev)
    flush = l2_flusher(torch, dev, l2) if B < 2 * l2 else None
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        clk.mark(True)
        with torch.cuda.stream(stream):
            for e0, e1 in ev:
                if flush is not None:
                    flush()
                e0.record(stream)
                graph.replay()
                e1.record(stream)
        torch.cuda.synchronize()
        clk.mark(False)
        time.sleep(0.05)
    if dist is not None:
        dist.barrier()
    step_ms = sum(e0.elapsed_time(e1) for e0, e1 in ev)
    if flush is None:  # back to back: one interval from the first start to the last end
        step_ms = ev[0][0].elapsed_time(ev[-1][1])
    ms = max_over_ranks(dist, step_ms / args.steps, dev)
    value = job_throughput(world, T, ms)
    l2_note = (f"L2 ({l2 / 1e6:.0f} MB) flushed before each step by a {2 * l2 / 1e6:.0f} MB write, outside the timed events"
               if flush is not None else
               f"no flush: a step's algorithmic bytes ({B / 1e9:.2f} GB) exceed twice the L2 ({l2 / 1e6:.0f} MB)")
    # tensor peak of the dtype the GEMMs run in: e4m3 at the nominal 2x of the measured bf16
    dtype_peak = bf16_peak * (2.0 if shape.wdtype == "fp8" else 1.0)
    t_roof = max(B / (hbm * 1e9), F / (dtype_peak * 1e12))
    layer_frac = t_roof / (ms / 1e3)

    # dominant kernel: the gate_up grouped GEMM, timed alone on its stream
    S = T * shape.top_k
    counts_t = torch.empty(shape.E, dtype=torch.int32, device=dev)
    offsets = torch.empty(shape.E + 1, dtype=torch.int32, device=dev)
    perm = torch.empty(S, dtype=torch.int32, device=dev)
    inv = torch.empty(S, dtype=torch.int32, device=dev)
    adt = torch.uint8 if shape.wdtype == "fp8" else torch.bfloat16
    x_perm = torch.empty((S, shape.H), dtype=adt, device=dev)
    act = torch.empty((S, shape.I), dtype=adt, device=dev)
    abytes = 1 if shape.wdtype == "fp8" else 2
    roof = dominant_kernel(moe, torch, shape, args.config, T, p, wts, tok, ids, touched, ws, stream, dev,
                           max(5, args.steps), flush, l2, hbm, bf16_peak, peak_src, plan,
                           (counts_t, offsets, perm, inv, x_perm, act))

    # per-stage times: each entry point on its own, CUDA events between them on the
    # stream, no graph (L2 flushed before each rep where the step is flushed)
    y_perm = torch.empty((S, shape.H), dtype=torch.bfloat16, device=dev)
    out_s = torch.empty((T, shape.H), dtype=torch.bfloat16, device=dev)
    sev = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(max(5, args.steps))]
    with torch.cuda.stream(stream):
        for evs in sev:
            if flush is not None:
                flush()
            evs[0].record(stream)
            moe.gate_topk(p, tok.logits, tok.bias, ids, tw, stream.cuda_stream)
            evs[1].record(stream)
            moe.align_permute(p, ids, tok.x, tok.a1_scale, counts_t, offsets, perm, inv, x_perm, ws,
                              stream.cuda_stream)
            evs[2].record(stream)
            moe.grouped_gemm_swiglu(p, wts, x_perm, offsets, act, ws, stream.cuda_stream)
            evs[3].record(stream)
            moe.grouped_gemm_down(p, wts, act, offsets, y_perm, ws, stream.cuda_stream)
            evs[4].record(stream)
            moe.unpermute_reduce(p, y_perm, inv, tw, out_s, ws, stream.cuda_stream)
            evs[5].record(stream)
    stream.synchronize()
    if moe.get_device_error(ws, stream.cuda_stream) != 0:
        raise RuntimeError("device error in the staged run")
    stage_names = ("gate_topk", "align_permute", "gate_up_swiglu", "down", "unpermute_reduce")
    stages_us = {n: sum(e[i].elapsed_time(e[i + 1]) for e in sev) / len(sev) * 1e3
                 for i, n in enumerate(stage_names)}
    # bytes the intermediates move (written once, read once): overhead, not algorithmic
    act_rw = S * shape.I * abytes * 2 + (S * shape.I * 2 * 2 if shape.act_scale == "dynamic" else 0)
    inter_bytes = {"x_perm": S * shape.H * abytes * 2, "act": act_rw, "y_perm": S * shape.H * 2 * 2,
                   "split_k_partials": (plan.splits_up * S * 2 * shape.I * 4 * 2 if plan.splits_up > 1 else 0) +
                   (plan.splits_down * S * shape.H * 4 * 2 if plan.splits_down > 1 else 0)}

    # end to end through the public call with host buffers: every step uploads its
    # inputs (x, logits) from pinned host memory, runs moe_forward and reads its
    # output back.  Steps are pipelined the way a serving loop would run them:
    # step i's upload overlaps step i-1's forward and step i-1's download overlaps
    # step i's forward (two device buffer sets; copies on their own streams).
    x_h = tok.x.cpu().pin_memory()
    l_h = tok.logits.cpu().pin_memory()
    o_h = [torch.empty((T, shape.H), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    x_d = [torch.empty_like(tok.x) for _ in range(2)]
    l_d = [torch.empty_like(tok.logits) for _ in range(2)]
    o_d = [torch.empty((T, shape.H), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("in", "comp", "out")}
    started = [False, False]

    def e2e_step(i):
        b = i & 1
        with torch.cuda.stream(s_in):
            if started[b]:
                s_in.wait_event(ev["comp"][b])  # step i-2's forward has read x_d[b]
            x_d[b].copy_(x_h, non_blocking=True)
            l_d[b].copy_(l_h, non_blocking=True)
            ev["in"][b].record(s_in)
        stream.wait_event(ev["in"][b])
        if started[b]:
            stream.wait_event(ev["out"][b])  # step i-2's download has read o_d[b]
        moe.forward(p, wts, x_d[b], l_d[b], tok.bias, o_d[b], ws, stream.cuda_stream)
        ev["comp"][b].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev["comp"][b])
            o_h[b].copy_(o_d[b], non_blocking=True)
            ev["out"][b].record(s_out)
        started[b] = True

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for i in range(args.steps):
        e2e_step(2 + i)
    e1.record(s_out)
    torch.cuda.synchronize()
    e_ms = max_over_ranks(dist, e0.elapsed_time(e1) / args.steps, dev)
    torch.cuda.synchronize()
    e2e_ok = bool(torch.equal(o_h[(2 + args.steps - 1) & 1], out.cpu()))  # same inputs -> same output

    sweep = []
    sweeps = {}
    if args.sweep and rank == 0:
        with ClockSampler(local) as sclk:
            sclk.mark(True)
            sweep = run_sweep(moe, torch, shape, w, codes, dev, stream, hbm, bf16_peak)
            sclk.mark(False)
        sweeps[args.config] = {"workload": WORKLOADS.get(args.config, args.config), "rows": sweep,
                               "clocks": sclk.summary(), "dominant_kernel_T4096": roof if T == 4096 else None}
        for cfg in args.sweep_configs:
            if cfg != args.config:
                sweeps[cfg] = sweep_config(moe, torch, cfg, dev, stream, local, hbm, bf16_peak, peak_src)

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": {"bf16": "bf16", "fp8": "e4m3", "int4": "bf16", "int8": "bf16"}[shape.wdtype],
        "data": "synthetic",
        "config": {"workload": WORKLOADS.get(args.config, args.config) + (f"_E{shape.E}" if args.E else ""), "T": T, "H": shape.H, "I": shape.I, "E": shape.E,
                   "top_k": shape.top_k, "gate": f"{shape.scoring} top-{shape.top_k}" +
                   (", renormalised" if shape.renormalize else "") +
                   (f", {shape.n_group} groups keep {shape.topk_group}" if shape.n_group else ""),
                   "weights": {"bf16": "bf16", "fp8": "e4m3 per-expert scale" +
                               (", dynamic per-tensor activation scales" if shape.act_scale == "dynamic" else ""),
                               "int4": "int4 group-128" + (" + zero points" if shape.zero_point else "") +
                                       (", codes paired once by moe_repack_int4" if shape.int4_order == "paired"
                                        else ""),
                               "int8": "int8 group-128" + (" + zero points" if shape.zero_point else "")}[shape.wdtype],
                   "global_batch": world * T, "parallelism": f"replicas x{world} (independent batches)",
                   "l2": l2_note,
                   "cuda_graph": True, "plan": {"bn_max": plan.bn_max_up, "splits_up": plan.splits_up,
                                                "splits_down": plan.splits_down, "stages_up": plan.stages_up,
                                                "sms": plan.num_sms}},
        "layer_roofline": {"t_roof_us": t_roof * 1e6, "frac": layer_frac, "touched_experts": touched,
                           "bytes": B, "flops": F},
        "stages_us": stages_us,
        "stages_note": "each entry point alone, CUDA events between them, no graph or PDL overlap",
        "intermediate_bytes": inter_bytes,
        "roofline": roof,
        "e2e": {"value": job_throughput(world, T, e_ms), "unit": UNIT,
                "h2d_bytes_per_step": int(x_h.numel() * 2 + l_h.numel() * 4),
                "d2h_bytes_per_step": int(o_h[0].numel() * 2), "ms_per_step": e_ms,
                "pipelined": "step i's upload and step i-1's download overlap forwards",
                "output_matches_device_run": e2e_ok},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk.summary(),
    }
    if args.tuning:
        line["config"]["planner_overrides"] = json.loads(args.tuning)
    if sweep:
        line["sweep"] = sweep
    if sweeps:
        line["sweeps"] = sweeps
        line["sweeps_note"] = ("per workload: layer tokens/s and roofline fraction for T = 1..4096 (CUDA graph, "
                               "20 reps per T, L2 flushed before each rep when its bytes could stay in L2), "
                               "nvidia-smi clocks sampled during that workload's sweep, and its gate_up GEMM "
                               "timed alone at T = 4096 against its bound")
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(shape, w, tok, args.cpu_sample)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def dominant_kernel(moe, torch, shape, config, T, p, wts, tok, ids, touched, ws, stream, dev, reps, flush, l2,
                    hbm, bf16_peak, peak_src, plan, bufs):
    """The gate_up grouped GEMM (the dominant kernel) timed alone on its stream
    with CUDA events: achieved rate against its roofline bound, and the DRAM
    traffic of a committed ncu summary taken on the current GEMM source."""
    counts_t, offsets, perm, inv, x_perm, act = bufs
    S = T * shape.top_k
    moe.align_permute(p, ids, tok.x, tok.a1_scale, counts_t, offsets, perm, inv, x_perm, ws, stream.cuda_stream)
    for _ in range(3):
        moe.grouped_gemm_swiglu(p, wts, x_perm, offsets, act, ws, stream.cuda_stream)
    up_flops = 2.0 * S * (2 * shape.I) * shape.H
    gbytes = (3.0 if shape.zero_point else 2.0) / shape.group_size  # scale (+ zero point) per group
    wbytes_per_elem = {"bf16": 2.0, "fp8": 1.0, "int4": 0.5 + gbytes, "int8": 1.0 + gbytes}[shape.wdtype]
    abytes = 1 if shape.wdtype == "fp8" else 2
    up_bytes = touched * (2 * shape.I * shape.H * wbytes_per_elem) + S * shape.H * abytes + S * shape.I * abytes
    kflush = (flush or l2_flusher(torch, dev, l2)) if up_bytes < 2 * l2 else None
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    with torch.cuda.stream(stream):
        for e0, e1 in kev:
            if kflush is not None:
                kflush()
            e0.record(stream)
            moe.grouped_gemm_swiglu(p, wts, x_perm, offsets, act, ws, stream.cuda_stream)
            e1.record(stream)
    stream.synchronize()
    if kflush is not None:
        k_ms = sum(e0.elapsed_time(e1) for e0, e1 in kev) / reps
    else:
        k_ms = kev[0][0].elapsed_time(kev[-1][1]) / reps
    dtype_peak = bf16_peak * (2.0 if shape.wdtype == "fp8" else 1.0)
    tensor_peak = dtype_peak
    t_tensor = up_flops / (tensor_peak * 1e12)
    t_hbm = up_bytes / (hbm * 1e9)
    if t_tensor >= t_hbm:
        roof = {"bound": "tensor", "achieved": up_flops / (k_ms / 1e3) / 1e12, "peak": tensor_peak,
                "unit": "TFLOP/s",
                "peak_kind": ("fp8 dense = 2x bf16 dense burst, " if shape.wdtype == "fp8" else "bf16 dense burst, ")
                + peak_src}
    else:
        roof = {"bound": "hbm", "achieved": up_bytes / (k_ms / 1e3) / 1e9, "peak": hbm,
                "unit": "GB/s", "peak_kind": f"HBM copy, {peak_src}"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["kernel"] = (f"grouped_gemm_wna16_kernel<{shape.wdtype}>" if shape.wdtype in ("int4", "int8")
                      else f"grouped_gemm_{'pair_' if plan.pair_up else ''}kernel<{shape.wdtype}>") + \
        (" (clusters of 2 CTAs)" if plan.pair_up else "") + \
        (" (2 MMA-issuing threads)" if plan.issuers_up == 2 else "") + " (gate_up + SwiGLU)" + \
        (" + absmax + e4m3 pass (dynamic scales)" if shape.act_scale == "dynamic" else "")
    roof["kernel_ms"] = k_ms
    roof["algorithmic"] = {"flops": up_flops, "bytes": up_bytes}
    roof["l2_flushed"] = kflush is not None
    roof["traffic"] = _traffic_for("grouped_gemm_up", config, T)
    return roof


def l2_bytes(torch, dev):
    props = torch.cuda.get_device_properties(dev)
    return int(getattr(props, "L2_cache_size", 0) or 128 * 1024 * 1024)


def l2_flusher(torch, dev, l2):
    """A callable that overwrites twice the L2 on the current stream."""
    buf = torch.empty((2 * l2,), dtype=torch.uint8, device=dev)
    state = {"v": 0}

    def flush():
        state["v"] = (state["v"] + 1) & 0x7F
        buf.fill_(state["v"])
    return flush


def sweep_config(moe, torch, cfg, dev, stream, local, hbm, bf16_peak, peak_src):
    """One more workload's batch sweep in the same process: its own weights
    (seed 0), its clocks, and its dominant kernel at T = 4096."""
    from synth import SHAPES, make_tokens, make_weights
    shape = SHAPES[cfg]
    w = make_weights(shape, dev, seed=0)
    codes = lib_codes(moe, shape, w)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        clk.mark(True)
        rows = run_sweep(moe, torch, shape, w, codes, dev, stream, hbm, bf16_peak)
        clk.mark(False)
    T = 4096
    tok = make_tokens(shape, T, dev, seed=0)
    p = moe.problem(T, shape.H, shape.I, shape.E, shape.top_k, scoring=shape.scoring,
                    renormalize=shape.renormalize, n_group=shape.n_group, topk_group=shape.topk_group,
                    routed_scaling_factor=shape.routed_scaling_factor, wdtype=lib_wdtype(shape),
                    act_scale=shape.act_scale)
    wts = moe.Weights(codes[0], codes[1], w.w13_scale, w.w2_scale, tok.a1_scale, tok.a2_scale, w.w13_zero,
                      w.w2_zero)
    ws = moe.alloc_workspace(p, dev)
    ids = torch.empty((T, shape.top_k), dtype=torch.int32, device=dev)
    tw = torch.empty((T, shape.top_k), dtype=torch.float32, device=dev)
    moe.gate_topk(p, tok.logits, tok.bias, ids, tw, stream.cuda_stream)
    stream.synchronize()
    touched = int(torch.unique(ids).numel())
    S = T * shape.top_k
    adt = torch.uint8 if shape.wdtype == "fp8" else torch.bfloat16
    bufs = (torch.empty(shape.E, dtype=torch.int32, device=dev), torch.empty(shape.E + 1, dtype=torch.int32, device=dev),
            torch.empty(S, dtype=torch.int32, device=dev), torch.empty(S, dtype=torch.int32, device=dev),
            torch.empty((S, shape.H), dtype=adt, device=dev), torch.empty((S, shape.I), dtype=adt, device=dev))
    l2 = l2_bytes(torch, dev)
    roof = dominant_kernel(moe, torch, shape, cfg, T, p, wts, tok, ids, touched, ws, stream, dev, 10, None, l2,
                           hbm, bf16_peak, peak_src, moe.get_plan(p), bufs)
    if moe.get_device_error(ws, stream.cuda_stream) != 0:
        raise RuntimeError(f"device error in the {cfg} sweep")
    out = {"workload": WORKLOADS.get(cfg, cfg), "rows": rows, "clocks": clk.summary(),
           "dominant_kernel_T4096": roof}
    del w, codes, wts, ws, bufs, tok
    torch.cuda.empty_cache()
    return out


def run_sweep(moe, torch, shape, w, codes, dev, stream, hbm, bf16_peak):
    """Per-T tokens/s and roofline fraction of the whole layer (CUDA graph, 20 reps;
    L2 flushed before each rep, outside its events, when the rep's bytes could stay in L2)."""
    from synth import T_SWEEP, make_tokens
    rows = []
    l2 = l2_bytes(torch, dev)
    flusher = None
    for T in T_SWEEP:
        tok = make_tokens(shape, T, dev, seed=0)
        p = moe.problem(T, shape.H, shape.I, shape.E, shape.top_k, scoring=shape.scoring,
                        renormalize=shape.renormalize, n_group=shape.n_group, topk_group=shape.topk_group,
                        routed_scaling_factor=shape.routed_scaling_factor, wdtype=lib_wdtype(shape),
                    act_scale=shape.act_scale)
        wts = moe.Weights(codes[0], codes[1], w.w13_scale, w.w2_scale, tok.a1_scale, tok.a2_scale,
                       w.w13_zero, w.w2_zero)
        ws = moe.alloc_workspace(p, dev)
        out = torch.empty((T, shape.H), dtype=torch.bfloat16, device=dev)
        with torch.cuda.stream(stream):
            moe.forward(p, wts, tok.x, tok.logits, tok.bias, out, ws, stream.cuda_stream)
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                moe.forward(p, wts, tok.x, tok.logits, tok.bias, out, ws, stream.cuda_stream)
            for _ in range(3):
                g.replay()
        ids = torch.empty((T, shape.top_k), dtype=torch.int32, device=dev)
        tw = torch.empty((T, shape.top_k), dtype=torch.float32, device=dev)
        moe.gate_topk(p, tok.logits, tok.bias, ids, tw, stream.cuda_stream)
        stream.synchronize()
        touched = int(torch.unique(ids).numel())
        B, F = layer_bytes_flops(shape, T, touched)
        reps = 20
        flush = None
        if B < 2 * l2:
            flusher = flusher or l2_flusher(torch, dev, l2)
            flush = flusher
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        with torch.cuda.stream(stream):
            for e0, e1 in evs:
                if flush is not None:
                    flush()
                e0.record(stream)
                g.replay()
                e1.record(stream)
        stream.synchronize()
        if flush is not None:
            ms = sum(e0.elapsed_time(e1) for e0, e1 in evs) / reps
        else:
            ms = evs[0][0].elapsed_time(evs[-1][1]) / reps
        tb, tf = B / (hbm * 1e9), F / (bf16_peak * (2.0 if shape.wdtype == "fp8" else 1.0) * 1e12)
        rows.append({"T": T, "us": ms * 1e3, "tokens_s": T / (ms / 1e3), "tflops": F / (ms / 1e3) / 1e12,
                     "gbs": B / (ms / 1e3) / 1e9, "bound": "hbm" if tb >= tf else "tensor",
                     "roofline_frac": max(tb, tf) / (ms / 1e3), "touched": touched,
                     "l2_flushed": flush is not None})
        del g, ws
    return rows


def _traffic_for(kernel, config, T):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel source (else null)."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{config}_T{T}.json")
    try:
        with open(path) as f:
            d = json.load(f)
        if d.get("source_sha256") != _gemm_source_hash():
            return None
        return d.get("dram_bytes_per_launch")
    except Exception:
        return None


def _gemm_source_hash():
    h = hashlib.sha256()
    for name in ("gemm.cu", "common.cuh", "kernels.h"):
        with open(os.path.join(ROOT, "mixture_experts_layer_gate_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


# ------------------------------------------------------------ CPU oracle

class _OracleRunner:
    """fp64 CPU oracle on a bounded token sample, decoded experts cached."""

    def __init__(self, shape, w, tok, sample):
        import numpy as np
        import oracle
        self.np, self.oracle = np, oracle
        from oracle.torch_io import np_of, bf16_bits
        T = tok.x.shape[0]
        n = min(sample, T)
        rows = np.linspace(0, T - 1, n).astype(np.int64)
        self.rows = rows
        self.x_bits = bf16_bits(tok.x)[rows]
        self.logits = np_of(tok.logits)[rows]
        self.bias = np_of(tok.bias)
        self.p = oracle.Problem(T=n, H=shape.H, I=shape.I, E=shape.E, top_k=shape.top_k, scoring=shape.scoring,
                                renormalize=shape.renormalize, n_group=shape.n_group,
                                topk_group=shape.topk_group, routed_scaling_factor=shape.routed_scaling_factor,
                                wdtype=shape.wdtype, group_size=shape.group_size, act_scale=shape.act_scale)
        self.a1 = None if tok.a1_scale is None else float(tok.a1_scale.cpu()[0])
        self.a2 = None if tok.a2_scale is None else float(tok.a2_scale.cpu()[0])
        self.cache = {}
        self._w = w
        outer = self

        class Cached(oracle.ExpertWeights):
            def __call__(self_inner, e):
                if e not in outer.cache:
                    t0 = time.perf_counter()
                    sub = oracle.ExpertWeights(outer.p, {e: np_of(w.w13[e])}, {e: np_of(w.w2[e])},
                                               None if w.w13_scale is None else {e: np_of(w.w13_scale[e])},
                                               None if w.w2_scale is None else {e: np_of(w.w2_scale[e])},
                                               None if w.w13_zero is None else {e: np_of(w.w13_zero[e])},
                                               None if w.w2_zero is None else {e: np_of(w.w2_zero[e])})
                    outer.cache[e] = sub(e)
                    self_inner.prep_seconds += time.perf_counter() - t0
                return outer.cache[e]

        self.experts = Cached(self.p, None, None)

    def step(self):
        st = {}
        self.oracle.forward(self.p, self.x_bits, self.logits, self.bias, self.experts, self.a1, self.a2, stats=st)
        return st["seconds"], len(self.rows)


def cpu_baseline(shape, w, tok, sample):
    r = _OracleRunner(shape, w, tok, sample)
    r.step()  # decode the touched experts (excluded from timing)
    secs, n = r.step()
    return {"value": n / secs, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{n} of the {tok.x.shape[0]} tokens (evenly spaced), fp64 numpy, expert decode excluded",
            "seconds": secs}


def run_reference(args):
    rank = _env_int("RANK", 0)
    if rank != 0:
        return
    import torch
    from synth import SHAPES, make_tokens, make_weights
    shape = SHAPES[args.config]
    dev = torch.device("cuda", _env_int("LOCAL_RANK", 0)) if torch.cuda.is_available() else torch.device("cpu")
    w = make_weights(shape, dev, seed=0)
    tok = make_tokens(shape, args.T, dev, seed=0)
    r = _OracleRunner(shape, w, tok, args.ref_sample)
    for _ in range(args.warmup):
        r.step()
    total, n = 0.0, 0
    t0 = time.perf_counter()
    for _ in range(args.steps):
        s, k = r.step()
        total += s
        n += k
    wall = time.perf_counter() - t0
    v = n / total
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT,
            "n_gpus": _env_int("WORLD_SIZE", 1), "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOADS.get(args.config, args.config), "T": args.T,
                       "sample_tokens_per_step": len(r.rows)},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                             "sample": f"{len(r.rows)} of {args.T} tokens per step, fp64 numpy, expert decode excluded"},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "wall_s": wall}
    print(json.dumps(line), flush=True)


def measure_tensor_peaks():
    """Dense GEMM throughput of the vendor library on this GPU, for the roofline
    denominators: cuBLASLt bf16 and e4m3 (per-tensor scales) n x n x n GEMMs,
    CUDA events around 20 back-to-back launches after 5 warm-up ones."""
    import torch
    dev = torch.device("cuda:0")
    res = {}
    for n in (8192, 16384):
        a8 = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn)
        b8 = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn).t()
        one = torch.ones((), device=dev)
        a16 = torch.randn(n, n, device=dev, dtype=torch.bfloat16)
        b16 = torch.randn(n, n, device=dev, dtype=torch.bfloat16)
        row = {}
        for name, fn in (("e4m3", lambda: torch._scaled_mm(a8, b8, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)),
                         ("bf16", lambda: a16 @ b16)):
            for _ in range(5):
                fn()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(20):
                fn()
            e1.record()
            torch.cuda.synchronize()
            row[name + "_tflops"] = 2.0 * n ** 3 / (e0.elapsed_time(e1) / 20 / 1e3) / 1e12
        res[str(n)] = row
    print(json.dumps({"tensor_peaks": res}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default=CONFIG_NAME)
    ap.add_argument("--T", type=int, default=4096)
    ap.add_argument("--E", type=int, default=0, help="override the expert count (profiling small cases)")
    ap.add_argument("--no-sweep", dest="sweep", action="store_false")
    ap.add_argument("--tuning", default=None,
                    help="planner overrides as JSON (moe_set_tuning), e.g. '{\"full_box\": 1}'; for experiments")
    ap.add_argument("--sweep-configs", default=None,
                    help="comma-separated further workloads to sweep in the same run (default with the "
                         "Mixtral headline: qwen2,dsv3,dsv3_paired,scout,qwen2_tp4,dsv3_tp8,tiny; else none)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-sample", type=int, default=4096)
    ap.add_argument("--ref-sample", type=int, default=16)
    ap.add_argument("--measure-tensor-peaks", action="store_true",
                    help="print the library's dense bf16 / e4m3 GEMM throughput and exit")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.sweep_configs is None:
        args.sweep_configs = "qwen2,dsv3,dsv3_paired,scout,qwen2_tp4,dsv3_tp8,tiny" if args.config == CONFIG_NAME else ""
    args.sweep_configs = [c for c in args.sweep_configs.split(",") if c]
    if args.measure_tensor_peaks:
        measure_tensor_peaks()
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
