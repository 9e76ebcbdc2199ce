"""Benchmark of the fused MoE expert forward on GB300.

Workload: the Mixtral-8x7B-shaped prefill layer (M=4096 tokens, H=4096,
I=14336, E=8, top-2, bf16; weights N(0, 0.02), router softmax top-2 of N(0,1)
logits), seeded synthetic inputs resident in HBM.  One step = one pass of the
whole path over the batch: routing + permute, grouped GEMM1 with the fused
SiLU-and-mul, grouped GEMM2, weighted unpermute-reduce -- the same launches
fused_experts makes, issued through the staged C-ABI entry points so CUDA
events can bracket each stage on the launching stream.  The fused_experts
call itself is timed as well (fused_call_ms).  The weights (2.82 GB) are far
larger than L2, so no flush is needed between steps.

The same run then measures the other workloads the same way, each with its
own inputs, and reports them under "workloads": Mixtral-shaped decode (M=64),
the DeepSeek-class FP8 layer (M=8192, H=7168, I=2048, E=256, top-8, 128x128
fp32 block scales, skewed routing), the same shape with MXFP4 W4A8 weights
(M=2048, uniform routing) and with MXFP8 1x32 weights; plus a dense e4m3
GEMM probe (torch._scaled_mm) as a measured FP8 denominator beside the
nominal one.  --no-extra times the --workload alone.

Metric: routed tokens/s (M * top-k per second), whole job over all ranks.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
       torchrun ... bench.py --gpus N ...  (replicas: one independent layer per GPU)

--impl reference times the fp64 CPU oracle (oracle/, test infrastructure) on
the host cores, one token of the same workload per step.
"""
from __future__ import annotations

import argparse
import csv
import io
import json
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused-MoE fwd routed tokens/s; % of tensor-core/HBM roofline (1 GB300)"
UNIT = "routed tokens/s"
WORKLOAD = "mixtral"


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p["bf16_tflops_sustained"], "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


_LABEL = {"mixtral": "Mixtral-8x7B-shaped prefill", "decode": "Mixtral-8x7B-shaped decode",
          "dsfp8": "DeepSeek-class FP8 (128x128 block scales, skewed routing)",
          "mxfp4": "DeepSeek-class MXFP4 W4A8", "mxfp8": "DeepSeek-class MXFP8 (1x32)",
          "tiny": "tiny"}


def _workload(args):
    from moe_synth import get_config
    # the batched layout runs the decode workload's rows (reference arm: the
    # same per-row expert MLPs through the oracle)
    cfg = get_config("decode" if args.workload == "decode_batched" else args.workload)
    if args.tokens:
        cfg = cfg.with_(M=args.tokens, name=f"{cfg.name}-M{args.tokens}")
    if args.experts:
        cfg = cfg.with_(E=args.experts, name=f"{cfg.name}-E{args.experts}")
    return cfg


def _config_dict(cfg, n):
    base = cfg.name.split("-")[0]
    return {"workload": f"{cfg.name}: {_LABEL.get(base, base)} M={cfg.M} H={cfg.H} "
                        f"I={cfg.I} E={cfg.E} top-{cfg.topk} {cfg.quant}",
            "M": cfg.M, "H": cfg.H, "I": cfg.I, "E": cfg.E, "topk": cfg.topk,
            "block_size": cfg.block_size, "routed_tokens_per_gpu": cfg.R,
            "quant": cfg.quant, "act_scale_fmt": cfg.act_scale_fmt,
            "l2": "inputs larger than L2 (expert weights >= 2.8 GB per GPU), no flush",
            "parallelism": f"replicas x{n}"}


class ClockSampler:
    """nvidia-smi samples (200 ms) while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                self.out = ""
        return False

    def summary(self, under_load_frac=0.5):
        if self.proc is None or not getattr(self, "out", ""):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        rows = [r for r in csv.reader(io.StringIO(self.out)) if len(r) >= 9]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = sorted(float(r[1]) for r in rows)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[j] for r in rows for j in range(4)
                          if r[5 + j].strip().lower() == "active"})
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": float(rows[0][2]),
                "samples": len(rows), "power_w_max": max(float(r[3]) for r in rows),
                "reasons": reasons}


def _gpu_id(dev):
    import torch
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return str(dev)


def max_over_ranks(values, world, device="cpu"):
    """Element-wise maximum of a list of floats over all ranks (the job's
    time is its slowest rank's); a no-op for one rank."""
    import torch
    import torch.distributed as dist
    t = torch.tensor(values, dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# --------------------------------------------------------------- CPU oracle
def _oracle_arrays(d, cfg):
    """Host copies of the inputs for the oracle (setup, outside any timed
    region); bf16 weights are converted to fp64 once here."""
    import numpy as np
    f = (lambda t: None if t is None else
         (t.float().cpu().numpy() if t.dtype.is_floating_point else t.cpu().numpy()))
    # the oracle takes the weight scales as generated (not a prepacked copy)
    a = dict(x=f(d["x"]), topk_ids=f(d["topk_ids"]), topk_weights=f(d["topk_weights"]),
             w13=f(d["w13"]), w2=f(d["w2"]), w13_scale=f(d.get("w13_scale_raw", d["w13_scale"])),
             w2_scale=f(d.get("w2_scale_raw", d["w2_scale"])))
    if cfg.quant == "bf16":
        a["w13"] = a["w13"].astype(np.float64)
        a["w2"] = a["w2"].astype(np.float64)
    return a


def _time_oracle(arrs, tokens, cfg):
    from oracle import experts
    t0 = time.perf_counter()
    experts.fused_experts_per_token(**arrs, tokens=tokens, quant=cfg.quant,
                                    act_scale_fmt=cfg.act_scale_fmt,
                                    apply_router_weight_on_input=cfg.apply_router_weight_on_input)
    return time.perf_counter() - t0


_KERNEL_SOURCES = {
    "bf16": ["gemm_bf16.cu", "moe_common.cuh", "tile_sched.cuh"],
    "bf16_2sm": ["gemm_bf16_2sm.cu", "moe_common.cuh", "tile_sched.cuh"],
    "fp8": ["gemm_fp8.cu", "moe_common.cuh", "tile_sched.cuh", "e4m3_pack.cuh"],
    "mxfp4": ["gemm_mxfp4.cu", "mx_common.cuh", "moe_common.cuh", "tile_sched.cuh",
              "e4m3_pack.cuh"],
    "mxfp8": ["gemm_mxfp4.cu", "mx_common.cuh", "moe_common.cuh", "tile_sched.cuh",
              "e4m3_pack.cuh"],
}


def gemm1_kernel(cfg):
    """(source key, kernel label) of the GEMM1 launch the library picks for cfg:
    the bf16 GEMMs run on SM pairs once the experts average two 128-row blocks."""
    if cfg.quant == "fp8":
        return "fp8", "k_ggemm_fp8 (GEMM1)"
    if cfg.quant == "mxfp4":
        return "mxfp4", "k_ggemm_mxfp4<fused act + e4m3 quant> (GEMM1)"
    if cfg.quant == "mxfp8":
        return "mxfp8", "k_ggemm_mxfp4<MX8, fused act + 1x32 quant> (GEMM1, e4m3 weights)"
    if cfg.M * cfg.topk >= 2 * 128 * cfg.E:
        return "bf16_2sm", "k_ggemm_bf16_2sm<fused SiLU-and-mul> (GEMM1, SM pairs)"
    return "bf16", "k_ggemm_bf16<fused SiLU-and-mul> (GEMM1)"


def kernel_source_sha(kind):
    """sha256 over the sources of the GEMM kernel `kind` (a key of _KERNEL_SOURCES)."""
    import hashlib
    h = hashlib.sha256()
    for f in _KERNEL_SOURCES[kind]:
        with open(os.path.join(ROOT, "mixture_experts_ffn_align_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def _traffic(cfg):
    """DRAM bytes (read + write) per GEMM1 launch from the committed ncu record
    in profiles/gemm1_dram_traffic.json, if it was taken on this workload with
    the current kernel sources; else None."""
    try:
        with open(os.path.join(ROOT, "profiles", "gemm1_dram_traffic.json")) as f:
            recs = json.load(f)
    except Exception:
        return None
    kind = gemm1_kernel(cfg)[0]
    for r in recs:
        if (r.get("kernel") == kind and r.get("workload") == cfg.name
                and r.get("source_sha") == kernel_source_sha(kind)):
            return r["dram_bytes_per_launch"]
    return None


def gemm_bytes(cfg, S):
    """Algorithmic DRAM bytes of one launch of each grouped GEMM, with S the
    used rows of the padded layout: the weights and their scales read once,
    the used activation rows (and their scales) read once, the output written
    once -- GEMM1 writes z (the fused activation; bf16, or e4m3 codes + fp32
    scales) except in the FP8-block mode, where it writes H1 (bf16); GEMM2
    reads z and writes Y2 (bf16)."""
    E, H, I, q = cfg.E, cfg.H, cfg.I, cfg.quant
    wb = {"bf16": 2, "fp8": 1, "mxfp4": 0.5, "mxfp8": 1}[q]
    ab = 2 if q == "bf16" else 1
    g = 32 if q == "mxfp8" else 128

    def wscales(N, K):
        if q == "fp8":
            return E * (N // 128) * (K // 128) * 4
        return E * N * (K // 32) if q in ("mxfp4", "mxfp8") else 0

    def act(rows, K):
        return rows * K * ab + (rows * (K // g) * 4 if q != "bf16" else 0)

    w13 = E * 2 * I * H * wb + wscales(2 * I, H)
    w2 = E * H * I * wb + wscales(H, I)
    out1 = S * 2 * I * 2 if q == "fp8" else act(S, I)
    return {"gemm1": w13 + act(S, H) + out1, "gemm2": w2 + act(S, I) + S * H * 2,
            "w13": w13, "w2": w2}


def _gemm1_roofline(cfg, peaks, peak, ratio, flops, nbytes, w13_bytes, ms):
    """Roofline object of GEMM1: tensor-bound when its FLOPs take at least as
    long at the tensor peak as its algorithmic bytes at the HBM peak, else
    HBM-bound (decode, and the E = 256 layers whose weights outweigh their
    FLOPs)."""
    t_flop = flops / (peak * 1e12)
    t_mem = nbytes / (peaks["hbm_gbs"] * 1e9)
    tflops = flops / (ms * 1e-3) / 1e12
    gbs = nbytes / (ms * 1e-3) / 1e9
    common = {"kernel": gemm1_kernel(cfg)[1], "traffic": _traffic(cfg),
              "tensor_frac": tflops / peak, "hbm_frac": gbs / peaks["hbm_gbs"],
              "weight_hbm_frac": w13_bytes / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"]}
    if t_flop >= t_mem:
        return {"bound": "tensor", "achieved": tflops, "peak": peak, "unit": "TFLOP/s",
                "frac": tflops / peak,
                "peak_source": f"bf16 x {ratio:g} ({peaks['source']})",
                "algorithmic_per_launch": f"2*R*H*2I = {flops:.4e} FLOP", **common}
    return {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": gbs / peaks["hbm_gbs"], "peak_source": f"hbm_gbs ({peaks['source']})",
            "algorithmic_per_launch": f"weights + scales, used activation rows in, output out "
                                      f"= {nbytes:.4e} B", **common}


def _cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count()


def run_reference(args):
    """--impl reference: the fp64 oracle on the host cores, one token of the
    workload per step (its two routed items through their experts)."""
    import torch
    from moe_synth import make_inputs
    world, rank, _ = _dist()
    if rank != 0:
        return
    cfg = _workload(args)
    d = make_inputs(cfg, "cpu")
    arrs = _oracle_arrays(d, cfg)
    for s in range(args.warmup):
        _time_oracle(arrs, [s % cfg.M], cfg)
    total = 0.0
    for s in range(args.steps):
        total += _time_oracle(arrs, [(args.warmup + s) % cfg.M], cfg)
    routed = args.steps * cfg.topk
    value = routed / total
    sample = (f"{args.steps} steps x 1 token ({cfg.topk} routed items) of the {cfg.name} "
              "workload, per-token fp64 oracle, weights converted once outside timing")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": _config_dict(cfg, 1),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": _cores(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


# ------------------------------------------------------------------ our arm
def _stage_plan(moe, p, cfg, d, b, stream):
    """The launches of one step, as (name, callable) pairs, in the order
    fused_experts issues them."""
    import torch
    x, ids, wts, w13, w2 = d["x"], d["topk_ids"], d["topk_weights"], d["w13"], d["w2"]
    q = cfg.quant != "bf16"
    plan = [("align_permute", lambda: moe.moe_align_permute(
        p, x, ids, wts if cfg.apply_router_weight_on_input else None, b["sorted_ids"],
        b["block_expert_ids"], b["expert_offsets"], b["num_post_padded"], b["inv_perm"],
        b["x_perm"], b["x_perm_scale"], b["align_ws"], stream=stream))]
    if not q:
        plan.append(("gemm1_silu_mul", lambda: moe.grouped_gemm_w13(
            p, b["x_perm"], None, w13, None, b["block_expert_ids"], b["num_post_padded"],
            b["z"], None, fuse_act=True, stream=stream)))
    elif cfg.quant in ("mxfp4", "mxfp8"):
        # the block-scaled GEMM1 writes the quantised activation itself
        plan.append(("gemm1_act_quant", lambda: moe.grouped_gemm_w13(
            p, b["x_perm"], b["x_perm_scale"], w13, d["w13_scale"], b["block_expert_ids"],
            b["num_post_padded"], b["z"], b["z_scale"], fuse_act=True, stream=stream)))
    else:
        plan.append(("gemm1", lambda: moe.grouped_gemm_w13(
            p, b["x_perm"], b["x_perm_scale"], w13, d["w13_scale"], b["block_expert_ids"],
            b["num_post_padded"], b["h1"], stream=stream)))
        plan.append(("act_mul_quant", lambda: moe.act_mul_quant(
            p, b["h1"], b["num_post_padded"], b["z"], b["z_scale"], stream=stream)))
    splits = moe.moe_gemm2_splits(p)
    if splits > 1 and not cfg.apply_router_weight_on_input:
        # decode-sized bf16: GEMM2 in K slices over all SMs (as fused_experts)
        b["partial"] = torch.empty(moe.moe_gemm2_partial_bytes(p, splits) // 4,
                                   dtype=torch.float32, device=x.device)
        plan.append(("gemm2_split_k", lambda: moe.grouped_gemm_w2_split(
            p, b["z"], w2, b["block_expert_ids"], b["num_post_padded"], b["sorted_ids"],
            splits, b["partial"], stream=stream)))
        plan.append(("unpermute_reduce", lambda: moe.unpermute_reduce_split(
            p, b["partial"], splits, b["inv_perm"], wts, b["y"], stream=stream)))
        return plan
    plan.append(("gemm2", lambda: moe.grouped_gemm_w2(
        p, b["z"], b["z_scale"], w2, d["w2_scale"], b["block_expert_ids"],
        b["num_post_padded"], b["y2"], stream=stream)))
    plan.append(("unpermute_reduce", lambda: moe.unpermute_reduce(
        p, b["y2"], b["inv_perm"], wts, b["y"], stream=stream)))
    return plan


def _peak_for(peaks, q, timed_s):
    """Tensor peak of a GEMM timed over a region of timed_s seconds: the
    measured burst bf16 rate when the region is short (< 1 s: the clocks do
    not reach the power cap's steady state), else the sustained one; FP8
    contractions take 2 x that (the recipe's nominal FP8 / bf16 ratio)."""
    burst = timed_s < 1.0
    ratio = 2.0 if q else 1.0
    base = peaks["bf16_tflops"] if burst else peaks["bf16_tflops_sustained"]
    name = "bf16_tflops (burst)" if burst else "bf16_tflops_sustained"
    return base * ratio, ratio, f"{name} x {ratio:g} ({peaks['source']}; timed region " \
                                f"{timed_s:.3f} s)"


def fp8_probe(dev):
    """Dense e4m3 GEMM throughput of torch._scaled_mm (cuBLASLt), 8192^3, best
    of 10 launches timed with CUDA events: a measured FP8 denominator shown
    beside the nominal 2 x bf16 one.  None where the call is unavailable."""
    import torch
    try:
        n = 8192
        g = torch.Generator(device=dev).manual_seed(0)
        a = torch.randn(n, n, device=dev, generator=g).to(torch.float8_e4m3fn)
        b = torch.randn(n, n, device=dev, generator=g).to(torch.float8_e4m3fn).t()
        one = torch.ones((), device=dev)
        f = lambda: torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
        for _ in range(3):
            f()
        best = None
        for _ in range(10):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            f()
            e1.record()
            e1.synchronize()
            ms = e0.elapsed_time(e1)
            best = ms if best is None else min(best, ms)
        return {"tflops": 2.0 * n ** 3 / (best * 1e-3) / 1e12, "ms": best,
                "how": "torch._scaled_mm e4m3 x e4m3 -> bf16, 8192^3, best of 10 (CUDA events)"}
    except Exception as ex:       # noqa: BLE001 -- reported, not fatal
        return {"tflops": None, "error": str(ex)[:200]}


def _measure(moe, cfg, args, dev, world, rank, full, fp8_tflops=None):
    """One workload: inputs generated on the device, W warm-up steps, K timed
    steps of the stage plan (CUDA events per stage on the launching stream),
    then the fused_experts call and the end-to-end host-buffer entry.  With
    ``full`` also the router timing.  Returns (rank 0's record, ms_per_step)."""
    import torch
    import torch.distributed as dist
    from moe_synth import make_inputs

    if rank > 0:
        cfg = cfg.with_(seed=cfg.seed + 100 * rank)
    d = make_inputs(cfg, dev)
    p = moe.Problem.from_config(cfg)
    if cfg.quant in ("mxfp4", "mxfp8") and not args.raw_scales:
        # load time, outside any timed region: the weight scales rewritten once
        # into the block-scaled MMA's operand layout (moe_prepack_weights)
        s13 = torch.empty(moe.moe_prepacked_scale_bytes(p, 0), dtype=torch.uint8, device=dev)
        s2 = torch.empty(moe.moe_prepacked_scale_bytes(p, 1), dtype=torch.uint8, device=dev)
        moe.moe_prepack_weights(p, d["w13_scale"], d["w2_scale"], s13, s2)
        d["w13_scale_raw"], d["w2_scale_raw"] = d["w13_scale"], d["w2_scale"]
        d["w13_scale"], d["w2_scale"] = s13, s2
        p = moe.Problem.from_config(cfg, weight_scales_prepacked=True)
    b = moe.stage_buffers(p, dev)
    ws = torch.empty(moe.moe_workspace_bytes(p), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    x, ids, wts, w13, w2 = d["x"], d["topk_ids"], d["topk_weights"], d["w13"], d["w2"]
    w13s, w2s = d["w13_scale"], d["w2_scale"]
    plan = _stage_plan(moe, p, cfg, d, b, stream)
    # routing (one CTA, or hist/scan/scatter) + permute, then one launch per
    # remaining stage
    launches_per_step = moe.moe_align_permute_launches(p) + (len(plan) - 1)

    def barrier():
        torch.cuda.synchronize(dev)
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    for _ in range(args.warmup):
        for _, fn in plan:
            fn()
    st = moe.moe_sync_status(stream)
    if st != 0:
        raise RuntimeError(f"device status {moe.moe_status_string(st)}")

    n_st = len(plan)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(n_st + 1)]
           for _ in range(args.steps)]
    barrier()
    with ClockSampler(_gpu_id(dev)) as clk:
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for s in range(args.steps):
            ev = evs[s]
            for i, (_, fn) in enumerate(plan):
                ev[i].record(stream)
                fn()
            ev[n_st].record(stream)
        end.record(stream)
        barrier()
    elapsed_ms = start.elapsed_time(end)
    if moe.moe_sync_status(stream) != 0:
        raise RuntimeError("device error in the timed region")
    stage_ms = {name: sum(e[i].elapsed_time(e[i + 1]) for e in evs) / args.steps
                for i, (name, _) in enumerate(plan)}
    S_used = int(b["num_post_padded"].item())     # after the timed region

    # the fused_experts call itself (same kernels, one entry point)
    f_steps = max(3, args.steps // 4)
    for _ in range(3):
        moe.fused_experts(p, x, w13, w13s, w2, w2s, wts, ids, b["y"], ws, stream=stream)
    barrier()
    fs, fe = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    fs.record(stream)
    for _ in range(f_steps):
        moe.fused_experts(p, x, w13, w13s, w2, w2s, wts, ids, b["y"], ws, stream=stream)
    fe.record(stream)
    barrier()
    fused_ms = fs.elapsed_time(fe) / f_steps

    # end to end through the C ABI from pinned host buffers
    hws = torch.empty(moe.moe_host_workspace_bytes(p), dtype=torch.uint8, device=dev)
    hx, hid, hw = x.cpu().pin_memory(), ids.cpu().pin_memory(), wts.cpu().pin_memory()
    hy = torch.empty_like(hx).pin_memory()
    e_steps = max(3, args.steps // 4)
    for _ in range(3):
        moe.fused_experts_from_host(p, hx, hid, hw, hy, w13, w13s, w2, w2s, hws, stream=stream)
    barrier()
    t0 = time.perf_counter()
    for _ in range(e_steps):
        moe.fused_experts_from_host(p, hx, hid, hw, hy, w13, w13s, w2, w2s, hws, stream=stream)
    torch.cuda.synchronize(dev)
    e2e_s = (time.perf_counter() - t0) / e_steps
    h2d = hx.numel() * 2 + hid.numel() * 4 + hw.numel() * 4
    d2h = hy.numel() * 2
    if moe.moe_sync_status(stream) != 0:
        raise RuntimeError("device error in the e2e region")

    router = None
    if full:
        # the step before the path (not in the step): the router on logits of
        # this workload's shape, softmax + renormalise
        gen = torch.Generator(device=dev).manual_seed(cfg.seed)
        logits = torch.randn(cfg.M, cfg.E, device=dev, generator=gen)
        r_w = torch.empty(cfg.M, cfg.topk, dtype=torch.float32, device=dev)
        r_ids = torch.empty(cfg.M, cfg.topk, dtype=torch.int32, device=dev)
        for _ in range(3):
            moe.moe_topk_router(logits, cfg.topk, r_w, r_ids, stream=stream)
        barrier()
        # a launch is a few microseconds of GPU work, less than its host-side
        # call: time 20 launches captured in a CUDA graph
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):          # captured on torch's side stream
            for _ in range(20):
                moe.moe_topk_router(logits, cfg.topk, r_w, r_ids)
        graph.replay()
        barrier()
        rs, re_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        r_reps = 10
        rs.record(stream)
        for _ in range(r_reps):
            graph.replay()
        re_.record(stream)
        barrier()
        router_ms = rs.elapsed_time(re_) / (20 * r_reps)
        router_bytes = cfg.M * cfg.E * 4 + cfg.M * cfg.topk * 8
        router = {"ms": router_ms, "bytes": router_bytes,
                  "gbs": router_bytes / (router_ms * 1e-3) / 1e9,
                  "note": "moe_topk_router on [M, E] fp32 logits (softmax, renormalise); "
                          "the step before the path, not part of a step"}

    # max over ranks
    elapsed_ms, e2e_s, fused_ms = max_over_ranks([elapsed_ms, e2e_s, fused_ms], world, dev)
    ms = elapsed_ms / args.steps
    R = cfg.R
    out = None
    if rank == 0:
        peaks = _peaks()
        q = cfg.quant != "bf16"
        gemm1_flops = 2.0 * R * cfg.H * 2 * cfg.I      # padding rows not counted
        gemm2_flops = 2.0 * R * cfg.I * cfg.H
        g1 = [n for n, _ in plan if n.startswith("gemm1")][0]
        g2 = [n for n, _ in plan if n.startswith("gemm2")][0]
        peak, ratio, peak_src = _peak_for(peaks, q, elapsed_ms * 1e-3)
        gb = gemm_bytes(cfg, S_used)
        g2_tf = gemm2_flops / (stage_ms[g2] * 1e-3) / 1e12
        roof = _gemm1_roofline(cfg, peaks, peak, ratio, gemm1_flops, gb["gemm1"], gb["w13"],
                               stage_ms[g1])
        roof["peak_source"] = peak_src if roof["bound"] == "tensor" else roof["peak_source"]
        sust = peaks["bf16_tflops_sustained"] * ratio
        roof["tensor_frac_vs_sustained"] = roof["tensor_frac"] * peak / sust
        if q and fp8_tflops:
            roof["tensor_frac_vs_fp8_probe"] = roof["tensor_frac"] * peak / fp8_tflops
        out = {
            "metric": METRIC, "value": world * R / (ms * 1e-3), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": {"bf16": "bf16", "fp8": "e4m3 (fp32 accumulate)",
                      "mxfp4": "e2m1 x e4m3", "mxfp8": "e4m3 x e4m3 (E8M0 / 32)"}[cfg.quant],
            "data": "synthetic (seeded; random-init weights)",
            "config": _config_dict(cfg, world),
            "tflops": (gemm1_flops + gemm2_flops) / (ms * 1e-3) / 1e12,
            "stages_ms": stage_ms,
            "fused_call_ms": fused_ms,
            "roofline": roof,
            "gemm2_roofline": {"kernel": g2, "achieved": g2_tf, "frac": g2_tf / peak,
                               "hbm_frac": gb["gemm2"] / (stage_ms[g2] * 1e-3) / 1e9 /
                               peaks["hbm_gbs"],
                               "weight_hbm_frac": gb["w2"] / (stage_ms[g2] * 1e-3) / 1e9 /
                               peaks["hbm_gbs"]},
            "used_rows": S_used,
            "e2e": {"value": world * R / e2e_s, "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_s * 1e3,
                    "path": "fused_experts_from_host on pinned host buffers: topk ids/weights "
                            "copied in; x read and y written in place in host memory by the "
                            "permute and reduce kernels (each row once, over the host link)"},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clk.summary(),
        }
        if router is not None:
            out["router"] = router
        if world == 1 and full and not args.no_cpu_baseline:
            arrs = _oracle_arrays(d, cfg)
            t2 = _time_oracle(arrs, [0, 1], cfg)   # also warms the BLAS threads
            # about 15 s of CPU work, at least 4 tokens
            n_tok = int(min(cfg.M - 2, max(4, round(15.0 / max(t2 / 2, 1e-3)))))
            tokens = list(range(2, 2 + n_tok))
            secs = _time_oracle(arrs, tokens, cfg)
            out["cpu_baseline"] = {
                "value": len(tokens) * cfg.topk / secs, "unit": UNIT, "cores": _cores(),
                "kind": "oracle",
                "sample": f"{len(tokens)} tokens ({len(tokens) * cfg.topk} routed items) of the "
                          f"{cfg.name} workload through the per-token fp64 oracle, weights "
                          f"decoded once outside timing; {secs:.1f} s"}
    del d, b, ws, hws
    torch.cuda.empty_cache()
    return out


# the other workloads measured in the same default run, after the headline
EXTRA_WORKLOADS = ("decode", "dsfp8", "mxfp4", "mxfp8")


def run_ours(args):
    import torch
    import torch.distributed as dist

    import mixture_experts_ffn_align_gb300 as moe

    world, rank, local = _dist()
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    moe.lib()
    moe.moe_debug_set_bf16_gemm_form(args.gemm_form)

    cfg = _workload(args)
    probe = fp8_probe(dev) if rank == 0 and world == 1 and not args.no_extra else None
    fp8_tf = probe["tflops"] if probe else None
    out = _measure(moe, cfg, args, dev, world, rank, True, fp8_tf)
    extra = {}
    if world == 1 and not args.no_extra and args.workload == WORKLOAD and not args.tokens \
            and not args.experts:
        from moe_synth import get_config
        for name in EXTRA_WORKLOADS:
            rec = _measure(moe, get_config(name), args, dev, world, rank, False, fp8_tf)
            keep = ("value", "unit", "ms_per_step", "dtype", "config", "tflops", "stages_ms",
                    "fused_call_ms", "roofline", "gemm2_roofline", "used_rows", "e2e",
                    "gpu_launches", "clocks")
            extra[name] = {k: rec[k] for k in keep}
    if rank == 0:
        if extra:
            out["workloads"] = extra
        if probe is not None:
            out["fp8_probe"] = probe
        print(json.dumps(out), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_batched(args):
    """The batched expert layout at the Mixtral-shaped decode size: x [E, T, H]
    with the decode routing's per-expert counts, T = 128; one step = one
    fused_experts_batched call (count-to-block kernel, GEMM1 with SiLU-and-mul,
    GEMM2), counts read on the device."""
    import torch
    import torch.distributed as dist

    import mixture_experts_ffn_align_gb300 as moe
    from moe_synth import get_config, make_inputs

    world, rank, local = _dist()
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    moe.lib()
    cfg = get_config("decode")
    if rank > 0:
        cfg = cfg.with_(seed=cfg.seed + 100 * rank)
    d = make_inputs(cfg, dev)
    counts = torch.bincount(d["topk_ids"].reshape(-1).long(), minlength=cfg.E)
    T = 128 * max(1, -(-int(counts.max()) // 128))
    cnt = counts.to(torch.int32)
    g = torch.Generator(device=dev).manual_seed(cfg.seed)
    x_b = torch.randn(cfg.E, T, cfg.H, device=dev, generator=g).to(torch.bfloat16)
    y_b = torch.empty_like(x_b)
    p = moe.Problem.from_config(cfg)
    ws = torch.empty(moe.moe_batched_workspace_bytes(p, T), dtype=torch.uint8, device=dev)
    expected_m = (cfg.M * cfg.topk + cfg.E) // cfg.E      # the pages' expected_m, one dispatcher
    stream = torch.cuda.current_stream(dev)
    routed = int(counts.sum())

    def step():
        moe.fused_experts_batched(p, x_b, cnt, d["w13"], None, d["w2"], None, y_b, ws,
                                  expected_m=expected_m, stream=stream)

    def barrier():
        torch.cuda.synchronize(dev)
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    for _ in range(args.warmup):
        step()
    if moe.moe_sync_status(stream) != 0:
        raise RuntimeError("device error in the warm-up")
    barrier()
    with ClockSampler(_gpu_id(dev)) as clk:
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for _ in range(args.steps):
            step()
        end.record(stream)
        barrier()
    elapsed_ms = start.elapsed_time(end)
    if moe.moe_sync_status(stream) != 0:
        raise RuntimeError("device error in the timed region")
    # end to end: the layout and counts from pinned host memory, the result back
    hx = x_b.cpu().pin_memory()
    hc = cnt.cpu().pin_memory()
    hy = torch.empty_like(hx).pin_memory()
    e_steps = max(3, args.steps // 4)

    def e2e_step():
        x_b.copy_(hx, non_blocking=True)
        cnt.copy_(hc, non_blocking=True)
        step()
        hy.copy_(y_b, non_blocking=True)

    for _ in range(3):
        e2e_step()
    barrier()
    t0 = time.perf_counter()
    for _ in range(e_steps):
        e2e_step()
    torch.cuda.synchronize(dev)
    e2e_s = (time.perf_counter() - t0) / e_steps
    elapsed_ms, e2e_s = max_over_ranks([elapsed_ms, e2e_s], world, dev)
    ms = elapsed_ms / args.steps
    if rank == 0:
        peaks = _peaks()
        used = int((counts > 0).sum())
        wbytes = used * 3 * cfg.I * cfg.H * 2          # w13 + w2 of the experts with tokens
        gbs = wbytes / (ms * 1e-3) / 1e9
        out = {
            "metric": METRIC, "value": world * routed / (ms * 1e-3), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded; random-init weights)",
            "config": {"workload": f"decode_batched: Mixtral-8x7B-shaped decode in the batched "
                                   f"layout [E={cfg.E}, T={T}, H={cfg.H}], I={cfg.I}, per-expert "
                                   f"counts of M={cfg.M} top-{cfg.topk} routing",
                       "E": cfg.E, "T": T, "H": cfg.H, "I": cfg.I, "routed_tokens_per_gpu": routed,
                       "expected_m": expected_m, "quant": "bf16",
                       "l2": "inputs larger than L2 (expert weights 2.8 GB per GPU), no flush",
                       "parallelism": f"replicas x{world}"},
            "roofline": {"bound": "hbm", "kernel": "fused_experts_batched step (the weights of "
                                                   "every expert with tokens, once)",
                         "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / peaks["hbm_gbs"], "traffic": None,
                         "peak_source": f"hbm_gbs ({peaks['source']})",
                         "algorithmic_per_launch": f"3*I*H*2 B x {used} experts = {wbytes:.4e} B"},
            "e2e": {"value": world * routed / e2e_s, "unit": UNIT,
                    "h2d_bytes_per_step": hx.numel() * 2 + hc.numel() * 4,
                    "d2h_bytes_per_step": hy.numel() * 2, "ms_per_step": e2e_s * 1e3},
            "gpu_launches": 3 * args.steps,
            "clocks": clk.summary(),
        }
        if world == 1 and not args.no_cpu_baseline:
            # the same per-row expert MLPs: the decode workload's tokens through
            # the per-token oracle (each routed item is one row of the layout)
            arrs = _oracle_arrays(d, cfg)
            t2 = _time_oracle(arrs, [0, 1], cfg)
            n_tok = int(min(cfg.M - 2, max(4, round(15.0 / max(t2 / 2, 1e-3)))))
            tokens = list(range(2, 2 + n_tok))
            secs = _time_oracle(arrs, tokens, cfg)
            out["cpu_baseline"] = {
                "value": len(tokens) * cfg.topk / secs, "unit": UNIT, "cores": _cores(),
                "kind": "oracle",
                "sample": f"{len(tokens)} tokens ({len(tokens) * cfg.topk} routed rows) of the "
                          f"decode workload through the per-token fp64 oracle, weights decoded "
                          f"once outside timing; {secs:.1f} s"}
        print(json.dumps(out), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=WORKLOAD,
                    choices=["mixtral", "decode", "dsfp8", "mxfp4", "mxfp8", "tiny",
                             "decode_batched"])
    ap.add_argument("--tokens", type=int, default=0,
                    help="override M (smaller cases for profiling captures)")
    ap.add_argument("--experts", type=int, default=0,
                    help="override E (smaller cases for profiling captures)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--gemm-form", choices=["auto", "single", "pairs"], default="auto",
                    help="force the bf16 / FP8-block GEMM form (profiling comparisons)")
    ap.add_argument("--raw-scales", action="store_true",
                    help="MXFP4 / MXFP8: use the weight scales as generated instead of "
                         "prepacked ones")
    ap.add_argument("--no-extra", action="store_true",
                    help="time only --workload (no FP8 probe, no other workloads)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.workload == "decode_batched":
        run_batched(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
