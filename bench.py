"""Throughput of the MoE-layer forward pass on B300 (one JSON line on stdout).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one pass of the whole hot path over one batch: router logits ->
routing -> dispatch layout -> permute -> grouped SwiGLU FFN -> combine, each a
call of the C library on the current stream, with CUDA events between the
calls so every stage is timed live inside the timed region.  Inputs are
resident in HBM before timing starts; the per-step working set (22.5 GB of
expert weights at the DeepSeek-V3 shape) is far larger than the 126 MB L2.

``e2e`` repeats the measurement through moe_layer_forward_host: the host->device
copy of x from pinned memory, the layer and the device->host copy of y are all
inside its timed region, every step; two streams take alternate steps so one
step's copies overlap the other's compute.

Under torchrun (N > 1) every rank runs an independent replica of the layer
(the path has no data exchange on one node: the expert-parallel traffic is
computed as the n_ij matrix only); the time is the max over ranks and the value
counts the tokens of all ranks.

``--impl reference`` times the CPU oracle instead (rank 0 only), on a bounded
sample of the same workload per step.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s at DeepSeek-V3 shape; permute GB/s & GEMM % of peak"
# DRAM bytes (read + write) of the grouped FFN's two launches over its
# algorithmic bytes, from one ncu capture of the 32-expert DeepSeek-V3-shaped
# layer (deepseek_v3_e32_T512: 2.9703 GB measured / 2.9696 GB algorithmic, the
# kernel with separate weight and token rings).  Both scale with the touched
# experts and kept rows, so a full launch's traffic is this ratio times its
# algorithmic bytes.  Re-measure whenever the kernel changes.
FFN_TRAFFIC_RATIO = 1.0002
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def workload_config(w):
    return {"workload": w.name, "T": w.T, "h": w.h, "E": w.E, "K": w.K, "I": w.I, "shared_I": w.shared_I,
            "n_redundant": w.n_redundant, "fp8": w.fp8,
            "score": w.score,
            "n_groups": w.n_groups, "topk_groups": w.topk_groups, "capacity": w.capacity, "ep_size": w.ep_size,
            "l2": "inputs larger than L2: every step streams all touched expert weights (GBs) through the 126 MB L2",
            "parallelism": "replicas"}


# ---------------------------------------------------------------------------- ranks
def max_over_ranks(value: float, world: int, device) -> float:
    """The largest `value` over all ranks (one scalar all-reduce; timing only)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_rank: int, world: int, steps: int, max_ms: float) -> float:
    """Whole-job tokens/s: every rank's tokens over the slowest rank's time."""
    return world * tokens_per_rank * steps / (max_ms / 1e3)


# ---------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, path: str = None):
        """Samples GPU `index` every 100 ms into `path` (a temporary file if None)."""
        self.index = index
        self.proc = None
        if path is None:
            import tempfile
            fd, path = tempfile.mkstemp(prefix=f"moe_clocks_{index}_", suffix=".csv")
            os.close(fd)
        self.path = path

    def __enter__(self):
        os.makedirs(os.path.dirname(os.path.abspath(self.path)), exist_ok=True)
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            self.proc.wait(timeout=10)
            self.fh.close()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), float(parts[2]), parts[4:8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        loaded = [r for r in rows if r[2] > 300.0] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in loaded for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": max(r[1] for r in rows),
                "samples": len(loaded), "power_w_max": max(r[2] for r in rows), "reasons": reasons}


# ---------------------------------------------------------------------------- our arm
def run_ours(args, rank, world, local_rank):
    import numpy as np
    import torch
    import torch.distributed as dist

    import expert_dispatch_bias_b300 as moe
    from synth import device, workloads

    torch.cuda.set_device(local_rank)
    w = workloads.ALL.get(args.workload) or workloads.EXTRA[args.workload]
    cfg = moe.config_from(w)
    inp = device.layer_inputs(w)
    dt = inp["x"].dtype
    R = moe.moe_rows(cfg)
    T, K, E, N = w.T, w.K, w.E, w.ep_size
    i32 = dict(dtype=torch.int32, device="cuda")
    logits = torch.empty(T, E, device="cuda")
    ids = torch.empty(T, K, **i32)
    wts = torch.empty(T, K, device="cuda")
    lay = moe.alloc_layout(cfg)
    ws_layout = moe.alloc_workspace(cfg, moe.MOE_OP_LAYOUT)
    ws_ffn = moe.alloc_workspace(cfg, moe.MOE_OP_FFN)
    ws_logits = moe.alloc_workspace(cfg, moe.MOE_OP_LOGITS)
    xp = torch.empty(R, w.h, dtype=dt, device="cuda")
    yp = torch.empty(R, w.h, dtype=dt, device="cuda")
    y = torch.empty(T, w.h, dtype=dt, device="cuda")
    stream = torch.cuda.current_stream()
    shared = w.shared_I > 0  # the whole block: routed layer plus the shared expert
    if shared:
        ys = torch.empty(T, w.h, dtype=dt, device="cuda")
        ws_shared = moe.alloc_workspace(cfg, moe.MOE_OP_SHARED)
    eplb = w.n_redundant > 0  # replicas: plan once from this batch's logical expert loads (not timed)
    if eplb:
        moe.moe_router_logits(cfg, inp["x"], inp["w_r"], inp["logit_offset"], logits, ws_logits)
        moe.moe_route(cfg, logits, inp["sel_bias"], ids, wts)
        counts = torch.bincount(ids.view(-1).long(), minlength=E).cpu().numpy()
        plan_h = moe.moe_eplb_plan(E, N, w.n_redundant, counts)
        plan = {k: torch.from_numpy(v).cuda() for k, v in plan_h.items() if k != "rank_load"}
        pids = torch.empty(T, K, **i32)
    fp8 = w.fp8  # FP8 experts: weights quantised once here (not timed)
    if fp8:
        q13 = torch.empty(inp["w13"].shape, dtype=torch.uint8, device="cuda")
        s13 = torch.empty(E, 2 * w.I, dtype=torch.float32, device="cuda")
        q2 = torch.empty(inp["w2"].shape, dtype=torch.uint8, device="cuda")
        s2 = torch.empty(E, w.h, dtype=torch.float32, device="cuda")
        moe.moe_quantize_fp8(inp["w13"].view(-1, w.h), q13.view(-1, w.h), s13.view(-1))
        moe.moe_quantize_fp8(inp["w2"].view(-1, w.I), q2.view(-1, w.I), s2.view(-1))
        del inp["w13"], inp["w2"]
        torch.cuda.synchronize()
        xq = torch.empty(R, w.h, dtype=torch.uint8, device="cuda")
        sxp = torch.empty(R, dtype=torch.float32, device="cuda")
        ws_ffn = moe.alloc_workspace(cfg, moe.MOE_OP_FFN_FP8)
    # `--fused-permute`: the FFN gathers its rows from x (moe_grouped_ffn_gather)
    # instead of the layer's explicit permute
    gather = args.fused_permute and not fp8 and not eplb
    stages = (("logits", "route") + (("eplb_map",) if eplb else ()) + ("layout",)
              + (("ffn",) if gather else ("permute", "ffn")) + (("shared",) if shared else ()) + ("combine",))
    n_ev = len(stages) + 1

    def step(ev=None):
        n = [0]

        def rec():
            if ev is not None:
                ev[n[0]].record(stream)
            n[0] += 1

        rec()
        moe.moe_router_logits(cfg, inp["x"], inp["w_r"], inp["logit_offset"], logits, ws_logits)
        rec()
        moe.moe_route(cfg, logits, inp["sel_bias"], ids, wts)
        rec()
        lids = ids
        if eplb:
            moe.moe_eplb_map(cfg, ids, plan["rep_offsets"], plan["rep_phys"], pids)
            rec()
            lids = pids
        moe.moe_dispatch_layout(cfg, lids, lay.counts, lay.kept, lay.offsets, lay.slot, lay.row_src, lay.n_ij,
                                lay.rank_bytes, lay.stats, ws_layout)
        rec()
        if fp8:
            moe.moe_permute_fp8(cfg, inp["x"], lay.slot, xq, sxp)
            rec()
        elif not gather:
            moe.moe_permute(cfg, inp["x"], lay.slot, lay.row_src, xp)
            rec()
        if fp8:
            moe.moe_grouped_ffn_fp8(cfg, xq, sxp, lay.offsets, lay.kept, q13, s13, q2, s2, yp, ws_ffn)
        elif gather:  # the permutation fused into the FFN: rows read from x through row_src
            moe.moe_grouped_ffn_gather(cfg, inp["x"], lay.row_src, lay.offsets, lay.kept, inp["w13"], inp["w2"],
                                       yp, ws_ffn)
        elif eplb:
            moe.moe_grouped_ffn_mapped(cfg, xp, lay.offsets, lay.kept, plan["phys_to_log"], inp["w13"], inp["w2"],
                                       yp, ws_ffn)
        else:
            moe.moe_grouped_ffn(cfg, xp, lay.offsets, lay.kept, inp["w13"], inp["w2"], yp, ws_ffn)
        rec()
        if shared:
            moe.moe_shared_ffn(cfg, inp["x"], inp["w13s"], inp["w2s"], ys, ws_shared)
            rec()
            moe.moe_combine_add(cfg, yp, lay.slot, wts, ys, y)
        else:
            moe.moe_combine(cfg, yp, lay.slot, wts, y)
        rec()

    for _ in range(args.warmup):
        step()
    st = moe.moe_check()
    if st != 0:
        raise RuntimeError(f"device error during warm-up: {moe.STATUS[st]}")
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(n_ev)] for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    launches0 = moe.moe_launch_count()  # the library counts every kernel it launches
    with ClockSampler(local_rank, args.clocks_csv) as clk:
        for i in range(args.steps):
            step(events[i])
        torch.cuda.synchronize()
    timed_launches = moe.moe_launch_count() - launches0
    if world > 1:
        dist.barrier()
    st = moe.moe_check()
    if st != 0:
        raise RuntimeError(f"device error in the timed region: {moe.STATUS[st]}")
    total_ms = events[0][0].elapsed_time(events[-1][n_ev - 1])
    per_stage = {s: statistics.mean(events[i][j].elapsed_time(events[i][j + 1]) for i in range(args.steps))
                 for j, s in enumerate(stages)}
    total_ms = max_over_ranks(total_ms, world, "cuda")
    clocks = clk.summary()

    # ---- end to end through the public call with host buffers.  Two streams
    # take alternate steps, each with its own workspace and pinned buffers, so
    # the host<->device copies of one step overlap the compute of the other.
    op_host = (moe.MOE_OP_BLOCK_HOST if shared else moe.MOE_OP_LAYER if eplb else moe.MOE_OP_LAYER_FP8 if fp8
               else moe.MOE_OP_LAYER_HOST)
    dev_io = eplb or fp8  # layer calls that take device activations: copies on the lane's stream around them
    lanes = [dict(stream=torch.cuda.Stream(), x=inp["x"].cpu().pin_memory(),
                  y=torch.empty(T, w.h, dtype=dt).pin_memory(), ws=moe.alloc_workspace(cfg, op_host),
                  xd=torch.empty_like(inp["x"]) if dev_io else None, yd=torch.empty_like(y) if dev_io else None)
             for _ in range(2)]

    def e2e_step(i):
        ln = lanes[i % len(lanes)]
        if fp8:
            with torch.cuda.stream(ln["stream"]):
                ln["xd"].copy_(ln["x"], non_blocking=True)
                moe.moe_layer_forward_fp8(cfg, ln["xd"], inp["w_r"], inp["logit_offset"], inp["sel_bias"], q13, s13,
                                          q2, s2, ln["yd"], None, ln["ws"], stream=ln["stream"])
                ln["y"].copy_(ln["yd"], non_blocking=True)
        elif eplb:
            with torch.cuda.stream(ln["stream"]):
                ln["xd"].copy_(ln["x"], non_blocking=True)
                moe.moe_layer_forward_eplb(cfg, ln["xd"], inp["w_r"], inp["logit_offset"], inp["sel_bias"],
                                           inp["w13"], inp["w2"], plan["rep_offsets"], plan["rep_phys"],
                                           plan["phys_to_log"], ln["yd"], None, ln["ws"], stream=ln["stream"])
                ln["y"].copy_(ln["yd"], non_blocking=True)
        elif shared:
            moe.moe_block_forward_host(cfg, ln["x"], inp["w_r"], inp["logit_offset"], inp["sel_bias"], inp["w13"],
                                       inp["w2"], inp["w13s"], inp["w2s"], ln["y"], ln["ws"], stream=ln["stream"])
        else:
            moe.moe_layer_forward_host(cfg, ln["x"], inp["w_r"], inp["logit_offset"], inp["sel_bias"], inp["w13"],
                                       inp["w2"], ln["y"], ln["ws"], stream=ln["stream"])

    for i in range(max(2, args.warmup)):
        e2e_step(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    e0.record(stream)
    for ln in lanes:
        ln["stream"].wait_event(e0)
    for i in range(args.steps):
        e2e_step(i)
    for ln in lanes:
        stream.wait_stream(ln["stream"])
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    e2e_ms = max_over_ranks(e2e_ms, world, "cuda")
    if moe.moe_check() != 0:
        raise RuntimeError("device error in the end-to-end run")
    if not torch.equal(lanes[0]["y"].to(y.device), y):
        raise RuntimeError("the end-to-end layer output differs from the device-resident one")

    if rank != 0:
        return None

    # ---- algorithmic work of the step (from the layout of the last step)
    kept = lay.kept.cpu().numpy().astype(np.int64)
    stats = moe.stats_dict(lay.stats)
    rows_kept = int(kept.sum())
    ds = 2 if w.dtype == "bf16" else 4
    touched = int((kept > 0).sum())
    if eplb:  # replicas share their logical expert's weights: count each touched logical expert once
        touched = len(set(plan_h["phys_to_log"][kept > 0].tolist()))
    if fp8:  # E4M3 weights (+ float32 row scales); E4M3 rows in, bf16 intermediate out, re-quantised, bf16 out
        weight_bytes = touched * (3 * w.h * w.I + 4 * (2 * w.I + w.h))
        ffn_bytes = weight_bytes + rows_kept * (w.h + 4 + 2 * w.I * 2 + w.I * 2 + 4 + 2 * w.h)
    else:
        weight_bytes = touched * 3 * w.h * w.I * ds
        ffn_bytes = weight_bytes + rows_kept * (2 * w.h + 2 * w.I) * ds
    ffn_flops = 6.0 * w.h * w.I * rows_kept
    tokens_with_rows = int((lay.slot.view(T, K) >= 0).any(dim=1).sum().item())
    permute_bytes = (tokens_with_rows + rows_kept) * w.h * ds  # not moved when the FFN gathers from x
    combine_bytes = (rows_kept + T) * w.h * ds
    peaks, peak_kind = measured_peaks()
    hbm = float(peaks["hbm_gbs"])
    # FP8 dense tensor peak taken as twice the measured bf16 one (the nominal ratio)
    tc_peak = float(peaks["bf16_tflops_sustained"]) * (2.0 if fp8 else 1.0)
    ffn_s = per_stage["ffn"] / 1e3
    ffn_gbs = ffn_bytes / ffn_s / 1e9
    # the FFN is compute-bound when its arithmetic intensity is above the ridge of
    # the measured peaks (Mixtral: ~1000 rows per expert), else bound by HBM
    tensor_bound = ffn_flops / ffn_bytes > tc_peak * 1e12 / (hbm * 1e9)
    # FFN_TRAFFIC_RATIO was captured on the bf16 weights-as-M kernel (experts
    # expected to see at most 160 rows); other variants report no traffic
    expected_rows = (min(w.capacity, T) if w.capacity > 0 else -(-T * K // (E + w.n_redundant)))
    traffic_known = not fp8 and w.dtype == "bf16" and expected_rows <= 160
    ffn_tflops = ffn_flops / ffn_s / 1e12
    ms = total_ms / args.steps
    out = {
        "metric": METRIC,
        "value": job_throughput(T, world, args.steps, total_ms),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e4m3" if fp8 else w.dtype,
        "data": "synthetic: seeded counter-based generator (x~N(0,1), weights~N(0,1/h)), no dataset",
        "config": workload_config(w),
        "e2e": {"value": job_throughput(T, world, args.steps, e2e_ms), "unit": "tokens/s",
                "h2d_bytes_per_step": T * w.h * ds, "d2h_bytes_per_step": T * w.h * ds},
        "gpu_launches": timed_launches,
        "roofline": {"kernel": "grouped SwiGLU FFN (gate/up + down tcgen05 GEMMs)",
                     "bound": "tensor" if tensor_bound else "hbm",
                     "achieved": ffn_tflops if tensor_bound else ffn_gbs,
                     "peak": tc_peak if tensor_bound else hbm,
                     "unit": "TFLOP/s" if tensor_bound else "GB/s",
                     "frac": ffn_tflops / tc_peak if tensor_bound else ffn_gbs / hbm,
                     "peak_source": peak_kind + (" (bf16 sustained" + (" x 2 for FP8" if fp8 else "") + ")"
                                                 if tensor_bound else " (HBM copy)"),
                     "achieved_gbs": ffn_gbs, "algorithmic_bytes": ffn_bytes, "algorithmic_flops": ffn_flops,
                     "traffic": FFN_TRAFFIC_RATIO * ffn_bytes if traffic_known else None,
                     "traffic_source": ("ncu DRAM bytes / algorithmic bytes on deepseek_v3_e32_T512, scaled to this "
                                        "launch's algorithmic bytes") if traffic_known else
                                       "not captured for this FFN variant since its last change",
                     "tensor_tflops": ffn_tflops,
                     "tensor_frac_of_sustained": ffn_tflops / tc_peak},
        "stages_ms": per_stage,
        "permute_gbs": permute_bytes / (per_stage["permute"] / 1e3) / 1e9 if "permute" in per_stage else None,
        "permute_fused_into_ffn": gather,
        "combine_gbs": combine_bytes / (per_stage["combine"] / 1e3) / 1e9,
        "layout": {"dropped": stats["dropped"], "experts_touched": stats["experts_touched"],
                   "balancedness": stats["balancedness"], "offdiag_rows": stats["offdiag_rows"]},
        "clocks": clocks,
    }
    return out


# ---------------------------------------------------------------------------- the oracle (CPU)
def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info()]
        return max(n) if n else os.cpu_count()
    except Exception:  # noqa: BLE001
        return os.cpu_count()


def oracle_sample_time(w, sample_tokens: int, seed: int):
    """Seconds the oracle takes for the whole index path on all T tokens plus the
    FFN and combine of ``sample_tokens`` tokens, and the tokens/s extrapolated
    from that sample.  Input generation (synth) is outside the timed parts."""
    import numpy as np

    import oracle
    from synth import workloads

    x = workloads.host_x(w)
    wr = workloads.host_router_weight(w)
    bias = workloads.host_sel_bias(w)
    off = workloads.host_logit_offset(w)
    t0 = time.perf_counter()
    L = oracle.router_logits(x, wr, w.dtype, off)
    ids, wts, _, _ = oracle.route(L, w, bias)
    lay = oracle.dispatch_layout(ids, w)
    t_index = time.perf_counter() - t0
    rng = np.random.default_rng(seed)
    tokens = np.sort(rng.choice(w.T, size=min(sample_tokens, w.T), replace=False))
    need = {}
    for t in tokens:
        for k in range(w.K):
            s = lay["slot"][t, k]
            if s >= 0:
                need.setdefault(int(ids[t, k]), []).append(int(s))
    weights = {e: (workloads.host_w13(w, e), workloads.host_w2(w, e)) for e in need}  # input generation
    shared_w = (workloads.host_w13s(w), workloads.host_w2s(w)) if w.shared_I > 0 else None
    t1 = time.perf_counter()
    xp = np.zeros((lay["rows"], w.h), dtype=x.dtype)
    for e, rows in need.items():
        for r in rows:
            xp[r] = x[lay["row_src"][r]]
    parts = oracle.grouped_ffn(xp, lay["offsets"], lay["kept"], lambda e: weights[e][0], lambda e: weights[e][1], w,
                               experts=sorted(need), rows={e: sorted(r) for e, r in need.items()})
    yp = np.zeros_like(xp)
    for e, (idx, val) in parts.items():
        yp[idx] = val
    if shared_w is not None:
        ys = oracle.shared_ffn(x[tokens], shared_w[0], shared_w[1], w)
        oracle.combine(yp, lay["slot"], wts, w, tokens=list(tokens), rounded=False) + oracle.to_f64(ys, w.dtype)
    else:
        oracle.combine(yp, lay["slot"], wts, w, tokens=list(tokens))
    t_sample = time.perf_counter() - t1
    total = t_index + t_sample * (w.T / len(tokens))
    return {"value": w.T / total, "index_s": t_index, "sample_s": t_sample, "tokens": len(tokens)}


def run_reference(args):
    from synth import workloads

    w = workloads.ALL.get(args.workload) or workloads.EXTRA[args.workload]
    vals = []
    for i in range(args.warmup + args.steps):
        r = oracle_sample_time(w, args.ref_sample, seed=i)
        if i >= args.warmup:
            vals.append(r)
    v = statistics.mean(r["value"] for r in vals)
    sample = (f"per step: routing, layout and index outputs for all {w.T} tokens, FFN + combine for "
              f"{vals[0]['tokens']} random tokens; tokens/s extrapolated to the full batch")
    return {
        "metric": METRIC, "impl": "reference", "value": v, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * w.T / v, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (same generator as ours)",
        "config": workload_config(w),
        "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": blas_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="deepseek_v3")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--ref-sample", type=int, default=1, help="tokens whose FFN the oracle evaluates per step")
    ap.add_argument("--cpu-sample", type=int, default=8, help="tokens in the cpu_baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--clocks-csv", default=None, help="where to keep the nvidia-smi samples of the timed region")
    ap.add_argument("--fused-permute", action="store_true",
                    help="gather the FFN's rows from x instead of permuting (bf16 weights-as-M layers)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3) if args.impl == "ours" else args.warmup

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    out = run_ours(args, rank, world, local_rank)
    if rank == 0 and out is not None:
        if world == 1 and not args.no_cpu_baseline:
            from synth import workloads
            w = workloads.ALL.get(args.workload) or workloads.EXTRA[args.workload]
            r = oracle_sample_time(w, args.cpu_sample, seed=1234)
            out["cpu_baseline"] = {
                "value": r["value"], "unit": "tokens/s", "cores": blas_threads(), "kind": "oracle",
                "sample": (f"routing, layout and index outputs for all tokens ({r['index_s']:.1f} s) plus FFN and "
                           f"combine of {r['tokens']} random tokens ({r['sample_s']:.1f} s), extrapolated to the "
                           f"full batch")}
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
