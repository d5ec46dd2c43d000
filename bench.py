#!/usr/bin/env python3
"""Benchmark of one DSA step (store keys -> indexer score -> causal top-k ->
sparse absorbed MLA) on GB300, printed as one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Workloads (synthetic, seeded; DeepSeek-V3.2 shapes):
  long_decode (default)  128 requests x 1 row, contexts ~U[65536, 131072]
  decode                 32 requests x 1 row, contexts ~U[4096, 16384]
  chunked_prefill        1 request, 8192 cached + 8192 new rows
  mixed_fp8              16 decode rows + two 2048-row chunks, fp8 caches, sinks
  tiny_prefill           2 requests, contexts 256 / 384 (small shapes)

`value` is whole-job throughput (decode rows/s, or prefill tokens/s) with the
caches and the step inputs resident in HBM; each step is timed with CUDA
events on the launching stream and L2 is flushed (256 MB write) between steps
outside the timed events.  `e2e` is the same metric through the public API
with host buffers: per step dsa_plan from host spans, pinned host-to-device
copies of the step's inputs, the step, and a device-to-host copy of its output;
for decode workloads the step is instead one CUDA graph over a capturable plan
(dsa_plan_update re-plans on the device from spans and a page table copied up
with the inputs), which is also timed device-resident as `captured_step`.
The end-to-end loop keeps two buffer sets with the copies on their own
streams, so each step's transfers overlap the neighbouring steps' kernels.
Decode workloads also time the prefill workloads (`--prefill`, default
chunked_prefill and mixed_fp8) in the same process at the same steps and
warm-up, reported under `prefill`: tokens/s, the stage split, and the
indexer's and the attention's TFLOP/s as fractions of the measured dense bf16
peak, with the clocks of that leg.
Block-sparse MSA workloads (`--msa`, default msa_decode and msa_prefill) are
timed the same way and reported under `msa`: store, index score, block
selection and GQA attention over the kept blocks.  Decode legs hold the
indexer and the attention against the measured HBM copy rate (each key and
kept row is read once); prefill legs hold the indexer against the dense bf16
peak and report the attention's gather rate (kept rows re-read by the rows of
one request come mostly from L2) beside its TFLOP/s.
`--impl reference` times the CPU oracle (the only reference this method has)
on a bounded sample of the same workload on the host cores.
Multi-GPU (torchrun): independent replicas, one per rank (weak scaling).
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
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from deepseek_sparse_attention_dsa_gb300 import workloads as W  # noqa: E402

METRIC = "DSA decode rows/s + prefill tokens/s at 1 GB300; % HBM / tensor-core roofline"
WORKLOADS = {"tiny_prefill": 0, "decode": 1, "chunked_prefill": 2, "long_decode": 3, "mixed_fp8": 4}


def rank_info():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


# ----------------------------------------------------------------------------
# algorithmic work (bytes / flops) of a workload
# ----------------------------------------------------------------------------
def algorithmic(wl):
    sh = wl.shape
    _, pos, _ = wl.row_table()
    vis = pos + 1
    nsel = np.minimum(vis, sh.topk)
    T = len(pos)
    idx_bytes = float(vis.sum()) * sh.index_row_bytes + T * (sh.index_heads * sh.index_dim * 2 + sh.index_heads * 4)
    lat_bytes = float(nsel.sum()) * sh.latent_row_bytes
    att_io = T * sh.heads * (sh.kv_lora_rank + sh.rope_dim) * 2 + T * sh.heads * sh.kv_lora_rank * 2 + T * sh.topk * 4
    store = T * sh.index_row_bytes * 2
    idx_flops = float(vis.sum()) * 2.0 * sh.index_heads * sh.index_dim
    att_flops = float(nsel.sum()) * 2.0 * sh.heads * (sh.kv_lora_rank + sh.rope_dim + sh.kv_lora_rank)
    return dict(index_bytes=idx_bytes, attend_bytes=lat_bytes + att_io, step_bytes=idx_bytes + lat_bytes + att_io + store,
                index_flops=idx_flops, attend_flops=att_flops, rows=T, keys=int(vis.sum()), selected=int(nsel.sum()))


def unit_of(wl):
    decode = all(s.q_len == 1 for s in wl.spans)
    return ("rows/s" if decode else "tokens/s"), decode


def workload_config(name, wl):
    sh = wl.shape
    ctxs = [s.ctx_end for s in wl.spans]
    return {"workload": name, "requests": len(wl.spans), "rows": wl.num_rows, "ctx_min": int(min(ctxs)),
            "ctx_max": int(max(ctxs)), "ctx_mean": float(np.mean(ctxs)), "topk": sh.topk,
            "indexer": "%dx%d %s" % (sh.index_heads, sh.index_dim, "fp8-132B" if sh.index_fmt else "bf16"),
            "mla": "H=%d %d+%d %s" % (sh.heads, sh.kv_lora_rank, sh.rope_dim, "fp8-656B" if sh.latent_fmt else "bf16"),
            "page_size": sh.page_size, "sink": bool(sh.has_sink), "seed": wl.seed,
            "l2": "flushed between steps (256 MB write outside the timed events)"}


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "samples": len(sm), "reasons": sorted(reasons)}


# ----------------------------------------------------------------------------
# our implementation
# ----------------------------------------------------------------------------
def timed_steps(ctx, plan, wl, ic, lc, st, scores, sel, out, flush, args, world, dev):
    """W untimed steps, then K steps each timed per stage with CUDA events on
    the launching stream (L2 flushed before each step, outside the events),
    with the clocks sampled meanwhile.  A step = store keys, index score,
    top-k, attend over a host plan built once."""
    sh = wl.shape
    stream = torch.cuda.current_stream(dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
    launches = [0]

    def step(record):
        if record:
            ev[0].record(stream)
        ctx.store_keys(plan, st.keys, ic)
        n = ctx.last_launch_count()
        if record:
            ev[1].record(stream)
        ctx.index_scores(plan, st.q, st.w, ic, scores)
        n += ctx.last_launch_count()
        if record:
            ev[2].record(stream)
        ctx.topk_from_scores(plan, scores, sel)
        n += ctx.last_launch_count()
        if record:
            ev[3].record(stream)
        ctx.attend(plan, sel, st.q_nope, st.q_pe, lc, st.sink, sh.sm_scale, out)
        n += ctx.last_launch_count()
        if record:
            ev[4].record(stream)
        launches[0] = n

    for _ in range(args.warmup):
        step(False)
    ctx.get_error()
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    stage = {"store": [], "index": [], "topk": [], "attend": [], "step": []}
    n_launch = 0
    with ClockSampler(dev.index) as clk:
        for _ in range(args.steps):
            flush.zero_()
            step(True)
            n_launch += launches[0]
            ev[4].synchronize()
            stage["store"].append(ev[0].elapsed_time(ev[1]))
            stage["index"].append(ev[1].elapsed_time(ev[2]))
            stage["topk"].append(ev[2].elapsed_time(ev[3]))
            stage["attend"].append(ev[3].elapsed_time(ev[4]))
            stage["step"].append(ev[0].elapsed_time(ev[4]))
    torch.cuda.synchronize(dev)
    ctx.get_error()
    return stage, n_launch, clk.summary()


def prefill_leg(args, name, rank, world, dev, flush):
    """A prefill workload timed like the headline step, in the same process
    and at the same steps and warm-up: tokens/s, the stage split, and the
    indexer's and the attention's TFLOP/s against the measured bf16 peak."""
    from deepseek_sparse_attention_dsa_gb300 import dsa
    wl = W.config(WORKLOADS[name], seed=1000 + WORKLOADS[name] + 7919 * rank)
    sh = wl.shape
    work = algorithmic(wl)
    ic = W.make_index_cache(wl, device=dev)
    lc = W.make_latent_cache(wl, device=dev)
    st = W.make_step_inputs(wl, device=dev)
    ctx = dsa.Context(sh, dev.index)
    plan = ctx.plan(wl.spans, wl.num_pages)
    scores = torch.empty(max(1, plan.num_scores), dtype=torch.float32, device=dev)
    sel = torch.empty(plan.num_rows, sh.topk, dtype=torch.int32, device=dev)
    out = torch.empty(plan.num_rows, sh.heads, sh.kv_lora_rank, dtype=torch.bfloat16, device=dev)
    stage, n_launch, clk = timed_steps(ctx, plan, wl, ic, lc, st, scores, sel, out, flush, args, world, dev)
    total_ms = float(sum(stage["step"]))
    if world > 1:
        t = torch.tensor([total_ms], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        total_ms = float(t.item())
    ms = total_ms / args.steps
    _, bf16, _, peak_kind = measured_peaks()
    idx_ms = statistics.mean(stage["index"])
    att_ms = statistics.mean(stage["attend"])
    idx_tf = work["index_flops"] / (idx_ms / 1e3) / 1e12
    att_tf = work["attend_flops"] / (att_ms / 1e3) / 1e12
    leg = {"workload": name, "value": round(work["rows"] * world / (ms / 1e3), 2), "unit": unit_of(wl)[0],
           "ms_per_step": round(ms, 4), "stages_ms": {k: round(statistics.mean(v), 4) for k, v in stage.items()},
           "index_tflops": round(idx_tf, 2), "index_frac": round(idx_tf / bf16, 4),
           "attend_tflops": round(att_tf, 2), "attend_frac": round(att_tf / bf16, 4),
           "peak_tflops": bf16, "peak_kind": peak_kind + " (bf16_tflops burst)",
           "index_flops_per_step": work["index_flops"], "attend_flops_per_step": work["attend_flops"],
           "gpu_launches": n_launch, "clocks": clk, "config": workload_config(name, wl)}
    plan.close()
    del ic, lc, st, scores, sel, out
    torch.cuda.empty_cache()
    return leg


def msa_work(wl, block_sel=None):
    """Algorithmic work of an MSA step.  Attention: every kept position read
    once (K and V of all kv heads), q in, out back, the block ids; flops of
    QK and PV over the kept positions.  Without a selection, the count assumes
    each row keeps min(topk_blocks, its blocks) full blocks."""
    sh, ms = wl.shape, wl.msa
    _, pos, _ = wl.row_table()
    vis = pos + 1
    T = len(pos)
    if block_sel is None:
        kept = np.minimum(vis, ms.topk_blocks * ms.block_size)
    else:
        kept = np.zeros(T, np.int64)
        for r in range(T):
            b = block_sel[r][block_sel[r] >= 0].astype(np.int64)
            kept[r] = int(np.clip(pos[r] + 1 - b * ms.block_size, 0, ms.block_size).sum())
    idx_bytes = float(vis.sum()) * sh.index_row_bytes + T * (sh.index_heads * sh.index_dim * 2 + sh.index_heads * 4)
    att_bytes = float(kept.sum()) * ms.kv_row_bytes + T * ms.q_heads * ms.head_dim * 2 * 2 + T * ms.topk_blocks * 4
    return dict(rows=T, index_bytes=idx_bytes, attend_bytes=att_bytes,
                step_bytes=idx_bytes + att_bytes + T * sh.index_row_bytes * 2,
                index_flops=float(vis.sum()) * 2.0 * sh.index_heads * sh.index_dim,
                attend_flops=float(kept.sum()) * 4.0 * ms.q_heads * ms.head_dim, kept=int(kept.sum()))


def msa_leg(args, name, rank, world, dev, flush, requests=0):
    """A block-sparse MSA workload (store keys, index score, block selection,
    GQA attention over the kept blocks) timed like the headline step;
    `requests` keeps the first N requests (profiler captures)."""
    from deepseek_sparse_attention_dsa_gb300 import dsa
    wl = W.msa_config(name, seed=2000 + W.MSA_CONFIG_NAMES.index(name) + 7919 * rank)
    if requests:
        wl = wl.sub_workload(range(min(requests, len(wl.spans))))
    sh, ms = wl.shape, wl.msa
    unit, decode = unit_of(wl)
    ic = W.make_index_cache(wl, device=dev)
    kv = W.make_kv_cache(wl, device=dev)
    st = W.make_step_inputs(wl, device=dev)
    q = W.make_msa_q(wl, device=dev)
    ctx = dsa.Context(sh, dev.index)
    plan = ctx.plan(wl.spans, wl.num_pages)
    bsel = torch.empty(plan.num_rows, ms.topk_blocks, dtype=torch.int32, device=dev)
    out = torch.empty(plan.num_rows, ms.q_heads, ms.head_dim, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    launches = [0]

    def step(record):
        if record:
            ev[0].record(stream)
        ctx.store_keys(plan, st.keys, ic)
        n = ctx.last_launch_count()
        if record:
            ev[1].record(stream)
        # index score and block selection in one call (block maxima straight
        # from the indexer's epilogue where the kernels allow it)
        ctx.msa_index_select(plan, ms, st.q, st.w, ic, bsel)
        n += ctx.last_launch_count()
        if record:
            ev[2].record(stream)
        ctx.msa_attend(plan, ms, bsel, q, kv, ms.sm_scale, out)
        n += ctx.last_launch_count()
        if record:
            ev[3].record(stream)
        launches[0] = n

    for _ in range(args.warmup):
        step(False)
    ctx.get_error()
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    stage = {"store": [], "index_select": [], "attend": [], "step": []}
    n_launch = 0
    with ClockSampler(dev.index) as clk:
        for _ in range(args.steps):
            flush.zero_()
            step(True)
            n_launch += launches[0]
            ev[3].synchronize()
            for k, (a, b) in zip(("store", "index_select", "attend", "step"), ((0, 1), (1, 2), (2, 3), (0, 3))):
                stage[k].append(ev[a].elapsed_time(ev[b]))
    torch.cuda.synchronize(dev)
    ctx.get_error()
    total_ms = float(sum(stage["step"]))
    if world > 1:
        t = torch.tensor([total_ms], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        total_ms = float(t.item())
    ms_step = total_ms / args.steps
    work = msa_work(wl, bsel.cpu().numpy())
    hbm, bf16, _, peak_kind = measured_peaks()
    idx_ms = statistics.mean(stage["index_select"])   # the indexer with the block selection behind it
    att_ms = statistics.mean(stage["attend"])
    att_gbs = work["attend_bytes"] / (att_ms / 1e3) / 1e9
    att_tf = work["attend_flops"] / (att_ms / 1e3) / 1e12
    idx_gbs = work["index_bytes"] / (idx_ms / 1e3) / 1e9
    idx_tf = work["index_flops"] / (idx_ms / 1e3) / 1e12
    leg = {"workload": name, "value": round(work["rows"] * world / (ms_step / 1e3), 2), "unit": unit,
           "ms_per_step": round(ms_step, 4), "stages_ms": {k: round(statistics.mean(v), 4) for k, v in stage.items()},
           "attend_kernel": "msa_attend_tc_kernel" if ctx.msa_attend_on_tensor_cores(plan, ms) else "msa_attend_simt_kernel",
           "attend_tflops": round(att_tf, 2), "attend_tensor_frac": round(att_tf / bf16, 4),
           "attend_bytes_per_step": work["attend_bytes"], "kept_positions": work["kept"],
           "peaks": {"hbm_gbs": hbm, "bf16_tflops": bf16, "kind": peak_kind},
           "gpu_launches": n_launch, "clocks": clk.summary(),
           "config": dict(workload_config(name, wl), msa="top %d blocks of %d, GQA %d q / %d kv heads x %d"
                          % (ms.topk_blocks, ms.block_size, ms.q_heads, ms.kv_heads, ms.head_dim))}
    if decode:
        leg.update(attend_gbs=round(att_gbs, 1), attend_hbm_frac=round(att_gbs / hbm, 4),
                   index_gbs=round(idx_gbs, 1), index_hbm_frac=round(idx_gbs / hbm, 4),
                   step_hbm_frac=round(work["step_bytes"] / (ms_step / 1e3) / 1e9 / hbm, 4))
    else:
        # prefill rows of a request re-read the same index keys and kept
        # blocks (mostly from L2): the indexer is held against the tensor peak
        # and the attention's byte rate is what it gathers into shared memory
        leg.update(index_tflops=round(idx_tf, 2), index_frac=round(idx_tf / bf16, 4),
                   attend_gather_gbs=round(att_gbs, 1))
    plan.close()
    del ic, kv, st, q, bsel, out
    torch.cuda.empty_cache()
    return leg


def run_msa(args, name, rank, world, local_rank):
    """`--workload msa_*`: the MSA step as the line itself (for profiler
    captures and standalone runs; the headline stays long_decode)."""
    from deepseek_sparse_attention_dsa_gb300 import build as lib_build
    lib_build.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    leg = msa_leg(args, name, rank, world, dev, flush, args.requests)
    hbm, bf16 = leg["peaks"]["hbm_gbs"], leg["peaks"]["bf16_tflops"]
    if "attend_hbm_frac" in leg:
        roof = {"kernel": leg["attend_kernel"], "bound": "hbm", "achieved": leg["attend_gbs"], "peak": hbm,
                "unit": "GB/s", "frac": leg["attend_hbm_frac"], "traffic": None,
                "peak_kind": leg["peaks"]["kind"] + " (hbm_gbs)"}
    else:
        roof = {"kernel": leg["attend_kernel"], "bound": "tensor", "achieved": leg["attend_tflops"], "peak": bf16,
                "unit": "TFLOP/s", "frac": leg["attend_tensor_frac"], "traffic": None,
                "peak_kind": leg["peaks"]["kind"] + " (bf16_tflops burst)"}
    line = {"metric": METRIC, "value": leg["value"], "unit": leg["unit"], "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": leg["ms_per_step"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded counter-based generator; no dataset or weights)",
            "config": dict(leg["config"], requests_kept=args.requests or None),
            "roofline": roof,
            "stages_ms": leg["stages_ms"], "gpu_launches": leg["gpu_launches"], "clocks": leg["clocks"], "msa": leg}
    return line


def run_ours(args, name, rank, world, local_rank):
    from deepseek_sparse_attention_dsa_gb300 import build as lib_build
    from deepseek_sparse_attention_dsa_gb300 import dsa

    lib_build.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    wl = W.config(WORKLOADS[name], seed=1000 + WORKLOADS[name] + 7919 * rank, page_start=args.page_start)
    if args.requests:
        # the first N requests only: a smaller case of the same workload for profiler captures
        wl = wl.sub_workload(range(min(args.requests, len(wl.spans))))
    sh = wl.shape
    unit, decode = unit_of(wl)
    work = algorithmic(wl)

    ic = W.make_index_cache(wl, device=dev)
    lc = W.make_latent_cache(wl, device=dev)
    st = W.make_step_inputs(wl, device=dev)
    ctx = dsa.Context(sh, local_rank)
    stream = torch.cuda.current_stream(dev)
    t0 = time.perf_counter()
    plan = ctx.plan(wl.spans, wl.num_pages)
    torch.cuda.synchronize(dev)
    plan_ms = (time.perf_counter() - t0) * 1e3
    scores = torch.empty(max(1, plan.num_scores), dtype=torch.float32, device=dev)
    sel = torch.empty(plan.num_rows, sh.topk, dtype=torch.int32, device=dev)
    out = torch.empty(plan.num_rows, sh.heads, sh.kv_lora_rank, dtype=torch.bfloat16, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
    stage, n_launch, clk_summary = timed_steps(ctx, plan, wl, ic, lc, st, scores, sel, out, flush, args, world, dev)
    total_ms = float(sum(stage["step"]))
    if world > 1:
        t = torch.tensor([total_ms], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        total_ms = float(t.item())
    ms_per_step = total_ms / args.steps
    units_per_step = work["rows"]

    # ---- decode: the step as one CUDA graph over a capturable plan, which
    # re-plans on the device every step (spans, pages and counts in device
    # memory), so no host work sits between the kernels.  Reported beside the
    # step above (`captured_step`); the end-to-end number uses it.
    graph = None
    captured = None
    if decode and not args.eager:
        graph = capture_decode_step(ctx, wl, ic, lc, st, sel, out, dev)
        for _ in range(args.warmup):
            graph["replay"]()
        torch.cuda.synchronize(dev)
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)
        g_ms = []
        with ClockSampler(local_rank) as gclk:
            for _ in range(args.steps):
                flush.zero_()
                ev[0].record(stream)
                graph["replay"]()
                ev[1].record(stream)
                ev[1].synchronize()
                g_ms.append(ev[0].elapsed_time(ev[1]))
        torch.cuda.synchronize(dev)
        ctx.get_error()
        counts = graph["plan"].read_counts()
        assert counts["valid"] and counts["rows"] == work["rows"], counts
        total_ms = float(sum(g_ms))
        if world > 1:
            t = torch.tensor([total_ms], device=dev)
            torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
            total_ms = float(t.item())
        g_step = total_ms / args.steps
        captured = {"ms_per_step": round(g_step, 4), "value": round(units_per_step * world / (g_step / 1e3), 2),
                    "unit": unit, "launches_per_step": graph["launches"],
                    "path": "CUDA graph: device re-plan + store + index/top-k + attend", "clocks": gclk.summary()}
    value = units_per_step * world / (ms_per_step / 1e3)

    # ---- fp8 index cache: the indexer with an e4m3 query as well (the step
    # above scores with the bf16 query)
    fp8q = None
    if sh.index_fmt == W.INDEX_FP8_132:
        codes, qscale = ctx.quantize_q(plan, st.q)
        qt, it = [], []
        for i in range(args.warmup + args.steps):
            flush.zero_()
            ev[0].record(stream)
            ctx.quantize_q(plan, st.q, codes, qscale)
            ev[1].record(stream)
            ctx.index_scores_fp8q(plan, codes, qscale, st.w, ic, scores)
            ev[2].record(stream)
            ev[2].synchronize()
            if i >= args.warmup:
                qt.append(ev[0].elapsed_time(ev[1]))
                it.append(ev[1].elapsed_time(ev[2]))
        ctx.get_error()
        fp8q = {"quantize_ms": round(statistics.mean(qt), 4), "index_ms": round(statistics.mean(it), 4),
                "index_tflops": round(work["index_flops"] / (statistics.mean(it) / 1e3) / 1e12, 2),
                "path": "dsa_quantize_q + dsa_index_scores_fp8q (e4m3 x e4m3 tensor cores)"}

    # ---- end to end through the public API with host buffers
    pinned = {k: getattr(st, k).cpu().pin_memory() for k in ("q", "w", "keys", "q_nope", "q_pe")}
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in pinned.values())
    d2h = out_h.numel() * out_h.element_size()
    dbuf = {k: torch.empty_like(getattr(st, k)) for k in pinned}

    e2e_loop = None
    if graph is not None:
        # per step: this step's inputs and its spans and page table to the
        # device, the captured step, the output back.  Two captured steps over
        # two buffer sets let step i's copies run on their own streams while
        # the neighbouring steps compute (as a serving loop would).
        pin_sp = {k: v.cpu().pin_memory() for k, v in graph["spans"].items()}
        h2d += sum(t.numel() * t.element_size() for t in pin_sp.values())
        sel2 = torch.empty_like(sel)
        out2 = torch.empty_like(out)
        graphs = [(graph, out), (capture_decode_step(ctx, wl, ic, lc, st, sel2, out2, dev), out2)]
        outs_h = [out_h, torch.empty(out.shape, dtype=out.dtype).pin_memory()]
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        s_comp = torch.cuda.current_stream(dev)
        ready = [torch.cuda.Event() for _ in range(2)]
        done = [torch.cuda.Event() for _ in range(2)]
        back = [torch.cuda.Event() for _ in range(2)]

        def e2e_loop(n):
            for i in range(n):
                b = i % 2
                g, o = graphs[b]
                if i >= 2:
                    s_in.wait_event(done[b])     # step i-2 has consumed buffer set b
                with torch.cuda.stream(s_in):
                    for k, v in pinned.items():
                        g["inputs"][k].copy_(v, non_blocking=True)
                    for k, v in pin_sp.items():
                        g["spans"][k].copy_(v, non_blocking=True)
                    ready[b].record(s_in)
                s_comp.wait_event(ready[b])
                if i >= 2:
                    s_comp.wait_event(back[b])   # step i-2's output has been read back
                with torch.cuda.stream(s_comp):
                    g["replay"]()
                    done[b].record(s_comp)
                s_out.wait_event(done[b])
                with torch.cuda.stream(s_out):
                    outs_h[b].copy_(o, non_blocking=True)
                    back[b].record(s_out)
            torch.cuda.synchronize(dev)

    if e2e_loop is None:
        # per step: a host plan from the spans, the inputs to the device, the
        # calls, the output back; two input / output buffer sets let a step's
        # copies run on their own streams while the neighbouring steps compute
        dbufs = [dbuf, {k: torch.empty_like(v) for k, v in dbuf.items()}]
        eouts = [out, torch.empty_like(out)]
        eouts_h = [out_h, torch.empty(out.shape, dtype=out.dtype).pin_memory()]
        e_in, e_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        e_comp = torch.cuda.current_stream(dev)
        e_ready = [torch.cuda.Event() for _ in range(2)]
        e_done = [torch.cuda.Event() for _ in range(2)]
        e_back = [torch.cuda.Event() for _ in range(2)]

        def e2e_loop(n):
            for i in range(n):
                b = i % 2
                if i >= 2:
                    e_in.wait_event(e_done[b])
                with torch.cuda.stream(e_in):
                    for k, v in pinned.items():
                        dbufs[b][k].copy_(v, non_blocking=True)
                    e_ready[b].record(e_in)
                p = ctx.plan(wl.spans, wl.num_pages, stream=e_comp)
                e_comp.wait_event(e_ready[b])
                if i >= 2:
                    e_comp.wait_event(e_back[b])
                d = dbufs[b]
                ctx.store_keys(p, d["keys"], ic, stream=e_comp)
                sl = ctx.index_topk(p, d["q"], d["w"], ic, sel, stream=e_comp)
                ctx.attend(p, sl, d["q_nope"], d["q_pe"], lc, st.sink, sh.sm_scale, eouts[b], stream=e_comp)
                e_done[b].record(e_comp)
                p.close()   # freed in stream order, after the step's kernels
                e_out.wait_event(e_done[b])
                with torch.cuda.stream(e_out):
                    eouts_h[b].copy_(eouts[b], non_blocking=True)
                    e_back[b].record(e_out)
            torch.cuda.synchronize(dev)

    e2e_loop(max(2, args.warmup))
    e2e_steps = max(3, min(args.steps, 20))
    if world > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    e2e_loop(e2e_steps)
    e2e_s = (time.perf_counter() - t0) / e2e_steps
    if world > 1:
        t = torch.tensor([e2e_s], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        e2e_s = float(t.item())
    ctx.get_error()

    hbm, bf16, bf16_sus, peak_kind = measured_peaks()
    idx_ms = statistics.mean(stage["index"])
    att_ms = statistics.mean(stage["attend"])
    if decode:
        achieved = work["index_bytes"] / (idx_ms / 1e3) / 1e9
        roof = {"kernel": "index_tc_kernel (indexer score)", "bound": "hbm", "achieved": round(achieved, 1),
                "peak": hbm, "unit": "GB/s", "frac": round(achieved / hbm, 4),
                "traffic": profile_traffic("index_tc_kernel", name), "peak_kind": peak_kind + " (hbm_gbs)"}
    else:
        achieved = work["attend_flops"] / (att_ms / 1e3) / 1e12
        roof = {"kernel": "attend_tc_kernel (sparse MLA)", "bound": "tensor", "achieved": round(achieved, 1),
                "peak": bf16, "unit": "TFLOP/s", "frac": round(achieved / bf16, 4),
                "traffic": profile_traffic("attend_tc_kernel", name), "peak_kind": peak_kind + " (bf16_tflops burst)"}
    step_gbs = work["step_bytes"] / (ms_per_step / 1e3) / 1e9
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": unit, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if not sh.latent_fmt else "fp8+bf16",
        "data": "synthetic (seeded counter-based generator; no dataset or weights)",
        "config": workload_config(name, wl),
        "roofline": roof,
        "step_hbm": {"algorithmic_bytes": work["step_bytes"], "achieved_gbs": round(step_gbs, 1),
                     "frac": round(step_gbs / hbm, 4)},
        "stages_ms": {k: round(statistics.mean(v), 4) for k, v in stage.items()},
        "index_tflops": round(work["index_flops"] / (idx_ms / 1e3) / 1e12, 2),
        "attend_tflops": round(work["attend_flops"] / (att_ms / 1e3) / 1e12, 2),
        "plan_ms": round(plan_ms, 3),
        "step_path": "calls over a host plan built once (store, index/top-k, attend)",
        "captured_step": captured,
        "fp8_query": fp8q,
        "e2e": {"value": round(units_per_step * world / e2e_s, 2), "unit": unit, "h2d_bytes_per_step": h2d,
                "path": ("per step: inputs + spans + page table to the device, the captured step (device re-plan), "
                         "output back; two buffer sets, copies on their own streams overlapping the neighbouring "
                         "steps" if graph is not None else
                         "per step: host plan, inputs to the device, the calls, output back; two buffer sets, "
                         "copies on their own streams overlapping the neighbouring steps"),
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_s * 1e3, 3)},
        "gpu_launches": n_launch,
        "clocks": clk_summary,
    }
    if args.prefill and decode and not args.requests and not args.page_start:
        line["prefill"] = [prefill_leg(args, p, rank, world, dev, flush) for p in args.prefill.split(",") if p]
    if args.msa and decode and not args.requests and not args.page_start:
        line["msa"] = [msa_leg(args, m, rank, world, dev, flush) for m in args.msa.split(",") if m]
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, args.cpu_rows)
    return line


def capture_decode_step(ctx, wl, ic, lc, st, sel, out, dev):
    """The decode step as one CUDA graph over a capturable plan: the plan is
    rewritten on the device from the spans and page table in device memory
    (dsa_plan_update), then store_keys, index_topk and attend run over it.
    Replaying the graph after rewriting those tensors serves the next step."""
    import math
    sh = wl.shape
    rows, pages, off = [], [], 0
    for s in wl.spans:
        rows.append([s.q_len, s.ctx_start, s.page_start, off, len(s.pages), 0])
        pages.append(np.asarray(s.pages, np.int32))
        off += len(s.pages)
    spans = {"num_spans": torch.tensor([len(rows)], dtype=torch.int32, device=dev),
             "spans": torch.tensor(rows, dtype=torch.int32, device=dev),
             "pages": torch.from_numpy(np.concatenate(pages)).to(dev)}
    max_scores = sum((s.ctx_start + 1 + s.ctx_end) * s.q_len // 2 for s in wl.spans)
    align = math.gcd(sh.page_size, *[int(s.page_start) for s in wl.spans])
    plan = ctx.plan_capturable(wl.num_rows, len(rows), max_scores, wl.num_pages, page_start_align=align)
    inputs = {k: getattr(st, k).clone() for k in ("q", "w", "keys", "q_nope", "q_pe")}
    launches = [0]

    def step():
        n = 0
        ctx.plan_update(plan, spans["num_spans"], spans["spans"], spans["pages"])
        n += ctx.last_launch_count()
        ctx.store_keys(plan, inputs["keys"], ic)
        n += ctx.last_launch_count()
        ctx.index_topk(plan, inputs["q"], inputs["w"], ic, sel)
        n += ctx.last_launch_count()
        ctx.attend(plan, sel, inputs["q_nope"], inputs["q_pe"], lc, st.sink, sh.sm_scale, out)
        n += ctx.last_launch_count()
        launches[0] = n

    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        step()   # outside the capture: one-time kernel attributes
    torch.cuda.current_stream(dev).wait_stream(side)
    torch.cuda.synchronize(dev)
    ctx.get_error()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    return {"plan": plan, "graph": g, "replay": g.replay, "inputs": inputs, "spans": spans, "launches": launches[0]}


def source_fingerprint(path):
    """sha256 (16 hex digits) of a CUDA source with its // comments and blank
    lines dropped: the code a profile was taken of, not its commentary."""
    import hashlib
    import re
    lines = []
    for ln in open(path, encoding="utf-8"):
        code = re.sub(r"//.*$", "", ln.rstrip("\n")).rstrip()
        if code:
            lines.append(code)
    return hashlib.sha256("\n".join(lines).encode()).hexdigest()[:16]


def profile_traffic(kernel, workload):
    """dram bytes per launch from a committed ncu summary of this kernel and
    workload, if its source fingerprint matches the current source."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "%s_%s.md" % (kernel.split("_kernel")[0], workload))
    if not os.path.exists(path):
        return None
    src = {"index_tc": "indexer.cu", "attend_tc": "attend.cu"}.get(kernel.split("_kernel")[0])
    fp = None
    if src:
        fp = source_fingerprint(os.path.join(ROOT, "deepseek_sparse_attention_dsa_gb300", "csrc", src))
    traffic, sha = None, None
    for ln in open(path):
        if ln.startswith("traffic_bytes_per_launch:"):
            traffic = float(ln.split(":")[1])
        if ln.startswith("source_sha256_16:"):
            sha = ln.split(":")[1].strip()
    if traffic is None or (fp is not None and sha != fp):
        return None
    return traffic


# ----------------------------------------------------------------------------
# CPU oracle baseline
# ----------------------------------------------------------------------------
def oracle_sample(wl, nrows):
    """A bounded sample of the workload for the oracle: its first spans
    covering about `nrows` rows (or the first `nrows` rows of one long chunk),
    with host copies of the inputs.  Inputs are generated on the GPU when one
    is present (the generator is bit-identical on both) and only the latent
    rows the sample's selection reads are filled."""
    import oracle
    take, rows = [], 0
    for i, s in enumerate(wl.spans):
        if rows >= nrows:
            break
        if rows + s.q_len > nrows and take:
            break
        take.append(i)
        rows += s.q_len
    sub = wl.sub_workload(take)
    if rows > nrows:
        sub.spans[0].q_len = nrows
        rows = nrows
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    ic = W.make_index_cache(sub, device=dev).cpu()
    st = W.make_step_inputs(sub, device=dev)
    st = W.StepInputs(*(None if x is None else x.cpu() for x in (st.q, st.w, st.keys, st.q_nope, st.q_pe, st.sink)))
    cache = oracle.store_keys(sub.shape, sub.spans, sub.num_pages, st.keys, ic)
    sc, off = oracle.index_scores(sub.shape, sub.spans, sub.num_pages, st.q, st.w, cache)
    sel = oracle.topk(sub.shape, sub.spans, sc, off)
    _, pos, _ = sub.row_table()
    toks = set()
    for r, s in enumerate(sub.spans):
        for i in range(s.q_len):
            row = s.q_start + i
            toks.update((s.token_base + sel[row][sel[row] >= 0]).tolist())
    lc = W.make_latent_cache(sub, device=dev, tokens=toks).cpu()
    return sub, ic, lc, st, rows, take


def cpu_baseline(wl, nrows):
    import oracle
    sub, ic, lc, st, rows, take = oracle_sample(wl, nrows)
    t0 = time.perf_counter()
    oracle.run_all(sub, ic, lc, st)
    dt = time.perf_counter() - t0
    return {"value": round(rows / dt, 4), "unit": unit_of(wl)[0], "cores": oracle.max_threads(), "kind": "oracle",
            "sample": "%d rows of the same workload (spans %s%s), store+score+select+attend, %.1f s"
                      % (rows, take[:4], "..." if len(take) > 4 else "", dt)}


def run_reference(args, name, rank, world):
    """The reference arm: the CPU oracle timed on the host cores, bounded samples."""
    if rank != 0:
        return None
    import oracle
    wl = W.config(WORKLOADS[name])
    unit, _ = unit_of(wl)
    sub, ic, lc, st, rows, take = oracle_sample(wl, args.cpu_rows)
    for _ in range(min(args.warmup, 1)):
        oracle.run_all(sub, ic, lc, st)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.run_all(sub, ic, lc, st)
    dt = (time.perf_counter() - t0) / args.steps
    v = rows / dt
    return {"impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": unit, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
            "config": workload_config(name, wl),
            "cpu_baseline": {"value": round(v, 4), "unit": unit, "cores": oracle.max_threads(), "kind": "oracle",
                             "sample": "%d rows per step (spans %s%s) of %s, store+score+select+attend"
                                       % (rows, take[:4], "..." if len(take) > 4 else "", name)},
            "e2e": {"value": round(v, 4), "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="long_decode", choices=sorted(WORKLOADS) + W.MSA_CONFIG_NAMES)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-rows", type=int, default=16)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--eager", action="store_true",
                    help="decode workloads: time the eager calls over a host plan instead of the captured step")
    ap.add_argument("--prefill", default="chunked_prefill,mixed_fp8",
                    help="decode workloads: prefill workloads timed in the same run (comma list; '' for none)")
    ap.add_argument("--msa", default="msa_decode,msa_prefill",
                    help="decode workloads: block-sparse MSA workloads timed in the same run (comma list; '' for none)")
    ap.add_argument("--page-start", type=int, default=0,
                    help="every request's token 0 at this slot of its first page (0 in the evaluation workloads)")
    ap.add_argument("--requests", type=int, default=0,
                    help="keep only the first N requests of the workload (profiler captures; not a bench line)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3) if args.impl == "ours" else args.warmup
    rank, world, local_rank = rank_info()
    if args.impl == "reference":
        if args.workload not in WORKLOADS:
            ap.error("--impl reference times the DSA workloads (%s)" % ", ".join(sorted(WORKLOADS)))
        line = run_reference(args, args.workload, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    if args.workload in W.MSA_CONFIG_NAMES:
        line = run_msa(args, args.workload, rank, world, local_rank)
    else:
        line = run_ours(args, args.workload, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
