"""Shared helpers for the parity tests: run a workload through the C ABI on
the GPU and through the oracle on the host, and compare under the acceptance
rules (selection exact or within 1e-5 relative of the k-th score; attention
max-abs <= 2e-2 for bf16 latents / 6e-2 for fp8 and rel-L2 <= 1e-2)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from deepseek_sparse_attention_dsa_gb300 import dsa
from deepseek_sparse_attention_dsa_gb300 import workloads as W

ATOL_BF16 = 2e-2
ATOL_FP8 = 6e-2
REL_L2 = 1e-2
TOPK_REL = 1e-5


def host_inputs(wl):
    return W.make_index_cache(wl), W.make_latent_cache(wl), W.make_step_inputs(wl)


def device_inputs(wl, device="cuda"):
    return (W.make_index_cache(wl, device=device), W.make_latent_cache(wl, device=device),
            W.make_step_inputs(wl, device=device))


def to_dev(x, device="cuda"):
    return None if x is None else x.to(device)


def gpu_pipeline(ctx, wl, index_cache, latent_cache, step, want_scores=True, selection=None):
    """store -> (scores) -> index_topk -> attend on the GPU; returns host numpy."""
    plan = ctx.plan(wl.spans, wl.num_pages)
    ctx.store_keys(plan, step.keys, index_cache)
    res = {}
    if want_scores:
        res["scores"] = ctx.index_scores(plan, step.q, step.w, index_cache).cpu().numpy()[:plan.num_scores]
    sel = ctx.index_topk(plan, step.q, step.w, index_cache)
    res["selection"] = sel.cpu().numpy()
    att_sel = sel if selection is None else torch.from_numpy(selection).to(sel.device)
    out = ctx.attend(plan, att_sel, step.q_nope, step.q_pe, latent_cache, step.sink, wl.shape.sm_scale)
    res["out"] = out.float().cpu().numpy()
    res["index_cache"] = index_cache.cpu()
    ctx.get_error()
    plan.close()
    return res


def check_scores(gpu, ref, offsets, rel=2e-5):
    for r in range(len(offsets) - 1):
        a, b = gpu[offsets[r]:offsets[r + 1]], ref[offsets[r]:offsets[r + 1]].astype(np.float64)
        scale = max(1e-30, float(np.abs(b).max()))
        err = np.abs(a.astype(np.float64) - b)
        assert (err <= rel * np.maximum(np.abs(b), scale * 0.05)).all(), (r, float(err.max()), scale)


def check_selection(gpu_sel, ref_sel, ref_scores, offsets, K, exact=False):
    """Same sets (exact), or differing positions within TOPK_REL of the k-th score."""
    T = gpu_sel.shape[0]
    for r in range(T):
        g = gpu_sel[r]
        nvalid = int((g >= 0).sum())
        assert (g[:nvalid] >= 0).all() and (g[nvalid:] == -1).all(), "valid entries first, -1 tail"
        assert np.all(np.diff(g[:nvalid]) > 0), "ascending positions"
        gs, os_ = set(g[:nvalid].tolist()), set(ref_sel[r][ref_sel[r] >= 0].tolist())
        assert len(gs) == len(os_), (r, len(gs), len(os_))
        if gs == os_:
            continue
        assert not exact, ("selection differs", r, sorted(gs ^ os_)[:10])
        s = ref_scores[offsets[r]:offsets[r + 1]].astype(np.float64)
        sk = min(s[j] for j in os_)
        for j in gs ^ os_:
            assert abs(s[j] - sk) <= TOPK_REL * abs(sk), (r, j, s[j], sk)


def check_attention(gpu_out, ref_out, fp8=False):
    atol = ATOL_FP8 if fp8 else ATOL_BF16
    d = np.abs(gpu_out.astype(np.float64) - ref_out)
    assert float(d.max()) <= atol, ("max abs", float(d.max()))
    rel = np.linalg.norm(gpu_out.astype(np.float64) - ref_out) / max(1e-30, np.linalg.norm(ref_out))
    assert rel <= REL_L2, ("rel L2", rel)
    return float(d.max()), float(rel)


def deepseek_small(seed=0, fp8=False, sink=False, page_start=0, integer=False, heads=128, decode_ctx=(2500, 5000, 3001, 700),
                   chunk=(2090, 40), kv_lora_rank=512):
    """DeepSeek-V3.2 shapes (indexer 64x128, topk 2048, MLA 128 x 512+64,
    page 64) at contexts the oracle finishes in seconds: a few decode rows
    and one prefill chunk that crosses topk."""
    sh = W.DSAShape(**dict(W.DEEPSEEK, heads=heads, kv_lora_rank=kv_lora_rank),
                    latent_fmt=W.LATENT_FP8_656 if fp8 else W.LATENT_BF16,
                    index_fmt=W.INDEX_FP8_132 if fp8 else W.INDEX_BF16, has_sink=sink)
    reqs = [(c - 1, 1) for c in decode_ctx] + ([chunk] if chunk else [])
    return W.build_workload("small", sh, reqs, seed, W.Distributions(w=("uniform", 0.0, 0.125), integer=integer),
                            page_start=page_start, spare_pages=3)
