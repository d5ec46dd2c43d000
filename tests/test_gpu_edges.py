"""Edge cases through the C ABI against the oracle: empty steps reach every
entry point and launch nothing; rows at the selection boundaries (a row at
position 0, rows that see topk-1, topk and topk+1 keys) select, pad and
attend exactly as the oracle; block-sparse MSA rows at block boundaries (one
position past a block, exactly topk_blocks blocks, one block more)."""
import numpy as np
import pytest
import torch

import oracle
from deepseek_sparse_attention_dsa_gb300 import dsa
from deepseek_sparse_attention_dsa_gb300 import workloads as W
from tests import harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from deepseek_sparse_attention_dsa_gb300 import build
    build.build()


def test_empty_steps_reach_every_call_and_launch_nothing():
    sh = W.DSAShape(**W.DEEPSEEK)
    ctx = dsa.Context(sh, 0)
    plan = ctx.plan([], cache_pages=1)
    assert plan.num_rows == 0 and plan.num_scores == 0
    dev = torch.device("cuda", 0)
    z = lambda *shape, dt=torch.bfloat16: torch.zeros(*shape, dtype=dt, device=dev)   # noqa: E731
    ic = z(1, sh.page_size, sh.index_dim)
    lc = z(1, sh.page_size, sh.kv_lora_rank + sh.rope_dim)
    ctx.store_keys(plan, z(0, sh.index_dim), ic)
    assert ctx.last_launch_count() == 0
    ctx.index_scores(plan, z(0, sh.index_heads, sh.index_dim), z(0, sh.index_heads, dt=torch.float32), ic,
                     z(1, dt=torch.float32))
    assert ctx.last_launch_count() == 0
    sel = ctx.index_topk(plan, z(0, sh.index_heads, sh.index_dim), z(0, sh.index_heads, dt=torch.float32), ic)
    assert sel.shape == (0, sh.topk) and ctx.last_launch_count() == 0
    out = ctx.attend(plan, sel, z(0, sh.heads, sh.kv_lora_rank), z(0, sh.heads, sh.rope_dim), lc, None, sh.sm_scale)
    assert out.shape[0] == 0 and ctx.last_launch_count() == 0
    ms = W.MSAShape()
    msa_ctx = dsa.Context(ms.index_shape(), 0)
    mplan = msa_ctx.plan([], cache_pages=1)
    bsel = msa_ctx.msa_select_blocks(mplan, ms, z(1, dt=torch.float32))
    assert bsel.shape == (0, ms.topk_blocks) and msa_ctx.last_launch_count() == 0
    mout = msa_ctx.msa_attend(mplan, ms, bsel, z(0, ms.q_heads, ms.head_dim), z(1, ms.page_size, ms.kv_row_elems),
                              ms.sm_scale)
    assert mout.shape[0] == 0 and msa_ctx.last_launch_count() == 0
    ctx.get_error()
    msa_ctx.get_error()


def test_rows_at_the_selection_boundaries():
    """Rows at positions 0, 2046, 2047, 2048 and 4096 (topk 2048): one key;
    topk-1 keys (every key kept, one -1); exactly topk (every key, no -1);
    topk+1 (the first row that drops a key); and a longer row."""
    wl = H.deepseek_small(seed=61, decode_ctx=(1, 2047, 2048, 2049, 4097), chunk=None)
    ic, lc, st = H.host_inputs(wl)
    ref = oracle.run_all(wl, ic, lc, st)
    ctx = dsa.Context(wl.shape, 0)
    dev = W.StepInputs(*(H.to_dev(x) for x in (st.q, st.w, st.keys, st.q_nope, st.q_pe, st.sink)))
    got = H.gpu_pipeline(ctx, wl, ic.cuda(), lc.cuda(), dev)
    H.check_scores(got["scores"], ref["scores"], ref["offsets"])
    H.check_selection(got["selection"], ref["selection"], ref["scores"], ref["offsets"], wl.shape.topk)
    counts = (got["selection"] >= 0).sum(axis=1)
    assert counts.tolist() == [1, 2047, 2048, 2048, 2048]
    ref_e2e = oracle.attend(wl.shape, wl.spans, wl.num_pages, got["selection"], st.q_nope, st.q_pe, lc, st.sink)
    H.check_attention(got["out"], ref_e2e)
    plan = ctx.plan(wl.spans, wl.num_pages)
    assert plan.needs_selection   # the rows at 2048 and 4096 see more than topk keys


def test_msa_rows_at_block_boundaries():
    """Rows at positions 0, 127, 128, 2047 and 2048 with blocks of 128 and
    topk_blocks 16: one block; one full block; a second block holding a single
    visible position; exactly 16 blocks (all kept); 17 blocks (one dropped)."""
    ms = W.MSAShape(q_heads=16, kv_heads=2)
    wl = W.build_workload("msa_edges", ms.index_shape(), [(0, 1), (127, 1), (128, 1), (2047, 1), (2048, 1)], 2201,
                          W.Distributions(w=("uniform", 0.0, 1.0 / 8)))
    wl.msa = ms
    ic, kv, st, q = (W.make_index_cache(wl), W.make_kv_cache(wl), W.make_step_inputs(wl), W.make_msa_q(wl))
    ref = oracle.msa_run_all(wl, ic, kv, st, q)
    ctx = dsa.Context(wl.shape, 0)
    plan = ctx.plan(wl.spans, wl.num_pages)
    icd = ic.cuda()
    ctx.store_keys(plan, st.keys.cuda(), icd)
    sel = ctx.msa_index_select(plan, ms, st.q.cuda(), st.w.cuda(), icd)
    out = ctx.msa_attend(plan, ms, sel, q.cuda(), kv.cuda(), ms.sm_scale)
    ctx.get_error()
    g = sel.cpu().numpy()
    H.check_selection(g, ref["selection"], ref["block_scores"], ref["block_offsets"], ms.topk_blocks)
    assert (g >= 0).sum(axis=1).tolist() == [1, 1, 2, 16, 16]
    ref_e2e = oracle.msa_attend(ms, wl.spans, wl.num_pages, g, q, kv)
    H.check_attention(out.float().cpu().numpy(), ref_e2e)
