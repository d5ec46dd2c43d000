"""GPU parity for block-sparse MSA (LLMServingSim, "Sparse attention (DSA and
block-sparse MSA)", MiniMax-M3 column): the CUDA block selection and GQA
attention through the C ABI against the CPU oracle on the same seeded inputs,
at small sizes (every row) and at the msa_decode workload's full size
(sampled rows recomputed by the oracle)."""
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


def _inputs(wl, device="cpu"):
    return (W.make_index_cache(wl, device=device), W.make_kv_cache(wl, device=device),
            W.make_step_inputs(wl, device=device), W.make_msa_q(wl, device=device))


def _run(wl, expect_tc=True, exact_selection=False):
    ms = wl.msa
    ic, kv, st, q = _inputs(wl)
    ref = oracle.msa_run_all(wl, ic, kv, st, q)
    ctx = dsa.Context(wl.shape, 0)
    plan = ctx.plan(wl.spans, wl.num_pages)
    assert ctx.msa_attend_on_tensor_cores(plan, ms) == expect_tc
    icd, kvd, qd = ic.cuda(), kv.cuda(), q.cuda()
    ctx.store_keys(plan, st.keys.cuda(), icd)
    scores = ctx.index_scores(plan, st.q.cuda(), st.w.cuda(), icd)
    sel = ctx.msa_select_blocks(plan, ms, scores)
    sel2 = ctx.msa_index_select(plan, ms, st.q.cuda(), st.w.cuda(), icd)
    out = ctx.msa_attend(plan, ms, sel, qd, kvd, ms.sm_scale)
    ctx.get_error()
    assert torch.equal(sel, sel2)
    H.check_scores(scores.cpu().numpy()[:plan.num_scores], ref["scores"], ref["offsets"])
    # the GPU's blocks against the oracle's, under the block scores the oracle computed
    H.check_selection(sel.cpu().numpy(), ref["selection"], ref["block_scores"], ref["block_offsets"],
                      ms.topk_blocks, exact=exact_selection)
    # the selection of the oracle's own scores is the oracle's, exactly
    sel_o = ctx.msa_select_blocks(plan, ms, torch.from_numpy(ref["scores"]).cuda())
    ctx.get_error()
    H.check_selection(sel_o.cpu().numpy(), ref["selection"], ref["block_scores"], ref["block_offsets"],
                      ms.topk_blocks, exact=True)
    # end to end: the oracle attends over the GPU's selection
    ref_e2e = oracle.msa_attend(ms, wl.spans, wl.num_pages, sel.cpu().numpy(), q, kv)
    H.check_attention(out.float().cpu().numpy(), ref_e2e)
    # decoupled: the GPU attends over the oracle's selection (score-ordered)
    out_o = ctx.msa_attend(plan, ms, torch.from_numpy(ref["selection"]).cuda(), qd, kvd, ms.sm_scale)
    ctx.get_error()
    H.check_attention(out_o.float().cpu().numpy(), ref["out"])
    plan.close()
    return ref


def test_msa_small():
    _run(W.msa_config("msa_small"))


def test_msa_integer_index_inputs_select_exactly():
    """Integer-valued index keys and queries make every token score exact, so
    the block selection must be the oracle's set exactly, ties included."""
    wl = W.msa_config("msa_small", seed=2101)
    wl.dist = W.Distributions(w=("uniform", 0.0, 1.0 / 8), integer=True)
    _run(wl, exact_selection=True)


def test_msa_page_start_off_the_box_boundary():
    """Token 0 at slots 5, 37 and 70: every block spans two tiles of the
    attention; rows outside the kept blocks are masked and their V rows zeroed."""
    _run(W.msa_config("msa_small", seed=2102, page_start=[5, 37, 70]))


def test_msa_more_heads_per_group_and_one_kv_head():
    """Other tensor-core instances: 32 query heads on one kv head (N = 32), 40
    heads over 2 kv heads (a group of 20 padded to 32)."""
    for qh, kh, seed in ((32, 1, 2103), (40, 2, 2104)):
        wl = W.msa_config("msa_small", seed=seed)
        wl.msa = W.MSAShape(topk_blocks=4, q_heads=qh, kv_heads=kh)
        _run(wl)


@pytest.mark.parametrize("q_heads,kv_heads,page_start",
                         [(8, 2, 0), (32, 1, [13, 0, 70, 101, 3]), (16, 4, [5, 37, 0, 64, 0]),
                          (40, 2, [0, 9, 0, 0, 77])])
def test_msa_rows_walked_by_persistent_ctas(q_heads, kv_heads, page_start):
    """541 rows, more than the SMs: each CTA of the persistent grid walks three
    or four rows (its two tile-list buffers reused, the next row's Q and
    loads overlapping the current row's tail, each row's output written
    during the next row when two O buffers fit, at the row's end otherwise),
    with one or two softmax groups (odd and even kv head counts), rows of a
    single tile (one step per group) and token 0 on and off the box
    boundary; every row against the oracle."""
    ms = W.MSAShape(topk_blocks=4, q_heads=q_heads, kv_heads=kv_heads)
    reqs = [(600, 200), (900, 150), (1499, 1), (300, 60), (0, 130)]
    wl = W.build_workload("msa_rows", ms.index_shape(), reqs, 2110 + kv_heads,
                          W.Distributions(w=("uniform", 0.0, 1.0 / 8)), page_start=page_start)
    wl.msa = ms
    _run(wl)


@pytest.mark.parametrize("page_start,block_size", [(0, 128), ([5, 37, 70, 101], 128), ([3, 0, 63, 29], 64)])
def test_msa_block_maxima_from_the_indexer_epilogue(page_start, block_size):
    """Decode-only steps take the indexer's block-maximum epilogue (no token
    scores): its selection equals the score path's exactly and matches the
    oracle.  Token 0 off the 32-key boundary puts warps across block edges;
    blocks of 64 put two blocks in one 128-key tile."""
    sh = W.MSAShape(block_size=block_size, topk_blocks=6, q_heads=8, kv_heads=2,
                    head_dim=128 if block_size == 128 else 64,
                    sm_scale=1.0 / np.sqrt(128.0 if block_size == 128 else 64.0))
    wl = W.build_workload("msa_fused", sh.index_shape(), [(1499, 1), (699, 1), (2999, 1), (130, 1)], 2106,
                          W.Distributions(w=("uniform", 0.0, 1.0 / 8)), page_start=page_start)
    wl.msa = sh
    ic, kv, st, q = _inputs(wl)
    ref = oracle.msa_run_all(wl, ic, kv, st, q)
    ctx = dsa.Context(wl.shape, 0)
    plan = ctx.plan(wl.spans, wl.num_pages)
    icd = ic.cuda()
    ctx.store_keys(plan, st.keys.cuda(), icd)
    fused = ctx.msa_index_select(plan, sh, st.q.cuda(), st.w.cuda(), icd)
    scores = ctx.index_scores(plan, st.q.cuda(), st.w.cuda(), icd)
    via_scores = ctx.msa_select_blocks(plan, sh, scores)
    ctx.get_error()
    assert torch.equal(fused, via_scores)
    H.check_selection(fused.cpu().numpy(), ref["selection"], ref["block_scores"], ref["block_offsets"],
                      sh.topk_blocks)


def test_msa_radix_selection_exact_on_integer_inputs():
    """Rows of 260-550 blocks take the radix path of the block selection;
    integer-valued index inputs on a 4 x 32 indexer make every token score
    exact and small, so block maxima tie at the k-th block (two of the rows
    drop a tie there) and the kept set must be the oracle's exactly (ties to
    the lower block), through the indexer's block-maximum epilogue and
    through stored scores alike."""
    sh = W.MSAShape(topk_blocks=16, q_heads=8, kv_heads=2, index_heads=4, index_dim=32)
    wl = W.build_workload("msa_radix", sh.index_shape(), [(33300, 1), (70000, 1), (47999, 1)], 2107,
                          W.Distributions(w=("uniform", 0.0, 1.0 / 8), integer=True))
    wl.msa = sh
    ic, kv, st, q = _inputs(wl)
    ref = oracle.msa_run_all(wl, ic, kv, st, q)
    ctx = dsa.Context(wl.shape, 0)
    plan = ctx.plan(wl.spans, wl.num_pages)
    icd = ic.cuda()
    ctx.store_keys(plan, st.keys.cuda(), icd)
    fused = ctx.msa_index_select(plan, sh, st.q.cuda(), st.w.cuda(), icd)
    scores = ctx.index_scores(plan, st.q.cuda(), st.w.cuda(), icd)
    via_scores = ctx.msa_select_blocks(plan, sh, scores)
    ctx.get_error()
    assert torch.equal(fused, via_scores)
    H.check_selection(fused.cpu().numpy(), ref["selection"], ref["block_scores"], ref["block_offsets"],
                      sh.topk_blocks, exact=True)
    out = ctx.msa_attend(plan, sh, fused, q.cuda(), kv.cuda(), sh.sm_scale)
    ctx.get_error()
    H.check_attention(out.float().cpu().numpy(), ref["out"])


def test_msa_cuda_core_shapes():
    """Shapes outside the tensor-core kernel (head_dim 64, blocks of 64) run the
    CUDA-core kernel, checked the same way."""
    wl = W.msa_config("msa_small", seed=2105)
    wl.msa = W.MSAShape(block_size=64, topk_blocks=6, q_heads=8, kv_heads=2, head_dim=64,
                        sm_scale=1.0 / np.sqrt(64.0))
    _run(wl, expect_tc=False)


def _full_size_sampled_rows(name, nsample, seed):
    """The whole MSA step of `name` at full size on the GPU, in the bench's
    launch configuration (the fused index-select call), with the score path
    beside it; `nsample` sampled rows recomputed by the oracle."""
    wl = W.msa_config(name)
    ms, sh = wl.msa, wl.shape
    dev = torch.device("cuda", 0)
    ic = W.make_index_cache(wl, device=dev)
    kv = W.make_kv_cache(wl, device=dev)
    st = W.make_step_inputs(wl, device=dev)
    q = W.make_msa_q(wl, device=dev)
    ctx = dsa.Context(sh, 0)
    plan = ctx.plan(wl.spans, wl.num_pages)
    assert ctx.msa_attend_on_tensor_cores(plan, ms)
    ctx.store_keys(plan, st.keys, ic)
    sel = ctx.msa_index_select(plan, ms, st.q, st.w, ic)
    scores = ctx.index_scores(plan, st.q, st.w, ic)
    sel_s = ctx.msa_select_blocks(plan, ms, scores)
    out = ctx.msa_attend(plan, ms, sel, q, kv, ms.sm_scale)
    ctx.get_error()
    # block maxima from the indexer's epilogue select what the stored scores select
    assert torch.equal(sel, sel_s)
    span_of, pos_all, _ = wl.row_table()
    off_all = np.zeros(wl.num_rows + 1, np.int64)
    np.cumsum(pos_all + 1, out=off_all[1:])
    rng = np.random.default_rng(seed)
    for row in rng.choice(wl.num_rows, size=nsample, replace=False):
        row = int(row)
        span_i = int(span_of[row])
        rw = wl.row_workload(span_i, row - wl.spans[span_i].q_start)
        ric = W.make_index_cache(rw)
        rst = W.make_step_inputs(rw)
        cache = oracle.store_keys(sh, rw.spans, rw.num_pages, rst.keys, ric)
        sc, off = oracle.index_scores(sh, rw.spans, rw.num_pages, rst.q, rst.w, cache)
        H.check_scores(scores[off_all[row]:off_all[row + 1]].cpu().numpy(), sc, off)
        bsc, boff = oracle.msa_block_scores(ms, rw.spans, sc, off)
        osel = oracle.msa_select(ms, rw.spans, bsc, boff)
        g_sel = sel[row:row + 1].cpu().numpy()
        H.check_selection(g_sel, osel, bsc, boff, ms.topk_blocks)
        # attention over the GPU's blocks, recomputed from the rows they hold
        p = int(pos_all[row])
        toks = set()
        for b in g_sel[0][g_sel[0] >= 0]:
            toks.update(rw.spans[0].token_base + np.arange(b * ms.block_size, min((b + 1) * ms.block_size, p + 1)))
        rkv = W.make_kv_cache(rw, tokens=toks)
        rq = W.make_msa_q(rw)
        ref = oracle.msa_attend(ms, rw.spans, rw.num_pages, g_sel, rq, rkv)
        H.check_attention(out[row:row + 1].float().cpu().numpy(), ref)


def test_msa_decode_full_size_sampled_rows():
    """msa_decode at full size (128 rows at 64K-128K, top 16 blocks of 128, 64
    query heads over 4 kv heads): 16 sampled rows recomputed by the oracle."""
    _full_size_sampled_rows("msa_decode", 16, 7)


def test_msa_prefill_full_size_sampled_rows():
    """msa_prefill at full size (one request, 8,192 new rows after 8,192
    cached; multi-row indexer groups): 12 sampled rows recomputed by the
    oracle."""
    _full_size_sampled_rows("msa_prefill", 12, 8)
