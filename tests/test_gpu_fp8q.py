"""GPU: the indexer with an fp8 query (dsa_quantize_q, dsa_index_scores_fp8q,
dsa_index_topk_fp8q) against the CPU oracle: the query codes and scales byte
for byte, the scores within the parity tolerance, the selection under the
tie rule; on a capturable plan too; refused for the bf16 index format."""
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


@pytest.mark.parametrize("page_start", [0, 8])
def test_fp8_query_matches_the_oracle(page_start):
    wl = H.deepseek_small(seed=41 + page_start, fp8=True, page_start=page_start, decode_ctx=(2500, 5000, 700),
                          chunk=(2090, 40))
    ic, lc, st = H.host_inputs(wl)
    ctx = dsa.Context(wl.shape, 0)
    plan = ctx.plan(wl.spans, wl.num_pages)
    icd = ic.clone().cuda()
    ctx.store_keys(plan, st.keys.cuda(), icd)
    codes, scales = ctx.quantize_q(plan, st.q.cuda())
    ref_codes, ref_scales = oracle.quantize_rows(st.q, 128)
    assert np.array_equal(codes.cpu().numpy().reshape(-1), ref_codes)
    assert np.array_equal(scales.cpu().numpy().reshape(-1), ref_scales)
    scores = ctx.index_scores_fp8q(plan, codes, scales, st.w.cuda(), icd)
    sel = ctx.index_topk_fp8q(plan, codes, scales, st.w.cuda(), icd)
    ctx.get_error()
    cache = oracle.store_keys(wl.shape, wl.spans, wl.num_pages, st.keys, ic)
    ref, off = oracle.index_scores_fp8q(wl.shape, wl.spans, wl.num_pages, ref_codes, ref_scales, st.w, cache)
    H.check_scores(scores.cpu().numpy()[:int(off[-1])], ref, off)
    H.check_selection(sel.cpu().numpy(), oracle.topk(wl.shape, wl.spans, ref, off), ref, off, wl.shape.topk)


def test_fp8_query_on_a_capturable_plan_equals_the_host_plan():
    wl = H.deepseek_small(seed=43, fp8=True, decode_ctx=(2500, 5000, 3001, 700), chunk=None)
    ic, lc, st = H.host_inputs(wl)
    ctx = dsa.Context(wl.shape, 0)
    plan = ctx.plan(wl.spans, wl.num_pages)
    icd = ic.clone().cuda()
    ctx.store_keys(plan, st.keys.cuda(), icd)
    codes, scales = ctx.quantize_q(plan, st.q.cuda())
    sel_h = ctx.index_topk_fp8q(plan, codes, scales, st.w.cuda(), icd)
    R, T = 6, wl.num_rows
    cap = ctx.plan_capturable(R, 6, R * 6000, wl.num_pages, page_start_align=64)
    rows, pages, o = [], [], 0
    for s in wl.spans:
        rows.append([s.q_len, s.ctx_start, s.page_start, o, len(s.pages), 0])
        pages.append(np.asarray(s.pages, np.int32))
        o += len(s.pages)
    sp = np.zeros((6, 6), np.int32)
    sp[:len(rows)] = rows
    ctx.plan_update(cap, torch.tensor([len(rows)], dtype=torch.int32, device="cuda"), torch.from_numpy(sp).cuda(),
                    torch.from_numpy(np.concatenate(pages)).cuda())
    qpad = torch.zeros((R,) + tuple(st.q.shape[1:]), dtype=torch.bfloat16, device="cuda")
    qpad[:T] = st.q.cuda()
    wpad = torch.zeros((R, wl.shape.index_heads), dtype=torch.float32, device="cuda")
    wpad[:T] = st.w.cuda()
    c2 = torch.full((R, wl.shape.index_heads, 128), 7, dtype=torch.uint8, device="cuda")
    s2 = torch.full((R, wl.shape.index_heads), -3.0, dtype=torch.float32, device="cuda")
    ctx.quantize_q(cap, qpad, c2, s2)
    sel_c = ctx.index_topk_fp8q(cap, c2, s2, wpad, icd)
    ctx.get_error()
    assert torch.equal(c2[:T], codes) and torch.equal(s2[:T], scales)
    assert bool((c2[T:] == 7).all()) and bool((s2[T:] == -3.0).all())   # padding rows untouched
    assert torch.equal(sel_c[:T].cpu(), sel_h.cpu())


def test_fp8_query_needs_the_fp8_index_format():
    wl = H.deepseek_small(seed=44, decode_ctx=(900,), chunk=None)
    ctx = dsa.Context(wl.shape, 0)
    plan = ctx.plan(wl.spans, wl.num_pages)
    T = wl.num_rows
    codes = torch.zeros((T, 64, 128), dtype=torch.uint8, device="cuda")
    scales = torch.ones((T, 64), dtype=torch.float32, device="cuda")
    with pytest.raises(dsa.DSAError) as e:
        ctx.index_scores_fp8q(plan, codes, scales, torch.zeros((T, 64), device="cuda"),
                              torch.zeros(16, dtype=torch.uint8, device="cuda"))
    assert e.value.status == 7
