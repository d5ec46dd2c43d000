"""GPU: capturable plans (dsa_plan_capturable / dsa_plan_update).  The device
planner must give the same rows, work and results as the host planner: bit
for bit on decode rows, within the parity tolerances against the oracle on
prefill-chunk rows (the capturable plan scores those one row at a time); a
CUDA graph of update + store + index/top-k + attend must replay correctly
after the spans in device memory are rewritten; padding rows are never
written; invalid spans empty the plan and are reported."""
import numpy as np
import pytest
import torch

import oracle
from deepseek_sparse_attention_dsa_gb300 import dsa
from deepseek_sparse_attention_dsa_gb300 import workloads as W
from tests import harness as H

pytestmark = pytest.mark.gpu

SENTINEL = -7


@pytest.fixture(scope="module", autouse=True)
def built():
    from deepseek_sparse_attention_dsa_gb300 import build
    build.build()


def _device_spans(wl, max_spans, max_page_ids=None):
    """(num_spans (1,), spans (max_spans, 6), pages) int32 device tensors for wl."""
    rows, pages, off = [], [], 0
    for s in wl.spans:
        rows.append([s.q_len, s.ctx_start, s.page_start, off, len(s.pages), 0])
        pages.append(np.asarray(s.pages, np.int32))
        off += len(s.pages)
    sp = np.zeros((max_spans, dsa.DEVICE_SPAN_FIELDS), np.int32)
    sp[:len(rows)] = np.asarray(rows, np.int32)
    pg = np.concatenate(pages).astype(np.int32)
    if max_page_ids is not None:
        pg = np.concatenate([pg, np.zeros(max_page_ids - pg.size, np.int32)])
    return (torch.tensor([len(rows)], dtype=torch.int32, device="cuda"), torch.from_numpy(sp).cuda(),
            torch.from_numpy(pg).cuda())


def _padded(x, rows):
    """x (T, ...) on the device, padded with zeros to `rows` rows."""
    out = torch.zeros((rows,) + tuple(x.shape[1:]), dtype=x.dtype, device="cuda")
    out[:x.shape[0]] = x.cuda()
    return out


def _host_path(ctx, wl, ic, lc, st):
    plan = ctx.plan(wl.spans, wl.num_pages)
    icd, lcd = ic.clone().cuda(), lc.cuda()
    ctx.store_keys(plan, st.keys.cuda(), icd)
    sel = ctx.index_topk(plan, st.q.cuda(), st.w.cuda(), icd)
    sink = st.sink.cuda() if st.sink is not None else None
    out = ctx.attend(plan, sel, st.q_nope.cuda(), st.q_pe.cuda(), lcd, sink, wl.shape.sm_scale)
    ctx.get_error()
    return sel.cpu(), out.cpu(), icd.cpu()


def test_decode_rows_match_the_host_plan_bit_for_bit():
    wl = H.deepseek_small(seed=21, decode_ctx=(2500, 5000, 3001, 700, 4100), chunk=None)
    ic, lc, st = H.host_inputs(wl)
    ctx = dsa.Context(wl.shape, 0)
    sel_h, out_h, ic_h = _host_path(ctx, wl, ic, lc, st)

    R, T, K = 8, wl.num_rows, wl.shape.topk
    max_scores = R * 6000
    plan = ctx.plan_capturable(R, 8, max_scores, wl.num_pages)
    assert plan.num_rows == R and plan.num_scores == max_scores and plan.capturable
    ns, spans, pages = _device_spans(wl, 8)
    ctx.plan_update(plan, ns, spans, pages)
    c = plan.read_counts()
    assert c["valid"] and c["rows"] == T and c["num_scores"] == sum(s.ctx_start + 1 for s in wl.spans)
    icd, lcd = ic.clone().cuda(), lc.cuda()
    ctx.store_keys(plan, _padded(st.keys, R), icd)
    sel = torch.full((R, K), SENTINEL, dtype=torch.int32, device="cuda")
    ctx.index_topk(plan, _padded(st.q, R), _padded(st.w, R), icd, selection=sel)
    out = torch.full((R, wl.shape.heads, wl.shape.kv_lora_rank), 3.0, dtype=torch.bfloat16, device="cuda")
    ctx.attend(plan, sel, _padded(st.q_nope, R), _padded(st.q_pe, R), lcd, None, wl.shape.sm_scale, out)
    ctx.get_error()
    assert torch.equal(icd.cpu(), ic_h)
    assert torch.equal(sel[:T].cpu(), sel_h)
    assert torch.equal(out[:T].cpu(), out_h)
    assert bool((sel[T:] == SENTINEL).all()) and bool((out[T:] == 3.0).all())   # padding untouched
    ref = oracle.attend(wl.shape, wl.spans, wl.num_pages, sel_h.numpy(), st.q_nope, st.q_pe, lc, None)
    H.check_attention(out[:T].float().cpu().numpy(), ref)


def test_chunk_rows_match_the_oracle():
    """A step with decode rows and a prefill chunk that crosses topk, split
    attention rows included: scores, selection and attention against the oracle."""
    wl = H.deepseek_small(seed=22, sink=True, decode_ctx=(2300, 900), chunk=(2040, 24))
    ic, lc, st = H.host_inputs(wl)
    ref = oracle.run_all(wl, ic, lc, st)
    ctx = dsa.Context(wl.shape, 0)
    R = wl.num_rows + 5
    max_scores = int(ref["offsets"][-1]) + 10000
    plan = ctx.plan_capturable(R, 4, max_scores, wl.num_pages)
    ns, spans, pages = _device_spans(wl, 4)
    ctx.plan_update(plan, ns, spans, pages)
    icd, lcd = ic.clone().cuda(), lc.cuda()
    ctx.store_keys(plan, _padded(st.keys, R), icd)
    scores = torch.zeros(max_scores, dtype=torch.float32, device="cuda")
    ctx.index_scores(plan, _padded(st.q, R), _padded(st.w, R), icd, scores=scores)
    sel = ctx.index_topk(plan, _padded(st.q, R), _padded(st.w, R), icd)
    out = ctx.attend(plan, sel, _padded(st.q_nope, R), _padded(st.q_pe, R), lcd, st.sink.cuda(), wl.shape.sm_scale)
    ctx.get_error()
    T = wl.num_rows
    n = int(ref["offsets"][-1])
    H.check_scores(scores[:n].cpu().numpy(), ref["scores"], ref["offsets"])
    H.check_selection(sel[:T].cpu().numpy(), ref["selection"], ref["scores"], ref["offsets"], wl.shape.topk)
    ref_e2e = oracle.attend(wl.shape, wl.spans, wl.num_pages, sel[:T].cpu().numpy(), st.q_nope, st.q_pe, lc, st.sink)
    H.check_attention(out[:T].float().cpu().numpy(), ref_e2e)
    assert plan.read_counts()["split_rows"] >= 0


@pytest.mark.parametrize("fp8", [False, True])
def test_odd_page_starts_match_the_oracle(fp8):
    """A capturable plan with alignment 1 and spans starting at slots 3, 37 and
    61 (bf16 and fp8 keys): the device planner gives the same tile leads as the
    host planner, the indexer stays on the tensor cores, and scores,
    selection and attention match the oracle."""
    wl = H.deepseek_small(seed=27 + fp8, fp8=fp8, sink=fp8, page_start=[3, 37, 61],
                          decode_ctx=(2500, 5000, 700), chunk=None)
    ic, lc, st = H.host_inputs(wl)
    ref = oracle.run_all(wl, ic, lc, st)
    ctx = dsa.Context(wl.shape, 0)
    R = wl.num_rows + 2
    max_scores = int(ref["offsets"][-1]) + 3000
    plan = ctx.plan_capturable(R, 4, max_scores, wl.num_pages)   # page_start_align 1
    assert plan.index_tensor_cores
    ns, spans, pages = _device_spans(wl, 4)
    ctx.plan_update(plan, ns, spans, pages)
    icd, lcd = ic.clone().cuda(), lc.cuda()
    ctx.store_keys(plan, _padded(st.keys, R), icd)
    scores = torch.zeros(max_scores, dtype=torch.float32, device="cuda")
    ctx.index_scores(plan, _padded(st.q, R), _padded(st.w, R), icd, scores=scores)
    sel = ctx.index_topk(plan, _padded(st.q, R), _padded(st.w, R), icd)
    sink = st.sink.cuda() if st.sink is not None else None
    out = ctx.attend(plan, sel, _padded(st.q_nope, R), _padded(st.q_pe, R), lcd, sink, wl.shape.sm_scale)
    ctx.get_error()
    T = wl.num_rows
    n = int(ref["offsets"][-1])
    H.check_scores(scores[:n].cpu().numpy(), ref["scores"], ref["offsets"])
    H.check_selection(sel[:T].cpu().numpy(), ref["selection"], ref["scores"], ref["offsets"], wl.shape.topk)
    ref_e2e = oracle.attend(wl.shape, wl.spans, wl.num_pages, sel[:T].cpu().numpy(), st.q_nope, st.q_pe, lc, st.sink)
    H.check_attention(out[:T].float().cpu().numpy(), ref_e2e, fp8)
    # the host plan of the same step gives bit-identical decode scores
    hplan = ctx.plan(wl.spans, wl.num_pages)
    hs = ctx.index_scores(hplan, st.q.cuda(), st.w.cuda(), icd)
    ctx.get_error()
    assert torch.equal(hs[:n].cpu(), scores[:n].cpu())


def test_graph_replay_follows_the_spans_in_device_memory():
    """Capture update + store + index/top-k + attend once; replay it for two
    different decode steps (other contexts, fewer requests) whose spans, pages,
    caches and inputs are rewritten in place; each replay equals the host path."""
    A = H.deepseek_small(seed=23, decode_ctx=(2500, 5000, 3001, 700), chunk=None)
    B = H.deepseek_small(seed=24, decode_ctx=(4100, 1800, 2900), chunk=None)
    sh = A.shape
    R, S, K = 6, 6, sh.topk
    NP = max(A.num_pages, B.num_pages)
    max_ids = sum(len(s.pages) for s in A.spans) + sum(len(s.pages) for s in B.spans)
    ctx = dsa.Context(sh, 0)
    plan = ctx.plan_capturable(R, S, R * 6000, NP)
    # the buffers the graph is captured on
    ic0, lc0, _ = H.host_inputs(A)
    icd = torch.zeros((NP,) + tuple(ic0.shape[1:]), dtype=ic0.dtype, device="cuda")
    lcd = torch.zeros((NP,) + tuple(lc0.shape[1:]), dtype=lc0.dtype, device="cuda")
    q = torch.zeros((R, sh.index_heads, sh.index_dim), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((R, sh.index_heads), dtype=torch.float32, device="cuda")
    keys = torch.zeros((R, sh.index_dim), dtype=torch.bfloat16, device="cuda")
    qn = torch.zeros((R, sh.heads, sh.kv_lora_rank), dtype=torch.bfloat16, device="cuda")
    qp = torch.zeros((R, sh.heads, sh.rope_dim), dtype=torch.bfloat16, device="cuda")
    sel = torch.full((R, K), SENTINEL, dtype=torch.int32, device="cuda")
    out = torch.zeros((R, sh.heads, sh.kv_lora_rank), dtype=torch.bfloat16, device="cuda")
    ns, spans, pages = _device_spans(A, S, max_ids)

    def step():
        ctx.plan_update(plan, ns, spans, pages)
        ctx.store_keys(plan, keys, icd)
        ctx.index_topk(plan, q, w, icd, selection=sel)
        ctx.attend(plan, sel, qn, qp, lcd, None, sh.sm_scale, out)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()   # warm-up outside the capture (one-time kernel attributes)
    torch.cuda.current_stream().wait_stream(side)
    ctx.get_error()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()

    for wl in (A, B):
        ic, lc, st = H.host_inputs(wl)
        sel_h, out_h, ic_h = _host_path(ctx, wl, ic, lc, st)
        T = wl.num_rows
        icd.zero_()
        icd[:wl.num_pages] = ic.cuda()
        lcd.zero_()
        lcd[:wl.num_pages] = lc.cuda()
        for dst, src in ((q, st.q), (w, st.w), (keys, st.keys), (qn, st.q_nope), (qp, st.q_pe)):
            dst.zero_()
            dst[:T] = src.cuda()
        sel.fill_(SENTINEL)
        n2, s2, p2 = _device_spans(wl, S, max_ids)
        ns.copy_(n2)
        spans.copy_(s2)
        pages.copy_(p2)
        g.replay()
        torch.cuda.synchronize()
        ctx.get_error()
        assert plan.read_counts()["rows"] == T
        assert torch.equal(icd[:wl.num_pages].cpu(), ic_h)
        assert torch.equal(sel[:T].cpu(), sel_h)
        assert bool((sel[T:] == SENTINEL).all())
        assert torch.equal(out[:T].cpu(), out_h)


@pytest.mark.parametrize("bad", ["q_len", "page_off", "short_pages", "num_spans", "rows", "align"])
def test_invalid_spans_empty_the_plan_and_are_reported(bad):
    wl = H.deepseek_small(seed=25, decode_ctx=(2500, 900), chunk=None)
    ic, lc, st = H.host_inputs(wl)
    ctx = dsa.Context(wl.shape, 0)
    R, S = 4, 3
    plan = ctx.plan_capturable(R, S, R * 4000, wl.num_pages, page_start_align=64)
    ns, spans, pages = _device_spans(wl, S)
    ctx.plan_update(plan, ns, spans, pages)   # a valid update first
    assert plan.read_counts()["rows"] == 2
    sp = spans.cpu()
    if bad == "q_len":
        sp[1, 0] = 0
    elif bad == "page_off":
        sp[1, 3] = pages.numel()
    elif bad == "short_pages":
        sp[0, 4] = 1
    elif bad == "num_spans":
        ns.fill_(S + 1)
    elif bad == "rows":
        sp[1, 0] = R   # 1 + R rows
    elif bad == "align":
        sp[0, 2] = 8
    spans.copy_(sp)
    ctx.plan_update(plan, ns, spans, pages)
    with pytest.raises(dsa.DSAError) as e:
        ctx.get_error()
    assert e.value.status == 9
    c = plan.read_counts()
    assert c["rows"] == 0 and not c["valid"] and c["attend_units"] == 0 and c["index_items"] == 0
    sel = torch.full((R, wl.shape.topk), SENTINEL, dtype=torch.int32, device="cuda")
    icd = ic.clone().cuda()
    ctx.store_keys(plan, _padded(st.keys, R), icd)
    ctx.index_topk(plan, _padded(st.q, R), _padded(st.w, R), icd, selection=sel)
    out = torch.full((R, wl.shape.heads, wl.shape.kv_lora_rank), 3.0, dtype=torch.bfloat16, device="cuda")
    ctx.attend(plan, sel, _padded(st.q_nope, R), _padded(st.q_pe, R), lc.cuda(), None, wl.shape.sm_scale, out)
    ctx.get_error()
    assert bool((sel == SENTINEL).all()) and bool((out == 3.0).all())
    assert torch.equal(icd.cpu(), ic)   # an emptied plan stores nothing


def test_fp8_caches_sink_and_shared_layer_match_the_host_plan():
    """fp8 index / latent caches, an attention sink, split rows, and a SHARED
    layer attending over the selection the capturable plan's FULL layer wrote."""
    wl = H.deepseek_small(seed=26, fp8=True, sink=True, decode_ctx=(2500, 5000, 700), chunk=None)
    ic, lc, st = H.host_inputs(wl)
    ctx = dsa.Context(wl.shape, 0)
    sel_h, out_h, ic_h = _host_path(ctx, wl, ic, lc, st)
    R, T = 4, wl.num_rows
    plan = ctx.plan_capturable(R, 4, R * 6000, wl.num_pages)
    ns, spans, pages = _device_spans(wl, 4)
    ctx.plan_update(plan, ns, spans, pages)
    icd, lcd = ic.clone().cuda(), lc.cuda()
    ctx.store_keys(plan, _padded(st.keys, R), icd)
    sel = ctx.index_topk(plan, _padded(st.q, R), _padded(st.w, R), icd)
    out = ctx.attend(plan, sel, _padded(st.q_nope, R), _padded(st.q_pe, R), lcd, st.sink.cuda(), wl.shape.sm_scale)
    shared = ctx.attend_shared(plan, _padded(st.q_nope, R), _padded(st.q_pe, R), lcd, st.sink.cuda(),
                               wl.shape.sm_scale)
    ctx.get_error()
    assert torch.equal(icd.cpu(), ic_h)
    assert torch.equal(sel[:T].cpu(), sel_h)
    assert torch.equal(out[:T].cpu(), out_h)
    assert torch.equal(shared[:T].cpu(), out_h)   # same queries, same recorded selection
    assert plan.read_counts()["split_rows"] > 0
