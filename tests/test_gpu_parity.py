"""GPU parity: the CUDA library (through the C ABI) against the CPU oracle on
the same seeded inputs, at sizes the oracle finishes in seconds that still
span several tiles and a ragged tail."""
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


def _run(wl, attend_with_oracle_selection=True, exact_selection=False):
    ic, lc, st = H.host_inputs(wl)
    ref = oracle.run_all(wl, ic, lc, st)
    ctx = dsa.Context(wl.shape, 0)
    dev = W.StepInputs(*(H.to_dev(x) for x in (st.q, st.w, st.keys, st.q_nope, st.q_pe, st.sink)))
    got = H.gpu_pipeline(ctx, wl, ic.cuda(), lc.cuda(), dev)
    # the stored cache is the oracle's, byte for byte
    assert np.array_equal(got["index_cache"].view(torch.uint8).numpy().reshape(-1),
                          ref["index_cache"].reshape(-1))
    H.check_scores(got["scores"], ref["scores"], ref["offsets"])
    H.check_selection(got["selection"], ref["selection"], ref["scores"], ref["offsets"], wl.shape.topk,
                      exact=exact_selection)
    fp8 = wl.shape.latent_fmt == W.LATENT_FP8_656
    # end to end: the oracle attends over the GPU's selection (same rows, same set)
    ref_e2e = oracle.attend(wl.shape, wl.spans, wl.num_pages, got["selection"], st.q_nope, st.q_pe, lc, st.sink)
    H.check_attention(got["out"], ref_e2e, fp8)
    if attend_with_oracle_selection:
        # decoupled: the GPU attends over the oracle's selection
        plan = ctx.plan(wl.spans, wl.num_pages)
        out = ctx.attend(plan, torch.from_numpy(ref["selection"]).cuda(), dev.q_nope, dev.q_pe, lc.cuda(), dev.sink,
                         wl.shape.sm_scale)
        ctx.get_error()
        H.check_attention(out.float().cpu().numpy(), ref["out"], fp8)
    return ctx, ref, got


def test_tiny_prefill_config():
    _run(W.config(0))


def test_tiny_prefill_integer_inputs_bit_exact():
    wl = W.config(0)
    wl.dist = W.Distributions(integer=True)
    ic, lc, st = H.host_inputs(wl)
    ref = oracle.run_all(wl, ic, lc, st)
    ctx = dsa.Context(wl.shape, 0)
    dev = W.StepInputs(*(H.to_dev(x) for x in (st.q, st.w, st.keys, st.q_nope, st.q_pe, st.sink)))
    got = H.gpu_pipeline(ctx, wl, ic.cuda(), lc.cuda(), dev)
    assert np.array_equal(got["scores"], ref["scores"])
    H.check_selection(got["selection"], ref["selection"], ref["scores"], ref["offsets"], wl.shape.topk, exact=True)


def test_deepseek_shapes_bf16():
    _run(H.deepseek_small(seed=1))


def test_deepseek_shapes_integer_bit_exact():
    wl = H.deepseek_small(seed=2, integer=True, decode_ctx=(2300, 4100), chunk=(2040, 24))
    ic, lc, st = H.host_inputs(wl)
    cache = oracle.store_keys(wl.shape, wl.spans, wl.num_pages, st.keys, ic)
    sc, off = oracle.index_scores(wl.shape, wl.spans, wl.num_pages, st.q, st.w, cache)
    sel = oracle.topk(wl.shape, wl.spans, sc, off)
    ctx = dsa.Context(wl.shape, 0)
    plan = ctx.plan(wl.spans, wl.num_pages)
    icd = ic.cuda()
    ctx.store_keys(plan, st.keys.cuda(), icd)
    g_sc = ctx.index_scores(plan, st.q.cuda(), st.w.cuda(), icd).cpu().numpy()[:plan.num_scores]
    assert np.array_equal(g_sc, sc)
    g_sel = ctx.index_topk(plan, st.q.cuda(), st.w.cuda(), icd).cpu().numpy()
    ctx.get_error()
    H.check_selection(g_sel, sel, sc, off, wl.shape.topk, exact=True)


def test_deepseek_shapes_page_start_and_sink():
    _run(H.deepseek_small(seed=3, sink=True, page_start=8, decode_ctx=(2049, 3333), chunk=(1990, 70)))


def test_deepseek_shapes_fewer_heads():
    _run(H.deepseek_small(seed=4, heads=64, decode_ctx=(2600,), chunk=(2040, 16)))


@pytest.mark.parametrize("kv_lora_rank,heads,fp8", [(256, 128, False), (128, 128, False), (256, 40, False),
                                                  (512, 72, True), (256, 128, True)])
def test_attention_other_latent_widths(kv_lora_rank, heads, fp8):
    """The tensor-core attention at its other latent widths (each CTA of the
    pair owns 128 or 64 latent columns instead of 256) and with fewer heads
    than the 128 TMEM lanes (40 and 72 split a warp of heads); fp8 latents of
    width 256 take the CUDA-core kernel."""
    _run(H.deepseek_small(seed=20 + kv_lora_rank // 64 + heads + fp8, kv_lora_rank=kv_lora_rank, heads=heads,
                          fp8=fp8, sink=fp8, decode_ctx=(2300, 700), chunk=(2040, 12)))


def test_fp8_formats():
    _run(H.deepseek_small(seed=5, fp8=True, sink=True, decode_ctx=(2200, 2900), chunk=(2030, 24)))


@pytest.mark.parametrize("fp8", [False, True])
def test_any_page_start_stays_on_tensor_cores(fp8):
    """Spans whose token 0 sits at any slot of a page (page_start 3, 37, 0, 61
    and 70, which also skips the first page's start): key tiles start on the
    box boundary below page_start, the epilogue drops the rows before token 0,
    and the plan keeps the tensor-core indexer (bf16 and fp8 keys)."""
    wl = H.deepseek_small(seed=50 + fp8, fp8=fp8, sink=fp8, page_start=[3, 37, 0, 61, 70],
                          decode_ctx=(2049, 130, 4097, 700), chunk=(1990, 70))
    ctx, ref, got = _run(wl)
    plan = ctx.plan(wl.spans, wl.num_pages)
    assert plan.index_tensor_cores and plan.info.index_box_rows == 64
    plan.close()


def test_fp8_power_of_two_scales():
    """An extra exactness case: fp8 rows packed with power-of-two scales, under
    which the attention producers' code x scale is exact in bf16 and the fp8-key
    epilogue's factored scale is exact; the tolerances are the same."""
    wl = H.deepseek_small(seed=6, fp8=True, sink=True, decode_ctx=(2200, 2900), chunk=(2030, 24))
    wl.dist = W.Distributions(w=("uniform", 0.0, 0.125), fp8_scale="pow2")
    _run(wl)


def test_fp8_page_start_ragged():
    """fp8 keys and latents with spans starting mid-page, a context shorter than
    one key tile and chunks whose tails leave partial tiles and groups."""
    _run(H.deepseek_small(seed=7, fp8=True, page_start=8, decode_ctx=(2049, 130, 4097), chunk=(1990, 70)))


def test_topk_from_oracle_scores_is_exact():
    """Given the oracle's own fp32 scores, the GPU selection is the oracle's set exactly."""
    for wl in (W.config(0), H.deepseek_small(seed=6, decode_ctx=(9000, 2049, 2048, 100), chunk=(2000, 100))):
        ic, lc, st = H.host_inputs(wl)
        cache = oracle.store_keys(wl.shape, wl.spans, wl.num_pages, st.keys, ic)
        sc, off = oracle.index_scores(wl.shape, wl.spans, wl.num_pages, st.q, st.w, cache)
        sel = oracle.topk(wl.shape, wl.spans, sc, off)
        ctx = dsa.Context(wl.shape, 0)
        plan = ctx.plan(wl.spans, wl.num_pages)
        g = ctx.topk_from_scores(plan, torch.from_numpy(sc).cuda()).cpu().numpy()
        H.check_selection(g, sel, sc, off, wl.shape.topk, exact=True)


def test_topk_ties_and_signed_zero():
    """Many equal scores (including -0.0 vs +0.0): the earliest positions win."""
    sh = W.DSAShape(**W.DEEPSEEK)
    n = 5000
    wl = W.build_workload("ties", sh, [(n - 1, 1), (n - 1, 1)], seed=9)
    off = np.array([0, n, 2 * n], np.int64)
    rng = np.random.default_rng(0)
    a = rng.integers(0, 3, size=n).astype(np.float32)          # three values, massive ties
    b = np.zeros(n, np.float32)
    b[rng.random(n) < 0.5] = -0.0
    b[:100] = 1.0
    sc = np.concatenate([a, b])
    ref = oracle.topk(sh, wl.spans, sc, off)
    ctx = dsa.Context(sh, 0)
    plan = ctx.plan(wl.spans, wl.num_pages)
    g = ctx.topk_from_scores(plan, torch.from_numpy(sc).cuda()).cpu().numpy()
    H.check_selection(g, ref, sc, off, sh.topk, exact=True)


def test_topk_paths():
    """Rows that take each path of the selection kernel: every key a candidate,
    a strided sample, a sample the data fools (fallback to exact passes over
    the row), a row longer than the position bitmap, and threshold ties below,
    equal to and above what the tie ranking holds."""
    sh = W.DSAShape(**W.DEEPSEEK)
    K = sh.topk
    rng = np.random.default_rng(11)
    rows = []
    rows.append(rng.standard_normal(8000).astype(np.float32))                     # all candidates
    rows.append(rng.standard_normal(100000).astype(np.float32))                   # sampled
    rows.append(rng.standard_normal(300000).astype(np.float32))                   # past the bitmap
    fool = (rng.random(50000) * 10 + 1).astype(np.float32)
    fool[:: 50000 // 4096] = 0.0                                                  # the sample sees only zeros
    rows.append(fool)
    for n_tie, n_top in ((3000, 1000), (1500, 1000), (1048, 1000)):               # ties > cap, <= cap, == need
        r = (rng.random(20000) * 0.5).astype(np.float32)
        idx = rng.permutation(20000)
        r[idx[:n_top]] = (2.0 + rng.random(n_top)).astype(np.float32)
        r[idx[n_top:n_top + n_tie]] = 1.0
        rows.append(r)
    reqs = [(len(r) - 1, 1) for r in rows]
    wl = W.build_workload("topk_paths", sh, reqs, seed=12)
    off = np.zeros(len(rows) + 1, np.int64)
    off[1:] = np.cumsum([len(r) for r in rows])
    sc = np.concatenate(rows)
    ref = oracle.topk(sh, wl.spans, sc, off)
    ctx = dsa.Context(sh, 0)
    plan = ctx.plan(wl.spans, wl.num_pages)
    assert plan.num_scores == len(sc)
    g = ctx.topk_from_scores(plan, torch.from_numpy(sc).cuda()).cpu().numpy()
    ctx.get_error()
    H.check_selection(g, ref, sc, off, K, exact=True)


def test_topk_many_rows_per_cta():
    """More rows than the persistent selection grid holds CTAs, so each CTA
    selects several rows in turn (its shared memory reused between rows)."""
    sh = W.DSAShape(**W.DEEPSEEK)
    rng = np.random.default_rng(13)
    lens = rng.integers(2049, 12000, size=700)
    rows = [rng.standard_normal(int(n)).astype(np.float32) for n in lens]
    wl = W.build_workload("topk_many", sh, [(len(r) - 1, 1) for r in rows], seed=14)
    off = np.zeros(len(rows) + 1, np.int64)
    off[1:] = np.cumsum([len(r) for r in rows])
    sc = np.concatenate(rows)
    ref = oracle.topk(sh, wl.spans, sc, off)
    ctx = dsa.Context(sh, 0)
    plan = ctx.plan(wl.spans, wl.num_pages)
    g = ctx.topk_from_scores(plan, torch.from_numpy(sc).cuda()).cpu().numpy()
    ctx.get_error()
    H.check_selection(g, ref, sc, off, sh.topk, exact=True)


def test_topk_many_short_rows_four_ctas_per_sm():
    """More rows than two per SM, none longer than 32,768 keys: the selection
    runs 256-thread CTAs, four per SM, with the smaller shared-memory
    capacities (4,096 candidates, a 1,024-key sample, a 65,536-position
    bitmap).  Rows of every path: fewer keys than topk, every key a candidate,
    a strided sample, a sample the data fools, and threshold ties below, equal
    to and above what the tie ranking holds."""
    sh = W.DSAShape(**W.DEEPSEEK)
    rng = np.random.default_rng(17)
    rows = []
    rows += [rng.standard_normal(int(n)).astype(np.float32) for n in rng.integers(100, 2048, size=20)]
    rows += [rng.standard_normal(int(n)).astype(np.float32) for n in rng.integers(2049, 4096, size=120)]
    rows += [rng.standard_normal(int(n)).astype(np.float32) for n in rng.integers(4097, 32768, size=200)]
    rows.append(rng.standard_normal(32768).astype(np.float32))
    for _ in range(8):
        fool = (rng.random(30000) * 10 + 1).astype(np.float32)
        fool[:: 30000 // 1024] = 0.0                                              # the sample sees only zeros
        rows.append(fool)
    for n_tie, n_top in ((3000, 1000), (1500, 1000), (1048, 1000)) * 4:        # ties > cap, <= cap, == need
        r = (rng.random(20000) * 0.5).astype(np.float32)
        idx = rng.permutation(20000)
        r[idx[:n_top]] = (2.0 + rng.random(n_top)).astype(np.float32)
        r[idx[n_top:n_top + n_tie]] = 1.0
        rows.append(r)
    order = rng.permutation(len(rows))
    rows = [rows[i] for i in order]
    assert len(rows) > 2 * 152 and max(len(r) for r in rows) <= 32768
    wl = W.build_workload("topk_short", sh, [(len(r) - 1, 1) for r in rows], seed=18)
    off = np.zeros(len(rows) + 1, np.int64)
    off[1:] = np.cumsum([len(r) for r in rows])
    sc = np.concatenate(rows)
    ref = oracle.topk(sh, wl.spans, sc, off)
    ctx = dsa.Context(sh, 0)
    plan = ctx.plan(wl.spans, wl.num_pages)
    g = ctx.topk_from_scores(plan, torch.from_numpy(sc).cuda()).cpu().numpy()
    ctx.get_error()
    H.check_selection(g, ref, sc, off, sh.topk, exact=True)


def test_quantize_on_store_bit_exact():
    """bf16 rows quantised into the 132-byte index rows and 656-byte latent rows
    give the oracle's bytes exactly (scales, codes, ties to even, saturation,
    zero groups, copied rope), and the pipeline over the quantised caches
    matches the oracle."""
    wl = H.deepseek_small(seed=15, fp8=True, sink=True, page_start=8, decode_ctx=(2049, 700), chunk=(1990, 40))
    sh = wl.shape
    ic, lc, st = H.host_inputs(wl)
    T = wl.num_rows
    rng = np.random.default_rng(16)
    keys = rng.standard_normal((T, 128)).astype(np.float32) * 3
    keys[0] = 0.0                                        # an all-zero group
    keys[1, 5] = 1e4                                     # one large value
    keys[2, :] = -0.0
    lat = rng.standard_normal((T, 576)).astype(np.float32)
    lat[3, 128:256] = 0.0
    kb, lb = torch.from_numpy(keys).to(torch.bfloat16), torch.from_numpy(lat).to(torch.bfloat16)
    ref_ic = oracle.quantize_store_keys(sh, wl.spans, wl.num_pages, kb, ic)
    ref_lc = oracle.quantize_store_latents(sh, wl.spans, wl.num_pages, lb, lc)
    ctx = dsa.Context(sh, 0)
    plan = ctx.plan(wl.spans, wl.num_pages)
    g_ic, g_lc = ic.cuda(), lc.cuda()
    ctx.quantize_store_keys(plan, kb.cuda(), g_ic)
    ctx.quantize_store_latents(plan, lb.cuda(), g_lc)
    ctx.get_error()
    assert np.array_equal(g_ic.cpu().numpy().reshape(-1), ref_ic.reshape(-1))
    assert np.array_equal(g_lc.cpu().numpy().reshape(-1), ref_lc.reshape(-1))
    # selection and attention over the quantised caches
    sc, off = oracle.index_scores(sh, wl.spans, wl.num_pages, st.q, st.w, ref_ic)
    sel = oracle.topk(sh, wl.spans, sc, off)
    g_sel = ctx.index_topk(plan, st.q.cuda(), st.w.cuda(), g_ic).cpu().numpy()
    H.check_selection(g_sel, sel, sc, off, sh.topk)
    ref_out = oracle.attend(sh, wl.spans, wl.num_pages, sel, st.q_nope, st.q_pe, ref_lc, st.sink)
    out = ctx.attend(plan, torch.from_numpy(sel).cuda(), st.q_nope.cuda(), st.q_pe.cuda(), g_lc,
                     None if st.sink is None else st.sink.cuda(), sh.sm_scale)
    ctx.get_error()
    H.check_attention(out.float().cpu().numpy(), ref_out, True)


def test_quantize_on_store_rejects_bf16_formats():
    wl = H.deepseek_small(seed=17, decode_ctx=(300,), chunk=None)
    ctx = dsa.Context(wl.shape, 0)
    plan = ctx.plan(wl.spans, wl.num_pages)
    keys = torch.zeros(wl.num_rows, 128, dtype=torch.bfloat16, device="cuda")
    cache = torch.zeros(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(dsa.DSAError):
        ctx.quantize_store_keys(plan, keys, cache)


def test_full_and_shared_layers():
    """A forward of four layers over one plan: FULL, SHARED, FULL, SHARED.  Each
    SHARED layer attends with its own queries and latents over the selection
    the last FULL layer wrote (IndexShare); a FULL layer's selection replaces it."""
    base = H.deepseek_small(seed=18, sink=True, decode_ctx=(2300, 900), chunk=(2040, 24))
    layers = [W.Workload(base.name, base.shape, base.spans, base.num_pages, 18 + 97 * i, base.dist) for i in range(4)]
    full = [True, False, True, False]
    ctx = dsa.Context(base.shape, 0)
    plan = ctx.plan(base.spans, base.num_pages)
    with pytest.raises(dsa.DSAError):              # no FULL layer yet
        ctx.attend_shared(plan, torch.zeros(1, device="cuda", dtype=torch.bfloat16),
                          torch.zeros(1, device="cuda", dtype=torch.bfloat16),
                          torch.zeros(1, device="cuda", dtype=torch.bfloat16))
    last_sel = None
    for wl, is_full in zip(layers, full):
        ic, lc, st = H.host_inputs(wl)
        dev = W.StepInputs(*(H.to_dev(x) for x in (st.q, st.w, st.keys, st.q_nope, st.q_pe, st.sink)))
        lcd = lc.cuda()
        if is_full:
            icd = ic.cuda()
            ctx.store_keys(plan, dev.keys, icd)
            sel = ctx.index_topk(plan, dev.q, dev.w, icd)
            cache = oracle.store_keys(wl.shape, wl.spans, wl.num_pages, st.keys, ic)
            sc, off = oracle.index_scores(wl.shape, wl.spans, wl.num_pages, st.q, st.w, cache)
            H.check_selection(sel.cpu().numpy(), oracle.topk(wl.shape, wl.spans, sc, off), sc, off, wl.shape.topk)
            out = ctx.attend(plan, sel, dev.q_nope, dev.q_pe, lcd, dev.sink)
            last_sel = sel
        else:
            out = ctx.attend_shared(plan, dev.q_nope, dev.q_pe, lcd, dev.sink)
        ctx.get_error()
        ref = oracle.attend(wl.shape, wl.spans, wl.num_pages, last_sel.cpu().numpy(), st.q_nope, st.q_pe, lc, st.sink)
        H.check_attention(out.float().cpu().numpy(), ref, False)


def test_bounds_errors_are_reported_not_faulted():
    """Selected positions past the row or below -1 set DSA_ERR_BOUNDS and are skipped."""
    wl = H.deepseek_small(seed=7, decode_ctx=(3000,), chunk=None)
    ic, lc, st = H.host_inputs(wl)
    ctx = dsa.Context(wl.shape, 0)
    plan = ctx.plan(wl.spans, wl.num_pages)
    sel = torch.full((1, wl.shape.topk), -1, dtype=torch.int32)
    sel[0, :10] = torch.arange(10)
    sel[0, 10] = 3000           # row 0 sits at position 2999
    sel[0, 11] = -5
    out = ctx.attend(plan, sel.cuda(), st.q_nope.cuda(), st.q_pe.cuda(), lc.cuda(), None, wl.shape.sm_scale)
    with pytest.raises(dsa.DSAError) as e:
        ctx.get_error()
    assert e.value.status == 5
    ctx.get_error()  # the word was cleared
    ref_sel = sel.numpy().copy()
    ref_sel[0, 10:12] = -1
    ref = oracle.attend(wl.shape, wl.spans, wl.num_pages, ref_sel, st.q_nope, st.q_pe, lc, None)
    H.check_attention(out.float().cpu().numpy(), ref)


def test_empty_step_and_launch_count():
    sh = W.DSAShape(**W.DEEPSEEK)
    ctx = dsa.Context(sh, 0)
    plan = ctx.plan([], cache_pages=1)
    assert plan.num_rows == 0
    wl = H.deepseek_small(seed=8, decode_ctx=(2500,), chunk=None)
    ic, lc, st = H.device_inputs(wl)
    plan = ctx.plan(wl.spans, wl.num_pages)
    ctx.index_topk(plan, st.q, st.w, ic)
    assert ctx.last_launch_count() == 2
    ctx.get_error()


@pytest.mark.parametrize("fp8", [False, True])
def test_generator_is_identical_on_gpu(fp8):
    wl = H.deepseek_small(seed=10, fp8=fp8, sink=True, decode_ctx=(700,), chunk=(100, 5))
    a = H.host_inputs(wl)
    b = H.device_inputs(wl)
    for x, y in zip(a[:2], b[:2]):
        assert torch.equal(x.view(torch.uint8), y.cpu().view(torch.uint8))
    for x, y in zip(a[2].__dict__.values(), b[2].__dict__.values()):
        if x is not None:
            assert torch.equal(x.contiguous().view(torch.uint8), y.cpu().contiguous().view(torch.uint8))
