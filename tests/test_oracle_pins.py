"""Pins of the CPU oracle to facts outside itself (no GPU).

Each test ties one oracle function to a closed form, an invariant, a brute-force
enumeration or a library routine, chosen so that a plausible mistake (a dropped
relu, a swapped head weight, a transposed operand, a wrong slot mapping, a
reversed tie-break, a misplaced fp8 scale, a sink multiplied by the scale) makes
at least one of them fail.
"""
import itertools
import math

import numpy as np
import pytest
import torch

import oracle
from deepseek_sparse_attention_dsa_gb300 import workloads as W
from tests.dsa_cases import bf16, make_case, phys_rows, tiny_shape


# ----------------------------------------------------------------------------
# fp8 e4m3 (OCP FP8 "E4M3FN")
# ----------------------------------------------------------------------------
def test_e4m3_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_values(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert set(np.nonzero(nan)[0]) == {0x7F, 0xFF}


def test_e4m3_spec_points():
    v = oracle.e4m3_values([0x7E, 0x01, 0x08, 0x38, 0xB8, 0x80, 0x07])
    assert v[0] == 448.0                 # largest finite: 1.75 * 2^8
    assert v[1] == 2.0 ** -9             # smallest subnormal: 1/8 * 2^-6
    assert v[2] == 2.0 ** -6             # smallest normal
    assert v[3] == 1.0 and v[4] == -1.0
    assert v[5] == 0.0 and math.copysign(1.0, v[5]) < 0
    assert v[6] == 7.0 / 8.0 * 2.0 ** -6  # largest subnormal


def test_e4m3_encode_inverts_every_code():
    """Encoding the value of every finite code gives the code back (-0 -> 0x80)."""
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = oracle.e4m3_values(codes).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(vals), codes)


def test_e4m3_encode_matches_torch_cast():
    """Round to nearest even, as torch's float32 -> float8_e4m3fn cast, over the finite range."""
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.standard_normal(3000) * 40, rng.standard_normal(2000) * 1e-2,
                        (rng.random(1000) - 0.5) * 890]).astype(np.float32)
    x = x[np.abs(x) < 448]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_encode(x), ref)


def test_e4m3_encode_ties_and_saturation():
    v = oracle.e4m3_values(np.arange(0x7F, dtype=np.uint8))       # 0 .. 448, increasing
    mids = ((v[:-1] + v[1:]) / 2).astype(np.float32)               # exact midpoints
    want = np.array([c if c % 2 == 0 else c + 1 for c in range(0x7E)], dtype=np.uint8)
    assert np.array_equal(oracle.e4m3_encode(mids), want)          # ties go to the even code
    assert np.array_equal(oracle.e4m3_encode(-mids), want | 0x80)
    assert list(oracle.e4m3_encode([448.0, 449.0, 1e6, -500.0])) == [0x7E, 0x7E, 0x7E, 0xFE]


def test_quantize_keys_and_latents_bounds():
    """Each group's largest magnitude maps to +-448 * scale; every value is within
    half an E4M3 step (times the scale) of its dequantised code; an all-zero
    group gets scale 1; rope values are copied bit for bit."""
    sh = tiny_shape(index_dim=128, page_size=4, kv_lora_rank=512, rope_dim=64, index_fmt=W.INDEX_FP8_132,
                    latent_fmt=W.LATENT_FP8_656)
    case = make_case(sh, [(0, 3)], num_pages=1)
    rng = np.random.default_rng(5)
    keys = rng.standard_normal((3, 128)).astype(np.float32) * np.array([[1.0], [1e-3], [0.0]], np.float32)
    kb = bf16(keys)
    kc = oracle.quantize_store_keys(sh, case.spans, 1, kb, np.zeros(4 * 132, np.uint8))
    codes = kc[:4 * 128].reshape(4, 128)[:3]
    scales = kc[4 * 128:].view(np.float32)[:3]
    kf = kb.float().numpy()
    for r in range(3):
        amax = np.abs(kf[r]).max()
        assert scales[r] == (np.float32(amax) / np.float32(448) if amax > 0 else 1.0)
        deq = oracle.e4m3_values(codes[r]) * scales[r]
        if amax > 0:
            i = np.argmax(np.abs(kf[r]))
            assert codes[r][i] & 0x7F == 0x7E
        q = kf[r] / scales[r]
        step = np.where(np.abs(q) < 2.0 ** -6, 2.0 ** -9, 2.0 ** (np.floor(np.log2(np.maximum(np.abs(q), 1e-30))) - 3))
        assert np.all(np.abs(deq - kf[r]) <= 0.5 * step * scales[r] * (1 + 1e-6) + 1e-30)
    lat = rng.standard_normal((3, 576)).astype(np.float32)
    lat[1, :128] = 0.0
    lb = bf16(lat)
    lc = oracle.quantize_store_latents(sh, case.spans, 1, lb, np.zeros(4 * 656, np.uint8)).reshape(4, 656)
    lf = lb.float().numpy()
    for r in range(3):
        sc = lc[r, 512:528].view(np.float32)
        for g in range(4):
            amax = np.abs(lf[r, 128 * g:128 * (g + 1)]).max()
            assert sc[g] == (np.float32(amax) / np.float32(448) if amax > 0 else 1.0)
        assert np.array_equal(lc[r, 528:656].view(np.uint16), lb.view(torch.int16).numpy()[r, 512:].view(np.uint16))
    assert lc[1, :128].max() == 0 and lc[1, 512:516].view(np.float32)[0] == 1.0


# ----------------------------------------------------------------------------
# slot mapping (DSASpan: page_start is the first token's offset in the pages)
# ----------------------------------------------------------------------------
def test_store_keys_slot_mapping_literal():
    # page_size 2, pages [3, 1], page_start 1: positions 0, 1, 2 sit at slots 1, 2, 3,
    # i.e. (page 3, slot 1), (page 1, slot 0), (page 1, slot 1) -> physical rows 7, 2, 3.
    sh = tiny_shape(index_dim=2, page_size=2)
    case = make_case(sh, [(0, 3)], pages=[[3, 1]], page_start=1, num_pages=4)
    keys = bf16([[1, 2], [3, 4], [5, 6]])
    cache = torch.zeros(4, 2, 2, dtype=torch.bfloat16)
    out = oracle.store_keys(sh, case.spans, 4, keys, cache).view(np.uint16)
    flat = torch.from_numpy(out.reshape(8, 2).astype(np.int16)).view(torch.bfloat16).float().numpy()
    expect = np.zeros((8, 2))
    expect[7] = [1, 2]
    expect[2] = [3, 4]
    expect[3] = [5, 6]
    assert np.array_equal(flat, expect)


def test_store_keys_fp8_page_blocked_literal():
    # fp8 index rows: each page = [page_size x 128 codes][page_size x fp32 scale]
    sh = tiny_shape(index_dim=128, page_size=2, index_fmt=W.INDEX_FP8_132)
    case = make_case(sh, [(0, 3)], pages=[[1, 0]], page_start=0, num_pages=2)
    keys = np.zeros((3, 132), np.uint8)
    for r in range(3):
        keys[r, :128] = 10 + r
        keys[r, 128:] = np.frombuffer(np.float32(r + 0.5).tobytes(), np.uint8)
    cache = np.zeros((2, 2 * 132), np.uint8)
    out = oracle.store_keys(sh, case.spans, 2, keys, cache).reshape(2, 264)
    # position 0 -> page 1 slot 0, position 1 -> page 1 slot 1, position 2 -> page 0 slot 0
    assert (out[1, 0:128] == 10).all() and (out[1, 128:256] == 11).all() and (out[0, 0:128] == 12).all()
    assert np.frombuffer(out[1, 256:260].tobytes(), np.float32)[0] == 0.5
    assert np.frombuffer(out[1, 260:264].tobytes(), np.float32)[0] == 1.5
    assert np.frombuffer(out[0, 256:260].tobytes(), np.float32)[0] == 2.5
    assert (out[0, 128:256] == 0).all()


# ----------------------------------------------------------------------------
# indexer score: sum_h w[h] * relu(q[h] . k)   (mstar index_topk)
# ----------------------------------------------------------------------------
def _score_case(index_fmt=W.INDEX_BF16, page_start=2, pages=((5, 0, 3, 1),)):
    """Row r (positions 6..9 of one request) has q[r,0] = (r+1, 0, 2), q[r,1] = (-1, 0, 0),
    w[r] = (1, 5); key j = (j - 5, 7, 0).  Closed form:
        score(r, j) = (r+1) * relu(j - 5) + 5 * relu(5 - j),  j = 0 .. pos(r)."""
    Di = 3 if index_fmt == W.INDEX_BF16 else 128
    sh = tiny_shape(index_dim=Di, page_size=4, index_fmt=index_fmt)
    case = make_case(sh, [(6, 4)], pages=[list(pages[0])], page_start=page_start, num_pages=6)
    keys_log = np.zeros((10, Di), np.float32)
    keys_log[:, 0] = np.arange(10) - 5
    keys_log[:, 1] = 7
    rows = phys_rows(case, 0, np.arange(10))
    if index_fmt == W.INDEX_BF16:
        cache = np.zeros((6 * 4, Di), np.float32)
        cache[rows] = keys_log
        cache = bf16(cache).view(6, 4, Di)
        step_keys = bf16(keys_log[6:10])
    else:
        # e4m3 codes of (j - 5) / 2 and 3.5 with scale 2: e4m3 holds k/2 exactly
        codes = torch.from_numpy(keys_log / 2.0).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        scale = np.frombuffer(np.float32(2.0).tobytes(), np.uint8)
        cache = np.zeros((6, 4 * (Di + 4)), np.uint8)
        for j in range(6):  # history only; the step stores positions 6..9
            pg, sl = divmod(int(rows[j]), 4)
            cache[pg, sl * Di:(sl + 1) * Di] = codes[j]
            cache[pg, 4 * Di + 4 * sl: 4 * Di + 4 * sl + 4] = scale
        step_keys = np.concatenate([codes[6:10], np.tile(scale, (4, 1))], axis=1)
    q = np.zeros((4, 2, Di), np.float32)
    for r in range(4):
        q[r, 0, 0], q[r, 0, 2], q[r, 1, 0] = r + 1, 2, -1
    w = np.tile(np.array([1.0, 5.0], np.float32), (4, 1))
    return sh, case, cache, step_keys, bf16(q), torch.from_numpy(w)


@pytest.mark.parametrize("index_fmt", [W.INDEX_BF16, W.INDEX_FP8_132])
def test_score_closed_form(index_fmt):
    sh, case, cache, step_keys, q, w = _score_case(index_fmt)
    cache = oracle.store_keys(sh, case.spans, case.num_pages, step_keys, cache)
    scores, off = oracle.index_scores(sh, case.spans, case.num_pages, q, w, cache)
    for r in range(4):
        p = 6 + r
        j = np.arange(p + 1)
        expect = (r + 1) * np.maximum(j - 5, 0) + 5 * np.maximum(5 - j, 0)
        assert np.array_equal(scores[off[r]:off[r + 1]], expect.astype(np.float32)), r


def test_score_paging_invariance():
    """The same logical keys under other page tables and page_start give the same scores."""
    a = _score_case(page_start=0, pages=((0, 1, 2),))
    b = _score_case(page_start=2, pages=((5, 0, 3, 1),))
    outs = []
    for sh, case, cache, step_keys, q, w in (a, b):
        cache = oracle.store_keys(sh, case.spans, case.num_pages, step_keys, cache)
        outs.append(oracle.index_scores(sh, case.spans, case.num_pages, q, w, cache)[0])
    assert np.array_equal(outs[0], outs[1])


def test_score_negative_weight_and_rounding_once():
    """A negative head weight subtracts (it is not clipped), and the fp64 sum is
    rounded to fp32 once: 1 + 2^-30 - 1 survives as 2^-30 only when summed in
    double before rounding (fp32 partial sums would lose it)."""
    sh = tiny_shape(index_heads=3, index_dim=1, page_size=4)
    case = make_case(sh, [(0, 1)])
    cache = bf16(np.ones((1, 4, 1))).view(1, 4, 1)
    q = bf16(np.ones((1, 3, 1)))
    w = torch.tensor([[1.0, 2.0 ** -30, -1.0]], dtype=torch.float32)
    cache = oracle.store_keys(sh, case.spans, 1, bf16([[1.0]]), cache)
    s, _ = oracle.index_scores(sh, case.spans, 1, q, w, cache)
    assert s[0] == np.float32(2.0 ** -30)


def test_score_integer_inputs_are_integers():
    wl = W.build_workload("int", W.DSAShape(index_heads=8, index_dim=64, topk=16, heads=2, kv_lora_rank=4,
                                            rope_dim=2, page_size=16, sm_scale=1.0),
                          [(30, 5), (100, 1)], seed=7, dist=W.Distributions(integer=True))
    ic = W.make_index_cache(wl)
    st = W.make_step_inputs(wl)
    cache = oracle.store_keys(wl.shape, wl.spans, wl.num_pages, st.keys, ic)
    s, _ = oracle.index_scores(wl.shape, wl.spans, wl.num_pages, st.q, st.w, cache)
    assert np.array_equal(s, np.round(s)) and (s >= 0).all()


# ----------------------------------------------------------------------------
# top-k: ties to the earlier position, -1 padding (mstar select_topk_causal)
# ----------------------------------------------------------------------------
def _topk_rows(score_rows, K):
    sh = tiny_shape(topk=K)
    case = make_case(sh, [(len(score_rows[0]) - 1, 1)] if len(score_rows) == 1 else
                     [(len(r) - 1, 1) for r in score_rows])
    off = np.zeros(len(score_rows) + 1, np.int64)
    off[1:] = np.cumsum([len(r) for r in score_rows])
    return oracle.topk(sh, case.spans, np.concatenate(score_rows).astype(np.float32), off)


def _defining_property(s, S, K):
    """S is the top-K set under (score desc, position asc) iff every member ranks
    before every non-member and |S| = min(K, n)."""
    n = len(s)
    if len(S) != min(K, n) or len(set(S)) != len(S):
        return False
    rest = [j for j in range(n) if j not in S]
    return all(s[i] > s[j] or (s[i] == s[j] and i < j) for i in S for j in rest)


def test_topk_brute_force_enumeration():
    rng = np.random.default_rng(3)
    for n in range(1, 8):
        for trial in range(6):
            s = rng.integers(0, 3, size=n).astype(np.float32)   # many ties
            for K in range(1, n + 2):
                sel = _topk_rows([s], K)[0]
                got = [int(x) for x in sel if x >= 0]
                assert (sel[len(got):] == -1).all()
                winners = [set(c) for c in itertools.combinations(range(n), min(K, n))
                           if _defining_property(s, list(c), K)]
                assert len(winners) == 1
                assert set(got) == winners[0]


def test_topk_tie_cases():
    n, K = 20, 5
    assert list(_topk_rows([np.zeros(n)], K)[0]) == [0, 1, 2, 3, 4]
    assert list(_topk_rows([np.arange(n, dtype=np.float32)], K)[0]) == [19, 18, 17, 16, 15]
    assert list(_topk_rows([-np.arange(n, dtype=np.float32)], K)[0]) == [0, 1, 2, 3, 4]
    s = np.zeros(n, np.float32)
    s[[3, 9, 12]] = 1.0
    assert list(_topk_rows([s], K)[0]) == [3, 9, 12, 0, 1]
    # -0.0 and +0.0 are equal scores: the earlier position wins
    s = np.full(4, -1.0, np.float32)
    s[1], s[2] = -0.0, 0.0
    assert list(_topk_rows([s], 1)[0]) == [1]


def test_topk_short_rows_pad():
    sel = _topk_rows([np.array([2.0, 1.0, 3.0], np.float32)], 6)[0]
    assert list(sel) == [2, 0, 1, -1, -1, -1]


def test_topk_random_invariants():
    rng = np.random.default_rng(11)
    rows = [rng.standard_normal(n).astype(np.float32).round(1) for n in (1, 7, 64, 65, 300)]
    K = 64
    sel = _topk_rows(rows, K)
    for s, srow in zip(rows, sel):
        got = [int(x) for x in srow if x >= 0]
        assert (srow[len(got):] == -1).all()
        assert all(0 <= j < len(s) for j in got)
        assert _defining_property(s, got, K)
        # canonical order: score descending, position ascending
        keys = [(-float(s[j]), j) for j in got]
        assert keys == sorted(keys)


def test_topk_packing_independence():
    """A request's selection does not depend on the batch it is packed in nor on its pages."""
    wl = W.build_workload("pack", W.DSAShape(index_heads=4, index_dim=32, topk=16, heads=2, kv_lora_rank=4,
                                             rope_dim=2, page_size=8, sm_scale=1.0),
                          [(40, 3), (0, 25), (70, 1)], seed=5, dist=W.Distributions(integer=True))
    full = oracle.run_all(wl, W.make_index_cache(wl), W.make_latent_cache(wl), W.make_step_inputs(wl))
    for order in ([2, 0], [1], [2, 1, 0]):
        sub = wl.sub_workload(order)
        got = oracle.run_all(sub, W.make_index_cache(sub), W.make_latent_cache(sub), W.make_step_inputs(sub))
        r_sub = 0
        for i in order:
            s = wl.spans[i]
            a = full["selection"][s.q_start:s.q_start + s.q_len]
            b = got["selection"][r_sub:r_sub + s.q_len]
            assert np.array_equal(a, b)
            assert np.array_equal(full["out"][s.q_start:s.q_start + s.q_len], got["out"][r_sub:r_sub + s.q_len])
            r_sub += s.q_len


# ----------------------------------------------------------------------------
# attend: absorbed MLA over the picked latents (mstar DSAManager.attend;
# ttnn sparse_sdpa for V = the leading kv_lora_rank columns and for the sink)
# ----------------------------------------------------------------------------
def _latent_case(H=2, L=4, Rd=2, ctx=6, q_len=3, sm_scale=0.7, seed=0, P=4, pages=None, page_start=1):
    sh = tiny_shape(heads=H, kv_lora_rank=L, rope_dim=Rd, page_size=P, sm_scale=sm_scale, topk=ctx + q_len)
    case = make_case(sh, [(ctx, q_len)], pages=pages, page_start=page_start)
    rng = np.random.default_rng(seed)
    n = ctx + q_len
    lat = rng.standard_normal((n, L + Rd)).astype(np.float32)
    cache = np.zeros((case.num_pages * P, L + Rd), np.float32)
    cache[phys_rows(case, 0, np.arange(n))] = lat
    qn = rng.standard_normal((q_len, H, L)).astype(np.float32)
    qp = rng.standard_normal((q_len, H, Rd)).astype(np.float32)
    return sh, case, bf16(lat).double(), bf16(cache).view(case.num_pages, P, L + Rd), bf16(qn), bf16(qp)


def test_attend_all_keys_equals_dense_causal_sdpa():
    """With every visible key selected, sparse absorbed MLA is dense causal MQA:
    q = [q_nope | q_pe], k = [c | k_pe], v = c, one KV head."""
    H, L, Rd, ctx, q_len = 3, 8, 4, 5, 4
    sh, case, lat, cache, qn, qp = _latent_case(H=H, L=L, Rd=Rd, ctx=ctx, q_len=q_len, pages=[[2, 0, 1]])
    K = sh.topk
    sel = np.full((q_len, K), -1, np.int32)
    for r in range(q_len):
        sel[r, :ctx + r + 1] = np.arange(ctx + r + 1)[::-1]   # any order
    out = oracle.attend(sh, case.spans, case.num_pages, sel, qn, qp, cache)
    q = torch.cat([qn.double(), qp.double()], dim=-1).transpose(0, 1)          # (H, q_len, L+R)
    k = lat.unsqueeze(0).expand(H, -1, -1)                                        # (H, n, L+R)
    v = lat[:, :L].unsqueeze(0).expand(H, -1, -1)
    mask = torch.zeros(q_len, ctx + q_len, dtype=torch.bool)
    for r in range(q_len):
        mask[r, :ctx + r + 1] = True
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=sh.sm_scale)
    np.testing.assert_allclose(out, ref.transpose(0, 1).numpy(), rtol=1e-12, atol=1e-12)


def test_attend_single_key_and_equal_latents():
    sh, case, lat, cache, qn, qp = _latent_case()
    sel = np.full((3, sh.topk), -1, np.int32)
    sel[:, 0] = 4
    out = oracle.attend(sh, case.spans, case.num_pages, sel, qn, qp, cache)
    assert np.array_equal(out, np.broadcast_to(lat[4, :sh.kv_lora_rank].numpy(), out.shape))
    # -1 entries in the middle are skipped
    sel2 = np.full((3, sh.topk), -1, np.int32)
    sel2[:, 2] = 4
    assert np.array_equal(oracle.attend(sh, case.spans, case.num_pages, sel2, qn, qp, cache), out)


def test_attend_uniform_logits_give_mean():
    sh, case, lat, cache, qn, qp = _latent_case()
    zero = torch.zeros_like(qn)
    sel = np.full((3, sh.topk), -1, np.int32)
    sel[:, :3] = [0, 2, 5]
    out = oracle.attend(sh, case.spans, case.num_pages, sel, zero, torch.zeros_like(qp), cache)
    mean = lat[[0, 2, 5], :sh.kv_lora_rank].numpy().mean(axis=0)
    np.testing.assert_allclose(out, np.broadcast_to(mean, out.shape), rtol=0, atol=1e-15)


def test_attend_sink_closed_forms():
    """The sink is a logit in scaled units that joins only the denominator:
    two keys with logit 0 and a sink 0 give (c_a + c_b) / 3; a sink at -1e30 is no sink."""
    sh, case, lat, cache, qn, qp = _latent_case(sm_scale=3.0)
    zero_n, zero_p = torch.zeros_like(qn), torch.zeros_like(qp)
    sel = np.full((3, sh.topk), -1, np.int32)
    sel[:, :2] = [1, 3]
    sink0 = torch.zeros(sh.heads)
    out = oracle.attend(sh, case.spans, case.num_pages, sel, zero_n, zero_p, cache, sink0)
    expect = (lat[1, :sh.kv_lora_rank] + lat[3, :sh.kv_lora_rank]).numpy() / 3.0
    np.testing.assert_allclose(out, np.broadcast_to(expect, out.shape), rtol=0, atol=1e-15)
    far = torch.full((sh.heads,), -1e30)
    a = oracle.attend(sh, case.spans, case.num_pages, sel, qn, qp, cache, far)
    b = oracle.attend(sh, case.spans, case.num_pages, sel, qn, qp, cache, None)
    np.testing.assert_allclose(a, b, rtol=0, atol=0)
    # sink equal to the single key's logit: output is half the latent
    sel1 = np.full((3, sh.topk), -1, np.int32)
    sel1[:, 0] = 2
    lg = (qn.double() @ lat[2, :sh.kv_lora_rank] + qp.double() @ lat[2, sh.kv_lora_rank:]) * sh.sm_scale
    r0 = oracle.attend(sh, case.spans, case.num_pages, sel1[:1], qn[:1], qp[:1], cache, lg[0].float())
    half = 0.5 * lat[2, :sh.kv_lora_rank].numpy()
    np.testing.assert_allclose(r0[0], np.broadcast_to(half, r0[0].shape), rtol=1e-6, atol=1e-6)


def test_attend_fp8_656_row_layout():
    """A 656-byte row is [512 e4m3 | 4 fp32 scales, one per 128 | 64 bf16 rope]: with one
    selected key the output is the dequantised c exactly."""
    L, Rd, P = 512, 64, 2
    sh = tiny_shape(heads=2, kv_lora_rank=L, rope_dim=Rd, page_size=P, topk=4, latent_fmt=W.LATENT_FP8_656)
    assert sh.latent_row_bytes == 656
    case = make_case(sh, [(1, 1)], pages=[[1]], num_pages=2)
    rng = np.random.default_rng(2)
    codes = rng.integers(0, 256, size=(L,), dtype=np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x10   # no NaN codes
    scales = np.array([0.5, 2.0, 3.0, 0.25], np.float32)
    rope = bf16(rng.standard_normal(Rd)).view(torch.int16).numpy().view(np.uint8)
    row = np.concatenate([codes, scales.view(np.uint8), rope])
    cache = np.zeros((2, P, 656), np.uint8)
    cache[1, 1] = row    # position 1 -> slot 1 of page 1
    qn = bf16(rng.standard_normal((1, 2, L)))
    qp = bf16(rng.standard_normal((1, 2, Rd)))
    sel = np.array([[1, -1, -1, -1]], np.int32)
    out = oracle.attend(sh, case.spans, 2, sel, qn, qp, cache)
    deq = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy() * np.repeat(scales.astype(np.float64), 128)
    assert np.array_equal(out[0, 0], deq) and np.array_equal(out[0, 1], deq)


def test_attend_rejects_noncausal_selection():
    sh, case, lat, cache, qn, qp = _latent_case()
    sel = np.full((3, sh.topk), -1, np.int32)
    sel[0, 0] = 7            # row 0 sits at position 6
    with pytest.raises(oracle.OracleError):
        oracle.attend(sh, case.spans, case.num_pages, sel, qn, qp, cache)


def test_short_history_raises():
    sh = tiny_shape(page_size=4)
    case = make_case(sh, [(6, 2)], pages=[[0]], num_pages=1)     # 8 tokens need 2 pages
    with pytest.raises(oracle.OracleError):
        oracle.store_keys(sh, case.spans, 1, bf16(np.zeros((2, 3))), torch.zeros(1, 4, 3, dtype=torch.bfloat16))


# ----------------------------------------------------------------------------
# byte identities stated on the pages
# ----------------------------------------------------------------------------
def test_format_sizes_match_pages():
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "format_sizes.txt")
    facts = {}
    for line in open(path):
        line = line.split("#")[0].strip()
        if line:
            k, v = line.split("=")
            facts[k.strip()] = int(v)
    bf = W.DSAShape(**W.DEEPSEEK)
    f8 = W.DSAShape(**W.DEEPSEEK, latent_fmt=W.LATENT_FP8_656, index_fmt=W.INDEX_FP8_132)
    assert bf.latent_row_bytes == facts["mla_latent_bf16"]
    assert f8.latent_row_bytes == facts["mla_latent_fp8_packed"]
    assert f8.index_row_bytes == facts["dsa_index_fp8"]
    assert facts["selected_tokens"] == bf.topk


# ---------------------------------------------------------------- fp8 query
def _fp8_index_case(seed, index_heads=2, index_dim=8):
    """A tiny fp8-index case: two requests, random non-NaN key codes, signed scales."""
    sh = tiny_shape(index_heads=index_heads, index_dim=index_dim, page_size=4, index_fmt=W.INDEX_FP8_132)
    case = make_case(sh, [(0, 6), (3, 2)])
    rng = np.random.default_rng(seed)
    P, D = sh.page_size, index_dim
    npg = case.num_pages
    cache = np.zeros(npg * P * (D + 4), np.uint8)
    for pg in range(npg):
        base = pg * P * (D + 4)
        codes = rng.integers(0, 0x7F, size=P * D).astype(np.uint8) | (rng.integers(0, 2, size=P * D) << 7).astype(np.uint8)
        cache[base:base + P * D] = codes
        cache[base + P * D:base + P * (D + 4)] = (rng.choice([0.25, 0.5, -1.0, 2.0], size=P).astype(np.float32)).view(np.uint8)
    T = sum(s.q_len for s in case.spans)
    w = rng.uniform(0, 1, size=(T, index_heads)).astype(np.float32)
    return sh, case, cache, w, rng


def test_fp8_query_equals_the_bf16_query_it_decodes_to():
    """q = e4m3(code) * 2^k is exact in bf16, so the fp8-query score must equal the
    bf16-query score of the decoded values bit for bit (same fp64 products)."""
    sh, case, cache, w, rng = _fp8_index_case(31)
    T, Hi, D = w.shape[0], sh.index_heads, sh.index_dim
    codes = (rng.integers(0, 0x77, size=(T, Hi, D)).astype(np.uint8) | (rng.integers(0, 2, size=(T, Hi, D)) << 7)).astype(np.uint8)
    scales = rng.choice([0.125, 0.5, 1.0, 4.0], size=(T, Hi)).astype(np.float32)
    qv = oracle.e4m3_values(codes.reshape(-1)).reshape(T, Hi, D) * scales[:, :, None]
    q_bf16 = bf16(qv.astype(np.float32))
    assert np.array_equal(q_bf16.float().numpy(), qv.astype(np.float32))   # exact in bf16
    s_ref, off = oracle.index_scores(sh, case.spans, case.num_pages, q_bf16, w, cache)
    s_f8, off2 = oracle.index_scores_fp8q(sh, case.spans, case.num_pages, codes, scales, w, cache)
    assert np.array_equal(off, off2)
    assert np.array_equal(s_f8, s_ref)
    assert np.any(s_ref > 0) and np.any(s_ref == 0)   # both sides of the relu are exercised


def test_fp8_query_scale_sign_and_size():
    """A negative query scale is the sign-flipped code (relu sees -q); a power-of-two
    scale multiplies every score by itself (relu is positively homogeneous)."""
    sh, case, cache, w, rng = _fp8_index_case(32)
    T, Hi, D = w.shape[0], sh.index_heads, sh.index_dim
    codes = rng.integers(0, 0x77, size=(T, Hi, D)).astype(np.uint8)
    ones = np.ones((T, Hi), np.float32)
    s1, _ = oracle.index_scores_fp8q(sh, case.spans, case.num_pages, codes, ones, w, cache)
    s4, _ = oracle.index_scores_fp8q(sh, case.spans, case.num_pages, codes, 4 * ones, w, cache)
    assert np.array_equal(s4, 4 * s1)
    sneg, _ = oracle.index_scores_fp8q(sh, case.spans, case.num_pages, codes, -ones, w, cache)
    sflip, _ = oracle.index_scores_fp8q(sh, case.spans, case.num_pages, codes ^ 0x80, ones, w, cache)
    assert np.array_equal(sneg, sflip)
    assert not np.array_equal(sneg, s1)


def test_quantize_rows_recovers_representable_rows():
    """Rows made of E4M3 values times 2^k whose largest magnitude is 448 * 2^k come
    back as the same codes with scale 2^k; an all-zero row gets scale 1."""
    rng = np.random.default_rng(33)
    codes = rng.integers(0, 0x7E, size=(5, 128)).astype(np.uint8) | (rng.integers(0, 2, size=(5, 128)) << 7).astype(np.uint8)
    codes[:, 17] = 0x7E                                   # +448 in every row
    k = np.array([-3, 0, 2, 5, -1])
    vals = oracle.e4m3_values(codes.reshape(-1)).reshape(5, 128) * np.ldexp(1.0, k)[:, None]
    vals[4] = 0.0
    got_codes, got_scales = oracle.quantize_rows(bf16(vals.astype(np.float32)), 128)
    got_codes = got_codes.reshape(5, 128)
    assert np.array_equal(got_scales[:4], np.ldexp(1.0, k[:4]).astype(np.float32))
    assert np.array_equal(got_codes[:4], codes[:4])
    assert got_scales[4] == 1.0 and not np.any(got_codes[4] & 0x7F)


# ----------------------------------------------------------------------------
# block-sparse MSA (LLMServingSim, "Sparse attention (DSA and block-sparse
# MSA)", MiniMax-M3 column): block scores, block selection, GQA attention
# ----------------------------------------------------------------------------
def _msa_rows(positions):
    """Single-row spans at the given positions (pages are not read here)."""
    sh = tiny_shape()
    return make_case(sh, [(int(p), 1) for p in positions]).spans


def test_msa_block_scores_closed_form_and_causal_tail():
    """Token scores s_j = j: a block's score is its last visible position,
    min(b*bs + bs - 1, pos); blocks past pos do not exist and positions past
    pos inside the last block are not read (a spike there is ignored)."""
    ms = W.MSAShape(block_size=4)
    pos = [10, 3, 0, 17]
    spans = _msa_rows(pos)
    rows = []
    for p in pos:
        s = np.arange(p + 1, dtype=np.float32)
        rows.append(s)
    off = np.zeros(len(rows) + 1, np.int64)
    off[1:] = np.cumsum([len(r) for r in rows])
    bs, boff = oracle.msa_block_scores(ms, spans, np.concatenate(rows), off)
    for r, p in enumerate(pos):
        got = bs[boff[r]:boff[r + 1]]
        assert len(got) == p // 4 + 1
        assert list(got) == [float(min(4 * b + 3, p)) for b in range(p // 4 + 1)]
    # a spike at position 9 of a row at pos 10 lifts block 2 only; the next
    # row's first score (a larger spike) lies where position 11 would be and
    # must not reach it
    s = np.zeros(11 + 3, np.float32)
    s[9] = 5.0
    s[11] = 50.0
    bs, boff = oracle.msa_block_scores(ms, _msa_rows([10, 2]), s, np.array([0, 11, 14]))
    assert list(bs[:3]) == [0.0, 0.0, 5.0] and list(bs[3:]) == [50.0]


def test_msa_selection_with_unit_blocks_is_the_token_selection():
    """block_size 1: every block is one position, so the block selection is the
    DSA token selection (itself pinned by brute force above)."""
    rng = np.random.default_rng(5)
    pos = [0, 6, 40, 41]
    rows = [rng.integers(0, 4, size=p + 1).astype(np.float32) for p in pos]   # ties
    off = np.zeros(len(rows) + 1, np.int64)
    off[1:] = np.cumsum([len(r) for r in rows])
    spans = _msa_rows(pos)
    for k in (1, 5, 16):
        ms = W.MSAShape(block_size=1, topk_blocks=k)
        bs, boff = oracle.msa_block_scores(ms, spans, np.concatenate(rows), off)
        assert np.array_equal(bs, np.concatenate(rows))
        sel = oracle.msa_select(ms, spans, bs, boff)
        ref = oracle.topk(tiny_shape(topk=k), spans, np.concatenate(rows), off)
        assert np.array_equal(sel, ref)


def test_msa_selection_ties_padding_and_order():
    ms = W.MSAShape(block_size=4, topk_blocks=3)
    # equal block scores: the lowest blocks win
    spans = _msa_rows([23])
    sel = oracle.msa_select(ms, spans, np.zeros(6, np.float32), np.array([0, 6]))
    assert list(sel[0]) == [0, 1, 2]
    # fewer blocks than topk_blocks: all of them, then -1
    spans = _msa_rows([5])
    sel = oracle.msa_select(ms, spans, np.array([1.0, 2.0], np.float32), np.array([0, 2]))
    assert list(sel[0]) == [1, 0, -1]
    # rank order: score descending, block ascending
    spans = _msa_rows([27])
    sel = oracle.msa_select(ms, spans, np.array([3, 1, 3, 9, 0, 3, 2], np.float32), np.array([0, 7]))
    assert list(sel[0]) == [3, 0, 2]


def _gqa_case(q_heads=4, kv_heads=2, D=8, bs=4, P=4, page_start=1, ctx=13, q_len=3, seed=0, pages=None):
    ms = W.MSAShape(index_heads=2, index_dim=8, page_size=P, block_size=bs, topk_blocks=16, q_heads=q_heads,
                    kv_heads=kv_heads, head_dim=D, sm_scale=0.3)
    case = make_case(tiny_shape(page_size=P), [(ctx, q_len)], pages=pages, page_start=page_start)
    rng = np.random.default_rng(seed)
    n = ctx + q_len
    kvv = rng.standard_normal((n, 2 * kv_heads * D)).astype(np.float32)
    cache = np.zeros((case.num_pages * P, 2 * kv_heads * D), np.float32)
    cache[phys_rows(case, 0, np.arange(n))] = kvv
    q = rng.standard_normal((q_len, q_heads, D)).astype(np.float32)
    return ms, case, bf16(kvv).double(), bf16(cache).view(case.num_pages, P, -1), bf16(q)


def test_msa_attend_every_block_equals_dense_causal_gqa():
    """With every block selected, MSA attention is dense causal GQA: computed
    here by torch's scaled_dot_product_attention in fp64, K and V taken from
    the row layout [K heads | V heads], query head h on kv head h // group."""
    qh, kh, D, ctx, q_len = 6, 2, 8, 13, 3
    ms, case, kvv, cache, q = _gqa_case(q_heads=qh, kv_heads=kh, D=D, ctx=ctx, q_len=q_len, pages=[[3, 0, 4, 1, 2]])
    nblk = (ctx + q_len - 1) // ms.block_size + 1
    sel = np.full((q_len, ms.topk_blocks), -1, np.int32)
    for r in range(q_len):
        nb = (ctx + r) // ms.block_size + 1
        sel[r, :nb] = np.arange(nb)[::-1]   # any order
    assert nblk <= ms.topk_blocks
    out = oracle.msa_attend(ms, case.spans, case.num_pages, sel, q, cache)
    n = ctx + q_len
    k = kvv[:, :kh * D].view(n, kh, D).transpose(0, 1).repeat_interleave(qh // kh, dim=0)   # (qh, n, D)
    v = kvv[:, kh * D:].view(n, kh, D).transpose(0, 1).repeat_interleave(qh // kh, dim=0)
    mask = torch.zeros(q_len, n, dtype=torch.bool)
    for r in range(q_len):
        mask[r, :ctx + r + 1] = True
    ref = torch.nn.functional.scaled_dot_product_attention(q.double().transpose(0, 1), k, v, attn_mask=mask,
                                                           scale=ms.sm_scale)
    assert np.allclose(out, ref.transpose(0, 1).numpy(), rtol=1e-12, atol=1e-12)


def test_msa_attend_head_groups_read_their_kv_head():
    """V of kv head g constant g + 1: every query head of group g outputs g + 1."""
    qh, kh, D = 8, 4, 4
    ms, case, kvv, cache, q = _gqa_case(q_heads=qh, kv_heads=kh, D=D, ctx=9, q_len=2)
    c = cache.clone().float().view(-1, 2 * kh * D)
    for g in range(kh):
        c[:, (kh + g) * D:(kh + g + 1) * D] = g + 1
    sel = np.array([[0, 2, -1, -1] + [-1] * 12, [1, -1, -1, -1] + [-1] * 12], np.int32)
    out = oracle.msa_attend(ms, case.spans, case.num_pages, sel, q, bf16(c.numpy()).view(cache.shape))
    for h in range(qh):
        assert np.allclose(out[:, h, :], h // (qh // kh) + 1, rtol=0, atol=1e-14)   # softmax weights sum to 1


def test_msa_attend_uniform_logits_give_the_mean_of_visible_values():
    """q = 0: equal logits, so each head outputs the mean V over the visible
    positions of its selected blocks (the row at position 13 with blocks 1 and
    3 of size 4 sees positions 4..7 and 12..13)."""
    ms, case, kvv, cache, q = _gqa_case(ctx=13, q_len=1, kv_heads=1, q_heads=2)
    sel = np.array([[3, 1] + [-1] * 14], np.int32)
    out = oracle.msa_attend(ms, case.spans, case.num_pages, sel, torch.zeros_like(q), cache)
    D = ms.head_dim
    vis = [4, 5, 6, 7, 12, 13]
    mean = kvv[vis][:, D:2 * D].mean(dim=0).numpy()
    assert np.allclose(out[0, 0], mean, rtol=0, atol=1e-14) and np.allclose(out[0, 1], mean, rtol=0, atol=1e-14)


def test_msa_attend_rejects_blocks_past_the_row():
    ms, case, kvv, cache, q = _gqa_case(ctx=13, q_len=1)
    sel = np.array([[4] + [-1] * 15], np.int32)   # the row at position 13 has blocks 0..3
    with pytest.raises(oracle.OracleError):
        oracle.msa_attend(ms, case.spans, case.num_pages, sel, q, cache)
