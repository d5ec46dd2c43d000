"""dsa_index_topk_static: index + top-k for callers that cannot allocate device
memory while serving (their process reserves HBM up front in its own pool).
Its scores live in the library's fixed device array instead of the context's
scratch.  Checked through the C ABI against dsa_index_topk on two calls in a
row (a larger step, then a smaller one that reuses the array's stale
contents) and on a third, larger step, with the device's free memory
unchanged around the calls; the size limit is checked too.  Collected last on
purpose."""
import ctypes

import numpy as np
import pytest
import torch

from deepseek_sparse_attention_dsa_gb300 import dsa
from deepseek_sparse_attention_dsa_gb300 import workloads as W
from tests import harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from deepseek_sparse_attention_dsa_gb300 import build
    build.build()


def _call_static(ctx, plan, q, w, cache, sel):
    L = dsa.load()
    return L.dsa_index_topk_static(ctx.handle, plan.handle, ctypes.c_void_p(q.data_ptr()),
                                   ctypes.c_void_p(w.data_ptr()), ctypes.c_void_p(cache.data_ptr()),
                                   ctypes.c_void_p(sel.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_static_entry_matches_index_topk_twice():
    """Two calls in a row (the second over the first's stale scores), then a
    third on a larger plan; each must equal dsa_index_topk.  Around the calls
    after the first, the device's free memory must not move: the entry point
    makes the driver allocate nothing (its array was taken by dsa_create)."""
    sh = W.DSAShape(**W.DEEPSEEK)
    ctx = dsa.Context(sh, 0)
    first = H.deepseek_small(seed=31, decode_ctx=(9000, 4100, 2500), chunk=(2100, 36))
    second = H.deepseek_small(seed=32, decode_ctx=(3000,), chunk=(1500, 8))
    third = H.deepseek_small(seed=33, decode_ctx=(12000, 7000, 5000, 300), chunk=(3000, 40))
    for i, wl in enumerate((first, second, third)):
        ic, _, st = H.device_inputs(wl)
        plan = ctx.plan(wl.spans, wl.num_pages)
        ctx.store_keys(plan, st.keys, ic)
        # the regular call first: it loads every kernel the static call uses
        ref = ctx.index_topk(plan, st.q, st.w, ic)
        got = torch.full_like(ref, -7)
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        assert _call_static(ctx, plan, st.q, st.w, ic, got) == dsa.DSA_OK
        torch.cuda.synchronize()
        free_after = torch.cuda.mem_get_info()[0]
        ctx.get_error()
        assert torch.equal(got, ref)
        if i > 0:
            assert free_after == free_before, "the static entry point changed the device's free memory"
        plan.close()


def test_static_entry_rejects_plans_over_the_limit():
    sh = W.DSAShape(**W.DEEPSEEK)
    ctx = dsa.Context(sh, 0)
    L = dsa.load()
    # two decode rows with 2M + 2M + 2 visible keys exceed 4M scores
    P = sh.page_size
    n = 2 * 1024 * 1024
    npg = -(-(n + 1) // P)

    class S:
        pass

    spans = []
    for i in range(2):
        s = S()
        s.q_start, s.q_len, s.ctx_start, s.page_start = i, 1, n, 0
        s.pages = np.arange(npg, dtype=np.int32)
        spans.append(s)
    plan = ctx.plan(spans, npg)
    assert plan.num_scores > dsa_static_max()
    sel = torch.empty(2, sh.topk, dtype=torch.int32, device="cuda")
    q = torch.zeros(2, sh.index_heads, sh.index_dim, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(2, sh.index_heads, dtype=torch.float32, device="cuda")
    cache = torch.zeros(1, dtype=torch.bfloat16, device="cuda")
    assert _call_static(ctx, plan, q, w, cache, sel) == 8   # DSA_ERR_SCRATCH_LIMIT, nothing launched
    assert ctx.last_launch_count() == 0
    assert b"DSA_STATIC_SCORES_MAX" in L.dsa_status_str(8)


def dsa_static_max():
    return 4 * 1024 * 1024
