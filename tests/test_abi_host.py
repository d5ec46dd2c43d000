"""The C-ABI library on the host (no GPU): it builds, loads, exports every
symbol include/dsa.h declares, and its planner validates spans as the header
states (a host-only context, device -1, makes no CUDA call)."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch  # noqa: F401  (loads the CUDA runtime the library links against)

from deepseek_sparse_attention_dsa_gb300 import build as dsa_build
from deepseek_sparse_attention_dsa_gb300 import dsa
from deepseek_sparse_attention_dsa_gb300 import workloads as W
from tests.dsa_cases import tiny_shape

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    dsa_build.build()
    return dsa.load()


def header_functions():
    text = open(os.path.join(ROOT, "include", "dsa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dsa_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = header_functions()
    assert "dsa_plan" in names and "dsa_attend" in names and "dsa_index_topk" in names
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) <= set(dsa.EXPORTED)


def test_status_strings(lib):
    for s in range(10):
        assert lib.dsa_status_str(s) and lib.dsa_status_str(s) != b"unknown status"
    assert lib.dsa_status_str(10) == b"unknown status"


def _host_ctx(shape=None):
    return dsa.Context(shape or W.DSAShape(**W.DEEPSEEK), device=-1)


class S:
    def __init__(self, q_start, q_len, ctx_start, pages, page_start=0):
        self.q_start, self.q_len, self.ctx_start, self.pages, self.page_start = q_start, q_len, ctx_start, pages, page_start


def _status(fn):
    try:
        fn()
    except dsa.DSAError as e:
        return e.status
    return 0


def test_create_rejects_bad_configs(lib):
    bad = W.DSAShape(**dict(W.DEEPSEEK, page_size=0))
    assert _status(lambda: dsa.Context(bad, device=-1)) == 1
    odd = W.DSAShape(**dict(W.DEEPSEEK, index_dim=3))          # rows not a multiple of 16 bytes
    assert _status(lambda: dsa.Context(odd, device=-1)) == 7
    fp8 = W.DSAShape(**dict(W.DEEPSEEK, index_dim=64), index_fmt=W.INDEX_FP8_132)   # fp8 rows are 128 + 4
    assert _status(lambda: dsa.Context(fp8, device=-1)) == 7


def test_plan_validation(lib):
    ctx = _host_ctx()
    P = 64
    pg = np.arange(4, dtype=np.int32)
    ok = ctx.plan([S(0, 1, 100, pg[:2]), S(1, 3, 0, pg[2:3])], cache_pages=4)
    assert ok.num_rows == 4 and not ok.needs_selection
    assert ok.num_scores == 101 + (1 + 2 + 3)
    # spans must tile rows in order
    assert _status(lambda: ctx.plan([S(1, 1, 0, pg[:1])], 4)) == 1
    assert _status(lambda: ctx.plan([S(0, 2, 0, pg[:1]), S(1, 1, 0, pg[1:2])], 4)) == 1
    assert _status(lambda: ctx.plan([S(0, 0, 0, pg[:1])], 4)) == 1
    assert _status(lambda: ctx.plan([S(0, 1, -1, pg[:1])], 4)) == 1
    assert _status(lambda: ctx.plan([S(0, 1, 0, pg[:1], page_start=-8)], 4)) == 1
    # too few pages for ctx_start + q_len tokens (mstar IndexKeyStore.history raises)
    assert _status(lambda: ctx.plan([S(0, 1, P, pg[:1])], 4)) == 2
    assert _status(lambda: ctx.plan([S(0, 1, P - 8, pg[:1], page_start=8)], 4)) == 2
    # page ids must exist in the cache
    assert _status(lambda: ctx.plan([S(0, 1, 0, np.array([4], np.int32))], 4)) == 1
    assert _status(lambda: ctx.plan([S(0, 1, 0, np.array([-1], np.int32))], 4)) == 1
    # empty step
    empty = ctx.plan([], cache_pages=4)
    assert empty.num_rows == 0 and empty.num_scores == 0


def test_plan_needs_selection_and_units(lib):
    ctx = _host_ctx()
    K = W.DEEPSEEK["topk"]
    pg = np.arange(64, dtype=np.int32)
    short = ctx.plan([S(0, 1, K - 1, pg[:32])], cache_pages=64)      # sees exactly topk keys
    assert not short.needs_selection
    long = ctx.plan([S(0, 1, K, pg[:33])], cache_pages=64)           # sees topk + 1
    assert long.needs_selection
    # attention: the rows' key tiles (64 keys each), in order, are cut into
    # contiguous ranges of ceil(S / n) tiles for n = min(76, ceil(S / 16))
    # persistent clusters (152 SMs); a row crossed by a cut is one unit per
    # piece.  One decode row of 32 tiles: two clusters of 16, two units.
    assert long.info.attend_splits_max == 2 and long.info.attend_units == 2
    wl = W.config(2)
    big = ctx.plan(wl.spans, wl.num_pages)
    tiles = 32 * wl.num_rows                  # every row selects 2048 keys
    n = min(76, -(-tiles // 16))
    per = -(-tiles // n)
    cuts_inside_rows = sum(1 for c in range(1, n) if (c * per) % 32 != 0)
    assert big.info.attend_units == wl.num_rows + cuts_inside_rows and big.info.attend_splits_max == 2
    assert big.num_scores == sum(range(8193, 16385))


def test_compute_calls_refuse_host_only_context(lib):
    ctx = _host_ctx()
    plan = ctx.plan([S(0, 1, 0, np.array([0], np.int32))], cache_pages=1)
    L = dsa.load()
    st = L.dsa_index_topk(ctx.handle, plan.handle, None, None, None, None, None)
    assert st == 1
    assert L.dsa_attend(ctx.handle, plan.handle, None, None, None, None, None, ctypes.c_float(1.0), None, None) == 1
    assert L.dsa_get_error(ctx.handle, None) == 1


def test_capturable_plan_calls_refuse_host_only_context_and_host_plans(lib):
    ctx = _host_ctx()
    assert _status(lambda: ctx.plan_capturable(8, 8, 1000, 10)) == 1
    L = dsa.load()
    h = ctypes.c_void_p()
    assert L.dsa_plan_capturable(None, 8, 8, 1000, 1, 10, None, ctypes.byref(h)) == 1
    assert L.dsa_plan_capturable(ctx.handle, 8, 8, 1000, 1, 10, None, None) == 1
    plan = ctx.plan([S(0, 1, 0, np.array([0], np.int32))], cache_pages=1)
    assert L.dsa_plan_update(ctx.handle, plan.handle, None, None, None, 0, None) == 1
    counts = (ctypes.c_int32 * 8)()
    assert L.dsa_plan_read_counts(plan.handle, ctypes.byref(counts)) == 1   # a host plan has no device counts


def test_indexer_stays_on_tensor_cores_for_any_page_start(lib):
    """Key tiles start on the box boundary below a span's page_start, so the
    box height depends on the page size only and any page_start keeps the
    tensor-core indexer; a page size that is not a multiple of 8 cannot."""
    ctx = _host_ctx()
    pg = np.arange(8, dtype=np.int32)
    for ps in (0, 1, 3, 37, 63, 64, 70):
        plan = ctx.plan([S(0, 1, 200, pg[:6], page_start=ps), S(1, 5, 9, pg[6:8], page_start=(ps * 7) % 64)],
                        cache_pages=8)
        assert plan.info.index_box_rows == 64 and plan.index_tensor_cores, ps
    tiny = W.config(0)
    plan = _host_ctx(tiny.shape).plan([S(0, 2, 0, np.arange(2, dtype=np.int32), page_start=5)], cache_pages=2)
    assert plan.info.index_box_rows == 16 and plan.index_tensor_cores
    small_pages = W.DSAShape(**dict(W.DEEPSEEK, page_size=4))
    plan = _host_ctx(small_pages).plan([S(0, 1, 10, np.arange(3, dtype=np.int32), page_start=1)], cache_pages=3)
    assert plan.info.index_box_rows == 4 and not plan.index_tensor_cores


def _att_schedule(positions, topk, num_sms=152):
    """The persistent attention schedule, written out: the rows' key tiles (64
    keys each) in row order are cut into n = min(SMs / 2, ceil(S / 16))
    contiguous ranges of ceil(S / n) tiles (n recomputed from that length); a
    row a cut crosses is one unit per piece.  Returns (units, largest pieces
    per row)."""
    tiles = [-(-min(topk, p + 1) // 64) for p in positions]
    S = sum(tiles)
    n = max(1, min(num_sms // 2, -(-S // 16)))
    per = max(1, -(-S // n))
    units, most, off = 0, 0, 0
    for t in tiles:
        pieces = (off + t - 1) // per - off // per + 1
        units += pieces
        most = max(most, pieces)
        off += t
    return units, most


@pytest.mark.parametrize("rows", [
    [0],                          # one tile
    [2047],                       # one full row: two clusters of 16 tiles
    [70000] * 16,                 # 16 decode rows: 32 clusters of 16 tiles, every row cut once
    [100000] * 128,               # long decode: 76 clusters of 54 tiles
    list(range(0, 640, 1)),       # 640 short rows of 1..10 tiles
    [5000] * 3 + list(range(2047, 2047 + 40)),   # decode rows and a chunk
])
def test_attention_schedule_units(lib, rows):
    """The plan's attention units follow the persistent schedule's definition
    (written out here): every row a range boundary crosses is one unit per
    piece."""
    ctx = _host_ctx()
    K = W.DEEPSEEK["topk"]
    pg = np.arange(2048, dtype=np.int32)
    spans, q = [], 0
    for p in rows:
        npg = (p + 1 + 63) // 64
        spans.append(S(q, 1, p, pg[:npg]))
        q += 1
    plan = ctx.plan(spans, cache_pages=2048)
    units, most = _att_schedule(rows, K)
    assert plan.info.attend_units == units and plan.info.attend_splits_max == most
