"""CPU oracle for DeepSeek Sparse Attention over a paged MLA cache.

TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the CPU
baseline leg of bench.py may import this package.  It shares no code with the
CUDA library (deepseek_sparse_attention_dsa_gb300), and the library never
imports it.

The arithmetic lives in dsa_oracle.c (plain loops in double precision, OpenMP
over rows).  This wrapper only marshals numpy / torch-CPU arrays and derives the
per-row table (position, page list, page_start) from the request spans itself,
following the DSASpan definition on the mstar page
"mstar.engine.resources.dsa.manager": a span's q_len rows start at row q_start,
its first row sits at position ctx_start, and its token 0 is page_start slots
into its page list.

Functions (all return numpy arrays):
  store_keys(shape, spans, num_pages, keys, cache)      -> cache with this step's keys written
  index_scores(shape, spans, num_pages, q, w, cache)    -> (scores fp32 concatenated, offsets)
  topk(shape, spans, scores, offsets)                   -> (T, topk) int32, -1 padded
  attend(shape, spans, num_pages, sel, q_nope, q_pe, latent_cache, sink) -> (T, H, L) float64
  e4m3_values(codes)                                    -> float64 values of e4m3 bytes
  e4m3_encode(values)                                   -> e4m3 codes of fp32 values
  quantize_store_keys / quantize_store_latents          -> caches with this step's bf16 rows quantised
  msa_block_scores(msa, spans, scores, offsets)         -> (block scores fp32, block offsets)
  msa_select(msa, spans, block_scores, block_offsets)   -> (T, topk_blocks) int32 block ids, -1 padded
  msa_attend(msa, spans, num_pages, sel, q, kv_cache)   -> (T, q_heads, head_dim) float64

Parity status of each function is recorded in the docstring of each test in
tests/test_oracle_pins.py.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_lib = None

OK, BAD_ARG, SHORT_HISTORY, BAD_PAGE, BAD_SELECTION, NOMEM = range(6)
_ERRORS = {BAD_ARG: "bad argument", SHORT_HISTORY: "span pages do not reach a needed position",
           BAD_PAGE: "page id outside the cache", BAD_SELECTION: "selected position outside 0..pos",
           NOMEM: "out of host memory"}


class OracleError(RuntimeError):
    pass


class _Rows(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("page_size", ctypes.c_int32), ("num_pages", ctypes.c_int32),
                ("pos", ctypes.c_void_p), ("page_off", ctypes.c_void_p), ("npages", ctypes.c_void_p),
                ("page_start", ctypes.c_void_p), ("pages", ctypes.c_void_p)]


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        L.oracle_e4m3_value.restype = ctypes.c_double
        L.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
        L.oracle_store_keys.argtypes = [ctypes.POINTER(_Rows), ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
        L.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        L.oracle_e4m3_encode.restype = ctypes.c_uint8
        L.oracle_quantize_store_keys.argtypes = [ctypes.POINTER(_Rows), ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
        L.oracle_quantize_store_latents.argtypes = [ctypes.POINTER(_Rows), ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                                    ctypes.c_void_p]
        L.oracle_index_scores.argtypes = [ctypes.POINTER(_Rows), ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
        L.oracle_index_scores_fp8q.argtypes = [ctypes.POINTER(_Rows), ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                               ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                               ctypes.c_void_p, ctypes.c_void_p]
        L.oracle_quantize_rows.argtypes = [ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
        L.oracle_topk.argtypes = [ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
        L.oracle_attend.argtypes = [ctypes.POINTER(_Rows), ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                    ctypes.c_double, ctypes.c_void_p]
        L.oracle_msa_block_scores.argtypes = [ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                              ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
        L.oracle_msa_attend.argtypes = [ctypes.POINTER(_Rows), ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                        ctypes.c_double, ctypes.c_void_p]
        L.oracle_set_num_threads.argtypes = [ctypes.c_int]
        L.oracle_max_threads.restype = ctypes.c_int
        _lib = L
    return _lib


def set_num_threads(n: int) -> None:
    lib().oracle_set_num_threads(int(n))


def max_threads() -> int:
    return int(lib().oracle_max_threads())


def _np(x, dtype=None):
    """torch (CPU) or numpy -> contiguous numpy, reinterpreting bf16 as uint16."""
    if hasattr(x, "detach"):
        import torch
        x = x.detach()
        if x.device.type != "cpu":
            raise ValueError("the oracle takes host arrays")
        if x.dtype == torch.bfloat16:
            x = x.view(torch.int16)
        x = x.contiguous().numpy()
    x = np.ascontiguousarray(x)
    if dtype is not None:
        x = x.view(dtype) if x.dtype.itemsize == np.dtype(dtype).itemsize else x.astype(dtype)
    return x


def _check(status):
    if status != OK:
        raise OracleError(_ERRORS.get(status, "error %d" % status))


class RowTable:
    """Per-row positions and page lists, built from the spans (DSASpan reading)."""

    def __init__(self, spans, page_size: int, num_pages: int):
        spans = list(spans)
        T = sum(int(s.q_len) for s in spans)
        expect = 0
        for s in spans:
            if int(s.q_start) != expect or int(s.q_len) <= 0 or int(s.ctx_start) < 0 or int(s.page_start) < 0:
                raise OracleError(_ERRORS[BAD_ARG])
            expect += int(s.q_len)
        self.T = T
        self.pos = np.empty(T, np.int64)
        self.page_off = np.empty(T, np.int64)
        self.npages = np.empty(T, np.int64)
        self.page_start = np.empty(T, np.int64)
        page_lists, off = [], 0
        for s in spans:
            pg = np.asarray(s.pages, dtype=np.int32)
            sl = slice(int(s.q_start), int(s.q_start) + int(s.q_len))
            self.pos[sl] = int(s.ctx_start) + np.arange(int(s.q_len))
            self.page_off[sl] = off
            self.npages[sl] = len(pg)
            self.page_start[sl] = int(s.page_start)
            page_lists.append(pg)
            off += len(pg)
        self.pages = np.concatenate(page_lists) if page_lists else np.zeros(1, np.int32)
        self.struct = _Rows(T, int(page_size), int(num_pages), self.pos.ctypes.data, self.page_off.ctypes.data,
                            self.npages.ctypes.data, self.page_start.ctypes.data, self.pages.ctypes.data)

    def score_offsets(self) -> np.ndarray:
        off = np.zeros(self.T + 1, np.int64)
        np.cumsum(self.pos + 1, out=off[1:])
        return off


def e4m3_values(codes) -> np.ndarray:
    codes = np.asarray(codes, dtype=np.uint8).reshape(-1)
    L = lib()
    return np.array([L.oracle_e4m3_value(int(c)) for c in codes], dtype=np.float64)


def store_keys(shape, spans, num_pages, keys, cache) -> np.ndarray:
    rt = RowTable(spans, shape.page_size, num_pages)
    k = _np(keys).view(np.uint8)
    out = _np(cache).view(np.uint8).copy()
    _check(lib().oracle_store_keys(ctypes.byref(rt.struct), int(shape.index_fmt), int(shape.index_dim),
                                   k.ctypes.data, out.ctypes.data))
    return out


def e4m3_encode(values) -> np.ndarray:
    """fp32 values -> E4M3 codes (round to nearest even, saturating at 448)."""
    v = np.asarray(values, dtype=np.float32).reshape(-1)
    L = lib()
    return np.array([L.oracle_e4m3_encode(float(x)) for x in v], dtype=np.uint8)


def quantize_store_keys(shape, spans, num_pages, keys_bf16, cache) -> np.ndarray:
    """bf16 index keys (T, index_dim) -> the 132-byte fp8 rows stored at each row's slot."""
    rt = RowTable(spans, shape.page_size, num_pages)
    k = _np(keys_bf16).view(np.uint16)
    out = _np(cache).view(np.uint8).copy()
    _check(lib().oracle_quantize_store_keys(ctypes.byref(rt.struct), int(shape.index_dim), k.ctypes.data,
                                            out.ctypes.data))
    return out


def quantize_store_latents(shape, spans, num_pages, latents_bf16, cache) -> np.ndarray:
    """bf16 latent rows (T, L + R) -> the 656-byte fp8 rows stored at each row's slot."""
    rt = RowTable(spans, shape.page_size, num_pages)
    a = _np(latents_bf16).view(np.uint16)
    out = _np(cache).view(np.uint8).copy()
    _check(lib().oracle_quantize_store_latents(ctypes.byref(rt.struct), int(shape.kv_lora_rank), int(shape.rope_dim),
                                               a.ctypes.data, out.ctypes.data))
    return out


def index_scores(shape, spans, num_pages, q, w, cache):
    rt = RowTable(spans, shape.page_size, num_pages)
    qa = _np(q).view(np.uint16)
    wa = _np(w, np.float32)
    ca = _np(cache).view(np.uint8)
    off = rt.score_offsets()
    scores = np.zeros(int(off[-1]), np.float32)
    _check(lib().oracle_index_scores(ctypes.byref(rt.struct), int(shape.index_heads), int(shape.index_dim),
                                     int(shape.index_fmt), qa.ctypes.data, wa.ctypes.data, ca.ctypes.data,
                                     off.ctypes.data, scores.ctypes.data))
    return scores, off


def quantize_rows(x_bf16, width: int):
    """bf16 values, rows of `width` -> (e4m3 codes uint8, one fp32 scale per row)
    by the quantize-on-store rule (fp8 query)."""
    a = _np(x_bf16).view(np.uint16).reshape(-1)
    n = a.size // width
    codes = np.empty(n * width, np.uint8)
    scales = np.empty(n, np.float32)
    _check(lib().oracle_quantize_rows(n, int(width), a.ctypes.data, codes.ctypes.data, scales.ctypes.data))
    return codes, scales


def index_scores_fp8q(shape, spans, num_pages, q_codes, q_scale, w, cache):
    """Indexer scores with an fp8 query: q = e4m3(q_codes) * q_scale per (row, head)."""
    rt = RowTable(spans, shape.page_size, num_pages)
    qc = _np(q_codes).view(np.uint8)
    qs = _np(q_scale, np.float32)
    wa = _np(w, np.float32)
    ca = _np(cache).view(np.uint8)
    off = rt.score_offsets()
    scores = np.zeros(int(off[-1]), np.float32)
    _check(lib().oracle_index_scores_fp8q(ctypes.byref(rt.struct), int(shape.index_heads), int(shape.index_dim),
                                          int(shape.index_fmt), qc.ctypes.data, qs.ctypes.data, wa.ctypes.data,
                                          ca.ctypes.data, off.ctypes.data, scores.ctypes.data))
    return scores, off


def topk(shape, spans, scores, offsets) -> np.ndarray:
    rt = RowTable(spans, shape.page_size, 1)
    sc = np.ascontiguousarray(scores, dtype=np.float32)
    off = np.ascontiguousarray(offsets, dtype=np.int64)
    sel = np.empty((rt.T, int(shape.topk)), np.int32)
    _check(lib().oracle_topk(rt.T, int(shape.topk), rt.pos.ctypes.data, sc.ctypes.data, off.ctypes.data,
                             sel.ctypes.data))
    return sel


def attend(shape, spans, num_pages, sel, q_nope, q_pe, latent_cache, sink=None) -> np.ndarray:
    rt = RowTable(spans, shape.page_size, num_pages)
    s = _np(sel, np.int32)
    qn = _np(q_nope).view(np.uint16)
    qp = _np(q_pe).view(np.uint16)
    ca = _np(latent_cache).view(np.uint8)
    sk = None if sink is None else _np(sink, np.float32)
    out = np.zeros((rt.T, int(shape.heads), int(shape.kv_lora_rank)), np.float64)
    _check(lib().oracle_attend(ctypes.byref(rt.struct), int(shape.heads), int(shape.kv_lora_rank),
                               int(shape.rope_dim), int(s.shape[1]), int(shape.latent_fmt), s.ctypes.data,
                               qn.ctypes.data, qp.ctypes.data, ca.ctypes.data,
                               None if sk is None else sk.ctypes.data, float(shape.sm_scale), out.ctypes.data))
    return out


def run_all(wl, index_cache, latent_cache, step):
    """store -> score -> select -> attend for a whole workload (host arrays)."""
    sh = wl.shape
    cache = store_keys(sh, wl.spans, wl.num_pages, step.keys, index_cache)
    scores, off = index_scores(sh, wl.spans, wl.num_pages, step.q, step.w, cache)
    sel = topk(sh, wl.spans, scores, off)
    out = attend(sh, wl.spans, wl.num_pages, sel, step.q_nope, step.q_pe, latent_cache, step.sink)
    return dict(index_cache=cache, scores=scores, offsets=off, selection=sel, out=out)


# ----------------------------------------------------------------------------
# block-sparse MSA (LLMServingSim, "Sparse attention (DSA and block-sparse
# MSA)", MiniMax-M3 column)
# ----------------------------------------------------------------------------
def msa_block_offsets(spans, block_size: int) -> np.ndarray:
    rt = RowTable(spans, 1, 1)
    off = np.zeros(rt.T + 1, np.int64)
    np.cumsum(rt.pos // int(block_size) + 1, out=off[1:])
    return off


def msa_block_scores(msa, spans, scores, offsets):
    """Largest token score of each block of block_size positions the row sees."""
    rt = RowTable(spans, 1, 1)
    sc = np.ascontiguousarray(scores, dtype=np.float32)
    off = np.ascontiguousarray(offsets, dtype=np.int64)
    boff = msa_block_offsets(spans, msa.block_size)
    bs = np.zeros(int(boff[-1]), np.float32)
    _check(lib().oracle_msa_block_scores(rt.T, int(msa.block_size), rt.pos.ctypes.data, sc.ctypes.data,
                                         off.ctypes.data, boff.ctypes.data, bs.ctypes.data))
    return bs, boff


def msa_select(msa, spans, block_scores, block_offsets) -> np.ndarray:
    """The causal top-k of the DSA selection, over a row's blocks: the
    topk_blocks highest block scores, ties to the lower block, -1 padded."""
    rt = RowTable(spans, 1, 1)
    last = np.ascontiguousarray(rt.pos // int(msa.block_size), dtype=np.int64)   # the row's last block
    bs = np.ascontiguousarray(block_scores, dtype=np.float32)
    boff = np.ascontiguousarray(block_offsets, dtype=np.int64)
    sel = np.empty((rt.T, int(msa.topk_blocks)), np.int32)
    _check(lib().oracle_topk(rt.T, int(msa.topk_blocks), last.ctypes.data, bs.ctypes.data, boff.ctypes.data,
                             sel.ctypes.data))
    return sel


def msa_attend(msa, spans, num_pages, sel, q, kv_cache) -> np.ndarray:
    """GQA attention over the visible positions of the selected blocks."""
    rt = RowTable(spans, msa.page_size, num_pages)
    s = _np(sel, np.int32)
    qa = _np(q).view(np.uint16)
    ca = _np(kv_cache).view(np.uint8)
    out = np.zeros((rt.T, int(msa.q_heads), int(msa.head_dim)), np.float64)
    _check(lib().oracle_msa_attend(ctypes.byref(rt.struct), int(msa.q_heads), int(msa.kv_heads), int(msa.head_dim),
                                   int(msa.block_size), int(s.shape[1]), s.ctypes.data, qa.ctypes.data,
                                   ca.ctypes.data, float(msa.sm_scale), out.ctypes.data))
    return out


def msa_run_all(wl, index_cache, kv_cache, step, q):
    """store -> token scores -> block scores -> block selection -> GQA attention."""
    sh, ms = wl.shape, wl.msa
    cache = store_keys(sh, wl.spans, wl.num_pages, step.keys, index_cache)
    scores, off = index_scores(sh, wl.spans, wl.num_pages, step.q, step.w, cache)
    bscores, boff = msa_block_scores(ms, wl.spans, scores, off)
    sel = msa_select(ms, wl.spans, bscores, boff)
    out = msa_attend(ms, wl.spans, wl.num_pages, sel, q, kv_cache)
    return dict(index_cache=cache, scores=scores, offsets=off, block_scores=bscores, block_offsets=boff,
                selection=sel, out=out)
