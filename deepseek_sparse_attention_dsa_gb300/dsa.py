"""Python binding of the C ABI in include/dsa.h (argument marshalling only).

Every computation runs in libdsa_gb300.so (CUDA, sm_103a).  Loading fails
loudly when the library has not been built: there is no CPU path.

    ctx = Context(shape, device=0)                 # dsa_create
    plan = ctx.plan(spans, cache_pages)            # dsa_plan
    ctx.store_keys(plan, keys, index_cache)        # dsa_store_keys
    sel = ctx.index_topk(plan, q, w, index_cache)  # dsa_index_topk
    out = ctx.attend(plan, sel, q_nope, q_pe, latent_cache, sink, sm_scale)   # dsa_attend
    ctx.get_error()                                # dsa_get_error (synchronises)

A decode step that re-plans on the device (capturable in a CUDA graph):

    plan = ctx.plan_capturable(max_rows, max_spans, max_scores, cache_pages)
    ctx.plan_update(plan, num_spans, spans, pages)  # device tensors, no sync
    ... then store_keys / index_topk / attend with max_rows-row buffers

fp8 query for the indexer (fp8 index cache): quantize_q, index_scores_fp8q,
index_topk_fp8q.  Quantize-on-store: quantize_store_keys / _latents.  SHARED
layers: attend_shared.

Tensors are torch tensors on the context's device, contiguous, in the dtypes
the header states; the calls run on torch's current CUDA stream unless a
stream is given.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import numpy as np
import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_build", "libdsa_gb300.so")

DSA_OK = 0
STATUS_NAMES = {0: "DSA_OK", 1: "DSA_ERR_INVALID_ARG", 2: "DSA_ERR_SHORT_HISTORY", 3: "DSA_ERR_OOM",
                4: "DSA_ERR_CUDA", 5: "DSA_ERR_BOUNDS", 6: "DSA_ERR_TIMEOUT", 7: "DSA_ERR_UNSUPPORTED",
                8: "DSA_ERR_SCRATCH_LIMIT", 9: "DSA_ERR_BAD_SPANS"}

EXPORTED = ["dsa_create", "dsa_destroy", "dsa_plan", "dsa_plan_destroy", "dsa_plan_get_info", "dsa_store_keys",
            "dsa_index_topk", "dsa_index_scores", "dsa_topk_from_scores", "dsa_attend", "dsa_get_error",
            "dsa_last_launch_count", "dsa_status_str", "dsa_index_topk_static", "dsa_last_cuda_error",
            "dsa_quantize_store_keys", "dsa_quantize_store_latents", "dsa_attend_shared", "dsa_plan_capturable",
            "dsa_plan_update", "dsa_plan_read_counts", "dsa_quantize_q", "dsa_index_scores_fp8q",
            "dsa_index_topk_fp8q", "dsa_selftest_wait_timeout", "dsa_msa_select_blocks", "dsa_msa_index_select",
            "dsa_msa_attend", "dsa_msa_attend_on_tensor_cores"]

# dsa_device_span_t: q_len, ctx_start, page_start, page_off, num_pages, reserved (int32 each)
DEVICE_SPAN_FIELDS = 6


class DSAError(RuntimeError):
    def __init__(self, status: int, what: str, detail: str = ""):
        self.status = status
        super().__init__("%s: %s (%s)%s" % (what, STATUS_NAMES.get(status, str(status)), _status_str(status),
                                           (" [" + detail + "]") if detail else ""))


class _Config(ctypes.Structure):
    _fields_ = [("index_heads", ctypes.c_int32), ("index_dim", ctypes.c_int32), ("topk", ctypes.c_int32),
                ("heads", ctypes.c_int32), ("kv_lora_rank", ctypes.c_int32), ("rope_dim", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("latent_fmt", ctypes.c_int32), ("index_fmt", ctypes.c_int32)]


class _Span(ctypes.Structure):
    _fields_ = [("request_id", ctypes.c_int64), ("q_start", ctypes.c_int32), ("q_len", ctypes.c_int32),
                ("ctx_start", ctypes.c_int32), ("page_start", ctypes.c_int32), ("pages", ctypes.c_void_p),
                ("num_pages", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class _MsaShape(ctypes.Structure):
    _fields_ = [("block_size", ctypes.c_int32), ("topk_blocks", ctypes.c_int32), ("q_heads", ctypes.c_int32),
                ("kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("reserved", ctypes.c_int32)]


def _msa_shape(ms) -> _MsaShape:
    return _MsaShape(int(ms.block_size), int(ms.topk_blocks), int(ms.q_heads), int(ms.kv_heads), int(ms.head_dim), 0)


class PlanInfo(ctypes.Structure):
    _fields_ = [("num_rows", ctypes.c_int32), ("num_spans", ctypes.c_int32), ("needs_selection", ctypes.c_int32),
                ("index_items", ctypes.c_int32), ("num_scores", ctypes.c_int64), ("attend_units", ctypes.c_int32),
                ("attend_splits_max", ctypes.c_int32), ("index_tensor_cores", ctypes.c_int32),
                ("index_box_rows", ctypes.c_int32)]


_lib = None


def library_path() -> str:
    return LIB_PATH


def load() -> ctypes.CDLL:
    """Load libdsa_gb300.so; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError("libdsa_gb300.so is not built (%s); run "
                           "`python -m deepseek_sparse_attention_dsa_gb300.build`" % LIB_PATH)
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    L.dsa_create.argtypes = [ctypes.POINTER(_Config), ctypes.c_int, ctypes.POINTER(vp)]
    L.dsa_destroy.argtypes = [vp]
    L.dsa_destroy.restype = None
    L.dsa_plan.argtypes = [vp, ctypes.POINTER(_Span), i32, i32, vp, ctypes.POINTER(vp)]
    L.dsa_plan_destroy.argtypes = [vp]
    L.dsa_plan_destroy.restype = None
    L.dsa_plan_get_info.argtypes = [vp, ctypes.POINTER(PlanInfo)]
    L.dsa_store_keys.argtypes = [vp, vp, vp, vp, vp]
    L.dsa_quantize_store_keys.argtypes = [vp, vp, vp, vp, vp]
    L.dsa_quantize_store_latents.argtypes = [vp, vp, vp, vp, vp]
    L.dsa_index_topk.argtypes = [vp, vp, vp, vp, vp, vp, vp]
    L.dsa_index_scores.argtypes = [vp, vp, vp, vp, vp, vp, vp]
    L.dsa_index_topk_static.argtypes = [vp, vp, vp, vp, vp, vp, vp]
    L.dsa_topk_from_scores.argtypes = [vp, vp, vp, vp, vp]
    L.dsa_attend.argtypes = [vp, vp, vp, vp, vp, vp, vp, ctypes.c_float, vp, vp]
    L.dsa_attend_shared.argtypes = [vp, vp, vp, vp, vp, vp, ctypes.c_float, vp, vp]
    L.dsa_plan_capturable.argtypes = [vp, i32, i32, i64, i32, i32, vp, ctypes.POINTER(vp)]
    L.dsa_plan_update.argtypes = [vp, vp, vp, vp, vp, i64, vp]
    L.dsa_plan_read_counts.argtypes = [vp, ctypes.POINTER(i32 * 8)]
    L.dsa_quantize_q.argtypes = [vp, vp, vp, vp, vp, vp]
    L.dsa_index_scores_fp8q.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp]
    L.dsa_index_topk_fp8q.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp]
    L.dsa_get_error.argtypes = [vp, vp]
    L.dsa_selftest_wait_timeout.argtypes = [vp, ctypes.c_uint64, vp, vp]
    msp = ctypes.POINTER(_MsaShape)
    L.dsa_msa_select_blocks.argtypes = [vp, vp, msp, vp, vp, vp]
    L.dsa_msa_index_select.argtypes = [vp, vp, msp, vp, vp, vp, vp, vp]
    L.dsa_msa_attend.argtypes = [vp, vp, msp, vp, vp, vp, ctypes.c_float, vp, vp]
    L.dsa_msa_attend_on_tensor_cores.argtypes = [vp, vp, msp]
    L.dsa_msa_attend_on_tensor_cores.restype = ctypes.c_int
    L.dsa_last_launch_count.argtypes = [vp]
    L.dsa_last_launch_count.restype = i32
    L.dsa_last_cuda_error.argtypes = [vp]
    L.dsa_last_cuda_error.restype = ctypes.c_char_p
    L.dsa_status_str.argtypes = [i32]
    L.dsa_status_str.restype = ctypes.c_char_p
    for name in ("dsa_create", "dsa_plan", "dsa_plan_get_info", "dsa_store_keys", "dsa_index_topk", "dsa_index_topk_static",
                 "dsa_index_scores", "dsa_topk_from_scores", "dsa_attend", "dsa_get_error", "dsa_quantize_store_keys",
                 "dsa_quantize_store_latents", "dsa_attend_shared", "dsa_plan_capturable", "dsa_plan_update",
                 "dsa_plan_read_counts", "dsa_quantize_q", "dsa_index_scores_fp8q", "dsa_index_topk_fp8q",
                 "dsa_selftest_wait_timeout", "dsa_msa_select_blocks", "dsa_msa_index_select", "dsa_msa_attend"):
        getattr(L, name).restype = i32
    _lib = L
    return L


def _status_str(s: int) -> str:
    try:
        return load().dsa_status_str(int(s)).decode()
    except Exception:
        return "?"


def _check(status: int, what: str, ctx_handle=None):
    if status != DSA_OK:
        detail = ""
        if ctx_handle is not None and status == 4:
            try:
                detail = load().dsa_last_cuda_error(ctx_handle).decode()
            except Exception:
                detail = ""
        raise DSAError(status, what, detail)


def _ptr(t: Optional[torch.Tensor], device: torch.device, dtypes, name: str):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch tensor" % name)
    if t.device != device:
        raise ValueError("%s is on %s, expected %s" % (name, t.device, device))
    if t.dtype not in dtypes:
        raise TypeError("%s has dtype %s, expected one of %s" % (name, t.dtype, dtypes))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


class Plan:
    """A step's rows (dsa_plan_t).  Keeps the spans' page arrays alive."""

    def __init__(self, ctx: "Context", handle: ctypes.c_void_p, keepalive, capturable: bool = False):
        self.ctx = ctx
        self.handle = handle
        self._keep = keepalive
        self.capturable = capturable
        info = PlanInfo()
        _check(load().dsa_plan_get_info(handle, ctypes.byref(info)), "dsa_plan_get_info")
        self.info = info

    @property
    def num_rows(self) -> int:
        return int(self.info.num_rows)

    @property
    def needs_selection(self) -> bool:
        return bool(self.info.needs_selection)

    @property
    def num_scores(self) -> int:
        return int(self.info.num_scores)

    @property
    def index_tensor_cores(self) -> bool:
        """True when the plan's index scores run on the tensor-core kernels."""
        return bool(self.info.index_tensor_cores)

    def read_counts(self) -> dict:
        """dsa_plan_read_counts (capturable plans; synchronises the device)."""
        c = (ctypes.c_int32 * 8)()
        _check(load().dsa_plan_read_counts(self.handle, ctypes.byref(c)), "dsa_plan_read_counts")
        return {"rows": c[0], "index_items": c[1], "attend_units": c[2], "split_rows": c[3], "slots": c[4],
                "valid": bool(c[5]), "splits": c[6], "num_scores": c[7]}

    def close(self):
        if self.handle:
            load().dsa_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Context:
    """dsa_ctx_t for one problem shape on one device (device=-1: host-only,
    planning and validation only)."""

    def __init__(self, shape, device: int = 0):
        L = load()
        cfg = _Config(shape.index_heads, shape.index_dim, shape.topk, shape.heads, shape.kv_lora_rank,
                      shape.rope_dim, shape.page_size, int(shape.latent_fmt), int(shape.index_fmt))
        h = ctypes.c_void_p()
        _check(L.dsa_create(ctypes.byref(cfg), int(device), ctypes.byref(h)), "dsa_create")
        self.handle = h
        self.shape = shape
        self.device_index = int(device)
        self.device = torch.device("cuda", device) if device >= 0 else torch.device("cpu")

    def close(self):
        if getattr(self, "handle", None):
            load().dsa_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -------------------------------------------------------------- planning
    def plan(self, spans: Sequence, cache_pages: int, stream=None) -> Plan:
        arr = (_Span * max(1, len(spans)))()
        keep = []
        for i, s in enumerate(spans):
            pg = np.ascontiguousarray(np.asarray(s.pages, dtype=np.int32))
            keep.append(pg)
            arr[i] = _Span(int(getattr(s, "request_id", i)), int(s.q_start), int(s.q_len), int(s.ctx_start),
                           int(getattr(s, "page_start", 0)), pg.ctypes.data if pg.size else None, int(pg.size), 0)
        h = ctypes.c_void_p()
        st = None if self.device_index < 0 else _stream(stream)
        _check(load().dsa_plan(self.handle, arr, len(spans), int(cache_pages), st, ctypes.byref(h)), "dsa_plan")
        return Plan(self, h, (arr, keep))

    def plan_capturable(self, max_rows: int, max_spans: int, max_scores: int, cache_pages: int,
                        page_start_align: int = 1, stream=None) -> Plan:
        """dsa_plan_capturable: a fixed-capacity plan that dsa_plan_update
        rewrites on the device (capturable in a CUDA graph)."""
        h = ctypes.c_void_p()
        st = None if self.device_index < 0 else _stream(stream)
        _check(load().dsa_plan_capturable(self.handle, int(max_rows), int(max_spans), int(max_scores),
                                          int(page_start_align), int(cache_pages), st, ctypes.byref(h)),
               "dsa_plan_capturable", self.handle)
        return Plan(self, h, None, capturable=True)

    def plan_update(self, plan: Plan, num_spans: torch.Tensor, spans: torch.Tensor, pages: torch.Tensor, stream=None):
        """dsa_plan_update: num_spans (1,) int32, spans (max_spans, 6) int32
        [q_len, ctx_start, page_start, page_off, num_pages, 0], pages int32;
        all on the device.  Enqueued on the stream; nothing synchronises."""
        d = self.device
        if spans.dim() != 2 or spans.shape[1] != DEVICE_SPAN_FIELDS:
            raise ValueError("spans must be (max_spans, %d) int32" % DEVICE_SPAN_FIELDS)
        plan._keep = (num_spans, spans, pages)   # the plan keeps pointing at the page array
        _check(load().dsa_plan_update(self.handle, plan.handle, _ptr(num_spans, d, (torch.int32,), "num_spans"),
                                      _ptr(spans, d, (torch.int32,), "spans"), _ptr(pages, d, (torch.int32,), "pages"),
                                      int(pages.numel()), _stream(stream)), "dsa_plan_update", self.handle)

    # -------------------------------------------------------------- compute
    def store_keys(self, plan: Plan, keys: torch.Tensor, index_cache: torch.Tensor, stream=None):
        d = self.device
        _check(load().dsa_store_keys(self.handle, plan.handle, _ptr(keys, d, (torch.bfloat16, torch.uint8), "keys"),
                                     _ptr(index_cache, d, (torch.bfloat16, torch.uint8), "index_cache"),
                                     _stream(stream)), "dsa_store_keys", self.handle)

    def quantize_store_keys(self, plan: Plan, keys_bf16: torch.Tensor, index_cache: torch.Tensor, stream=None):
        """bf16 index keys (T, 128) -> 132-byte fp8 rows at each row's slot (fp8 index format only)."""
        d = self.device
        _check(load().dsa_quantize_store_keys(self.handle, plan.handle, _ptr(keys_bf16, d, (torch.bfloat16,), "keys"),
                                              _ptr(index_cache, d, (torch.uint8,), "index_cache"), _stream(stream)),
               "dsa_quantize_store_keys", self.handle)

    def quantize_store_latents(self, plan: Plan, latents_bf16: torch.Tensor, latent_cache: torch.Tensor, stream=None):
        """bf16 latent rows (T, 512 + 64) -> 656-byte fp8 rows at each row's slot (fp8 latent format only)."""
        d = self.device
        _check(load().dsa_quantize_store_latents(self.handle, plan.handle,
                                                 _ptr(latents_bf16, d, (torch.bfloat16,), "latents"),
                                                 _ptr(latent_cache, d, (torch.uint8,), "latent_cache"), _stream(stream)),
               "dsa_quantize_store_latents", self.handle)

    def index_topk(self, plan: Plan, q, w, index_cache, selection=None, stream=None) -> torch.Tensor:
        d = self.device
        if selection is None:
            selection = torch.empty(plan.num_rows, self.shape.topk, dtype=torch.int32, device=d)
        _check(load().dsa_index_topk(self.handle, plan.handle, _ptr(q, d, (torch.bfloat16,), "q"),
                                     _ptr(w, d, (torch.float32,), "w"),
                                     _ptr(index_cache, d, (torch.bfloat16, torch.uint8), "index_cache"),
                                     _ptr(selection, d, (torch.int32,), "selection"), _stream(stream)),
               "dsa_index_topk", self.handle)
        return selection

    def index_topk_static(self, plan: Plan, q, w, index_cache, selection=None, stream=None) -> torch.Tensor:
        """dsa_index_topk_static: the same selection, with the scores kept in
        the library's fixed device array (no allocation in the call)."""
        d = self.device
        if selection is None:
            selection = torch.empty(plan.num_rows, self.shape.topk, dtype=torch.int32, device=d)
        _check(load().dsa_index_topk_static(self.handle, plan.handle, _ptr(q, d, (torch.bfloat16,), "q"),
                                            _ptr(w, d, (torch.float32,), "w"),
                                            _ptr(index_cache, d, (torch.bfloat16, torch.uint8), "index_cache"),
                                            _ptr(selection, d, (torch.int32,), "selection"), _stream(stream)),
               "dsa_index_topk_static", self.handle)
        return selection

    # ------------------------------------------------------ block-sparse MSA
    def msa_select_blocks(self, plan: Plan, msa, scores, block_sel=None, stream=None) -> torch.Tensor:
        """dsa_msa_select_blocks: token scores -> (T, topk_blocks) int32 block ids."""
        d = self.device
        if block_sel is None:
            block_sel = torch.empty(plan.num_rows, int(msa.topk_blocks), dtype=torch.int32, device=d)
        ms = _msa_shape(msa)
        _check(load().dsa_msa_select_blocks(self.handle, plan.handle, ctypes.byref(ms),
                                            _ptr(scores, d, (torch.float32,), "scores"),
                                            _ptr(block_sel, d, (torch.int32,), "block_sel"), _stream(stream)),
               "dsa_msa_select_blocks", self.handle)
        return block_sel

    def msa_index_select(self, plan: Plan, msa, q, w, index_cache, block_sel=None, stream=None) -> torch.Tensor:
        """dsa_msa_index_select: index scores (context scratch) + block selection."""
        d = self.device
        if block_sel is None:
            block_sel = torch.empty(plan.num_rows, int(msa.topk_blocks), dtype=torch.int32, device=d)
        ms = _msa_shape(msa)
        _check(load().dsa_msa_index_select(self.handle, plan.handle, ctypes.byref(ms), _ptr(q, d, (torch.bfloat16,), "q"),
                                           _ptr(w, d, (torch.float32,), "w"),
                                           _ptr(index_cache, d, (torch.bfloat16, torch.uint8), "index_cache"),
                                           _ptr(block_sel, d, (torch.int32,), "block_sel"), _stream(stream)),
               "dsa_msa_index_select", self.handle)
        return block_sel

    def msa_attend(self, plan: Plan, msa, block_sel, q, kv_cache, sm_scale: float, out=None, stream=None):
        """dsa_msa_attend: GQA attention over the kept blocks -> (T, q_heads, head_dim) bf16."""
        d = self.device
        if out is None:
            out = torch.empty(plan.num_rows, int(msa.q_heads), int(msa.head_dim), dtype=torch.bfloat16, device=d)
        ms = _msa_shape(msa)
        _check(load().dsa_msa_attend(self.handle, plan.handle, ctypes.byref(ms),
                                     _ptr(block_sel, d, (torch.int32,), "block_sel"),
                                     _ptr(q, d, (torch.bfloat16,), "q"),
                                     _ptr(kv_cache, d, (torch.bfloat16,), "kv_cache"), ctypes.c_float(sm_scale),
                                     _ptr(out, d, (torch.bfloat16,), "out"), _stream(stream)),
               "dsa_msa_attend", self.handle)
        return out

    def msa_attend_on_tensor_cores(self, plan: Plan, msa) -> bool:
        ms = _msa_shape(msa)
        return bool(load().dsa_msa_attend_on_tensor_cores(self.handle, plan.handle, ctypes.byref(ms)))

    def quantize_q(self, plan: Plan, q_bf16, codes=None, scales=None, stream=None):
        """dsa_quantize_q: the indexer query (T, 64, 128) bf16 -> (codes uint8 of the
        same shape, scales (T, 64) fp32), one scale per (row, head)."""
        d = self.device
        if codes is None:
            codes = torch.empty(q_bf16.shape, dtype=torch.uint8, device=d)
        if scales is None:
            scales = torch.empty(q_bf16.shape[:-1], dtype=torch.float32, device=d)
        _check(load().dsa_quantize_q(self.handle, plan.handle, _ptr(q_bf16, d, (torch.bfloat16,), "q"),
                                     _ptr(codes, d, (torch.uint8,), "q_codes"),
                                     _ptr(scales, d, (torch.float32,), "q_scale"), _stream(stream)),
               "dsa_quantize_q", self.handle)
        return codes, scales

    def index_scores_fp8q(self, plan: Plan, q_codes, q_scale, w, index_cache, scores=None, stream=None):
        """dsa_index_scores_fp8q: scores with an e4m3 query (fp8 index cache)."""
        d = self.device
        if scores is None:
            scores = torch.empty(max(1, plan.num_scores), dtype=torch.float32, device=d)
        _check(load().dsa_index_scores_fp8q(self.handle, plan.handle, _ptr(q_codes, d, (torch.uint8,), "q_codes"),
                                            _ptr(q_scale, d, (torch.float32,), "q_scale"),
                                            _ptr(w, d, (torch.float32,), "w"),
                                            _ptr(index_cache, d, (torch.uint8,), "index_cache"),
                                            _ptr(scores, d, (torch.float32,), "scores"), _stream(stream)),
               "dsa_index_scores_fp8q", self.handle)
        return scores

    def index_topk_fp8q(self, plan: Plan, q_codes, q_scale, w, index_cache, selection=None, stream=None):
        """dsa_index_topk_fp8q: score with an e4m3 query, then the causal top-k."""
        d = self.device
        if selection is None:
            selection = torch.empty(plan.num_rows, self.shape.topk, dtype=torch.int32, device=d)
        _check(load().dsa_index_topk_fp8q(self.handle, plan.handle, _ptr(q_codes, d, (torch.uint8,), "q_codes"),
                                          _ptr(q_scale, d, (torch.float32,), "q_scale"),
                                          _ptr(w, d, (torch.float32,), "w"),
                                          _ptr(index_cache, d, (torch.uint8,), "index_cache"),
                                          _ptr(selection, d, (torch.int32,), "selection"), _stream(stream)),
               "dsa_index_topk_fp8q", self.handle)
        return selection

    def index_scores(self, plan: Plan, q, w, index_cache, scores=None, stream=None) -> torch.Tensor:
        d = self.device
        if scores is None:
            scores = torch.empty(max(1, plan.num_scores), dtype=torch.float32, device=d)
        _check(load().dsa_index_scores(self.handle, plan.handle, _ptr(q, d, (torch.bfloat16,), "q"),
                                       _ptr(w, d, (torch.float32,), "w"),
                                       _ptr(index_cache, d, (torch.bfloat16, torch.uint8), "index_cache"),
                                       _ptr(scores, d, (torch.float32,), "scores"), _stream(stream)),
               "dsa_index_scores", self.handle)
        return scores

    def topk_from_scores(self, plan: Plan, scores, selection=None, stream=None) -> torch.Tensor:
        d = self.device
        if selection is None:
            selection = torch.empty(plan.num_rows, self.shape.topk, dtype=torch.int32, device=d)
        _check(load().dsa_topk_from_scores(self.handle, plan.handle, _ptr(scores, d, (torch.float32,), "scores"),
                                           _ptr(selection, d, (torch.int32,), "selection"), _stream(stream)),
               "dsa_topk_from_scores", self.handle)
        return selection

    def attend(self, plan: Plan, selection, q_nope, q_pe, latent_cache, sink=None, sm_scale=None, out=None,
               stream=None) -> torch.Tensor:
        d = self.device
        sh = self.shape
        if sm_scale is None:
            sm_scale = sh.sm_scale
        if out is None:
            out = torch.empty(plan.num_rows, sh.heads, sh.kv_lora_rank, dtype=torch.bfloat16, device=d)
        _check(load().dsa_attend(self.handle, plan.handle, _ptr(selection, d, (torch.int32,), "selection"),
                                 _ptr(q_nope, d, (torch.bfloat16,), "q_nope"), _ptr(q_pe, d, (torch.bfloat16,), "q_pe"),
                                 _ptr(latent_cache, d, (torch.bfloat16, torch.uint8), "latent_cache"),
                                 _ptr(sink, d, (torch.float32,), "sink"), float(sm_scale),
                                 _ptr(out, d, (torch.bfloat16,), "out"), _stream(stream)), "dsa_attend", self.handle)
        return out

    def attend_shared(self, plan: Plan, q_nope, q_pe, latent_cache, sink=None, sm_scale=None, out=None,
                      stream=None) -> torch.Tensor:
        """A SHARED layer: attend over the selection the last FULL layer wrote for this plan."""
        d = self.device
        sh = self.shape
        if sm_scale is None:
            sm_scale = sh.sm_scale
        if out is None:
            out = torch.empty(plan.num_rows, sh.heads, sh.kv_lora_rank, dtype=torch.bfloat16, device=d)
        _check(load().dsa_attend_shared(self.handle, plan.handle, _ptr(q_nope, d, (torch.bfloat16,), "q_nope"),
                                        _ptr(q_pe, d, (torch.bfloat16,), "q_pe"),
                                        _ptr(latent_cache, d, (torch.bfloat16, torch.uint8), "latent_cache"),
                                        _ptr(sink, d, (torch.float32,), "sink"), float(sm_scale),
                                        _ptr(out, d, (torch.bfloat16,), "out"), _stream(stream)),
               "dsa_attend_shared", self.handle)
        return out

    def get_error(self, stream=None):
        _check(load().dsa_get_error(self.handle, _stream(stream)), "dsa_get_error", self.handle)

    def last_launch_count(self) -> int:
        return int(load().dsa_last_launch_count(self.handle))
