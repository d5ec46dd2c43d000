"""Seeded synthetic inputs for DeepSeek Sparse Attention over a paged MLA cache.

This module only *makes inputs*: request spans, page tables and the tensors a
step reads (index keys, indexer queries and head weights, MLA latents, MLA
queries, attention sinks).  It holds none of the method's arithmetic (no
scoring, no selection, no attention); the CUDA library and the CPU oracle both
consume what it produces, and neither is imported here.

Every value is a pure function of (seed, stream, logical element id), computed
with a counter-based integer hash ("lowbias32", C. Wellons' 32-bit integer
hash: xor-shift 16, multiply 0x7feb352d, xor-shift 15, multiply 0x846ca68b,
xor-shift 16) in int64 torch arithmetic that never overflows.  The same code
therefore yields bit-identical tensors on the CPU and on a GPU, and any slice of
a large workload (one request's keys, a handful of latent rows) can be
regenerated on the host without touching the device copy.

Logical ids are position based: a request's token at position ``pos`` has id
``token_base + pos``, so a row's inputs do not depend on how the batch is
packed or which physical pages hold it.

Distributions: "N(0, s)" is an Irwin-Hall(4) approximation of a normal with
standard deviation ``s`` (four 16-bit uniforms; exact integer sum, one fp64
scale, fp32 then bf16 round-to-nearest-even), "U(a, b)" is a 24-bit uniform.

Formats (per token, per layer):
  * bf16 index key            : index_dim bf16                       (256 B at dim 128)
  * fp8 index key  (132 B)    : 128 e4m3 + one fp32 scale, stored page-blocked:
                                each page is [page_size x 128 codes][page_size x fp32]
  * bf16 latent   (1,152 B)   : [kv_lora_rank | rope] bf16
  * fp8 latent    (656 B)     : [512 e4m3 | 4 fp32 scales (one per 128) | 64 bf16 rope]
fp8 packing uses, per group of values, scale = amax / 448 in fp32 (1 when
amax == 0) and round-to-nearest-even e4m3 codes of x / scale, saturating at
+-448 (torch's float8_e4m3fn cast) -- the rule of the library's quantise-on-
store.  ``Distributions.fp8_scale = "pow2"`` packs with power-of-two scales
instead, 2^(floor(log2 amax) - 7), under which code x scale is exact in bf16.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import List, Optional

import numpy as np
import torch

LATENT_BF16 = 0
LATENT_FP8_656 = 1
INDEX_BF16 = 0
INDEX_FP8_132 = 1

_M32 = 0xFFFFFFFF

# stream ids: one independent random stream per kind of tensor
S_INDEX_KEY, S_LATENT, S_Q, S_W, S_QNOPE, S_QPE, S_SINK, S_CTX, S_PAGES, S_KV, S_MSA_Q = range(1, 12)


# ----------------------------------------------------------------------------
# counter-based integer hash (works on python ints and on int64 tensors)
# ----------------------------------------------------------------------------
def _mul32(x, c: int):
    """(x * c) mod 2**32 for x in [0, 2**32) without int64 overflow."""
    lo, hi = c & 0xFFFF, c >> 16
    return (x * lo + ((x * hi) & 0xFFFF) * 65536) & _M32


def hash32(x):
    """lowbias32 integer hash of a 32-bit value (python int or int64 tensor)."""
    x = x ^ (x >> 16)
    x = _mul32(x, 0x7FEB352D)
    x = x ^ (x >> 15)
    x = _mul32(x, 0x846CA68B)
    x = x ^ (x >> 16)
    return x


def _stream_key(seed: int, stream: int, draw: int) -> int:
    k = hash32((seed * 0x9E3779B1) & _M32)
    k = hash32(k ^ ((stream * 0x85EBCA77) & _M32))
    return hash32(k ^ ((draw * 0xC2B2AE3D) & _M32))


def _bits(ids: torch.Tensor, seed: int, stream: int, draw: int) -> torch.Tensor:
    """32 random bits per logical id (ids: int64 tensor, values < 2**52)."""
    key = _stream_key(seed, stream, draw)
    h = hash32((ids & _M32) ^ key)
    if ids.numel() and int(ids.max()) > _M32:
        # ids at or above 2**32 fold their high word in with a second round;
        # the choice is per element, so a value never depends on its neighbours
        key_hi = hash32(key ^ 0x5BD1E995)
        hi = ids >> 32
        h = torch.where(hi != 0, hash32(h ^ _mul32((hi ^ key_hi) & _M32, 0x9E3779B1)), h)
    return h


def _normal(ids, seed, stream, std):
    """Irwin-Hall(4) normal with the given std, returned as fp32."""
    a = _bits(ids, seed, stream, 0)
    b = _bits(ids, seed, stream, 1)
    s = (a & 0xFFFF) + (a >> 16) + (b & 0xFFFF) + (b >> 16)       # exact, < 2**18
    x = (s - (1 << 17)).to(torch.float64) * (math.sqrt(3.0) / 65536.0)
    if std != 1.0:
        x = x * float(std)
    return x.to(torch.float32)


def _uniform(ids, seed, stream, lo, hi):
    u = (_bits(ids, seed, stream, 0) >> 8).to(torch.float32) * (1.0 / 16777216.0)
    if lo != 0.0 or hi != 1.0:
        u = u * float(hi - lo) + float(lo)
    return u


def _small_int(ids, seed, stream, lo, hi):
    """Integers uniformly in [lo, hi] as fp32 (exact)."""
    h = _bits(ids, seed, stream, 0)
    return (h % (hi - lo + 1) + lo).to(torch.float32)


def _to_bf16(x: torch.Tensor) -> torch.Tensor:
    return x.to(torch.float32).to(torch.bfloat16)


def _to_e4m3_bytes(x: torch.Tensor) -> torch.Tensor:
    return x.clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)


# ----------------------------------------------------------------------------
# problem description
# ----------------------------------------------------------------------------
@dataclass
class DSAShape:
    index_heads: int
    index_dim: int
    topk: int
    heads: int
    kv_lora_rank: int
    rope_dim: int
    page_size: int
    sm_scale: float
    latent_fmt: int = LATENT_BF16
    index_fmt: int = INDEX_BF16
    has_sink: bool = False

    @property
    def latent_dim(self) -> int:
        return self.kv_lora_rank + self.rope_dim

    @property
    def latent_row_bytes(self) -> int:
        if self.latent_fmt == LATENT_FP8_656:
            return self.kv_lora_rank + 4 * (self.kv_lora_rank // 128) + 2 * self.rope_dim
        return 2 * self.latent_dim

    @property
    def index_row_bytes(self) -> int:
        if self.index_fmt == INDEX_FP8_132:
            return self.index_dim + 4
        return 2 * self.index_dim


@dataclass
class MSAShape:
    """Block-sparse MSA (LLMServingSim, "Sparse attention (DSA and block-sparse
    MSA)", MiniMax-M3 column): the top ``topk_blocks`` blocks of
    ``block_size`` tokens per row, over plain GQA (``q_heads`` query heads
    sharing ``kv_heads`` key/value heads of ``head_dim``), with one bf16 index
    vector of ``index_dim`` per token.  The pages fix 16 blocks of 128 tokens,
    a bf16 index vector, and 2 x kv_heads x head_dim x 2 = 2,048 bytes of K and
    V per token (kv_heads x head_dim = 512); the 4 x 128 split, 64 query heads
    and the 64-head indexer query are readings."""
    index_heads: int = 64
    index_dim: int = 128
    page_size: int = 64
    block_size: int = 128
    topk_blocks: int = 16
    q_heads: int = 64
    kv_heads: int = 4
    head_dim: int = 128
    sm_scale: float = 1.0 / math.sqrt(128.0)

    @property
    def kv_row_elems(self) -> int:
        return 2 * self.kv_heads * self.head_dim

    @property
    def kv_row_bytes(self) -> int:
        return 2 * self.kv_row_elems

    def index_shape(self) -> "DSAShape":
        """The token-level indexer as a DSAShape (index fields and page size;
        the MLA fields stand in and are not read by the MSA calls)."""
        return DSAShape(index_heads=self.index_heads, index_dim=self.index_dim,
                        topk=self.block_size * self.topk_blocks, heads=self.q_heads, kv_lora_rank=self.head_dim,
                        rope_dim=0, page_size=self.page_size, sm_scale=self.sm_scale)


@dataclass
class Span:
    """One request's rows of a step: q_len rows from row q_start, the first at
    position ctx_start; ``pages`` are its cache pages and ``page_start`` the slot
    of its token 0 within them.  ``token_base`` is the logical id of its token 0."""
    request_id: int
    q_start: int
    q_len: int
    ctx_start: int
    pages: np.ndarray
    page_start: int = 0
    token_base: int = 0

    @property
    def ctx_end(self) -> int:
        return self.ctx_start + self.q_len


@dataclass
class Distributions:
    q_std: float = 1.0            # indexer queries
    k_std: float = 1.0            # index keys
    w: tuple = ("uniform", 0.0, 1.0)   # ("uniform", lo, hi) or ("normal", std)
    qn_std: float = 1.0           # MLA q_nope / q_pe
    lat_std: float = 0.5          # MLA latents
    sink_std: float = 1.0
    integer: bool = False         # q, k in {-3..3}, w in {0..3}: exact fp32 scores
    fp8_scale: str = "amax"       # fp8 rows: "amax" (scale = amax/448) or "pow2" (power-of-two scales)


@dataclass
class Workload:
    name: str
    shape: DSAShape
    spans: List[Span]
    num_pages: int
    seed: int
    dist: Distributions = field(default_factory=Distributions)
    msa: Optional[MSAShape] = None   # set for block-sparse MSA workloads

    @property
    def num_rows(self) -> int:
        return sum(s.q_len for s in self.spans)

    # ------------------------------------------------------------------ rows
    def row_table(self):
        """Per row: (span index, position, token id) as int64 numpy arrays."""
        T = self.num_rows
        span_of = np.empty(T, np.int64)
        pos = np.empty(T, np.int64)
        tok = np.empty(T, np.int64)
        for i, s in enumerate(self.spans):
            sl = slice(s.q_start, s.q_start + s.q_len)
            span_of[sl] = i
            pos[sl] = np.arange(s.ctx_start, s.ctx_end)
            tok[sl] = s.token_base + pos[sl]
        return span_of, pos, tok

    def slot_token_map(self) -> np.ndarray:
        """For every physical cache row (page * page_size + slot): the logical
        token id stored there, or -1.  Covers positions [0, ctx_end) of every
        request."""
        P = self.shape.page_size
        m = np.full(self.num_pages * P, -1, np.int64)
        for s in self.spans:
            n = s.ctx_end
            slots = s.page_start + np.arange(n, dtype=np.int64)
            rows = s.pages[slots // P].astype(np.int64) * P + slots % P
            m[rows] = s.token_base + np.arange(n, dtype=np.int64)
        return m

    def step_slot_mask(self) -> np.ndarray:
        """Boolean per physical row: True where the row holds one of this step's
        new tokens (positions ctx_start .. ctx_end-1), which the step stores."""
        P = self.shape.page_size
        m = np.zeros(self.num_pages * P, bool)
        for s in self.spans:
            pos = np.arange(s.ctx_start, s.ctx_end, dtype=np.int64)
            slots = s.page_start + pos
            rows = s.pages[slots // P].astype(np.int64) * P + slots % P
            m[rows] = True
        return m

    def row_workload(self, span_index: int, row_in_span: int) -> "Workload":
        """One row of one span as its own single-row step (pages renumbered,
        logical ids kept): the row sees the same keys and latents as in the
        full workload."""
        s = self.spans[span_index]
        sp = replace(s, q_start=0, q_len=1, ctx_start=s.ctx_start + row_in_span,
                     pages=np.arange(len(s.pages), dtype=np.int32))
        return Workload(self.name + "/row", self.shape, [sp], len(s.pages), self.seed, self.dist, self.msa)

    def sub_workload(self, span_indices) -> "Workload":
        """A workload holding only the given spans, re-packed from row 0 with
        pages renumbered 0..n-1.  Logical ids are kept, so every value is the same
        as in the full workload."""
        spans, q0, pbase = [], 0, 0
        for i in span_indices:
            s = self.spans[i]
            npg = len(s.pages)
            spans.append(replace(s, q_start=q0, pages=np.arange(pbase, pbase + npg, dtype=np.int32)))
            q0 += s.q_len
            pbase += npg
        return Workload(self.name + "/sub", self.shape, spans, pbase, self.seed, self.dist, self.msa)


# ----------------------------------------------------------------------------
# tensors
# ----------------------------------------------------------------------------
def _chunks(n: int, step: int):
    for a in range(0, n, step):
        yield a, min(n, a + step)


def _index_key_values(wl: Workload, tok: torch.Tensor) -> torch.Tensor:
    """fp32 logical index-key values, shape (len(tok), index_dim)."""
    D = wl.shape.index_dim
    ids = tok.view(-1, 1) * D + torch.arange(D, device=tok.device).view(1, -1)
    if wl.dist.integer:
        return _small_int(ids, wl.seed, S_INDEX_KEY, -3, 3)
    return _normal(ids, wl.seed, S_INDEX_KEY, wl.dist.k_std)


def _latent_values(wl: Workload, tok: torch.Tensor) -> torch.Tensor:
    Dl = wl.shape.latent_dim
    ids = tok.view(-1, 1) * Dl + torch.arange(Dl, device=tok.device).view(1, -1)
    return _normal(ids, wl.seed, S_LATENT, wl.dist.lat_std)


def _fp8_groups(x: torch.Tensor, group: int, scale_rule: str = "amax"):
    """Per-group e4m3 codes and fp32 scales.

    "amax" (the default): scale = amax / 448 in fp32 (1 if amax == 0), codes
    = e4m3 of the fp32 quotient x / scale, saturating at +-448 -- the same rule
    as the library's quantise-on-store.  IEEE fp32 division and torch's e4m3
    cast give the same bytes on the CPU and the GPU.
    "pow2": scale = 2^(floor(log2 amax) - 7), so the largest |x| / scale lies in
    [128, 256) and code x scale is exact in bf16 -- an extra exactness case."""
    n, d = x.shape
    g = x.to(torch.float32).view(n, d // group, group)
    amax = g.abs().amax(dim=2)
    if scale_rule == "pow2":
        _, e = torch.frexp(amax)                      # amax = m * 2^e, m in [0.5, 1)
        scale = torch.ldexp(torch.ones_like(amax), (e - 8).to(torch.int32))
    elif scale_rule == "amax":
        scale = amax / torch.tensor(448.0, dtype=torch.float32, device=amax.device)
    else:
        raise ValueError("fp8 scale rule %r" % (scale_rule,))
    scale = torch.where(amax > 0, scale, torch.ones_like(amax))
    codes = _to_e4m3_bytes(g / scale.unsqueeze(2)).view(n, d)
    return codes, scale.to(torch.float32)


def index_rows_bytes(wl: Workload, tok: torch.Tensor) -> torch.Tensor:
    """Index-key rows in cache format: (n, index_dim) bf16, or (n, 132) uint8
    = [128 e4m3 | fp32 scale] for the fp8 format."""
    x = _index_key_values(wl, tok)
    if wl.shape.index_fmt == INDEX_BF16:
        return _to_bf16(x)
    codes, scale = _fp8_groups(x, wl.shape.index_dim, wl.dist.fp8_scale)
    return torch.cat([codes, scale.contiguous().view(torch.uint8).view(-1, 4)], dim=1)


def latent_rows_bytes(wl: Workload, tok: torch.Tensor) -> torch.Tensor:
    """Latent rows in cache format: (n, L+R) bf16, or (n, 656) uint8."""
    x = _latent_values(wl, tok)
    sh = wl.shape
    if sh.latent_fmt == LATENT_BF16:
        return _to_bf16(x)
    L = sh.kv_lora_rank
    codes, scale = _fp8_groups(x[:, :L].contiguous(), 128, wl.dist.fp8_scale)
    rope = _to_bf16(x[:, L:].contiguous()).view(torch.uint8).view(-1, 2 * sh.rope_dim)
    return torch.cat([codes, scale.contiguous().view(torch.uint8).view(-1, 4 * (L // 128)), rope], dim=1)


def make_index_cache(wl: Workload, device="cpu", include_step: bool = False, chunk_rows: int = 1 << 20) -> torch.Tensor:
    """The paged index-key cache.  bf16: [num_pages, page_size, index_dim];
    fp8: [num_pages, page_size * 132] uint8, page-blocked.  History positions
    (< ctx_start) are filled; this step's positions only if ``include_step``
    (the step stores them itself); every other slot is zero."""
    sh = wl.shape
    P = sh.page_size
    m = wl.slot_token_map()
    if not include_step:
        m[wl.step_slot_mask()] = -1
    nrows = wl.num_pages * P
    if sh.index_fmt == INDEX_BF16:
        out = torch.zeros(nrows, sh.index_dim, dtype=torch.bfloat16, device=device)
    else:
        codes_all = torch.zeros(wl.num_pages, P, sh.index_dim, dtype=torch.uint8, device=device)
        scales_all = torch.zeros(wl.num_pages, P, 4, dtype=torch.uint8, device=device)
    for a, b in _chunks(nrows, chunk_rows):
        sel = np.nonzero(m[a:b] >= 0)[0]
        if len(sel) == 0:
            continue
        rows = torch.from_numpy(sel + a).to(device)
        tok = torch.from_numpy(m[a:b][sel]).to(device)
        v = index_rows_bytes(wl, tok)
        if sh.index_fmt == INDEX_BF16:
            out[rows] = v
        else:
            pg, sl = rows // P, rows % P
            codes_all[pg, sl] = v[:, : sh.index_dim]
            scales_all[pg, sl] = v[:, sh.index_dim:]
    if sh.index_fmt == INDEX_BF16:
        return out.view(wl.num_pages, P, sh.index_dim)
    return torch.cat([codes_all.view(wl.num_pages, -1), scales_all.view(wl.num_pages, -1)], dim=1).contiguous()


def make_latent_cache(wl: Workload, device="cpu", chunk_rows: int = 1 << 19, tokens=None) -> torch.Tensor:
    """The paged MLA latent cache with every position < ctx_end written (the
    caller writes a step's latents before attention).  bf16:
    [num_pages, page_size, L+R]; fp8: [num_pages, page_size, 656] uint8.
    ``tokens``: optional collection of logical token ids; only those rows are
    filled (the rest stay zero), to regenerate a few rows of a large cache."""
    sh = wl.shape
    P = sh.page_size
    m = wl.slot_token_map()
    if tokens is not None:
        keep = np.isin(m, np.asarray(sorted(tokens), dtype=np.int64))
        m[~keep] = -1
    nrows = wl.num_pages * P
    if sh.latent_fmt == LATENT_BF16:
        out = torch.zeros(nrows, sh.latent_dim, dtype=torch.bfloat16, device=device)
    else:
        out = torch.zeros(nrows, sh.latent_row_bytes, dtype=torch.uint8, device=device)
    for a, b in _chunks(nrows, chunk_rows):
        sel = np.nonzero(m[a:b] >= 0)[0]
        if len(sel) == 0:
            continue
        rows = torch.from_numpy(sel + a).to(device)
        tok = torch.from_numpy(m[a:b][sel]).to(device)
        out[rows] = latent_rows_bytes(wl, tok)
    return out.view(wl.num_pages, P, -1)


@dataclass
class StepInputs:
    q: torch.Tensor         # (T, Hi, Di) bf16 indexer queries
    w: torch.Tensor         # (T, Hi) fp32 head weights
    keys: torch.Tensor      # (T, Di) bf16 or (T, 132) uint8: this step's index keys
    q_nope: torch.Tensor    # (T, H, L) bf16
    q_pe: torch.Tensor      # (T, H, R) bf16
    sink: Optional[torch.Tensor]  # (H,) fp32 or None


def make_step_inputs(wl: Workload, device="cpu") -> StepInputs:
    sh, d = wl.shape, wl.dist
    _, _, tok_np = wl.row_table()
    tok = torch.from_numpy(tok_np).to(device)
    T = len(tok_np)
    Hi, Di, H, L, R = sh.index_heads, sh.index_dim, sh.heads, sh.kv_lora_rank, sh.rope_dim

    def ids(width):
        return tok.view(-1, 1) * width + torch.arange(width, device=device).view(1, -1)

    if d.integer:
        q = _small_int(ids(Hi * Di), wl.seed, S_Q, -3, 3)
        w = _small_int(ids(Hi), wl.seed, S_W, 0, 3)
    else:
        q = _normal(ids(Hi * Di), wl.seed, S_Q, d.q_std)
        if d.w[0] == "uniform":
            w = _uniform(ids(Hi), wl.seed, S_W, d.w[1], d.w[2])
        else:
            w = _normal(ids(Hi), wl.seed, S_W, d.w[1])
    q_nope = _normal(ids(H * L), wl.seed, S_QNOPE, d.qn_std)
    q_pe = _normal(ids(H * R), wl.seed, S_QPE, d.qn_std)
    sink = None
    if sh.has_sink:
        sink = _normal(torch.arange(H, device=device), wl.seed, S_SINK, d.sink_std)
    return StepInputs(
        q=_to_bf16(q).view(T, Hi, Di).contiguous(),
        w=w.view(T, Hi).contiguous(),
        keys=index_rows_bytes(wl, tok).contiguous(),
        q_nope=_to_bf16(q_nope).view(T, H, L).contiguous(),
        q_pe=_to_bf16(q_pe).view(T, H, R).contiguous(),
        sink=sink,
    )


def kv_rows(wl: Workload, tok: torch.Tensor) -> torch.Tensor:
    """GQA key/value rows of the given tokens: (n, 2 * kv_heads * head_dim)
    bf16, [K of kv heads 0..kv_heads-1 | V of the same heads], ~N(0, lat_std)."""
    width = wl.msa.kv_row_elems
    ids = tok.view(-1, 1) * width + torch.arange(width, device=tok.device).view(1, -1)
    return _to_bf16(_normal(ids, wl.seed, S_KV, wl.dist.lat_std))


def make_kv_cache(wl: Workload, device="cpu", chunk_rows: int = 1 << 18, tokens=None) -> torch.Tensor:
    """The paged GQA cache of an MSA workload, [num_pages, page_size,
    2 * kv_heads * head_dim] bf16, with every position < ctx_end written.
    ``tokens``: optional logical ids; only those rows are filled."""
    P = wl.shape.page_size
    m = wl.slot_token_map()
    if tokens is not None:
        keep = np.isin(m, np.asarray(sorted(tokens), dtype=np.int64))
        m[~keep] = -1
    nrows = wl.num_pages * P
    out = torch.zeros(nrows, wl.msa.kv_row_elems, dtype=torch.bfloat16, device=device)
    for a, b in _chunks(nrows, chunk_rows):
        sel = np.nonzero(m[a:b] >= 0)[0]
        if len(sel) == 0:
            continue
        rows = torch.from_numpy(sel + a).to(device)
        tok = torch.from_numpy(m[a:b][sel]).to(device)
        out[rows] = kv_rows(wl, tok)
    return out.view(wl.num_pages, P, -1)


def make_msa_q(wl: Workload, device="cpu") -> torch.Tensor:
    """GQA queries of an MSA workload, (T, q_heads, head_dim) bf16 ~N(0, qn_std)."""
    ms = wl.msa
    _, _, tok_np = wl.row_table()
    tok = torch.from_numpy(tok_np).to(device)
    width = ms.q_heads * ms.head_dim
    ids = tok.view(-1, 1) * width + torch.arange(width, device=device).view(1, -1)
    return _to_bf16(_normal(ids, wl.seed, S_MSA_Q, wl.dist.qn_std)).view(len(tok_np), ms.q_heads, ms.head_dim)


# ----------------------------------------------------------------------------
# workloads
# ----------------------------------------------------------------------------
def _uniform_ints(seed: int, stream: int, n: int, lo: int, hi: int) -> np.ndarray:
    h = _bits(torch.arange(n, dtype=torch.int64), seed, stream, 0)
    return (h % (hi - lo + 1) + lo).numpy()


def _page_permutation(seed: int, n: int) -> np.ndarray:
    h = _bits(torch.arange(n, dtype=torch.int64), seed, S_PAGES, 0)
    return np.argsort(h.numpy(), kind="stable").astype(np.int32)


def build_workload(name: str, shape: DSAShape, requests, seed: int,
                   dist: Optional[Distributions] = None, page_start=0,
                   spare_pages: int = 0, permute_pages: bool = True) -> Workload:
    """requests: list of (ctx_start, q_len); page_start: one value for every
    request or one per request.  Each request gets
    ceil((page_start + ctx_start + q_len) / page_size) pages from a seeded
    permutation of one pool; rows are packed in request order."""
    P = shape.page_size
    starts = [int(page_start)] * len(requests) if np.isscalar(page_start) else [int(x) for x in page_start]
    assert len(starts) == len(requests)
    need = [-(-(ps + c + q) // P) for (c, q), ps in zip(requests, starts)]
    total = sum(need) + spare_pages
    perm = _page_permutation(seed, total) if permute_pages else np.arange(total, dtype=np.int32)
    spans, q0, p0, tb = [], 0, 0, 0
    for i, ((c, q), n, ps) in enumerate(zip(requests, need, starts)):
        spans.append(Span(request_id=i, q_start=q0, q_len=q, ctx_start=c,
                          pages=perm[p0:p0 + n].copy(), page_start=ps, token_base=tb))
        q0 += q
        p0 += n
        tb += c + q + 1
    return Workload(name, shape, spans, total, seed, dist or Distributions())


DEEPSEEK = dict(index_heads=64, index_dim=128, topk=2048, heads=128, kv_lora_rank=512,
                rope_dim=64, page_size=64, sm_scale=1.0 / math.sqrt(192.0))

CONFIG_NAMES = ["tiny_prefill", "decode", "chunked_prefill", "long_decode", "mixed_fp8"]


def config(i: int, seed: Optional[int] = None, page_start=0) -> Workload:
    """The five evaluation workloads (seed defaults to 1000 + i).

    0 tiny_prefill    2 requests, contexts 256 / 384, every row queried; indexer 4x32,
                      topk 64; MLA H=8, 64+16, page 16, sm_scale 1/sqrt(80).
    1 decode          32 requests x 1 row, contexts ~U[4096, 16384]; DeepSeek-V3.2 shapes.
    2 chunked_prefill 1 request, 8192 cached + 8192 new rows (positions 8192..16383).
    3 long_decode     128 requests x 1 row, contexts ~U[65536, 131072].
    4 mixed_fp8       16 decode rows (contexts ~U[8192, 32768]) + two 2048-row chunks
                      ending at 4096 and 12288; fp8 656-B latents, 132-B index rows, sinks.

    page_start (0 in the evaluation workloads) moves every request's token 0 to
    that slot of its first page.
    """
    seed = 1000 + i if seed is None else seed
    name = CONFIG_NAMES[i]
    if i == 0:
        sh = DSAShape(index_heads=4, index_dim=32, topk=64, heads=8, kv_lora_rank=64, rope_dim=16,
                      page_size=16, sm_scale=1.0 / math.sqrt(80.0))
        return build_workload(name, sh, [(0, 256), (0, 384)], seed,
                              Distributions(w=("uniform", 0.0, 1.0)), page_start=page_start)
    if i == 1:
        ctx = _uniform_ints(seed, S_CTX, 32, 4096, 16384)
        return build_workload(name, DSAShape(**DEEPSEEK), [(int(c) - 1, 1) for c in ctx], seed,
                              Distributions(w=("uniform", 0.0, 1.0 / 8)), page_start=page_start)
    if i == 2:
        return build_workload(name, DSAShape(**DEEPSEEK), [(8192, 8192)], seed,
                              Distributions(w=("normal", 1.0)), page_start=page_start)
    if i == 3:
        ctx = _uniform_ints(seed, S_CTX, 128, 65536, 131072)
        return build_workload(name, DSAShape(**DEEPSEEK), [(int(c) - 1, 1) for c in ctx], seed,
                              Distributions(w=("uniform", 0.0, 1.0 / 8)), page_start=page_start)
    if i == 4:
        sh = DSAShape(**DEEPSEEK, latent_fmt=LATENT_FP8_656, index_fmt=INDEX_FP8_132, has_sink=True)
        ctx = _uniform_ints(seed, S_CTX, 16, 8192, 32768)
        reqs = [(int(c) - 1, 1) for c in ctx] + [(2048, 2048), (10240, 2048)]
        return build_workload(name, sh, reqs, seed, Distributions(w=("uniform", 0.0, 1.0 / 8)), page_start=page_start)
    raise ValueError(i)


MSA_CONFIG_NAMES = ["msa_small", "msa_decode", "msa_prefill"]


def msa_config(name: str, seed: Optional[int] = None, page_start=0) -> Workload:
    """Block-sparse MSA workloads (the pages give no MSA workload; these mirror
    the DSA ones at the MiniMax-M3 selection shape, top 16 blocks of 128):

    msa_small    3 requests: decode rows at contexts 1500 and 700 and a 96-row
                 chunk at positions 1024..1119; top 4 blocks of 128, 8 query
                 heads over 2 kv heads (selection spans several blocks, the
                 oracle runs in seconds).
    msa_decode   128 requests x 1 row, contexts ~U[65536, 131072]; top 16
                 blocks of 128, 64 query heads over 4 kv heads of 128.
    msa_prefill  1 request, 8192 cached + 8192 new rows; shapes as msa_decode.
    Index keys and queries as the DSA workloads (indexer 64 x 128 bf16); K, V
    ~N(0, 0.5), GQA queries ~N(0, 1)."""
    i = MSA_CONFIG_NAMES.index(name)
    seed = 2000 + i if seed is None else seed
    if name == "msa_small":
        ms = MSAShape(topk_blocks=4, q_heads=8, kv_heads=2)
        reqs = [(1499, 1), (699, 1), (1024, 96)]
    elif name == "msa_decode":
        ms = MSAShape()
        ctx = _uniform_ints(seed, S_CTX, 128, 65536, 131072)
        reqs = [(int(c) - 1, 1) for c in ctx]
    else:
        ms = MSAShape()
        reqs = [(8192, 8192)]
    wl = build_workload(name, ms.index_shape(), reqs, seed, Distributions(w=("uniform", 0.0, 1.0 / 8)),
                        page_start=page_start)
    wl.msa = ms
    return wl
