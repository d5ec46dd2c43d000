"""Small hand-built DSA problems for tests (explicit spans, pages and tensors).

Only builds inputs; computes nothing of the method.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np
import torch

from deepseek_sparse_attention_dsa_gb300.workloads import DSAShape, Span, INDEX_BF16, LATENT_BF16


@dataclass
class Case:
    shape: DSAShape
    spans: list
    num_pages: int


def tiny_shape(**kw):
    base = dict(index_heads=2, index_dim=3, topk=4, heads=2, kv_lora_rank=4, rope_dim=2, page_size=4,
                sm_scale=0.5, latent_fmt=LATENT_BF16, index_fmt=INDEX_BF16)
    base.update(kw)
    return DSAShape(**base)


def make_case(shape, requests, pages=None, page_start=0, num_pages=None):
    """requests: list of (ctx_start, q_len).  pages: optional list of page lists;
    by default each request takes the next pages of an identity pool."""
    P = shape.page_size
    spans, q0, p0 = [], 0, 0
    for i, (c, q) in enumerate(requests):
        need = -(-(page_start + c + q) // P)
        if pages is None:
            pg = np.arange(p0, p0 + need, dtype=np.int32)
        else:
            pg = np.asarray(pages[i], dtype=np.int32)
        spans.append(Span(request_id=i, q_start=q0, q_len=q, ctx_start=c, pages=pg, page_start=page_start))
        q0 += q
        p0 += need
    if num_pages is None:
        num_pages = max(int(s.pages.max()) + 1 for s in spans)
    return Case(shape, spans, num_pages)


def phys_rows(case, span_index, positions):
    """Physical cache rows of positions of one span (slot = page_start + pos)."""
    s = case.spans[span_index]
    P = case.shape.page_size
    slots = s.page_start + np.asarray(positions, dtype=np.int64)
    return s.pages[slots // P].astype(np.int64) * P + slots % P


def bf16(x):
    return torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
