"""Data-parallel sharding of a DSA step by request.

Every stage of the path (index-key store, indexer score, causal top-k, sparse
attention) reads only the request's own pages (mstar
"mstar.engine.resources.dsa.manager": each row scores its request's keys and
attends its request's latents), so requests can be spread over GPUs with each
request's pages local and no collective on the data path.  `shard_spans`
assigns whole requests to ranks, balancing the estimated bytes each rank
streams (visible index keys plus selected latent rows), and re-packs each
rank's spans from row 0 so they form a valid step on that rank.
"""
from __future__ import annotations

from dataclasses import replace
from typing import List, Sequence, Tuple


def request_cost(span, topk: int, index_row_bytes: int, latent_row_bytes: int) -> float:
    """Bytes the step streams for this request's rows: every visible index key
    once per row, and up to topk latent rows per row."""
    c0, n = int(span.ctx_start), int(span.q_len)
    keys = n * c0 + n * (n + 1) // 2                       # sum over rows of pos + 1
    sel = sum(min(topk, c0 + i + 1) for i in range(n))
    return float(keys) * index_row_bytes + float(sel) * latent_row_bytes


def assign_requests(costs: Sequence[float], world: int) -> List[List[int]]:
    """Longest-processing-time-first assignment of requests to `world` ranks;
    each rank's list keeps the requests' original order."""
    order = sorted(range(len(costs)), key=lambda i: (-costs[i], i))
    load = [0.0] * world
    owned: List[List[int]] = [[] for _ in range(world)]
    for i in order:
        r = min(range(world), key=lambda k: (load[k], k))
        owned[r].append(i)
        load[r] += costs[i]
    return [sorted(o) for o in owned]


def shard_spans(spans, world: int, topk: int, index_row_bytes: int, latent_row_bytes: int) -> List[Tuple[list, list]]:
    """For each rank: (original span indices, spans re-packed from row 0)."""
    costs = [request_cost(s, topk, index_row_bytes, latent_row_bytes) for s in spans]
    out = []
    for idx in assign_requests(costs, world):
        packed, q0 = [], 0
        for i in idx:
            packed.append(replace(spans[i], q_start=q0))
            q0 += int(spans[i].q_len)
        out.append((idx, packed))
    return out
