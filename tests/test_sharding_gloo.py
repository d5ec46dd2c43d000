"""The N>1 path on CPU: requests sharded over world_size 2 (gloo), each rank
computing its shard independently, gives exactly the single-process result;
the step time reduction is a MAX over ranks."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from deepseek_sparse_attention_dsa_gb300 import sharding
from deepseek_sparse_attention_dsa_gb300 import workloads as W


def _workload():
    sh = W.DSAShape(index_heads=4, index_dim=32, topk=24, heads=2, kv_lora_rank=16, rope_dim=8, page_size=8,
                    sm_scale=0.25)
    return W.build_workload("shard", sh, [(30, 1), (0, 20), (55, 3), (12, 1), (70, 1)], seed=21)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    wl = _workload()
    sh = wl.shape
    shards = sharding.shard_spans(wl.spans, world, sh.topk, sh.index_row_bytes, sh.latent_row_bytes)
    idx, spans = shards[rank]
    mine = W.Workload(wl.name, sh, spans, wl.num_pages, wl.seed, wl.dist)
    res = oracle.run_all(mine, W.make_index_cache(mine), W.make_latent_cache(mine), W.make_step_inputs(mine))
    # per-request results keyed by request id
    local = {}
    for s in spans:
        sl = slice(s.q_start, s.q_start + s.q_len)
        local[s.request_id] = (res["selection"][sl].copy(), res["out"][sl].copy())
    gathered = [None] * world
    dist.all_gather_object(gathered, local)
    t = torch.tensor([float(rank + 1)])
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    if rank == 0:
        merged = {}
        for g in gathered:
            assert not (set(g) & set(merged)), "a request on two ranks"
            merged.update(g)
        q.put((merged, float(t.item())))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_sharding_matches_single_process():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    merged, tmax = q.get(timeout=300)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert tmax == 2.0
    wl = _workload()
    full = oracle.run_all(wl, W.make_index_cache(wl), W.make_latent_cache(wl), W.make_step_inputs(wl))
    assert sorted(merged) == [s.request_id for s in wl.spans]
    for s in wl.spans:
        sl = slice(s.q_start, s.q_start + s.q_len)
        sel, out = merged[s.request_id]
        assert np.array_equal(sel, full["selection"][sl])
        assert np.array_equal(out, full["out"][sl])


def test_assignment_is_balanced_and_complete():
    costs = [10, 9, 8, 7, 6, 5, 4, 3, 2, 1]
    a = sharding.assign_requests(costs, 3)
    flat = sorted(i for o in a for i in o)
    assert flat == list(range(10))
    loads = [sum(costs[i] for i in o) for o in a]
    assert max(loads) - min(loads) <= max(costs)
    wl = _workload()
    sh = wl.shape
    shards = sharding.shard_spans(wl.spans, 2, sh.topk, sh.index_row_bytes, sh.latent_row_bytes)
    for idx, spans in shards:
        q0 = 0
        for s in spans:
            assert s.q_start == q0
            q0 += s.q_len
