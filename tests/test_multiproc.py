"""Multi-rank host logic on CPU (gloo, world size 2).

Each rank takes the segments longest-processing-time-first assigns to it, builds their
pairs (here with the float64 oracle, since this runs without a GPU), and the ranks
gather the pairs; the result must equal a single-process build of every segment, and
the assignment must satisfy the LPT bound.
"""
from __future__ import annotations

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from linear_attention_state_gb300.shard import lpt_assign, segments_of, worker_loads

LENS = [37, 120, 5, 64, 90, 1, 77, 33]
D = 4


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _segment_inputs(i):
    rng = np.random.default_rng(1000 + i)
    L = LENS[i]
    k = rng.standard_normal((L, D))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    v = rng.standard_normal((L, D))
    a = np.exp(-np.log1p(np.exp(rng.standard_normal(L))) / 8)
    b = 1 / (1 + np.exp(-rng.standard_normal(L)))
    return k, v, a, b


def _pair(i):
    import oracle
    k, v, a, b = _segment_inputs(i)
    return oracle.segment_pair("gated_delta", k, v, a, b)


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    owner = lpt_assign(LENS, world)
    mine = {i: _pair(i) for i in segments_of(rank, owner)}
    gathered = [None] * world
    dist.all_gather_object(gathered, mine)
    if rank == 0:
        merged = {}
        for g in gathered:
            merged.update(g)
        out.put({i: (T.tolist(), S.tolist()) for i, (T, S) in merged.items()})
    dist.barrier()
    dist.destroy_process_group()


def test_lpt_assignment_properties():
    for world in (1, 2, 3, 8):
        owner = lpt_assign(LENS, world)
        loads = worker_loads(LENS, owner, world)
        assert sum(loads) == sum(LENS)
        # LPT is within 4/3 of the optimum; the optimum is at least max(mean load, longest segment)
        lower = max(sum(LENS) / world, max(LENS))
        assert max(loads) <= 4 / 3 * lower + 1e-9
    assert lpt_assign([5, 5, 5, 5], 2) == [0, 1, 0, 1]
    with pytest.raises(ValueError):
        lpt_assign([1], 0)


def test_two_gloo_ranks_build_their_shards():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    merged = q.get(timeout=120)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert sorted(merged) == list(range(len(LENS)))
    for i in range(len(LENS)):
        T, S = _pair(i)
        assert np.array_equal(np.array(merged[i][0]), T)
        assert np.array_equal(np.array(merged[i][1]), S)
    assert torch.distributed.is_available()
