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


def _combine_worker(rank, world, port, combine_rank, out):
    from linear_attention_state_gb300.shard import CombinePlan, combine_pairs
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    plan = CombinePlan(LENS, world, combine_rank)
    mine = plan.segments_of(rank)
    pairs = [_pair(i) for i in mine]
    # [k, H = 1, d, d] per rank: this rank's segments in plan order (k may be 0)
    T_local = torch.tensor(np.array([p[0] for p in pairs]).reshape(len(mine), 1, D, D))
    S_local = torch.tensor(np.array([p[1] for p in pairs]).reshape(len(mine), 1, D, D))
    T_slots = S_slots = None
    if rank == combine_rank:
        T_slots = torch.full((len(LENS), 1, D, D), float("nan"), dtype=torch.float64)
        S_slots = torch.full((len(LENS), 1, D, D), float("nan"), dtype=torch.float64)
    combine_pairs(plan, rank, T_local, S_local, T_slots, S_slots)
    if rank == combine_rank:
        out.put((T_slots.tolist(), S_slots.tolist(), plan.owner))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world,combine_rank", [(2, 0), (3, 2)])
def test_cold_segments_scatter_and_combine_into_slots(world, combine_rank):
    """Cold segments built on the ranks LPT assigns them to arrive, by point-to-point transfers,
    in the combine rank's preallocated slots in request order, bit for bit."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_combine_worker, args=(r, world, port, combine_rank, q)) for r in range(world)]
    for p in procs:
        p.start()
    T_slots, S_slots, owner = q.get(timeout=120)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert len(set(owner)) == world  # every rank built something
    for i in range(len(LENS)):
        T, S = _pair(i)
        assert np.array_equal(np.array(T_slots[i][0]), T)
        assert np.array_equal(np.array(S_slots[i][0]), S)


def test_combine_plan_checks():
    from linear_attention_state_gb300.shard import CombinePlan
    with pytest.raises(ValueError):
        CombinePlan(LENS, 2, combine_rank=2)
    plan = CombinePlan(LENS, 3, combine_rank=1)
    assert sorted(i for r in range(3) for i in plan.segments_of(r)) == list(range(len(LENS)))
