"""Host-side partitioning of build units across ranks (one GPU per rank).

Segments of a request are independent build units (HYPIC reading notes, Method 7:
segment parallelism; paper Sec. 4.4).  Cold segments are spread over workers by
longest processing time first (paper Eq. (9)): sort by token count, largest first,
and give each to the worker with the least tokens so far, which approximately
minimises the largest per-worker total.  No data-path collective is needed: every
rank builds its own segments' pairs.
"""
from __future__ import annotations


def lpt_assign(lengths: list[int], n_workers: int) -> list[int]:
    """Worker index for each segment; ties go to the lower worker index, then the earlier segment."""
    if n_workers < 1:
        raise ValueError("n_workers must be >= 1")
    order = sorted(range(len(lengths)), key=lambda i: (-int(lengths[i]), i))
    load = [0] * n_workers
    owner = [0] * len(lengths)
    for i in order:
        w = min(range(n_workers), key=lambda k: (load[k], k))
        owner[i] = w
        load[w] += int(lengths[i])
    return owner


def worker_loads(lengths: list[int], owner: list[int], n_workers: int) -> list[int]:
    load = [0] * n_workers
    for L, w in zip(lengths, owner):
        load[w] += int(L)
    return load


def segments_of(rank: int, owner: list[int]) -> list[int]:
    return [i for i, w in enumerate(owner) if w == rank]


# ---- combine-side exchange -----------------------------------------------------------------
# With segment parallelism the cold segments of one request are built on several workers and their
# pairs go once to the worker that assembles the request (HYPIC reading notes, Method 7: scatter
# the cold segments, combine on one instance with one-sided writes into preallocated slots).  Here a
# worker is a rank of a torch.distributed group (one GPU per rank, NCCL for device tensors; gloo
# serves host tensors), and the one-sided write is a point-to-point send matched by a receive posted
# straight into the combine rank's slot: no staging copy and no collective over all ranks.

class CombinePlan:
    """Which rank builds each cold segment (longest processing time first) and which rank combines.

    Slot i of the combine rank's pair pool holds segment i (request order)."""

    def __init__(self, lengths: list[int], world: int, combine_rank: int = 0):
        if not 0 <= combine_rank < world:
            raise ValueError("combine_rank must be a rank of the group")
        self.lengths = [int(x) for x in lengths]
        self.world = world
        self.combine_rank = combine_rank
        self.owner = lpt_assign(self.lengths, world)

    def segments_of(self, rank: int) -> list[int]:
        return segments_of(rank, self.owner)


def combine_pairs(plan: CombinePlan, rank: int, T_local, S_local, T_slots=None, S_slots=None, group=None):
    """Deliver every rank's built pairs into the combine rank's preallocated slots.

    T_local, S_local: this rank's pairs, [k, H, ...] for its segments plan.segments_of(rank) in that
    order (k may be 0).  On the combine rank T_slots [n_seg, H, ...] and S_slots [n_seg, H, d, d] are
    filled in place (its own pairs by a local copy, the others' by receives posted directly into the
    slots); other ranks pass None.  All ranks call this together; pairs travel in ascending segment
    order, so sends and receives match without tags.  Returns when this rank's transfers are done.
    """
    import torch.distributed as dist

    mine = plan.segments_of(rank)
    if len(mine) != (0 if T_local is None else T_local.shape[0]):
        raise ValueError("T_local must hold this rank's segments in plan order")
    ops = []
    if rank == plan.combine_rank:
        if T_slots is None or S_slots is None or T_slots.shape[0] != len(plan.lengths):
            raise ValueError("the combine rank needs T_slots and S_slots with one slot per segment")
        for k, i in enumerate(mine):
            T_slots[i].copy_(T_local[k])
            S_slots[i].copy_(S_local[k])
        for i, w in enumerate(plan.owner):
            if w != rank:
                ops.append(dist.P2POp(dist.irecv, T_slots[i], w, group))
                ops.append(dist.P2POp(dist.irecv, S_slots[i], w, group))
    else:
        for k, i in enumerate(mine):
            ops.append(dist.P2POp(dist.isend, T_local[k].contiguous(), plan.combine_rank, group))
            ops.append(dist.P2POp(dist.isend, S_local[k].contiguous(), plan.combine_rank, group))
    if ops:
        for req in dist.batch_isend_irecv(ops):
            req.wait()
