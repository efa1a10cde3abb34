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
