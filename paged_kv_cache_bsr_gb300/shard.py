"""A paged batch spread over ranks, one GPU each.

Requests are independent, so a batch shards by request with no exchange: each
rank runs the requests ``partition_requests`` gives it and writes their rows.
A request too long for one rank's share shards by key range instead: each rank
attends to one contiguous run of its pages (``split_sequence``), and the one
exchange step is an all-gather of those partial (o, lse) states
(``allgather_states``), which merge_state folds into the full result
(``merge_gathered``) -- the same composition of partial attention states the
pages use for split-KV decode ("FlashInfer" guide, section 3 "FlashDecoding":
partial results combined by their log-sum-exp; fdeinterviews summary, "Load
balancing that survives CUDA graphs").
"""
from __future__ import annotations

import dataclasses
from typing import List, Sequence, Tuple

import torch


def request_costs(b) -> List[int]:
    """Work of every request of a paged batch in key pages x query rows x kv heads
    (for decode, its pages x kv heads: the unit the plans balance)."""
    return [int(b.kv_indptr[r + 1] - b.kv_indptr[r]) * max(1, int(b.qo_lens[r])) * b.num_kv_heads
            for r in range(b.batch)]


def partition_requests(costs: Sequence[int], world: int) -> List[List[int]]:
    """Requests onto ``world`` ranks, longest first onto the least-loaded rank (ties to
    the lower request and rank index); each rank's list in request order."""
    if world <= 0:
        raise ValueError("world must be positive")
    loads = [0] * world
    parts: List[List[int]] = [[] for _ in range(world)]
    for r in sorted(range(len(costs)), key=lambda i: (-int(costs[i]), i)):
        k = min(range(world), key=lambda j: (loads[j], j))
        parts[k].append(r)
        loads[k] += int(costs[r])
    return [sorted(p) for p in parts]


def split_sequence(b, request: int, world: int) -> list:
    """Request ``request``'s pages cut into ``world`` contiguous runs of near-equal
    length, each as a one-request batch over the same pool; its attention is the
    partial state of those keys (a run without pages gives o = 0, lse = -inf).
    The request must have one query row or a non-causal mask: a causal limit is
    measured from the end of the whole key range, which a run does not see."""
    qo = int(b.qo_lens[request])
    if b.causal and qo > 1:
        raise ValueError("a causal request with several query rows cannot be split by key range")
    lo, hi = int(b.kv_indptr[request]), int(b.kv_indptr[request + 1])
    n = hi - lo
    q0 = int(b.qo_indptr[request])
    pieces = []
    for k in range(world):
        a, e = lo + k * n // world, lo + (k + 1) * n // world
        if e > a:
            last = int(b.kv_last_page_len[request]) if e == hi else b.page_size
            kv_len = (e - a - 1) * b.page_size + last
        else:
            last, kv_len = 0, 0
        pieces.append(dataclasses.replace(
            b, q=b.q[q0:q0 + qo].clone(),
            qo_indptr=torch.tensor([0, qo], dtype=torch.int32),
            kv_indptr=torch.tensor([0, e - a], dtype=torch.int32),
            kv_indices=b.kv_indices[a:e].clone(),
            kv_last_page_len=torch.tensor([last], dtype=torch.int32),
            qo_lens=[qo], kv_lens=[kv_len], name=f"{b.name} keys {k}/{world}"))
    return pieces


def allgather_states(o: torch.Tensor, lse: torch.Tensor, group=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Every rank's partial state of the same rows, stacked rank by rank along a new
    first axis, on every rank: the one exchange step of a split sequence."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    os_ = [torch.empty_like(o) for _ in range(world)]
    ls = [torch.empty_like(lse) for _ in range(world)]
    dist.all_gather(os_, o.contiguous(), group=group)
    dist.all_gather(ls, lse.contiguous(), group=group)
    return torch.stack(os_), torch.stack(ls)


def merge_gathered(os_: torch.Tensor, lses: torch.Tensor, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Fold gathered partial states [world, rows, heads, d] / [world, rows, heads]
    into one with merge_state on the device, in rank order."""
    from . import api
    o, lse = os_[0].clone(), lses[0].clone()
    for k in range(1, os_.shape[0]):
        api.merge_state(o, lse, os_[k], lses[k], o, lse, stream=stream)
    return o, lse
