"""Run paged-KV attention on a workload through the C ABI (device marshalling only).

``DeviceBatch`` moves one paged batch to the GPU; ``decode``, ``prefill``,
``cascade`` and ``multi_level_cascade`` plan and launch through ``api.Plan`` and
return (o, lse) device tensors.  The arithmetic is all in libpkvbsr.so.
"""
from __future__ import annotations

import dataclasses
from typing import Optional, Sequence, Tuple

import torch

from . import api


@dataclasses.dataclass
class DeviceBatch:
    host: object               # the workloads.PagedBatch it came from
    q: torch.Tensor
    kv_data: torch.Tensor
    qo_indptr: torch.Tensor
    kv_indptr: torch.Tensor
    kv_indices: torch.Tensor
    kv_last_page_len: torch.Tensor

    @staticmethod
    def from_host(b, device: str = "cuda", kv_data: Optional[torch.Tensor] = None) -> "DeviceBatch":
        to = lambda t: t.to(device, non_blocking=False).contiguous()
        return DeviceBatch(host=b, q=to(b.q), kv_data=to(b.kv_data) if kv_data is None else kv_data,
                           qo_indptr=to(b.qo_indptr), kv_indptr=to(b.kv_indptr), kv_indices=to(b.kv_indices),
                           kv_last_page_len=to(b.kv_last_page_len))


def _limits_of(b, max_batch=None, max_total_q=None, max_kv_pages=None):
    return dict(max_batch=max_batch or max(b.batch, 1),
                max_total_q=max_total_q or max(b.total_q, 1),
                max_kv_pages=max_kv_pages or max(int(b.kv_indptr[-1]), 1))


def make_plan(b, kind: int, pipelined: bool = False, split_kv: bool = True, **limits) -> api.Plan:
    lim = _limits_of(b, **limits)
    return api.Plan(kind, num_qo_heads=b.num_qo_heads, num_kv_heads=b.num_kv_heads, head_dim=b.head_dim,
                    page_size=b.page_size, dtype=b.dtype, sm_scale=b.sm_scale, logits_cap=b.logits_cap,
                    causal=b.causal, pipelined=pipelined, split_kv=split_kv, **lim)


def plan_batch(plan: api.Plan, b, stream=None) -> None:
    plan.plan(b.kv_indptr, b.kv_last_page_len, b.num_pages,
              qo_indptr_h=b.qo_indptr if plan.kind != api.PLAN_DECODE else None,
              kv_indices_h=b.kv_indices, stream=stream)


def decode(db: DeviceBatch, plan: Optional[api.Plan] = None, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    b = db.host
    if plan is None:
        plan = make_plan(b, api.PLAN_DECODE)
        plan_batch(plan, b, stream)
    o = torch.empty_like(db.q)
    lse = torch.empty(db.q.shape[:2], dtype=torch.float32, device=db.q.device)
    plan.run(db.q, db.kv_data, db.kv_indices, db.kv_indptr, db.kv_last_page_len, o, lse, stream=stream)
    return o, lse


def prefill(db: DeviceBatch, plan: Optional[api.Plan] = None, stream=None,
            mask: Optional[torch.Tensor] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Batch prefill; ``mask`` is an optional packed custom mask on the device
    (``workloads.pack_mask`` layout), applied on top of the batch's causal flag."""
    b = db.host
    if plan is None:
        plan = make_plan(b, api.PLAN_PREFILL)
        plan_batch(plan, b, stream)
    o = torch.empty_like(db.q)
    lse = torch.empty(db.q.shape[:2], dtype=torch.float32, device=db.q.device)
    plan.run(db.q, db.kv_data, db.kv_indices, db.kv_indptr, db.kv_last_page_len, o, lse,
             qo_indptr=db.qo_indptr, mask=mask, stream=stream)
    return o, lse


def cascade(prefix: DeviceBatch, suffix: DeviceBatch, prefix_plan: Optional[api.Plan] = None,
            suffix_plan: Optional[api.Plan] = None, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Shared-prefix attention: one prefill over the prefix row block (all
    requests' queries, no mask), one decode over the per-request suffixes, and
    merge_state of the two states, all on the GPU."""
    o_p, l_p = prefill(prefix, prefix_plan, stream)
    o_s, l_s = decode(suffix, suffix_plan, stream)
    api.merge_state(o_p, l_p, o_s, l_s, o_p, l_p, stream=stream)
    return o_p, l_p


def append_kv(db: DeviceBatch, k_new: torch.Tensor, v_new: torch.Tensor, rope_theta: float = 0.0,
              q_out: Optional[torch.Tensor] = None, rotate_q: bool = True, error: Optional[torch.Tensor] = None,
              stream=None) -> Optional[torch.Tensor]:
    """Append stage: write the batch's new tokens (one per query row, rows by
    qo_indptr) into ``db.kv_data`` at the end of each request's page list, turning
    the keys (and the queries, into ``q_out`` or a new tensor) by RoPE when
    rope_theta > 0.  Returns the rotated queries (None with rotate_q False)."""
    b = db.host
    params = api.make_params(b.num_qo_heads, b.num_kv_heads, b.head_dim, b.page_size, b.dtype, b.sm_scale)
    if rotate_q and q_out is None:
        q_out = torch.empty_like(db.q)
    api.append_paged_kv(params, db.qo_indptr, db.kv_indptr, db.kv_indices, db.kv_last_page_len, k_new, v_new,
                        db.kv_data, db.q if rotate_q else None, q_out if rotate_q else None, rope_theta,
                        error=error, stream=stream)
    return q_out if rotate_q else None


def mixed(db: DeviceBatch, plan: Optional[api.Plan] = None, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """A batch mixing single-row (decode) and multi-row (prefill) requests in one
    call: the plan routes each request by its row count and splits the SMs, and one
    persistent launch runs both halves."""
    b = db.host
    if plan is None:
        plan = make_plan(b, api.PLAN_MIXED)
        plan_batch(plan, b, stream)
    o = torch.empty_like(db.q)
    lse = torch.empty(db.q.shape[:2], dtype=torch.float32, device=db.q.device)
    plan.run(db.q, db.kv_data, db.kv_indices, db.kv_indptr, db.kv_last_page_len, o, lse,
             qo_indptr=db.qo_indptr, stream=stream)
    return o, lse


def levels_mixed(db: DeviceBatch, n_levels: int, plan: Optional[api.Plan] = None, stream=None
                 ) -> Tuple[torch.Tensor, torch.Tensor]:
    """A prefix tree (or a cascade, n_levels = 2) as one mixed launch: ``db`` holds
    ``workloads.levels_as_mixed(levels)``.  Multi-row nodes run on the prefill half
    of the mixed kernel and single-row nodes on its decode half; one n-state
    merge_state then folds every level's rows into the last level's."""
    o, lse = mixed(db, plan, stream)
    R = db.q.shape[0] // n_levels
    o_out, l_out = o[(n_levels - 1) * R:], lse[(n_levels - 1) * R:]
    # every level's states at once, into the last level's rows
    api.merge_states(o, lse, n_levels, o_out, l_out, stream=stream)
    return o_out, l_out


def cascade_mixed(db: DeviceBatch, plan: Optional[api.Plan] = None, stream=None
                  ) -> Tuple[torch.Tensor, torch.Tensor]:
    """Cascade attention as one mixed launch (``workloads.cascade_as_mixed``)."""
    return levels_mixed(db, 2, plan, stream)


def level_kind(b) -> int:
    """A level whose nodes each hold one query row is plain decode; a level with
    multi-row blocks (a prefix shared by several requests) runs on the prefill
    kernel without a mask, so each node's KV is read once for all its rows."""
    return api.PLAN_DECODE if all(n == 1 for n in b.qo_lens) else api.PLAN_PREFILL


def multi_level_cascade(levels: Sequence[DeviceBatch], plans: Optional[Sequence[api.Plan]] = None,
                        stream=None, side_streams: Optional[Sequence] = None
                        ) -> Tuple[torch.Tensor, torch.Tensor]:
    """Attention over a prefix tree stored as one BSR matrix per level (greptalks
    summary, "Composable Formats for Shared Prefixes": one block-sparse matrix
    decomposed into several with different row-block sizes; fdeinterviews summary,
    "One format": shared prefixes as large row blocks, no data moved).

    Each level's batch groups the request rows into consecutive blocks (its nodes),
    each block against that node's pages; every level covers every row once.  Each
    level is computed on the GPU (prefill kernel for multi-row blocks, decode kernel
    for single rows) and the states are folded into level 0's buffers with
    merge_state.  With ``side_streams`` (one per level after the first) the levels
    run concurrently and join before the merges; the whole call is capturable in
    one CUDA graph.
    """
    if not levels:
        raise ValueError("multi_level_cascade needs at least one level")
    if plans is None:
        plans = []
        for db in levels:
            p = make_plan(db.host, level_kind(db.host))
            plan_batch(p, db.host, stream)
            plans.append(p)
    if len(plans) != len(levels):
        raise ValueError("one plan per level")
    if side_streams is not None and len(side_streams) < len(levels) - 1:
        raise ValueError("one side stream per level after the first")
    q = levels[0].q
    outs = [(torch.empty_like(q), torch.empty(q.shape[:2], dtype=torch.float32, device=q.device))
            for _ in levels]
    main = stream if stream is not None else torch.cuda.current_stream()

    def run(i, s):
        db, p = levels[i], plans[i]
        o, lse = outs[i]
        p.run(db.q, db.kv_data, db.kv_indices, db.kv_indptr, db.kv_last_page_len, o, lse,
              qo_indptr=db.qo_indptr if p.kind == api.PLAN_PREFILL else None, stream=s)

    if side_streams is None:
        for i in range(len(levels)):
            run(i, main)
    else:
        fork = torch.cuda.Event()
        fork.record(main)
        joins = []
        for i in range(1, len(levels)):
            s = side_streams[i - 1]
            s.wait_event(fork)
            run(i, s)
            ev = torch.cuda.Event()
            ev.record(s)
            joins.append(ev)
        run(0, main)
        for ev in joins:
            main.wait_event(ev)
    o0, l0 = outs[0]
    for o, lse in outs[1:]:
        api.merge_state(o0, l0, o, lse, o0, l0, stream=main)
    return o0, l0
