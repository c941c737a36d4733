"""Run paged-KV attention on a workload through the C ABI (device marshalling only).

``DeviceBatch`` moves one paged batch to the GPU; ``decode``, ``prefill`` and
``cascade`` plan and launch through ``api.Plan`` and return (o, lse) device
tensors.  The arithmetic is all in libpkvbsr.so.
"""
from __future__ import annotations

import dataclasses
from typing import Optional, Tuple

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


def make_plan(b, kind: int, **limits) -> api.Plan:
    lim = _limits_of(b, **limits)
    return api.Plan(kind, num_qo_heads=b.num_qo_heads, num_kv_heads=b.num_kv_heads, head_dim=b.head_dim,
                    page_size=b.page_size, dtype=b.dtype, sm_scale=b.sm_scale, logits_cap=b.logits_cap,
                    causal=b.causal, **lim)


def plan_batch(plan: api.Plan, b, stream=None) -> None:
    plan.plan(b.kv_indptr, b.kv_last_page_len, b.num_pages,
              qo_indptr_h=b.qo_indptr if plan.kind == api.PLAN_PREFILL else None,
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


def prefill(db: DeviceBatch, plan: Optional[api.Plan] = None, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    b = db.host
    if plan is None:
        plan = make_plan(b, api.PLAN_PREFILL)
        plan_batch(plan, b, stream)
    o = torch.empty_like(db.q)
    lse = torch.empty(db.q.shape[:2], dtype=torch.float32, device=db.q.device)
    plan.run(db.q, db.kv_data, db.kv_indices, db.kv_indptr, db.kv_last_page_len, o, lse,
             qo_indptr=db.qo_indptr, stream=stream)
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
