"""The decode entry point for callers that cannot allocate device memory.

pkv_batch_decode_paged_noalloc keeps its plan tables and fp32 partial states
in a static device array inside the library instead of a workspace the caller
allocates (for plug-ins whose framework owns all device memory, services under
a fixed memory budget, and code that must avoid cudaMalloc's implicit
synchronisation).  These tests call it through the C ABI and check that it
returns what pkv_batch_decode_paged returns on the same inputs, on two calls
in a row with different batches (the static array keeps the previous call's
contents), bit for bit in o and lse, and that a plan too large for the array is
refused.

This file is named to be collected after the main GPU tests.
"""
import pytest
import torch

from paged_kv_cache_bsr_gb300 import api, runner, workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_bsr_gb300 import build
    build.build()
    api.load()
    torch.cuda.set_device(0)


def _identical(o, lse, o_ref, lse_ref):
    """Both entry points run the same kernels on the same tables, so the outputs must
    agree bit for bit: a table or partial state misplaced in the static array would
    show here even where it stayed within the parity tolerance."""
    assert torch.isfinite(o.float()).all()
    assert torch.equal(o.view(torch.int16), o_ref.view(torch.int16))
    assert torch.equal(lse.view(torch.int32), lse_ref.view(torch.int32))


def test_noalloc_decode_matches_workspace_decode_on_two_calls():
    batches = [W.llama3_decode(seed=31, batch=24, poison=True),
               W.make_paged_batch(qo_lens=[1] * 5, kv_lens=[9000, 1, 0, 333, 4096], num_qo_heads=32,
                                  num_kv_heads=8, head_dim=128, page_size=16, dtype=torch.bfloat16, seed=32,
                                  poison=True)]
    max_pages = max(int(b.kv_indptr[-1]) for b in batches)
    plan = None
    for b in batches:
        db = runner.DeviceBatch.from_host(b)
        if plan is None:
            plan = runner.make_plan(b, api.PLAN_DECODE, max_batch=32, max_kv_pages=max_pages)
        # the existing entry point, with its caller-allocated workspace
        runner.plan_batch(plan, b)
        o_ref, lse_ref = runner.decode(db, plan)
        # the static-scratch entry point: plan on the host, then one call
        host_tables = torch.empty_like(plan.host_ws)  # ordinary (pageable) host memory
        api.plan_compute(plan.handle, b.batch, None, b.kv_indptr, b.kv_indices, b.kv_last_page_len, b.num_pages,
                         host_tables)
        o = torch.full_like(db.q, float("nan"))
        lse = torch.full(db.q.shape[:2], float("nan"), dtype=torch.float32, device=db.q.device)
        api.batch_decode_paged_noalloc(plan.handle, host_tables, db.q, db.kv_data, db.kv_indices, db.kv_indptr,
                                       db.kv_last_page_len, o, lse)
        torch.cuda.synchronize()
        assert plan.info().num_merge > 0  # the static array held fp32 partial states
        _identical(o, lse, o_ref, lse_ref)


def test_noalloc_refuses_plans_larger_than_its_scratch():
    b = W.make_paged_batch(qo_lens=[1] * 2, kv_lens=[100, 200], num_qo_heads=32, num_kv_heads=8, head_dim=128,
                           page_size=16, dtype=torch.bfloat16, seed=3)
    plan = runner.make_plan(b, api.PLAN_DECODE, max_batch=65536, max_kv_pages=1 << 20)
    dev_bytes, _ = api.plan_workspace_bytes(plan.handle)
    assert dev_bytes > (8 << 20)
    host_tables = torch.empty_like(plan.host_ws)
    api.plan_compute(plan.handle, b.batch, None, b.kv_indptr, b.kv_indices, b.kv_last_page_len, b.num_pages,
                     host_tables)
    db = runner.DeviceBatch.from_host(b)
    o = torch.empty_like(db.q)
    with pytest.raises(api.PkvError) as e:
        api.batch_decode_paged_noalloc(plan.handle, host_tables, db.q, db.kv_data, db.kv_indices, db.kv_indptr,
                                       db.kv_last_page_len, o, None)
    assert e.value.status == -4


def test_noalloc_refuses_tensor_core_decode_plans():
    """8 query heads per kv head at head_dim 128 decode on the tensor cores, whose
    prefill-sized partial states the static array cannot hold."""
    b = W.make_paged_batch(qo_lens=[1] * 2, kv_lens=[100, 200], num_qo_heads=64, num_kv_heads=8, head_dim=128,
                           page_size=16, dtype=torch.bfloat16, seed=3)
    plan = runner.make_plan(b, api.PLAN_DECODE)
    host_tables = torch.empty_like(plan.host_ws)
    api.plan_compute(plan.handle, b.batch, None, b.kv_indptr, b.kv_indices, b.kv_last_page_len, b.num_pages,
                     host_tables)
    db = runner.DeviceBatch.from_host(b)
    o = torch.empty_like(db.q)
    with pytest.raises(api.PkvError) as e:
        api.batch_decode_paged_noalloc(plan.handle, host_tables, db.q, db.kv_data, db.kv_indices, db.kv_indptr,
                                       db.kv_last_page_len, o, None)
    assert e.value.status == -3
