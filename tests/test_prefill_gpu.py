"""GPU parity of the tcgen05 paged prefill (causal ragged, split key ranges) and of
cascade attention (prefix row block + per-request suffix + merge_state) against the
fp64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_bsr_gb300 import api, runner, workloads as W
from gpu_util import assert_matches_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_bsr_gb300 import build
    build.build()
    oracle.build()
    api.load()
    torch.cuda.set_device(0)


def prefill_vs_oracle(b, what="", rows=None, **limits):
    db = runner.DeviceBatch.from_host(b)
    plan = runner.make_plan(b, api.PLAN_PREFILL, **limits)
    runner.plan_batch(plan, b)
    o, lse = runner.prefill(db, plan)
    torch.cuda.synchronize()
    assert plan.device_error() == 0
    ref_o, ref_lse = oracle.attention_of(b, rows=rows)
    if rows is not None:
        idx = torch.as_tensor(rows, dtype=torch.long, device=o.device)
        o, lse = o[idx], lse[idx]
    assert_matches_oracle(o, lse, ref_o, ref_lse, b.dtype, what)
    return plan


def batch(qo_lens, prefix, hq=8, hkv=2, P=16, dtype=torch.bfloat16, causal=True, seed=0, cap=0.0):
    kv = [q + p for q, p in zip(qo_lens, prefix)]
    return W.make_paged_batch(qo_lens=qo_lens, kv_lens=kv, num_qo_heads=hq, num_kv_heads=hkv, head_dim=128,
                              page_size=P, dtype=dtype, seed=seed, causal=causal, logits_cap=cap, poison=True)


def test_small_ragged_causal():
    prefill_vs_oracle(batch([1, 37, 200], [0, 5, 100], seed=1), "small causal")


@pytest.mark.parametrize("group", [1, 2, 4, 8])
def test_group_sizes(group):
    prefill_vs_oracle(batch([130, 7, 300], [17, 0, 64], hq=2 * group, hkv=2, seed=group), f"g{group}")


def test_fp16():
    prefill_vs_oracle(batch([100, 129], [3, 200], dtype=torch.float16, seed=2), "fp16")


def test_non_causal():
    prefill_vs_oracle(batch([50, 128, 300], [10, 70, 1], causal=False, seed=3), "non-causal")


@pytest.mark.parametrize("page_size", [8, 32, 64, 128])
def test_page_sizes(page_size):
    prefill_vs_oracle(batch([90, 257], [33, 5], P=page_size, seed=page_size), f"page {page_size}")


@pytest.mark.parametrize("page_size", [16, 1])
def test_rows_that_see_no_key_and_empty_requests(page_size):
    # causal with more rows than keys: the first qo - kv rows see nothing (o = 0, lse = -inf);
    # a request with no keys at all (no packed page either, with one-row pages)
    b = W.make_paged_batch(qo_lens=[10, 0, 3, 40, 6], kv_lens=[5, 9, 3, 1, 0], num_qo_heads=8, num_kv_heads=2,
                           head_dim=128, page_size=page_size, dtype=torch.bfloat16, seed=4, causal=True,
                           poison=True)
    prefill_vs_oracle(b, f"no keys, page {page_size}")


def test_softcap_prefill():
    prefill_vs_oracle(batch([77, 200], [100, 0], seed=5, cap=30.0), "softcap")


def test_split_key_range_is_merged():
    """Few query tiles and long keys: the plan cuts key ranges into chunks (partials + merge)."""
    b = W.make_paged_batch(qo_lens=[64], kv_lens=[9000], num_qo_heads=8, num_kv_heads=2, head_dim=128,
                           page_size=16, dtype=torch.bfloat16, seed=6, causal=False, poison=True)
    plan = prefill_vs_oracle(b, "split")
    assert plan.info().num_merge > 0 and plan.info().num_slots > 8


@pytest.mark.slow
def test_ragged_causal_prefill_full_size_every_row():
    """Batch 16, qo ~ U[128, 2048], kv = qo + U[0, 1024], 32/8 heads: every row of the
    measured batch (every work tile and every tile change on every CTA) against the
    oracle."""
    b = W.ragged_prefill(seed=1003, poison=True)
    prefill_vs_oracle(b, "ragged full size")


@pytest.mark.slow
def test_cascade_softcap_full_size_equals_full_attention():
    """64 requests sharing a 2048-token prefix (one large row block), suffixes U[50, 200],
    soft-cap 30: prefix prefill + suffix decode + merge_state vs non-cascade attention."""
    cb = W.cascade_decode(seed=1004, poison=True)
    kv = cb.full.kv_data.cuda()
    dp = runner.DeviceBatch.from_host(cb.prefix, kv_data=kv)
    ds = runner.DeviceBatch.from_host(cb.suffix, kv_data=kv)
    pplan = runner.make_plan(cb.prefix, api.PLAN_PREFILL)
    splan = runner.make_plan(cb.suffix, api.PLAN_DECODE)
    runner.plan_batch(pplan, cb.prefix)
    runner.plan_batch(splan, cb.suffix)
    o, lse = runner.cascade(dp, ds, pplan, splan)
    torch.cuda.synchronize()
    assert pplan.device_error() == 0 and splan.device_error() == 0
    ref_o, ref_lse = oracle.attention_of(cb.full)
    assert_matches_oracle(o, lse, ref_o, ref_lse, torch.bfloat16, "cascade")


@pytest.mark.parametrize("page_size", [16, 1])
def test_prefill_page_id_outside_the_pool_sets_the_error_bit(page_size):
    """A device page table with an id outside the pool: tensor loads use a page
    coordinate past the pool and the row gather zero-fills, so nothing outside
    kv_data is read; the page-index error bit is set, and the requests without the
    bad entry keep their exact results."""
    b = batch([40, 130, 77], [20, 300, 0], P=page_size, seed=41 + page_size)
    db = runner.DeviceBatch.from_host(b)
    plan = runner.make_plan(b, api.PLAN_PREFILL)
    runner.plan_batch(plan, b)
    bad = int(b.kv_indptr[1])  # the first page of request 1
    db.kv_indices[bad] = -3
    o, lse = runner.prefill(db, plan)
    torch.cuda.synchronize()
    assert plan.device_error() & 1
    rows = [i for r in (0, 2) for i in range(int(b.qo_indptr[r]), int(b.qo_indptr[r + 1]))]
    ref_o, ref_lse = oracle.attention_of(b, rows=rows)
    idx = torch.as_tensor(rows, dtype=torch.long, device=o.device)
    assert_matches_oracle(o[idx], lse[idx], ref_o, ref_lse, b.dtype, "other requests")


def test_prefill_page_permutation_is_bit_exact():
    b = batch([300, 45], [60, 200], seed=8)
    db = runner.DeviceBatch.from_host(b)
    plan = runner.make_plan(b, api.PLAN_PREFILL)
    runner.plan_batch(plan, b)
    o1, l1 = runner.prefill(db, plan)
    perm = torch.randperm(b.num_pages, generator=torch.Generator().manual_seed(5))
    kv2 = torch.empty_like(b.kv_data)
    kv2[perm] = b.kv_data
    b2 = W.PagedBatch(**{**b.__dict__, "kv_data": kv2, "kv_indices": perm[b.kv_indices.long()].to(torch.int32)})
    runner.plan_batch(plan, b2)
    o2, l2 = runner.prefill(runner.DeviceBatch.from_host(b2), plan)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("P", [16, 1])
def test_prefill_cuda_graph_replay_after_replanning(P):
    """Capture the prefill run calls once; re-plan another batch (same total query rows,
    same pool) into the same workspace and buffers; replay gives that batch's result.
    With one-row pages the captured calls include the packing copy, whose page count
    the replay reads from the re-planned tables."""
    hq, hkv, d = 8, 2, 128
    pool = 2560 // P
    gen = torch.Generator().manual_seed(21)
    kv = torch.randn(pool, 2, hkv, P, d, generator=gen).to(torch.bfloat16)

    def batch_with(qo_lens, kv_lens, seed):
        g = torch.Generator().manual_seed(seed)
        perm = torch.randperm(pool, generator=g)
        ip, ix, last, _ = W.build_page_table(kv_lens, P, perm)
        q = torch.randn(sum(qo_lens), hq, d, generator=g).to(torch.bfloat16)
        qo = torch.zeros(len(qo_lens) + 1, dtype=torch.int32)
        qo[1:] = torch.cumsum(torch.tensor(qo_lens), 0)
        return W.PagedBatch(page_size=P, num_qo_heads=hq, num_kv_heads=hkv, head_dim=d, dtype=torch.bfloat16,
                            q=q, kv_data=kv, qo_indptr=qo, kv_indptr=ip, kv_indices=ix, kv_last_page_len=last,
                            qo_lens=list(qo_lens), kv_lens=list(kv_lens), sm_scale=d ** -0.5, causal=True)

    a = batch_with([100, 300, 28], [150, 700, 28], 1)
    bb = batch_with([228, 200, 0], [500, 210, 7], 2)
    max_b, max_q = 3, 428
    plan = runner.make_plan(a, api.PLAN_PREFILL, max_batch=max_b, max_total_q=max_q, max_kv_pages=pool)
    dev = "cuda"
    kv_d = kv.to(dev)
    q_buf = torch.empty(max_q, hq, d, dtype=torch.bfloat16, device=dev)
    o_buf = torch.empty_like(q_buf)
    lse_buf = torch.empty(max_q, hq, dtype=torch.float32, device=dev)
    qo_buf = torch.zeros(max_b + 1, dtype=torch.int32, device=dev)
    ip_buf = torch.zeros(max_b + 1, dtype=torch.int32, device=dev)
    ix_buf = torch.zeros(pool, dtype=torch.int32, device=dev)
    last_buf = torch.zeros(max_b, dtype=torch.int32, device=dev)

    def load(b):
        q_buf.copy_(b.q)
        qo_buf.copy_(b.qo_indptr)
        ip_buf.copy_(b.kv_indptr)
        ix_buf[: b.kv_indices.numel()].copy_(b.kv_indices)
        last_buf.copy_(b.kv_last_page_len)

    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        load(a)
        runner.plan_batch(plan, a, stream=s)
        plan.run(q_buf, kv_d, ix_buf, ip_buf, last_buf, o_buf, lse_buf, qo_indptr=qo_buf, stream=s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        plan.run(q_buf, kv_d, ix_buf, ip_buf, last_buf, o_buf, lse_buf, qo_indptr=qo_buf, stream=s)
    for b in (bb, a, bb):
        with torch.cuda.stream(s):
            load(b)
            runner.plan_batch(plan, b, stream=s)
            g.replay()
        s.synchronize()
        ref_o, ref_lse = oracle.attention_of(b)
        assert_matches_oracle(o_buf, lse_buf, ref_o, ref_lse, torch.bfloat16, "prefill graph replay")
    assert plan.device_error() == 0


@pytest.mark.parametrize("page_size", [1, 2, 4])
def test_column_vector_pages(page_size):
    """Pages of 1, 2 or 4 rows (column-vector BSR) take the row-gather path."""
    prefill_vs_oracle(batch([90, 257, 1], [33, 5, 300], P=page_size, seed=20 + page_size), f"page {page_size}")


def test_column_vector_pages_split_and_softcap():
    b = W.make_paged_batch(qo_lens=[40], kv_lens=[5000], num_qo_heads=8, num_kv_heads=2, head_dim=128,
                           page_size=1, dtype=torch.float16, seed=24, causal=True, logits_cap=30.0, poison=True)
    plan = prefill_vs_oracle(b, "page 1 split")
    assert plan.info().num_merge > 0


@pytest.mark.parametrize("page_size", [1, 4])
def test_column_vector_pages_full_ragged_batch(page_size):
    """The full ragged batch on 1- and 4-row pages: every CTA walks several tiles, so
    each tile's last gathered block must be released before the next tile starts."""
    b = W.ragged_prefill(seed=1003, poison=True, page_size=page_size)
    rng = np.random.default_rng(1)
    rows = np.sort(rng.choice(b.total_q, size=1500, replace=False))
    plan = prefill_vs_oracle(b, f"ragged full size, page {page_size}", rows=rows)
    assert plan.info().active_workers > 0
