"""GPU parity of mixed batches (single-row decode requests and multi-row prefill
requests in one call: one persistent launch whose first CTAs run the tcgen05
prefill half and the rest the CUDA-core decode workers) against the fp64 oracle."""
import pytest
import torch

import oracle
from paged_kv_cache_bsr_gb300 import api, runner, workloads as W
from gpu_util import assert_matches_oracle, kernel_nodes

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_bsr_gb300 import build
    build.build()
    oracle.build()
    api.load()
    torch.cuda.set_device(0)


def mixed_vs_oracle(b, what, rows=None):
    db = runner.DeviceBatch.from_host(b)
    plan = runner.make_plan(b, api.PLAN_MIXED)
    runner.plan_batch(plan, b)
    o, lse = runner.mixed(db, plan)
    torch.cuda.synchronize()
    assert plan.device_error() == 0
    ref_o, ref_lse = oracle.attention_of(b, rows=rows)
    if rows is not None:
        idx = torch.as_tensor(rows, dtype=torch.long, device=o.device)
        o, lse = o[idx], lse[idx]
    assert_matches_oracle(o, lse, ref_o, ref_lse, b.dtype, what)
    return plan


def small_mixed(seed, hq=8, hkv=2, dtype=torch.bfloat16, n_decode=9, n_prefill=3):
    return W.mixed_batch(seed=seed, n_decode=n_decode, n_prefill=n_prefill, decode_lo=1, decode_hi=700, qo_lo=2,
                         qo_hi=300, prefix_lo=0, prefix_hi=200, num_qo_heads=hq, num_kv_heads=hkv, dtype=dtype,
                         poison=True)


@pytest.mark.parametrize("group,dtype", [(4, torch.bfloat16), (1, torch.float16), (8, torch.bfloat16)])
def test_small_mixed_batches(group, dtype):
    plan = mixed_vs_oracle(small_mixed(group, hq=2 * group, dtype=dtype), f"mixed g{group}")
    info = plan.info()
    if group == 8:  # single rows run on the tensor cores too: one prefill half on every SM
        assert info.decode_ctas == 0 and info.prefill_ctas == torch.cuda.get_device_properties(0).multi_processor_count
    else:
        assert info.prefill_ctas >= 1 and info.decode_ctas >= 1


@pytest.mark.parametrize("page_size,group,cap", [(1, 4, 0.0), (4, 2, 30.0), (2, 8, 0.0), (64, 1, 30.0)])
def test_mixed_page_sizes_and_cap(page_size, group, cap):
    """Pages of 1, 2 and 4 rows take the cp.async-gather instances of the mixed kernel;
    64-row pages and the soft-capped instances the others."""
    b = W.mixed_batch(seed=30 + page_size, n_decode=9, n_prefill=3, decode_lo=1, decode_hi=500, qo_lo=2,
                      qo_hi=260, prefix_lo=0, prefix_hi=150, num_qo_heads=2 * group, num_kv_heads=2,
                      page_size=page_size, poison=True)
    b = W.PagedBatch(**{**b.__dict__, "logits_cap": cap})
    plan = mixed_vs_oracle(b, f"mixed page {page_size} g{group} cap {cap}")
    info = plan.info()
    assert info.prefill_ctas >= 1 and info.decode_ctas >= 1


def test_mixed_is_one_attention_launch():
    """The run call launches the mixed kernel once (a CTA on every SM), then one merge
    kernel for both halves; neither the decode kernel nor the prefill kernel runs.  The
    two halves run as their own plans give the four launches that these two replace,
    which shows the count sees every kernel."""
    b = small_mixed(40)
    dec = [r for r in range(b.batch) if b.qo_lens[r] == 1]
    pre = [r for r in range(b.batch) if b.qo_lens[r] > 1]
    bd, bp = W.sub_batch(b, dec), W.sub_batch(b, pre)
    kv = b.kv_data.cuda()
    db, dd, dp = (runner.DeviceBatch.from_host(x, kv_data=kv) for x in (b, bd, bp))
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    s = torch.cuda.Stream()
    plans, outs = [], []
    with torch.cuda.stream(s):
        for x, kind in ((b, api.PLAN_MIXED), (bd, api.PLAN_DECODE), (bp, api.PLAN_PREFILL)):
            p = runner.make_plan(x, kind)
            runner.plan_batch(p, x, stream=s)
            plans.append(p)
        for x in (db, dd, dp):
            outs.append((torch.empty_like(x.q), torch.empty(x.q.shape[:2], dtype=torch.float32, device="cuda")))
    s.synchronize()

    def run(i, x):
        plans[i].run(x.q, kv, x.kv_indices, x.kv_indptr, x.kv_last_page_len, *outs[i], qo_indptr=x.qo_indptr,
                     stream=s)

    def kinds(nodes):
        return sorted(next((k for k in ("mixed_merge", "mixed_kernel", "prefill_merge", "decode_merge",
                                        "prefill_kernel", "decode_kernel") if k in name), name)
                      for name, _, _ in nodes)

    nodes = kernel_nodes(lambda: run(0, db), s)
    assert kinds(nodes) == ["mixed_kernel", "mixed_merge"], nodes  # both halves' merges in one launch
    assert [g for name, g, _ in nodes if "mixed_kernel" in name] == [(sms, 1, 1)], nodes
    halves = kernel_nodes(lambda: (run(1, dd), run(2, dp)), s)
    assert kinds(halves) == ["decode_kernel", "decode_merge", "prefill_kernel", "prefill_merge"], halves
    # the captured mixed launch still gives the oracle's result when run
    run(0, db)
    s.synchronize()
    assert plans[0].device_error() == 0
    ref_o, ref_lse = oracle.attention_of(b)
    assert_matches_oracle(outs[0][0], outs[0][1], ref_o, ref_lse, b.dtype, "mixed after capture")


@pytest.mark.parametrize("n_decode,n_prefill", [(7, 0), (0, 4)])
def test_mixed_batch_with_one_half(n_decode, n_prefill):
    mixed_vs_oracle(small_mixed(11, n_decode=n_decode, n_prefill=n_prefill), f"{n_decode}+{n_prefill}")


def test_mixed_with_softcap_and_split_decode():
    b = W.mixed_batch(seed=12, n_decode=3, n_prefill=2, decode_lo=30000, decode_hi=40000, qo_lo=100, qo_hi=200,
                      num_qo_heads=8, num_kv_heads=2, poison=True)
    b = W.PagedBatch(**{**b.__dict__, "logits_cap": 30.0})
    plan = mixed_vs_oracle(b, "mixed cap, long decodes")
    assert plan.info().num_merge > 0


def test_mixed_full_size():
    """60 decode requests (kv U[512, 4096]) and 4 prompt chunks (qo U[256, 2048] after
    a prefix U[0, 1024]), 32 q / 8 kv heads: every row of both halves."""
    mixed_vs_oracle(W.mixed_batch(seed=1007, poison=True), "mixed full size")


def test_mixed_graph_replay_after_replanning():
    """Capture the mixed run once; re-plan a batch with another decode/prefill mix of
    the same total rows (so another SM split, read by the kernel from the device
    tables); replay."""
    a = small_mixed(20, n_decode=10, n_prefill=2)
    total = a.total_q
    bb = W.mixed_batch(seed=21, n_decode=total - 2 * 50, n_prefill=2, decode_lo=1, decode_hi=700, qo_lo=50,
                       qo_hi=50, prefix_lo=0, prefix_hi=200, num_qo_heads=8, num_kv_heads=2, poison=True)
    assert bb.total_q == total
    pool = max(a.num_pages, bb.num_pages)

    def on_pool(b):
        kv = torch.zeros(pool, *b.kv_data.shape[1:], dtype=b.kv_data.dtype)
        kv[: b.num_pages] = b.kv_data
        return W.PagedBatch(**{**b.__dict__, "kv_data": kv})

    a, bb = on_pool(a), on_pool(bb)
    max_b = max(a.batch, bb.batch)
    plan = runner.make_plan(a, api.PLAN_MIXED, max_batch=max_b, max_total_q=total,
                            max_kv_pages=max(int(a.kv_indptr[-1]), int(bb.kv_indptr[-1])))
    dev = "cuda"
    q = torch.empty(total, 8, 128, dtype=torch.bfloat16, device=dev)
    kv = torch.empty(pool, *a.kv_data.shape[1:], dtype=torch.bfloat16, device=dev)
    o, lse = torch.empty_like(q), torch.empty(total, 8, dtype=torch.float32, device=dev)
    qo = torch.zeros(max_b + 1, dtype=torch.int32, device=dev)
    ip = torch.zeros(max_b + 1, dtype=torch.int32, device=dev)
    ix = torch.zeros(plan.limits.max_kv_pages, dtype=torch.int32, device=dev)
    last = torch.zeros(max_b, dtype=torch.int32, device=dev)

    def load(b):
        q.copy_(b.q)
        kv.copy_(b.kv_data)
        qo[: b.batch + 1].copy_(b.qo_indptr)
        ip[: b.batch + 1].copy_(b.kv_indptr)
        ix[: b.kv_indices.numel()].copy_(b.kv_indices)
        last[: b.batch].copy_(b.kv_last_page_len)

    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        load(a)
        runner.plan_batch(plan, a, stream=s)
        plan.run(q, kv, ix, ip, last, o, lse, qo_indptr=qo, stream=s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        plan.run(q, kv, ix, ip, last, o, lse, qo_indptr=qo, stream=s)
    for b in (bb, a):
        with torch.cuda.stream(s):
            load(b)
            runner.plan_batch(plan, b, stream=s)
            g.replay()
        s.synchronize()
        ref_o, ref_lse = oracle.attention_of(b)
        assert_matches_oracle(o, lse, ref_o, ref_lse, torch.bfloat16, "mixed graph replay")
    assert plan.device_error() == 0


def test_cascade_as_one_mixed_launch_full_size():
    """The 64-request soft-capped cascade as one mixed launch (prefix row block on the
    prefill kernel beside the suffixes on the decode kernel) + merge_state."""
    cb = W.cascade_decode(seed=1004, poison=True)
    m = W.cascade_as_mixed(cb.prefix, cb.suffix)
    db = runner.DeviceBatch.from_host(m)
    plan = runner.make_plan(m, api.PLAN_MIXED)
    runner.plan_batch(plan, m)
    o, lse = runner.cascade_mixed(db, plan)
    torch.cuda.synchronize()
    assert plan.device_error() == 0
    info = plan.info()
    assert info.prefill_ctas >= 1 and info.decode_ctas >= 1
    ref_o, ref_lse = oracle.attention_of(cb.full)
    assert_matches_oracle(o, lse, ref_o, ref_lse, torch.bfloat16, "cascade as mixed")
