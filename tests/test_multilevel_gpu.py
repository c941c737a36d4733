"""GPU parity of the multi-level cascade (parallel generation over a prefix tree):
each level's states come from the decode or prefill kernel through the C ABI and are
folded with merge_state; the result must equal full attention over every request's
whole path, computed by the fp64 oracle."""
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


def small_tree(seed=0, dtype=torch.bfloat16, cap=0.0, hq=8, hkv=2, samples=4):
    return W.parallel_generation(seed=seed, num_prompts=5, samples=samples, system_len=160, prompt_lo=40,
                                 prompt_hi=700, gen_lo=1, gen_hi=90, num_qo_heads=hq, num_kv_heads=hkv,
                                 dtype=dtype, logits_cap=cap, poison=True)


def device_levels(mb):
    kv = mb.full.kv_data.cuda()
    return [runner.DeviceBatch.from_host(lv, kv_data=kv) for lv in mb.levels]


def check(mb, o, lse, what):
    torch.cuda.synchronize()
    ref_o, ref_lse = oracle.attention_of(mb.full)
    assert_matches_oracle(o, lse, ref_o, ref_lse, mb.full.dtype, what)


@pytest.mark.parametrize("dtype,cap", [(torch.bfloat16, 0.0), (torch.float16, 0.0), (torch.bfloat16, 30.0)])
def test_three_levels_equal_full_attention(dtype, cap):
    mb = small_tree(seed=3, dtype=dtype, cap=cap)
    o, lse = runner.multi_level_cascade(device_levels(mb))
    check(mb, o, lse, f"3 levels {dtype} cap {cap}")


def test_levels_on_side_streams():
    mb = small_tree(seed=4, hq=16, hkv=2)
    dl = device_levels(mb)
    plans = []
    for lv in mb.levels:
        p = runner.make_plan(lv, runner.level_kind(lv))
        runner.plan_batch(p, lv)
        plans.append(p)
    side = [torch.cuda.Stream(), torch.cuda.Stream()]
    o, lse = runner.multi_level_cascade(dl, plans, side_streams=side)
    check(mb, o, lse, "side streams")
    assert all(p.device_error() == 0 for p in plans)


def test_level_kinds():
    mb = small_tree(seed=5)
    assert [runner.level_kind(lv) for lv in mb.levels] == [api.PLAN_PREFILL, api.PLAN_PREFILL, api.PLAN_DECODE]


def test_node_without_pages_contributes_nothing():
    """A prompt node with no pages (kv_len 0): its rows' state at that level is
    o = 0, lse = -inf, and the merge leaves the other levels' states unchanged."""
    mb = small_tree(seed=6)
    lv = mb.levels[1]
    counts = (lv.kv_indptr[1:] - lv.kv_indptr[:-1]).tolist()
    drop = 2
    keep = [i for i in range(len(counts)) if i != drop]
    pages = torch.cat([lv.kv_indices[int(lv.kv_indptr[i]):int(lv.kv_indptr[i + 1])] for i in keep])
    counts[drop] = 0
    ip = torch.zeros(len(counts) + 1, dtype=torch.int32)
    ip[1:] = torch.cumsum(torch.tensor(counts), 0)
    last = lv.kv_last_page_len.clone()
    last[drop] = 0
    kv_lens = list(lv.kv_lens)
    kv_lens[drop] = 0
    lv2 = W.PagedBatch(**{**lv.__dict__, "kv_indptr": ip, "kv_indices": pages, "kv_last_page_len": last,
                          "kv_lens": kv_lens})
    levels = [mb.levels[0], lv2, mb.levels[2]]
    kv = mb.full.kv_data.cuda()
    o, lse = runner.multi_level_cascade([runner.DeviceBatch.from_host(x, kv_data=kv) for x in levels])
    torch.cuda.synchronize()
    ref_o, ref_lse = oracle.cascade(*levels)
    assert_matches_oracle(o, lse, ref_o, ref_lse, torch.bfloat16, "empty node")
    # the level-1 state of the dropped node alone: zero output, -inf lse
    o1, l1 = runner.prefill(runner.DeviceBatch.from_host(lv2, kv_data=kv))
    torch.cuda.synchronize()
    rows = slice(int(lv2.qo_indptr[drop]), int(lv2.qo_indptr[drop + 1]))
    assert torch.all(o1[rows] == 0) and torch.all(torch.isneginf(l1[rows]))


def test_parallel_generation_full_size():
    """8 prompts x 8 samples = 64 requests, 32 q / 8 kv heads: system prompt 1024 tokens,
    prompts U[512, 2048], generated U[50, 200]."""
    mb = W.parallel_generation(seed=1005, poison=True)
    o, lse = runner.multi_level_cascade(device_levels(mb))
    check(mb, o, lse, "parallel generation")


def test_graph_capture_with_side_streams_replays():
    mb = small_tree(seed=7)
    dl = device_levels(mb)
    s = torch.cuda.Stream()
    side = [torch.cuda.Stream(), torch.cuda.Stream()]
    plans = []
    with torch.cuda.stream(s):
        for lv in mb.levels:
            p = runner.make_plan(lv, runner.level_kind(lv))
            runner.plan_batch(p, lv, stream=s)
            plans.append(p)
        o_e, l_e = runner.multi_level_cascade(dl, plans, stream=s, side_streams=side)
        o_e, l_e = o_e.clone(), l_e.clone()
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        o_g, l_g = runner.multi_level_cascade(dl, plans, stream=s, side_streams=side)
    for _ in range(3):
        o_g.zero_()
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(o_g, o_e) and torch.equal(l_g, l_e)


def test_parallel_generation_as_one_mixed_launch():
    """The full-size 3-level tree as one mixed launch (system prompt and shared prompts
    on the prefill kernel beside the own tokens on the decode kernel) + merge_state."""
    mb = W.parallel_generation(seed=1005, poison=True)
    m = W.levels_as_mixed(mb.levels)
    db = runner.DeviceBatch.from_host(m)
    plan = runner.make_plan(m, api.PLAN_MIXED)
    runner.plan_batch(plan, m)
    o, lse = runner.levels_mixed(db, 3, plan)
    torch.cuda.synchronize()
    assert plan.device_error() == 0
    ref_o, ref_lse = oracle.attention_of(mb.full)
    assert_matches_oracle(o, lse, ref_o, ref_lse, mb.full.dtype, "tree as one mixed launch")
