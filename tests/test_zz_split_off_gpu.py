"""GPU parity of batch decode with split-KV turned off (pkv_plan_set_split_kv).

Each (request, kv head) page list goes whole to one worker, longest first onto
the least-loaded worker, with no partial states and no merge.  These cases run
through the C ABI and compare with the fp64 oracle element by element.  The file
is named to be collected after the other GPU tests.
"""
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


def decode_vs_oracle(b, what):
    db = runner.DeviceBatch.from_host(b)
    plan = runner.make_plan(b, api.PLAN_DECODE, split_kv=False)
    runner.plan_batch(plan, b)
    o, lse = runner.decode(db, plan)
    torch.cuda.synchronize()
    assert plan.device_error() == 0
    ref_o, ref_lse = oracle.attention_of(b)
    assert_matches_oracle(o, lse, ref_o, ref_lse, b.dtype, what)
    return plan


def test_tiny_and_edge_decode_with_split_off():
    """Split-KV off: every (request, kv head) page list whole on one worker, with no
    partial states, gives the oracle's results (empty and one-token requests too)."""
    for b, what in ((W.tiny_decode(seed=1000, poison=True), "tiny, split off"),
                    (W.make_paged_batch(qo_lens=[1] * 5, kv_lens=[33, 0, 257, 1000, 1], num_qo_heads=8,
                                        num_kv_heads=2, head_dim=128, page_size=16, dtype=torch.bfloat16,
                                        seed=77, poison=True, pool_pages=90), "edge, split off")):
        plan = decode_vs_oracle(b, what)
        info = plan.info()
        assert info.num_merge == 0 and info.num_slots == 0 and info.num_work == b.batch * b.num_kv_heads


@pytest.mark.slow
def test_skewed_decode_full_size_with_split_off():
    """The skewed batch with split-KV off: the 131072-token request streams through
    one warp per kv head; results as the oracle's."""
    plan = decode_vs_oracle(W.skewed_decode(seed=1002, poison=True), "skewed, split off")
    info = plan.info()
    assert info.num_merge == 0 and info.num_slots == 0 and info.max_cost == 131072 // 16
