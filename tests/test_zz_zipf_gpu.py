"""GPU parity of batch decode on Zipf-distributed request lengths, the heavy-tailed
mix the pages' runtime scheduler is built to balance: 32 requests of 16 to 32768
tokens (P(len = k) proportional to k^-1.1), 32 q / 8 kv heads, head_dim 128, bf16,
page 16, a permuted and poisoned pool; split-KV on and off.  Every output element
against the fp64 oracle, through the C ABI.  The file is named to be collected
after the main GPU tests."""
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


@pytest.mark.parametrize("split_kv", [True, False])
def test_zipf_decode(split_kv):
    kv = W.zipf_lengths(32, 1.1, 16, 32768, seed=1009)
    b = W.make_paged_batch(qo_lens=[1] * 32, kv_lens=kv, num_qo_heads=32, num_kv_heads=8, head_dim=128,
                           page_size=16, dtype=torch.bfloat16, seed=1010, poison=True, name="zipf_decode")
    db = runner.DeviceBatch.from_host(b)
    plan = runner.make_plan(b, api.PLAN_DECODE, split_kv=split_kv)
    runner.plan_batch(plan, b)
    o, lse = runner.decode(db, plan)
    torch.cuda.synchronize()
    assert plan.device_error() == 0
    ref_o, ref_lse = oracle.attention_of(b)
    assert_matches_oracle(o, lse, ref_o, ref_lse, b.dtype, f"zipf, split {'on' if split_kv else 'off'}")
    info = plan.info()
    assert (info.num_merge > 0) == split_kv
