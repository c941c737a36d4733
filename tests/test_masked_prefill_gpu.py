"""GPU parity of the tcgen05 prefill with a packed custom mask (tree attention for
speculative decoding, arbitrary block-sparse patterns finer than a page) against
the fp64 oracle, through the C ABI."""
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


def random_masks(seed, qo_lens, kv_lens, causal, p=0.5):
    rng = np.random.default_rng(seed)
    out = []
    for n_q, kv in zip(qo_lens, kv_lens):
        m = rng.random((n_q, kv)) < p
        for i in range(n_q):
            lim = i + kv - n_q if causal else kv - 1
            if lim >= 0:
                m[i, rng.integers(0, lim + 1)] = True
        out.append(m)
    return out


def masked_vs_oracle(b, masks, what, rows=None):
    packed = W.pack_mask(masks)
    db = runner.DeviceBatch.from_host(b)
    plan = runner.make_plan(b, api.PLAN_PREFILL)
    runner.plan_batch(plan, b)
    o, lse = runner.prefill(db, plan, mask=packed.cuda())
    torch.cuda.synchronize()
    assert plan.device_error() == 0
    ref_o, ref_lse = oracle.attention_of(b, rows=rows, mask=packed)
    if rows is not None:
        idx = torch.as_tensor(rows, dtype=torch.long, device=o.device)
        o, lse = o[idx], lse[idx]
    assert_matches_oracle(o, lse, ref_o, ref_lse, b.dtype, what)
    return o, lse, plan


def batch(qo_lens, kv_lens, hq=8, hkv=2, P=16, dtype=torch.bfloat16, causal=False, seed=0, cap=0.0):
    return W.make_paged_batch(qo_lens=qo_lens, kv_lens=kv_lens, num_qo_heads=hq, num_kv_heads=hkv, head_dim=128,
                              page_size=P, dtype=dtype, seed=seed, causal=causal, logits_cap=cap, poison=True)


@pytest.mark.parametrize("group,dtype,causal", [(4, torch.bfloat16, False), (1, torch.float16, False),
                                                (8, torch.bfloat16, True), (2, torch.float16, True)])
def test_random_masks(group, dtype, causal):
    qo, kv = [5, 130, 40, 1], [77, 300, 40, 129]
    b = batch(qo, kv, hq=2 * group, hkv=2, dtype=dtype, causal=causal, seed=group)
    masked_vs_oracle(b, random_masks(group, qo, kv, causal), f"mask g{group} causal {causal}")


def test_mask_with_softcap():
    qo, kv = [70, 3], [200, 90]
    b = batch(qo, kv, seed=9, cap=30.0)
    masked_vs_oracle(b, random_masks(9, qo, kv, False), "mask + cap")


def test_all_ones_mask_equals_the_unmasked_kernel_bit_for_bit():
    qo, kv = [33, 200], [100, 260]
    b = batch(qo, kv, seed=3, causal=True)
    ones = [np.ones((a, c), bool) for a, c in zip(qo, kv)]
    o_m, l_m, plan = masked_vs_oracle(b, ones, "ones")
    o, l = runner.prefill(runner.DeviceBatch.from_host(b), plan)
    torch.cuda.synchronize()
    assert torch.equal(o, o_m) and torch.equal(l, l_m)


def test_lower_triangle_mask_equals_causal():
    qo, kv = [60, 129], [61, 300]
    tri = [np.arange(c)[None, :] <= np.arange(a)[:, None] + (c - a) for a, c in zip(qo, kv)]
    b = batch(qo, kv, seed=4, causal=False)
    o_m, l_m, _ = masked_vs_oracle(b, tri, "triangle")
    # the causal run plans fewer key blocks (its ranges end at the causal limit), so
    # the two runs split differently; both must match the causal oracle
    bc = W.PagedBatch(**{**b.__dict__, "causal": True})
    ref_o, ref_lse = oracle.attention_of(bc)
    assert_matches_oracle(o_m, l_m, ref_o, ref_lse, b.dtype, "triangle vs causal oracle")


def test_fully_masked_rows_and_empty_requests():
    qo, kv = [4, 0, 3], [50, 7, 20]
    masks = [np.ones((4, 50), bool), np.ones((0, 7), bool), np.ones((3, 20), bool)]
    masks[0][2] = False
    masks[2][:, :] = False
    b = batch(qo, kv, seed=5)
    o, lse, _ = masked_vs_oracle(b, masks, "masked rows")
    assert torch.all(o[2] == 0) and torch.all(torch.isneginf(lse[2]))
    assert torch.all(o[4:] == 0) and torch.all(torch.isneginf(lse[4:]))


def test_mask_on_split_key_ranges():
    """Few rows, long keys: the plan cuts the key range into chunks; each chunk reads
    its own part of the mask rows."""
    qo, kv = [32], [9000]
    b = batch(qo, kv, seed=6)
    _, _, plan = masked_vs_oracle(b, random_masks(6, qo, kv, False, p=0.3), "split + mask")
    assert plan.info().num_merge > 0


def test_tree_verify_small():
    tb = W.tree_verify(seed=7, batch=4, prefix_lo=20, prefix_hi=300, nodes=40, num_qo_heads=8, num_kv_heads=2,
                       poison=True)
    masked_vs_oracle(tb.batch, tb.matrices, "tree small")


def test_tree_verify_full_size():
    """16 requests, prefix U[512, 4096], 64-node draft trees, 32 q / 8 kv heads."""
    tb = W.tree_verify(seed=1006, poison=True)
    masked_vs_oracle(tb.batch, tb.matrices, "tree full size")


def test_short_mask_is_rejected():
    qo, kv = [10], [40]
    b = batch(qo, kv, seed=8)
    db = runner.DeviceBatch.from_host(b)
    plan = runner.make_plan(b, api.PLAN_PREFILL)
    runner.plan_batch(plan, b)
    short = torch.zeros(8, dtype=torch.uint8, device="cuda")  # 64 bits < 400
    with pytest.raises(api.PkvError):
        runner.prefill(db, plan, mask=short)


def test_tree_verify_on_single_token_pages():
    """Column-vector BSR (page size 1) with the tree mask: the tree's tokens and the
    prefix are single-token pages scattered over the pool."""
    tb = W.tree_verify(seed=8, batch=3, prefix_lo=50, prefix_hi=400, nodes=24, num_qo_heads=8, num_kv_heads=2,
                       page_size=1, poison=True)
    masked_vs_oracle(tb.batch, tb.matrices, "tree, page 1")
