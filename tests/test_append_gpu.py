"""GPU parity of the append stage (new tokens' K/V written into their pages) with
the fused rotary position embedding of keys and queries, against the fp64 oracle,
through the C ABI; and of attention run on the cache the append wrote."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_bsr_gb300 import api, runner, workloads as W
from gpu_util import assert_matches_oracle

pytestmark = pytest.mark.gpu

# |gpu - oracle| <= ULP_REL * |oracle| + ABS: one unit in the last place of the
# storage format (rounding the fp32 result) plus fp32 rotation error.
ULP_REL = {torch.bfloat16: 2.0 ** -8, torch.float16: 2.0 ** -11}
ABS = 2e-5
DT = {torch.bfloat16: "bf16", torch.float16: "f16"}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_bsr_gb300 import build
    build.build()
    oracle.build()
    api.load()
    torch.cuda.set_device(0)


def batch(qo_lens, kv_lens, hq=8, hkv=2, d=128, P=16, dtype=torch.bfloat16, seed=0, causal=False):
    return W.make_paged_batch(qo_lens=qo_lens, kv_lens=kv_lens, num_qo_heads=hq, num_kv_heads=hkv, head_dim=d,
                              page_size=P, dtype=dtype, seed=seed, causal=causal, poison=True)


def run_append(b, theta, in_place=False, seed=7):
    k_new, v_new = W.new_kv_rows(b, seed=seed)
    db = runner.DeviceBatch.from_host(b)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    q_out = db.q if in_place else None
    q_rot = runner.append_kv(db, k_new.cuda(), v_new.cuda(), theta, q_out=q_out, error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return db, q_rot, k_new, v_new


def check_pool(b, db, k_new, v_new, theta):
    """Written slots against the oracle (keys within a unit in the last place when
    rotated, exact otherwise; values exact); every other byte of the pool unchanged."""
    ref, page, slot = oracle.append_paged_kv(b.kv_data, b.qo_indptr, b.kv_indptr, b.kv_indices,
                                             b.kv_last_page_len, k_new, v_new, rope_theta=theta)
    got_t = db.kv_data.cpu()
    got = oracle.decode16(got_t)
    k_got, k_ref = got[page, 0, :, slot, :], ref[page, 0, :, slot, :]
    if theta > 0:
        bound = ULP_REL[b.dtype] * np.abs(k_ref) + ABS
        excess = np.abs(k_got - k_ref) - bound
        assert excess.max() <= 0, f"rotated keys off by {np.abs(k_got - k_ref).max():.3e}"
    else:
        np.testing.assert_array_equal(k_got, k_ref)
    np.testing.assert_array_equal(got[page, 1, :, slot, :], ref[page, 1, :, slot, :])
    written = np.zeros(b.kv_data.shape, dtype=bool)
    written[page, :, :, slot, :] = True
    raw_before = b.kv_data.view(torch.int16).numpy()
    raw_after = got_t.view(torch.int16).numpy()
    np.testing.assert_array_equal(raw_after[~written], raw_before[~written])
    return page, slot


def check_q(b, q_rot, theta, rows=None):
    _, pos, _, _ = oracle.append_positions(b.qo_indptr, b.kv_indptr, b.kv_last_page_len, b.kv_indices,
                                           b.page_size)
    got_t = q_rot.cpu()
    q = b.q
    if rows is not None:
        rows = np.asarray(rows, dtype=np.int64)
        idx = torch.from_numpy(rows)
        q, pos, got_t = q[idx], pos[rows], got_t[idx]
    ref = oracle.rope(q, pos, theta) if theta > 0 else oracle.decode16(q)
    got = oracle.decode16(got_t)
    if theta > 0:
        excess = np.abs(got - ref) - (ULP_REL[b.dtype] * np.abs(ref) + ABS)
        assert excess.max() <= 0, f"rotated queries off by {np.abs(got - ref).max():.3e}"
    else:
        np.testing.assert_array_equal(got, ref)


@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 128), (torch.float16, 64)])
def test_append_without_rope_is_an_exact_copy(dtype, d):
    b = batch([1, 5, 0, 17, 1], [1, 40, 9, 17, 300], d=d, dtype=dtype, seed=1)
    db, q_rot, k_new, v_new = run_append(b, 0.0)
    check_pool(b, db, k_new, v_new, 0.0)
    check_q(b, q_rot, 0.0)


@pytest.mark.parametrize("dtype,d,hq,hkv", [(torch.bfloat16, 128, 32, 8), (torch.float16, 128, 8, 8),
                                             (torch.bfloat16, 64, 16, 2), (torch.float16, 64, 3, 1)])
def test_append_with_rope(dtype, d, hq, hkv):
    b = batch([1, 33, 2, 100], [7, 33, 64, 130], hq=hq, hkv=hkv, d=d, dtype=dtype, seed=2)
    db, q_rot, k_new, v_new = run_append(b, 10000.0)
    check_pool(b, db, k_new, v_new, 10000.0)
    check_q(b, q_rot, 10000.0)


@pytest.mark.parametrize("P", [1, 8, 64])
def test_append_page_sizes(P):
    b = batch([3, 1, 20], [3, 50, 77], P=P, seed=P)
    db, q_rot, k_new, v_new = run_append(b, 500000.0)
    check_pool(b, db, k_new, v_new, 500000.0)
    check_q(b, q_rot, 500000.0)


def test_queries_rotated_in_place():
    b = batch([4, 9], [20, 9], seed=3)
    db, q_rot, _, _ = run_append(b, 10000.0, in_place=True)
    assert q_rot.data_ptr() == db.q.data_ptr()
    check_q(b, q_rot, 10000.0)


def test_positions_near_128k_keep_their_angles():
    """The new tokens of a 131072-token request turn by angles of ~1.3e5 rad at the
    highest frequency: the argument reduction must keep them accurate."""
    b = batch([8, 1], [131072, 3], hq=4, hkv=1, seed=4)
    db, q_rot, k_new, v_new = run_append(b, 10000.0)
    check_pool(b, db, k_new, v_new, 10000.0)
    check_q(b, q_rot, 10000.0)


def test_bad_page_id_is_flagged_and_not_written():
    b = batch([2, 3], [18, 40], seed=5)
    k_new, v_new = W.new_kv_rows(b)
    db = runner.DeviceBatch.from_host(b)
    bad = db.kv_indices.clone()
    p_last = int(b.kv_indptr[1]) - 1            # request 0's last page: holds both its new tokens
    bad[p_last] = b.num_pages + 5
    db2 = runner.DeviceBatch(host=b, q=db.q, kv_data=db.kv_data, qo_indptr=db.qo_indptr, kv_indptr=db.kv_indptr,
                             kv_indices=bad, kv_last_page_len=db.kv_last_page_len)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    runner.append_kv(db2, k_new.cuda(), v_new.cuda(), 10000.0, error=err)
    torch.cuda.synchronize()
    assert int(err.item()) & 1
    # request 1's tokens are written; request 0's slots and everything else unchanged
    only1 = W.PagedBatch(**{**b.__dict__, "qo_indptr": torch.tensor([0, 0, 3], dtype=torch.int32),
                            "qo_lens": [0, 3], "q": b.q[2:]})
    check_pool(only1, db, k_new[2:], v_new[2:], 10000.0)


def test_more_new_tokens_than_kv_len_is_flagged():
    b = batch([3, 2], [2, 40], seed=6)   # request 0 claims 3 new tokens but holds 2
    k_new, v_new = W.new_kv_rows(b)
    db = runner.DeviceBatch.from_host(b)
    before = db.kv_data.clone()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    runner.append_kv(db, k_new.cuda(), v_new.cuda(), 0.0, error=err)
    torch.cuda.synchronize()
    assert int(err.item()) & 16
    # request 1's two tokens still land
    diff = (db.kv_data.view(torch.int16) != before.view(torch.int16)).permute(0, 3, 1, 2, 4)
    changed = diff.reshape(diff.shape[0], diff.shape[1], -1).any(-1)   # [page, slot]
    assert int(changed.sum()) <= 2
    # none of request 0's slots (its single page) changed
    assert not bool(changed[int(b.kv_indices[0])].any())


def test_empty_append_is_a_no_op():
    b = batch([0, 0], [5, 9], seed=8)
    db = runner.DeviceBatch.from_host(b)
    empty = torch.empty(0, 2, 128, dtype=torch.bfloat16, device="cuda")
    before = db.kv_data.clone()
    runner.append_kv(db, empty, empty, 10000.0, rotate_q=False)
    torch.cuda.synchronize()
    assert torch.equal(before.view(torch.int16), db.kv_data.view(torch.int16))


def rope_pipeline_reference(b, theta, k_new, v_new):
    """Oracle of append -> attention: queries and keys rotated in fp64 and stored in
    the cache's dtype, then attention over the appended pool."""
    kv, page, slot = oracle.append_paged_kv(b.kv_data, b.qo_indptr, b.kv_indptr, b.kv_indices,
                                            b.kv_last_page_len, k_new, v_new, rope_theta=theta)
    _, pos, _, _ = oracle.append_positions(b.qo_indptr, b.kv_indptr, b.kv_last_page_len, b.kv_indices,
                                           b.page_size)
    name = DT[b.dtype]
    kv_st = torch.from_numpy(oracle.encode16(kv, name)).to(b.dtype)
    q_st = torch.from_numpy(oracle.encode16(oracle.rope(b.q, pos, theta), name)).to(b.dtype)
    ref = W.PagedBatch(**{**b.__dict__, "q": q_st, "kv_data": kv_st})
    return oracle.attention_of(ref)


def test_decode_step_with_rope_matches_oracle():
    """One decode step: append the new token of every request (keys turned by RoPE),
    turn the queries, then paged decode on the updated cache."""
    b = batch([1] * 12, list(np.random.default_rng(9).integers(20, 700, size=12)), hq=32, hkv=8, seed=9)
    k_new, v_new = W.new_kv_rows(b, seed=10)
    db = runner.DeviceBatch.from_host(b)
    q_rot = runner.append_kv(db, k_new.cuda(), v_new.cuda(), 500000.0)
    dq = runner.DeviceBatch(host=b, q=q_rot, kv_data=db.kv_data, qo_indptr=db.qo_indptr, kv_indptr=db.kv_indptr,
                            kv_indices=db.kv_indices, kv_last_page_len=db.kv_last_page_len)
    o, lse = runner.decode(dq)
    torch.cuda.synchronize()
    ref_o, ref_lse = rope_pipeline_reference(b, 500000.0, k_new, v_new)
    assert_matches_oracle(o, lse, ref_o, ref_lse, b.dtype, "rope decode step")


def test_causal_prefill_with_rope_matches_oracle():
    b = batch([37, 130, 1], [42, 190, 64], hq=8, hkv=2, seed=11, causal=True)
    k_new, v_new = W.new_kv_rows(b, seed=12)
    db = runner.DeviceBatch.from_host(b)
    q_rot = runner.append_kv(db, k_new.cuda(), v_new.cuda(), 10000.0)
    dq = runner.DeviceBatch(host=b, q=q_rot, kv_data=db.kv_data, qo_indptr=db.qo_indptr, kv_indptr=db.kv_indptr,
                            kv_indices=db.kv_indices, kv_last_page_len=db.kv_last_page_len)
    o, lse = runner.prefill(dq)
    torch.cuda.synchronize()
    ref_o, ref_lse = rope_pipeline_reference(b, 10000.0, k_new, v_new)
    assert_matches_oracle(o, lse, ref_o, ref_lse, b.dtype, "rope causal prefill")


def test_ragged_prefill_append_full_size():
    """The ragged causal prefill batch (16 requests, qo U[128, 2048], 32 q / 8 kv heads):
    all new K/V rows against the oracle, 3000 sampled query rows."""
    b = W.ragged_prefill(seed=1003, poison=True)
    db, q_rot, k_new, v_new = run_append(b, 10000.0)
    check_pool(b, db, k_new, v_new, 10000.0)
    rows = np.sort(np.random.default_rng(0).choice(b.total_q, size=3000, replace=False))
    check_q(b, q_rot, 10000.0, rows=rows)


def test_append_replays_in_a_cuda_graph():
    b = batch([1, 1, 1, 1], [10, 20, 30, 40], seed=13)
    k_new, v_new = W.new_kv_rows(b, seed=14)
    db = runner.DeviceBatch.from_host(b)
    kn, vn = k_new.cuda(), v_new.cuda()
    q_out = torch.empty_like(db.q)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        runner.append_kv(db, kn, vn, 10000.0, q_out=q_out, stream=s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        runner.append_kv(db, kn, vn, 10000.0, q_out=q_out, stream=s)
    db.kv_data.copy_(b.kv_data.cuda())
    q_out.zero_()
    g.replay()
    torch.cuda.synchronize()
    check_pool(b, db, k_new, v_new, 10000.0)
    check_q(b, q_out, 10000.0)
