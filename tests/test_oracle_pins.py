"""Pins for the fp64 oracle, against things other than the oracle itself.

Each test ties one part of the oracle to a fact the FlashInfer pages or plain
mathematics fix: the worked page-table example printed in the guide, a library
attention routine on contiguous K/V, closed forms, and invariants the pages
state (page permutation, split + merge, cascade = full attention).
"""
import json
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import logsumexp

import oracle
from paged_kv_cache_bsr_gb300 import workloads as W

HERE = os.path.dirname(os.path.abspath(__file__))


# --------------------------------------------------------------------------- helpers
def _scatter_to_pool(ks, vs, page_size, num_pages, gen, dtype, poison=True):
    """Build a paged pool from contiguous per-request K/V ([kv_len, Hkv, d] each).

    Pages are taken from a random permutation of the pool; unused pages and the
    tail of each last page hold NaN, so a wrong gather shows up.
    """
    hkv, d = ks[0].shape[1], ks[0].shape[2]
    pool = torch.full((num_pages, 2, hkv, page_size, d), float("nan"), dtype=torch.float64)
    perm = torch.randperm(num_pages, generator=gen).tolist()
    indptr, indices, last = [0], [], []
    nxt = 0
    for k, v in zip(ks, vs):
        n = k.shape[0]
        pages = (n + page_size - 1) // page_size
        for p in range(pages):
            phys = perm[nxt]
            nxt += 1
            indices.append(phys)
            lo, hi = p * page_size, min(n, (p + 1) * page_size)
            pool[phys, 0, :, : hi - lo, :] = k[lo:hi].permute(1, 0, 2)
            pool[phys, 1, :, : hi - lo, :] = v[lo:hi].permute(1, 0, 2)
        indptr.append(len(indices))
        last.append(n - (pages - 1) * page_size if pages else 0)
    if not poison:
        pool = torch.nan_to_num(pool, nan=0.0)
    return (pool.to(dtype), torch.tensor(indptr, dtype=torch.int32),
            torch.tensor(indices, dtype=torch.int32), torch.tensor(last, dtype=torch.int32))


def _sdpa_reference(q, ks, vs, qo_lens, scale, causal, masks=None):
    """torch SDPA in fp64 on contiguous K/V, one request at a time (GQA by repetition);
    ``masks``: optional boolean [qo_len, kv_len] per request, AND-ed with the causal rule."""
    hq = q.shape[1]
    outs = []
    row = 0
    for k, v, n_q in zip(ks, vs, qo_lens):
        g = hq // k.shape[1]
        qq = q[row:row + n_q].double().permute(1, 0, 2)            # [Hq, n_q, d]
        kk = k.double().repeat_interleave(g, dim=1).permute(1, 0, 2)  # [Hq, kv, d]
        vv = v.double().repeat_interleave(g, dim=1).permute(1, 0, 2)
        kv_len = k.shape[0]
        mask = torch.ones(n_q, kv_len, dtype=torch.bool)
        if causal:
            i = torch.arange(n_q)[:, None]
            j = torch.arange(kv_len)[None, :]
            mask = j <= i + (kv_len - n_q)
        if masks is not None:
            mask = mask & torch.as_tensor(masks[len(outs)], dtype=torch.bool)
        o = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, attn_mask=mask, scale=scale)
        outs.append(o.permute(1, 0, 2))
        row += n_q
    return torch.cat(outs).numpy()


def _random_case(seed, qo_lens, kv_lens, hq, hkv, d, page_size, dtype, extra_pages=5):
    gen = torch.Generator().manual_seed(seed)
    ks = [torch.randn(n, hkv, d, generator=gen).to(dtype) for n in kv_lens]
    vs = [torch.randn(n, hkv, d, generator=gen).to(dtype) for n in kv_lens]
    q = torch.randn(sum(qo_lens), hq, d, generator=gen).to(dtype)
    pages = sum((n + page_size - 1) // page_size for n in kv_lens) + extra_pages
    pool, indptr, indices, last = _scatter_to_pool(ks, vs, page_size, pages, gen, dtype)
    qo_indptr = torch.tensor(np.concatenate([[0], np.cumsum(qo_lens)]), dtype=torch.int32)
    return q, ks, vs, pool, qo_indptr, indptr, indices, last


# --------------------------------------------------------------------------- storage decoding
def test_decode16_matches_numpy_and_torch_for_every_code():
    codes = np.arange(1 << 16, dtype=np.uint16)
    f16 = oracle.decode16(codes, dtype="f16")
    ref16 = codes.view(np.float16).astype(np.float64)
    assert np.array_equal(np.isnan(f16), np.isnan(ref16))
    ok = ~np.isnan(ref16)
    assert np.array_equal(f16[ok], ref16[ok])
    bf = oracle.decode16(codes, dtype="bf16")
    refbf = torch.from_numpy(codes.view(np.int16)).view(torch.bfloat16).double().numpy()
    assert np.array_equal(np.isnan(bf), np.isnan(refbf))
    ok = ~np.isnan(refbf)
    assert np.array_equal(bf[ok], refbf[ok])


# --------------------------------------------------------------------------- worked example
def test_worked_example_page_table_and_gather():
    """Guide section 2 'Page-Level Attention': pages [5,12,3,8] and [1,7], page size 64."""
    with open(os.path.join(HERE, "golden", "worked_example_page_table.json")) as f:
        ex = json.load(f)
    P = ex["page_size"]
    kv_lens = [r["token_ranges"][-1][1] + 1 for r in ex["requests"]]
    perm = torch.tensor([p for r in ex["requests"] for p in r["pages"]])
    indptr, indices, last, used = W.build_page_table(kv_lens, P, perm)
    exp = ex["expected"]
    assert indptr.tolist() == exp["kv_indptr"]
    assert indices.tolist() == exp["kv_indices"]
    assert last.tolist() == exp["kv_last_page_len"]
    assert kv_lens == exp["kv_len"]

    # Every element of the pool encodes (page, slot); the gather must return, for
    # token t of a request, the page the example lists for t's range.
    num_pages = 16
    code = (torch.arange(num_pages)[:, None] * P + torch.arange(P)[None, :]).double()
    pool = code[:, None, None, :, None].expand(num_pages, 2, 1, P, 2).to(torch.float16).contiguous()
    for b, req in enumerate(ex["requests"]):
        for kv_sel in (0, 1):
            rows = oracle.gather(pool, indptr, indices, last, b, kv_sel, 0)
            assert rows.shape == (exp["kv_len"][b], 2)
            for page, (lo, hi) in zip(req["pages"], req["token_ranges"]):
                for t in range(lo, hi + 1):
                    assert rows[t, 0] == page * P + (t - lo)


# --------------------------------------------------------------------------- library routine
@pytest.mark.parametrize(
    "qo_lens,kv_lens,hq,hkv,d,P,causal,dtype",
    [
        ([1, 1, 1], [1, 17, 40], 4, 2, 16, 16, False, torch.float16),     # decode, ragged
        ([1, 1], [5, 33], 8, 1, 8, 3, False, torch.bfloat16),             # MQA, odd page
        ([1, 1, 1, 1], [16, 32, 15, 1], 4, 4, 16, 1, False, torch.float16),  # page size 1 (BC=1)
        ([4, 7, 1], [4, 20, 9], 4, 2, 16, 4, True, torch.bfloat16),       # causal, prefix
        ([5, 3], [5, 11], 2, 2, 8, 16, True, torch.float16),              # causal, prefix 0 and 8
        ([6, 2], [13, 2], 4, 1, 8, 5, False, torch.float16),              # non-causal prefill
    ],
)
def test_oracle_matches_sdpa_on_contiguous_kv(qo_lens, kv_lens, hq, hkv, d, P, causal, dtype):
    q, ks, vs, pool, qo_indptr, indptr, indices, last = _random_case(
        7 + sum(kv_lens), qo_lens, kv_lens, hq, hkv, d, P, dtype)
    scale = 1.0 / math.sqrt(d)
    o, lse = oracle.attention(q, pool, qo_indptr, indptr, indices, last, sm_scale=scale, causal=causal)
    ref = _sdpa_reference(q, ks, vs, qo_lens, scale, causal)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    np.testing.assert_allclose(o, ref, rtol=0, atol=1e-12)


def test_lse_matches_scipy_logsumexp_on_known_scores():
    # head_dim 1, q = 1, k_t = x_t, scale 1: the logits are exactly x_t.
    x = np.array([0.5, -1.25, 3.0, 2.0, -0.75, 1.5, 0.0], dtype=np.float64)
    n = x.size
    pool = torch.zeros(n, 2, 1, 1, 1, dtype=torch.float16)
    pool[:, 0, 0, 0, 0] = torch.from_numpy(x).half()
    pool[:, 1, 0, 0, 0] = torch.arange(n).half()
    q = torch.ones(1, 1, 1, dtype=torch.float16)
    idx = torch.arange(n, dtype=torch.int32).flip(0)  # logical token t at physical page n-1-t
    pool = pool.flip(0).contiguous()
    o, lse = oracle.attention(q, pool, torch.tensor([0, 1], dtype=torch.int32),
                              torch.tensor([0, n], dtype=torch.int32), idx,
                              torch.tensor([1], dtype=torch.int32), sm_scale=1.0)
    assert abs(lse[0, 0] - logsumexp(x)) < 1e-13
    w = np.exp(x - logsumexp(x))
    assert abs(o[0, 0, 0] - np.dot(w, np.arange(n))) < 1e-12
    # causal prefill over the same keys: row i of 3 rows sees keys t <= i + n - 3
    q3 = torch.ones(3, 1, 1, dtype=torch.float16)
    o3, l3 = oracle.attention(q3, pool, torch.tensor([0, 3], dtype=torch.int32),
                              torch.tensor([0, n], dtype=torch.int32), idx,
                              torch.tensor([1], dtype=torch.int32), sm_scale=1.0, causal=True)
    for i in range(3):
        assert abs(l3[i, 0] - logsumexp(x[: i + n - 3 + 1])) < 1e-13


# --------------------------------------------------------------------------- soft-capping
def _two_token_cap_case(scale, cap):
    pool = torch.zeros(2, 2, 1, 1, 1, dtype=torch.float16)
    pool[0, 0] = 1.0   # k_0 = 1 -> raw logit = scale
    pool[1, 0] = 0.0   # k_1 = 0 -> raw logit = 0
    pool[0, 1] = 2.0   # v_0
    pool[1, 1] = -1.0  # v_1
    q = torch.ones(1, 1, 1, dtype=torch.float16)
    return oracle.attention(q, pool, torch.tensor([0, 1], dtype=torch.int32),
                            torch.tensor([0, 2], dtype=torch.int32),
                            torch.tensor([0, 1], dtype=torch.int32),
                            torch.tensor([1], dtype=torch.int32), sm_scale=scale, logits_cap=cap)


def test_softcap_applies_after_scaling():
    # scale = cap * atanh(1/2): a capped logit of exactly cap / 2 = 15 (cap = 30),
    # which only holds when the scale is applied before cap * tanh(. / cap).
    cap = 30.0
    o, lse = _two_token_cap_case(cap * math.atanh(0.5), cap)
    expect = math.log(math.exp(15.0) + 1.0)
    assert abs(lse[0, 0] - expect) < 1e-12
    p0 = math.exp(15.0 - expect)
    assert abs(o[0, 0, 0] - (2.0 * p0 - (1 - p0))) < 1e-12


def test_softcap_saturates_to_plus_minus_cap():
    # raw logits of +-1000 become +-cap (tanh(1000/30) = 1 to double precision)
    o, lse = _two_token_cap_case(1000.0, 30.0)
    assert abs(lse[0, 0] - logsumexp([30.0, 0.0])) < 1e-12
    o, lse = _two_token_cap_case(-1000.0, 30.0)
    assert abs(lse[0, 0] - logsumexp([-30.0, 0.0])) < 1e-12


def test_softcap_with_huge_cap_is_plain_attention():
    b = W.tiny_decode(seed=5)
    o0, l0 = oracle.attention_of(b)
    b.logits_cap = 1e9
    o1, l1 = oracle.attention_of(b)
    np.testing.assert_allclose(o1, o0, atol=1e-9)
    np.testing.assert_allclose(l1, l0, atol=1e-9)


# --------------------------------------------------------------------------- closed forms
def test_uniform_v_gives_v():
    b = W.tiny_decode(seed=11)
    c = torch.randn(b.num_kv_heads, b.head_dim).half()
    b.kv_data[:, 1] = c[None, :, None, :]
    o, _ = oracle.attention_of(b)
    g = b.num_qo_heads // b.num_kv_heads
    want = c.double().repeat_interleave(g, 0).numpy()
    for r in range(o.shape[0]):
        np.testing.assert_allclose(o[r], want, rtol=0, atol=1e-13)


def test_zero_query_gives_log_count_and_mean():
    b = W.tiny_decode(seed=12)
    b.q.zero_()
    o, lse = oracle.attention_of(b)
    g = b.num_qo_heads // b.num_kv_heads
    for r, n in enumerate(b.kv_lens):
        np.testing.assert_allclose(lse[r], math.log(n), rtol=0, atol=1e-13)
        for h in range(b.num_qo_heads):
            v = oracle.gather(b.kv_data, b.kv_indptr, b.kv_indices, b.kv_last_page_len, r, 1, h // g)
            np.testing.assert_allclose(o[r, h], v.mean(axis=0), rtol=0, atol=1e-13)


def test_single_token_gives_v0_and_logit():
    b = W.make_paged_batch(qo_lens=[1, 1], kv_lens=[1, 1], num_qo_heads=4, num_kv_heads=2,
                           head_dim=32, page_size=16, dtype=torch.bfloat16, seed=3, poison=True)
    o, lse = oracle.attention_of(b)
    for r in range(2):
        for h in range(4):
            k0 = oracle.gather(b.kv_data, b.kv_indptr, b.kv_indices, b.kv_last_page_len, r, 0, h // 2)[0]
            v0 = oracle.gather(b.kv_data, b.kv_indptr, b.kv_indices, b.kv_last_page_len, r, 1, h // 2)[0]
            qv = b.q[r, h].double().numpy()
            assert abs(lse[r, h] - b.sm_scale * float(np.dot(qv, k0))) < 1e-12
            np.testing.assert_array_equal(o[r, h], v0)


def test_empty_request_gives_zero_and_minus_inf():
    b = W.make_paged_batch(qo_lens=[1, 1], kv_lens=[0, 5], num_qo_heads=2, num_kv_heads=1,
                           head_dim=8, page_size=4, dtype=torch.float16, seed=4)
    o, lse = oracle.attention_of(b)
    assert np.all(o[0] == 0) and np.all(np.isneginf(lse[0]))
    assert np.isfinite(lse[1]).all()


def test_causal_row_sees_exactly_end_aligned_keys():
    # K = 0 makes every visible key equally weighted; V = one-hot of the position
    # shows which keys row i saw: exactly t <= i + (kv_len - qo_len).
    qo, kv, P = 5, 12, 4
    pool = torch.zeros(3, 2, 1, P, 16, dtype=torch.float16)
    for t in range(kv):
        pool[t // P, 1, 0, t % P, t] = 1.0
    q = torch.randn(qo, 1, 16).half()
    o, _ = oracle.attention(q, pool, torch.tensor([0, qo], dtype=torch.int32),
                            torch.tensor([0, 3], dtype=torch.int32),
                            torch.tensor([0, 1, 2], dtype=torch.int32),
                            torch.tensor([P], dtype=torch.int32), sm_scale=1.0, causal=True)
    for i in range(qo):
        seen = np.nonzero(o[i, 0])[0]
        assert seen.tolist() == list(range(i + kv - qo + 1))
        np.testing.assert_allclose(o[i, 0, seen], 1.0 / seen.size, atol=1e-15)


# --------------------------------------------------------------------------- invariants
def test_page_permutation_leaves_output_unchanged():
    b = W.tiny_decode(seed=21)
    o0, l0 = oracle.attention_of(b)
    gen = torch.Generator().manual_seed(99)
    perm = torch.randperm(b.num_pages, generator=gen)
    new_kv = torch.empty_like(b.kv_data)
    new_kv[perm] = b.kv_data
    b.kv_data = new_kv
    b.kv_indices = perm[b.kv_indices.long()].to(torch.int32)
    o1, l1 = oracle.attention_of(b)
    np.testing.assert_array_equal(o1, o0)
    np.testing.assert_array_equal(l1, l0)


def _split_at_page(b, cut_pages):
    """Two page tables over the same pool: the first ``cut_pages[r]`` pages of each
    request (all full) and the rest."""
    ip, ix, last = b.kv_indptr.tolist(), b.kv_indices.tolist(), b.kv_last_page_len.tolist()
    a_ip, a_ix, a_last, c_ip, c_ix, c_last = [0], [], [], [0], [], []
    for r in range(b.batch):
        pages = ix[ip[r]:ip[r + 1]]
        k = cut_pages[r]
        a_ix += pages[:k]
        a_ip.append(len(a_ix))
        a_last.append(b.page_size if k else 0)
        c_ix += pages[k:]
        c_ip.append(len(c_ix))
        c_last.append(last[r] if len(pages) > k else 0)
    t = lambda x: torch.tensor(x, dtype=torch.int32)
    return (t(a_ip), t(a_ix), t(a_last)), (t(c_ip), t(c_ix), t(c_last))


def test_split_then_merge_equals_unsplit():
    b = W.tiny_decode(seed=31)
    o_full, l_full = oracle.attention_of(b)
    counts = (b.kv_indptr[1:] - b.kv_indptr[:-1]).tolist()
    cuts = [c // 2 for c in counts]
    (aip, aix, al), (cip, cix, cl) = _split_at_page(b, cuts)
    oa, la = oracle.attention(b.q, b.kv_data, b.qo_indptr, aip, aix, al, sm_scale=b.sm_scale)
    oc, lc = oracle.attention(b.q, b.kv_data, b.qo_indptr, cip, cix, cl, sm_scale=b.sm_scale)
    om, lm = oracle.merge_states([oa, oc], [la, lc])
    np.testing.assert_allclose(om, o_full, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lm, l_full, rtol=0, atol=1e-12)


def test_three_way_split_merge():
    b = W.make_paged_batch(qo_lens=[1, 1], kv_lens=[100, 47], num_qo_heads=4, num_kv_heads=2,
                           head_dim=16, page_size=8, dtype=torch.bfloat16, seed=8, poison=True)
    o_full, l_full = oracle.attention_of(b)
    (aip, aix, al), (rip, rix, rl) = _split_at_page(b, [3, 2])
    rest = W.PagedBatch(**{**b.__dict__, "kv_indptr": rip, "kv_indices": rix, "kv_last_page_len": rl})
    (bip, bix, bl), (cip, cix, cl) = _split_at_page(rest, [5, 1])
    parts = [oracle.attention(b.q, b.kv_data, b.qo_indptr, ip, ix, ll, sm_scale=b.sm_scale)
             for ip, ix, ll in [(aip, aix, al), (bip, bix, bl), (cip, cix, cl)]]
    om, lm = oracle.merge_states([p[0] for p in parts], [p[1] for p in parts])
    np.testing.assert_allclose(om, o_full, atol=1e-12)
    np.testing.assert_allclose(lm, l_full, atol=1e-12)


def test_cascade_equals_full_attention():
    cb = W.cascade_decode(seed=41, batch=6, prefix_len=64, suffix_lo=3, suffix_hi=40,
                          num_qo_heads=4, num_kv_heads=2, head_dim=16, poison=True)
    o_c, l_c = oracle.cascade(cb.prefix, cb.suffix)
    o_f, l_f = oracle.attention_of(cb.full)
    np.testing.assert_allclose(o_c, o_f, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l_c, l_f, rtol=0, atol=1e-12)


@pytest.mark.parametrize("cap", [0.0, 20.0])
def test_multi_level_cascade_equals_full_attention(cap):
    """Three levels (system prompt, per-group prompts, own tokens): the merge of the
    levels' states is attention over each request's whole path."""
    mb = W.parallel_generation(seed=42, num_prompts=3, samples=4, system_len=32, prompt_lo=8, prompt_hi=60,
                               gen_lo=1, gen_hi=30, num_qo_heads=4, num_kv_heads=2, head_dim=16, page_size=8,
                               logits_cap=cap, poison=True)
    batch = mb.full.batch
    for lv in mb.levels:
        assert int(lv.qo_indptr[-1]) == batch and lv.total_q == batch
    path_len = [0] * batch
    for lv in mb.levels:
        for n in range(lv.batch):
            for r in range(int(lv.qo_indptr[n]), int(lv.qo_indptr[n + 1])):
                path_len[r] += lv.kv_lens[n]
    assert path_len == mb.full.kv_lens
    o_c, l_c = oracle.cascade(*mb.levels)
    o_f, l_f = oracle.attention_of(mb.full)
    assert np.all(np.isfinite(o_f))
    np.testing.assert_allclose(o_c, o_f, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l_c, l_f, rtol=0, atol=1e-12)


# --------------------------------------------------------------------------- merge_state forms
def test_merge_state_closed_forms():
    rng = np.random.default_rng(0)
    o_a, o_b = rng.normal(size=(5, 3, 8)), rng.normal(size=(5, 3, 8))
    l_a = rng.normal(size=(5, 3))
    # an empty state (lse = -inf) is the identity, even with garbage o
    o, l = oracle.merge_states([o_a, np.full_like(o_b, np.nan)], [l_a, np.full_like(l_a, -np.inf)])
    np.testing.assert_array_equal(o, o_a)
    np.testing.assert_array_equal(l, l_a)
    # equal weights: the average, and lse + ln 2
    o, l = oracle.merge_states([o_a, o_b], [l_a, l_a])
    np.testing.assert_allclose(o, (o_a + o_b) / 2, atol=1e-15)
    np.testing.assert_allclose(l, l_a + math.log(2.0), atol=1e-15)
    # two empty states stay empty
    o, l = oracle.merge_states([o_a, o_b], [np.full_like(l_a, -np.inf)] * 2)
    assert np.all(o == 0) and np.all(np.isneginf(l))


# --------------------------------------------------------------------------- input checks
def test_oracle_rejects_malformed_tables():
    b = W.tiny_decode(seed=1)
    bad = b.kv_indices.clone()
    bad[0] = b.num_pages
    with pytest.raises(ValueError):
        oracle.attention(b.q, b.kv_data, b.qo_indptr, b.kv_indptr, bad, b.kv_last_page_len,
                         sm_scale=b.sm_scale)
    last = b.kv_last_page_len.clone()
    last[0] = b.page_size + 1
    with pytest.raises(ValueError):
        oracle.attention(b.q, b.kv_data, b.qo_indptr, b.kv_indptr, b.kv_indices, last,
                         sm_scale=b.sm_scale)


def test_poisoned_pool_never_reaches_outputs():
    b = W.tiny_decode(seed=51, poison=True)
    assert torch.isnan(b.kv_data.float()).any()
    o, lse = oracle.attention_of(b)
    assert np.isfinite(o).all() and np.isfinite(lse).all()


# --------------------------------------------------------------------------- append stage: rope, positions
def test_rope_closed_forms_fix_pairing_sign_and_frequencies():
    """Unit vectors: e_0 turns into (cos m, sin m) on the pair (0, d/2) (frequency 1);
    e_{d/2} into (-sin m, cos m); e_1 turns by m * theta^(-2/d)."""
    d, theta = 8, 10000.0
    m = np.array([0.0, 1.0, 7.0, 1000.0])
    e = np.zeros((4, 3, d))
    e[:, 0, 0] = 1.0
    e[:, 1, d // 2] = 1.0
    e[:, 2, 1] = 1.0
    r = oracle.rope(e, m, theta)
    np.testing.assert_allclose(r[:, 0, 0], np.cos(m), atol=1e-15)
    np.testing.assert_allclose(r[:, 0, d // 2], np.sin(m), atol=1e-15)
    np.testing.assert_allclose(r[:, 1, 0], -np.sin(m), atol=1e-15)
    np.testing.assert_allclose(r[:, 1, d // 2], np.cos(m), atol=1e-15)
    a1 = m * theta ** (-2.0 / d)  # = m / 10
    np.testing.assert_allclose(r[:, 2, 1], np.cos(a1), atol=1e-15)
    np.testing.assert_allclose(r[:, 2, 1 + d // 2], np.sin(a1), atol=1e-15)
    # every other coordinate of the three rows stays zero
    mask = np.ones_like(r, dtype=bool)
    mask[:, 0, [0, d // 2]] = mask[:, 1, [0, d // 2]] = mask[:, 2, [1, 1 + d // 2]] = False
    assert np.all(r[mask] == 0)


def test_rope_is_a_rotation_by_relative_position():
    """Position 0 is the identity, norms of each pair are kept, rotations compose
    (m then n is m + n), and <R(m) q, R(n) k> depends on m - n only."""
    rng = np.random.default_rng(3)
    d, theta = 16, 500.0
    x = rng.normal(size=(6, 2, d))
    np.testing.assert_array_equal(oracle.rope(x, np.zeros(6), theta), x)
    m = rng.integers(0, 5000, size=6).astype(np.float64)
    n = rng.integers(0, 5000, size=6).astype(np.float64)
    rx = oracle.rope(x, m, theta)
    pair_norm = lambda v: v[..., : d // 2] ** 2 + v[..., d // 2:] ** 2
    np.testing.assert_allclose(pair_norm(rx), pair_norm(x), rtol=1e-12)
    np.testing.assert_allclose(oracle.rope(rx, n, theta), oracle.rope(x, m + n, theta), atol=1e-9)
    q, k = rng.normal(size=(6, 1, d)), rng.normal(size=(6, 1, d))
    dots = lambda a, b: np.sum(oracle.rope(q, a, theta) * oracle.rope(k, b, theta), axis=-1)
    np.testing.assert_allclose(dots(m, n), dots(m + 37, n + 37), atol=1e-9)
    assert not np.allclose(dots(m, n), dots(m + 37, n))


def test_append_positions_worked_example():
    """P = 4.  Request 0: 2 pages, last 3 (kv_len 7), 2 new tokens -> positions 5, 6 =
    slots 1, 2 of its second page.  Request 1: 1 page, last 1, 1 new token -> position 0.
    Request 2: 3 full pages, nothing new.  Request 3: 2 pages, last 4, 5 new -> 3..7."""
    kv_indptr = [0, 2, 3, 6, 8]
    kv_indices = [9, 4, 7, 0, 1, 2, 5, 3]
    last = [3, 1, 4, 4]
    append_indptr = [0, 2, 3, 3, 8]
    req, pos, page, slot = oracle.append_positions(append_indptr, kv_indptr, last, kv_indices, 4)
    assert req.tolist() == [0, 0, 1, 3, 3, 3, 3, 3]
    assert pos.tolist() == [5, 6, 0, 3, 4, 5, 6, 7]
    assert page.tolist() == [4, 4, 7, 5, 3, 3, 3, 3]
    assert slot.tolist() == [1, 2, 0, 3, 0, 1, 2, 3]
    with pytest.raises(ValueError):
        oracle.append_positions([0, 9, 9, 9, 9], kv_indptr, last, kv_indices, 4)


def test_append_then_gather_reads_old_tokens_then_new():
    """After the append, the page-table gather of each request returns its earlier
    tokens unchanged followed by the new ones (rotated keys, plain values)."""
    b = W.make_paged_batch(qo_lens=[3, 1, 0, 9], kv_lens=[20, 1, 5, 9], num_qo_heads=4, num_kv_heads=2,
                           head_dim=16, page_size=8, dtype=torch.bfloat16, seed=11, poison=True)
    gen = torch.Generator().manual_seed(12)
    k_new = torch.randn(b.total_q, 2, 16, generator=gen).to(torch.bfloat16)
    v_new = torch.randn(b.total_q, 2, 16, generator=gen).to(torch.bfloat16)
    theta = 10000.0
    kv, page, slot = oracle.append_paged_kv(b.kv_data, b.qo_indptr, b.kv_indptr, b.kv_indices,
                                            b.kv_last_page_len, k_new, v_new, rope_theta=theta)
    req, pos, _, _ = oracle.append_positions(b.qo_indptr, b.kv_indptr, b.kv_last_page_len, b.kv_indices, 8)
    k_rot = oracle.rope(k_new, pos, theta)
    for r in range(b.batch):
        n_new = b.qo_lens[r]
        rows = np.nonzero(req == r)[0]
        for h in range(2):
            before_k = oracle.gather(b.kv_data, b.kv_indptr, b.kv_indices, b.kv_last_page_len, r, 0, h)
            p0, p1 = int(b.kv_indptr[r]), int(b.kv_indptr[r + 1])
            pages = b.kv_indices[p0:p1].long().numpy()
            after_k = kv[pages, 0, h].reshape(-1, 16)[: b.kv_lens[r]]
            after_v = kv[pages, 1, h].reshape(-1, 16)[: b.kv_lens[r]]
            old = b.kv_lens[r] - n_new
            np.testing.assert_array_equal(after_k[:old], before_k[:old])
            np.testing.assert_array_equal(after_k[old:], k_rot[rows, h])
            np.testing.assert_array_equal(after_v[old:], oracle.decode16(v_new)[rows, h])


def test_encode16_rounds_to_nearest_even():
    """Values a 32-bit float holds exactly round like torch's float -> bf16 / fp16
    conversion (round to nearest even); halfway cases go to the even neighbour;
    representable values and the special values come back unchanged."""
    rng = np.random.default_rng(5)
    v = np.concatenate([rng.normal(size=4000) * 10.0 ** rng.integers(-6, 5, size=4000),
                        [0.0, -0.0, np.inf, -np.inf, 65504.0, 65520.0, 1e-8, 6e-8]]).astype(np.float32)
    for name, td in (("bf16", torch.bfloat16), ("f16", torch.float16)):
        ref = torch.from_numpy(v).to(td).double().numpy()
        np.testing.assert_array_equal(oracle.encode16(v.astype(np.float64), name), ref)
    # 1 + 2^-8 is halfway between bf16 neighbours 1 and 1 + 2^-7: ties to even -> 1
    assert oracle.encode16(np.array([1 + 2.0 ** -8]), "bf16")[0] == 1.0
    assert oracle.encode16(np.array([1 + 3 * 2.0 ** -8]), "bf16")[0] == 1 + 2 * 2.0 ** -7
    # fp16: 1 + 2^-11 halfway -> 1, 2049 -> 2048 (ties to even), nan stays nan
    assert oracle.encode16(np.array([1 + 2.0 ** -11, 2049.0]), "f16").tolist() == [1.0, 2048.0]
    assert np.isnan(oracle.encode16(np.array([np.nan]), "bf16")[0])


# --------------------------------------------------------------------------- custom (tree) masks
def _random_masks(rng, qo_lens, kv_lens, causal, p=0.6):
    """Random boolean masks in which every row keeps at least one key the causal rule allows."""
    out = []
    for n_q, kv in zip(qo_lens, kv_lens):
        m = rng.random((n_q, kv)) < p
        for i in range(n_q):
            m[i, i + kv - n_q if causal else rng.integers(0, kv)] = True
        out.append(m)
    return out


@pytest.mark.parametrize("qo_lens,kv_lens,hq,hkv,P,causal", [
    ([3, 5, 1], [7, 40, 9], 4, 2, 4, False),
    ([6, 2], [6, 19], 2, 1, 1, True),       # page size 1 (column vectors), causal AND mask
    ([9], [33], 4, 4, 16, False),
])
def test_custom_mask_matches_sdpa_with_boolean_mask(qo_lens, kv_lens, hq, hkv, P, causal):
    """The packed mask (least significant bit first, requests back to back) selects
    exactly the keys a boolean attn_mask selects in torch SDPA."""
    q, ks, vs, pool, qo_indptr, indptr, indices, last = _random_case(
        31 + sum(kv_lens), qo_lens, kv_lens, hq, hkv, 16, P, torch.bfloat16)
    masks = _random_masks(np.random.default_rng(len(qo_lens)), qo_lens, kv_lens, causal)
    packed = W.pack_mask(masks)
    assert packed.numel() % 4 == 0
    o, lse = oracle.attention(q, pool, qo_indptr, indptr, indices, last, sm_scale=0.25, causal=causal, mask=packed)
    ref = _sdpa_reference(q, ks, vs, qo_lens, 0.25, causal, masks=masks)
    np.testing.assert_allclose(o, ref, rtol=0, atol=1e-12)
    # the mask changes the result: dropping it gives something else
    o2, _ = oracle.attention(q, pool, qo_indptr, indptr, indices, last, sm_scale=0.25, causal=causal)
    assert np.abs(o2 - o).max() > 1e-3


def test_mask_of_ones_is_no_mask_and_lower_triangle_is_causal():
    qo_lens, kv_lens = [4, 7], [10, 7]
    q, ks, vs, pool, qo_indptr, indptr, indices, last = _random_case(5, qo_lens, kv_lens, 4, 2, 16, 4,
                                                                      torch.float16)
    ones = W.pack_mask([np.ones((a, b), bool) for a, b in zip(qo_lens, kv_lens)])
    tri = W.pack_mask([np.arange(b)[None, :] <= np.arange(a)[:, None] + (b - a) for a, b in zip(qo_lens, kv_lens)])
    args = (q, pool, qo_indptr, indptr, indices, last)
    plain = oracle.attention(*args, sm_scale=0.3)
    causal = oracle.attention(*args, sm_scale=0.3, causal=True)
    for got, ref in ((oracle.attention(*args, sm_scale=0.3, mask=ones), plain),
                     (oracle.attention(*args, sm_scale=0.3, mask=tri), causal)):
        np.testing.assert_array_equal(got[0], ref[0])
        np.testing.assert_array_equal(got[1], ref[1])


def test_row_with_every_key_masked_gives_zero_and_minus_inf():
    qo_lens, kv_lens = [3], [9]
    q, ks, vs, pool, qo_indptr, indptr, indices, last = _random_case(6, qo_lens, kv_lens, 2, 2, 8, 4,
                                                                      torch.bfloat16)
    m = np.ones((3, 9), bool)
    m[1] = False
    o, lse = oracle.attention(q, pool, qo_indptr, indptr, indices, last, sm_scale=0.3, mask=W.pack_mask([m]))
    assert np.all(o[1] == 0) and np.all(np.isneginf(lse[1]))
    assert np.all(np.isfinite(lse[[0, 2]]))


def test_pack_mask_bit_order():
    """Bit k of byte j is entry 8 j + k (least significant first); requests follow
    each other with no padding; the buffer is padded to whole 32-bit words."""
    m1 = np.zeros((1, 3), bool)
    m1[0, 1] = True                      # entry 1
    m2 = np.zeros((2, 4), bool)
    m2[1, 2] = True                      # entry 3 + 4 + 2 = 9
    packed = W.pack_mask([m1, m2]).numpy()
    assert packed.tolist() == [0b10, 0b10, 0, 0]
    np.testing.assert_array_equal(np.unpackbits(packed, bitorder="little")[:11],
                                  np.concatenate([m1.reshape(-1), m2.reshape(-1)]))


def test_tree_verify_mask_is_prefix_plus_ancestors():
    """Tree verification: node i sees the whole prefix and exactly its ancestors and
    itself; against SDPA with the same boolean masks; a chain tree is causal."""
    tb = W.tree_verify(seed=3, batch=3, prefix_lo=5, prefix_hi=30, nodes=9, num_qo_heads=4, num_kv_heads=2,
                       head_dim=16, page_size=4, poison=True)
    for par, pre, m in zip(tb.parents, tb.prefix_lens, tb.matrices):
        for i in range(len(par)):
            anc = {i}
            j = par[i]
            while j >= 0:
                anc.add(j)
                j = par[j]
            assert m[i, :pre].all()
            assert set(np.nonzero(m[i, pre:])[0].tolist()) == anc
    o, _ = oracle.attention_of(tb.batch, mask=tb.mask)
    assert np.isfinite(o).all()
    chain = [np.arange(p + 9)[None, :] <= np.arange(9)[:, None] + p for p in tb.prefix_lens]
    oc, lc = oracle.attention_of(tb.batch, mask=W.pack_mask(chain))
    causal = W.PagedBatch(**{**tb.batch.__dict__, "causal": True})
    ocr, lcr = oracle.attention_of(causal)
    np.testing.assert_array_equal(oc, ocr)
    np.testing.assert_array_equal(lc, lcr)


def test_cascade_as_one_mixed_batch_equals_full_attention():
    """The mixed-batch form of a cascade (prefix row block + one-row suffix requests,
    queries listed twice) gives both partial states; their merge is full attention."""
    cb = W.cascade_decode(seed=43, batch=5, prefix_len=48, suffix_lo=2, suffix_hi=30, num_qo_heads=4,
                          num_kv_heads=2, head_dim=16, logits_cap=20.0, poison=True)
    m = W.cascade_as_mixed(cb.prefix, cb.suffix)
    assert m.qo_lens == [5, 1, 1, 1, 1, 1] and m.total_q == 10
    o, lse = oracle.attention_of(m)
    om, lm = oracle.merge_states([o[5:], o[:5]], [lse[5:], lse[:5]])
    of, lf = oracle.attention_of(cb.full)
    np.testing.assert_allclose(om, of, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lm, lf, rtol=0, atol=1e-12)


def test_prefix_tree_as_one_mixed_batch_equals_full_attention():
    """Three levels of a prefix tree as one mixed batch (every level's rows listed
    again): merging the levels' row blocks gives attention over each whole path."""
    mb = W.parallel_generation(seed=44, num_prompts=3, samples=4, system_len=32, prompt_lo=8, prompt_hi=60,
                               gen_lo=1, gen_hi=30, num_qo_heads=4, num_kv_heads=2, head_dim=16, page_size=8,
                               poison=True)
    m = W.levels_as_mixed(mb.levels)
    R = mb.full.batch
    assert m.total_q == 3 * R and m.batch == sum(lv.batch for lv in mb.levels)
    o, lse = oracle.attention_of(m)
    om, lm = oracle.merge_states([o[l * R:(l + 1) * R] for l in range(3)], [lse[l * R:(l + 1) * R] for l in range(3)])
    of, lf = oracle.attention_of(mb.full)
    np.testing.assert_allclose(om, of, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lm, lf, rtol=0, atol=1e-12)
