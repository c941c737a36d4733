"""The seeded synthetic workloads have the shapes, sizes and value distributions of the
five measured configurations: tiny decode, the Llama-3-8B-shaped decode batch, the
skewed long-context decode, the ragged causal prefill and the soft-capped cascade."""
import math

import pytest
import torch

from paged_kv_cache_bsr_gb300 import workloads as W


def check_page_table(b, pool_pages=None):
    """Each request's pages: ceil(kv_len / P) entries of a permuted pool, no page used twice,
    last_page_len the tokens of the final page; the pool as large as stated."""
    P = b.page_size
    counts = [(n + P - 1) // P for n in b.kv_lens]
    assert (b.kv_indptr[1:] - b.kv_indptr[:-1]).tolist() == counts
    last = [n - (c - 1) * P if c else 0 for n, c in zip(b.kv_lens, counts)]
    assert b.kv_last_page_len.tolist() == last
    ids = b.kv_indices.tolist()
    assert len(set(ids)) == len(ids) and all(0 <= i < b.num_pages for i in ids)
    assert b.num_pages == (sum(counts) if pool_pages is None else pool_pages)
    assert ids != sorted(ids)                     # drawn from a permutation, not in order
    assert b.kv_data.shape == (b.num_pages, 2, b.num_kv_heads, P, b.head_dim)
    assert b.q.shape == (b.total_q, b.num_qo_heads, b.head_dim)


def check_normal(t):
    """Values drawn from N(0, 1) and rounded to the storage type."""
    x = t.float().flatten()[:1 << 20]
    assert abs(x.mean().item()) < 0.01 and abs(x.std().item() - 1) < 0.01


def test_tiny_decode():
    b = W.tiny_decode(seed=1000)
    assert (b.batch, b.num_qo_heads, b.num_kv_heads, b.head_dim, b.page_size) == (4, 8, 2, 64, 16)
    assert b.dtype == torch.float16 and b.qo_lens == [1] * 4 and b.sm_scale == pytest.approx(1 / 8)
    assert all(1 <= n <= 256 for n in b.kv_lens)
    check_page_table(b, pool_pages=64)
    check_normal(b.kv_data)


@pytest.mark.slow
def test_llama3_8b_decode():
    b = W.llama3_decode(seed=1001)
    assert (b.batch, b.num_qo_heads, b.num_kv_heads, b.head_dim, b.page_size) == (64, 32, 8, 128, 16)
    assert b.dtype == torch.bfloat16 and b.qo_lens == [1] * 64
    assert b.sm_scale == pytest.approx(1 / math.sqrt(128))
    assert all(512 <= n <= 4096 for n in b.kv_lens) and max(b.kv_lens) - min(b.kv_lens) > 2000
    check_page_table(b)                             # pool = exactly the pages used
    assert b.kv_bytes() == sum(b.kv_lens) * 2 * 8 * 128 * 2
    check_normal(b.q)
    check_normal(b.kv_data)


@pytest.mark.slow
def test_skewed_long_context_decode():
    b = W.skewed_decode(seed=1002)
    assert (b.batch, b.num_qo_heads, b.num_kv_heads, b.head_dim, b.page_size) == (32, 32, 8, 128, 16)
    assert sorted(b.kv_lens) == [1024] * 31 + [131072]
    check_page_table(b)
    assert sum(b.kv_lens) * 4096 == b.kv_bytes()  # 162816 tokens x 4 KB


def test_ragged_causal_prefill():
    b = W.ragged_prefill(seed=1003)
    assert (b.batch, b.num_qo_heads, b.num_kv_heads, b.head_dim, b.page_size) == (16, 32, 8, 128, 16)
    assert b.causal and b.dtype == torch.bfloat16
    assert all(128 <= q <= 2048 for q in b.qo_lens)
    assert all(0 <= kv - q <= 1024 for q, kv in zip(b.qo_lens, b.kv_lens))
    assert b.qo_indptr.tolist() == [0] + torch.cumsum(torch.tensor(b.qo_lens), 0).tolist()
    check_page_table(b)
    check_normal(b.q)


def test_soft_capped_cascade():
    cb = W.cascade_decode(seed=1004)
    full, prefix, suffix = cb.full, cb.prefix, cb.suffix
    assert full.batch == 64 and full.logits_cap == 30.0 and full.page_size == 16
    assert (full.num_qo_heads, full.num_kv_heads, full.head_dim) == (32, 8, 128)
    # the prefix: 2048 tokens in 128 pages, stored once, first in every request's full view
    assert prefix.batch == 1 and prefix.qo_lens == [64] and prefix.kv_lens == [2048]
    pre_pages = prefix.kv_indices.tolist()
    assert len(pre_pages) == 128
    for r in range(64):
        lo = int(full.kv_indptr[r])
        assert full.kv_indices[lo:lo + 128].tolist() == pre_pages
    # each request's suffix: U[50, 200] tokens in its own pages
    assert all(50 <= n <= 200 for n in suffix.kv_lens)
    assert [f - 2048 for f in full.kv_lens] == suffix.kv_lens
    sfx = suffix.kv_indices.tolist()
    assert len(set(sfx)) == len(sfx) and not set(sfx) & set(pre_pages)
    assert full.num_pages == 128 + len(sfx)          # the pool holds the prefix once
    assert full.kv_data.data_ptr() == prefix.kv_data.data_ptr() == suffix.kv_data.data_ptr()
    check_page_table(suffix, pool_pages=full.num_pages)


def test_group8_decode():
    """64 q / 8 kv heads on the Llama-3-8B decode lengths (the tensor-core decode bench)."""
    b = W.group8_decode(seed=1008)
    assert (b.batch, b.num_qo_heads, b.num_kv_heads, b.head_dim, b.page_size) == (64, 64, 8, 128, 16)
    assert b.dtype == torch.bfloat16 and b.is_decode
    assert min(b.kv_lens) >= 512 and max(b.kv_lens) <= 4096
    assert b.num_pages == int(b.kv_indptr[-1])
    assert sorted(b.kv_indices.tolist()) == list(range(b.num_pages))

