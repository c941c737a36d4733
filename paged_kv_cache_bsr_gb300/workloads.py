"""Seeded synthetic workloads for paged (block-sparse row) KV-cache attention.

This module only builds inputs: page tables drawn from a randomly permuted
physical page pool, and Q/K/V drawn from N(0, 1) and rounded to the storage
dtype. It holds none of the attention arithmetic, so both the CUDA path and
the CPU oracle can be fed from it.

Layouts (FlashInfer pages: "Page-Level Attention", "The Interface"):
  q          [total_q, num_qo_heads, head_dim]            fp16 / bf16
  kv_data    [num_pages, 2, num_kv_heads, page_size, head_dim]   (K = 0, V = 1)
  qo_indptr  [batch + 1] int32   rows of request b are qo_indptr[b]:qo_indptr[b+1]
  kv_indptr  [batch + 1] int32   pages of request b are kv_indices[kv_indptr[b]:kv_indptr[b+1]]
  kv_indices [nnz_pages] int32   physical page ids (the BSR column indices)
  kv_last_page_len [batch] int32 valid slots of each request's last page, in [1, page_size]
                                 (0 only for a request with no pages)

Poisoning: when ``poison`` is set, pages of the pool no request references and
the slots past ``kv_last_page_len`` of each last page are filled with NaN/+inf/-inf,
so any read of them into a result shows up as a non-finite output.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence

import torch

__all__ = [
    "PagedBatch",
    "CascadeBatch",
    "build_page_table",
    "make_paged_batch",
    "tiny_decode",
    "llama3_decode",
    "group8_decode",
    "skewed_decode",
    "ragged_prefill",
    "cascade_decode",
    "MultiLevelBatch",
    "parallel_generation",
    "new_kv_rows",
    "pack_mask",
    "TreeBatch",
    "tree_verify",
    "mixed_batch",
    "sub_batch",
    "cascade_as_mixed",
    "levels_as_mixed",
    "WORKLOADS",
]


@dataclasses.dataclass
class PagedBatch:
    """One batch of requests over one paged KV pool (host tensors)."""

    page_size: int
    num_qo_heads: int
    num_kv_heads: int
    head_dim: int
    dtype: torch.dtype
    q: torch.Tensor
    kv_data: torch.Tensor
    qo_indptr: torch.Tensor
    kv_indptr: torch.Tensor
    kv_indices: torch.Tensor
    kv_last_page_len: torch.Tensor
    qo_lens: List[int]
    kv_lens: List[int]
    sm_scale: float
    logits_cap: float = 0.0
    causal: bool = False
    name: str = ""

    @property
    def batch(self) -> int:
        return len(self.kv_lens)

    @property
    def num_pages(self) -> int:
        return int(self.kv_data.shape[0])

    @property
    def total_q(self) -> int:
        return int(self.q.shape[0])

    @property
    def is_decode(self) -> bool:
        return all(n == 1 for n in self.qo_lens)

    def kv_bytes(self) -> int:
        """Bytes of K and V a decode pass must read: every valid token once per kv head."""
        elem = self.kv_data.element_size()
        return sum(self.kv_lens) * 2 * self.num_kv_heads * self.head_dim * elem


@dataclasses.dataclass
class CascadeBatch:
    """A shared-prefix batch seen three ways over the same pool (no data moves).

    ``full``   : every request's page list = shared prefix pages + its own suffix pages.
    ``prefix`` : one row block holding all requests' queries against the prefix pages.
    ``suffix`` : each request against its own suffix pages only.
    """

    full: PagedBatch
    prefix: PagedBatch
    suffix: PagedBatch
    prefix_len: int
    suffix_lens: List[int]


@dataclasses.dataclass
class MultiLevelBatch:
    """A prefix tree of KV over one pool, seen per level (no data moves).

    ``full``   : each request's page list = the pages of every level on its path.
    ``levels`` : level l groups the requests into consecutive row blocks (its nodes);
                 node n of level l attends, as one block of rows, to that node's own
                 pages.  Every level covers every request row exactly once, so the
                 merge of all levels' states is the full attention.
    """

    full: PagedBatch
    levels: List[PagedBatch]
    level_names: List[str]


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def _randn(shape, gen: torch.Generator, dtype: torch.dtype) -> torch.Tensor:
    return torch.randn(*shape, generator=gen, dtype=torch.float32).to(dtype)


def build_page_table(kv_lens: Sequence[int], page_size: int, perm: torch.Tensor):
    """Assign each request ceil(kv_len / page_size) pages taken in order from ``perm``.

    Returns (kv_indptr, kv_indices, kv_last_page_len, pages_used).
    """
    counts = [(int(n) + page_size - 1) // page_size for n in kv_lens]
    indptr = [0]
    for c in counts:
        indptr.append(indptr[-1] + c)
    used = indptr[-1]
    if used > perm.numel():
        raise ValueError(f"pool of {perm.numel()} pages cannot hold {used} pages")
    indices = perm[:used].to(torch.int32).clone()
    last = [int(n) - (c - 1) * page_size if c > 0 else 0 for n, c in zip(kv_lens, counts)]
    return (
        torch.tensor(indptr, dtype=torch.int32),
        indices,
        torch.tensor(last, dtype=torch.int32),
        used,
    )


def _poison_(kv_data: torch.Tensor, kv_indices: torch.Tensor, kv_indptr: torch.Tensor,
             kv_last: torch.Tensor, page_size: int) -> None:
    num_pages = kv_data.shape[0]
    referenced = torch.zeros(num_pages, dtype=torch.bool)
    referenced[kv_indices.long()] = True
    pattern = torch.tensor([float("nan"), float("inf"), float("-inf")], dtype=torch.float32)
    unref = (~referenced).nonzero().flatten()
    if unref.numel():
        flat = kv_data[unref].reshape(unref.numel(), -1)
        idx = torch.arange(flat.shape[1]) % 3
        flat[:] = pattern[idx].to(kv_data.dtype)
        kv_data[unref] = flat.reshape(kv_data[unref].shape)
    for b in range(kv_last.numel()):
        n = int(kv_indptr[b + 1] - kv_indptr[b])
        last = int(kv_last[b])
        if n == 0 or last >= page_size:
            continue
        page = int(kv_indices[int(kv_indptr[b + 1]) - 1])
        kv_data[page, :, :, last:, :] = float("nan")


def make_paged_batch(
    *,
    qo_lens: Sequence[int],
    kv_lens: Sequence[int],
    num_qo_heads: int,
    num_kv_heads: int,
    head_dim: int,
    page_size: int,
    dtype: torch.dtype,
    seed: int,
    pool_pages: Optional[int] = None,
    causal: bool = False,
    logits_cap: float = 0.0,
    sm_scale: Optional[float] = None,
    poison: bool = False,
    identity_pages: bool = False,
    name: str = "",
) -> PagedBatch:
    """Draw one batch: a random page permutation of the pool, then Q, K, V ~ N(0, 1)."""
    gen = _gen(seed)
    need = sum((int(n) + page_size - 1) // page_size for n in kv_lens)
    pool = need if pool_pages is None else int(pool_pages)
    pool = max(pool, 1)
    perm = torch.arange(pool, dtype=torch.int64) if identity_pages else torch.randperm(pool, generator=gen)
    kv_indptr, kv_indices, kv_last, _ = build_page_table(kv_lens, page_size, perm)
    qo_indptr = torch.zeros(len(qo_lens) + 1, dtype=torch.int32)
    qo_indptr[1:] = torch.cumsum(torch.tensor(list(qo_lens), dtype=torch.int64), 0).to(torch.int32)
    total_q = int(qo_indptr[-1])
    q = _randn((total_q, num_qo_heads, head_dim), gen, dtype)
    kv = _randn((pool, 2, num_kv_heads, page_size, head_dim), gen, dtype)
    if poison:
        _poison_(kv, kv_indices, kv_indptr, kv_last, page_size)
    return PagedBatch(
        page_size=page_size,
        num_qo_heads=num_qo_heads,
        num_kv_heads=num_kv_heads,
        head_dim=head_dim,
        dtype=dtype,
        q=q,
        kv_data=kv,
        qo_indptr=qo_indptr,
        kv_indptr=kv_indptr,
        kv_indices=kv_indices,
        kv_last_page_len=kv_last,
        qo_lens=[int(x) for x in qo_lens],
        kv_lens=[int(x) for x in kv_lens],
        sm_scale=(1.0 / math.sqrt(head_dim)) if sm_scale is None else float(sm_scale),
        logits_cap=float(logits_cap),
        causal=bool(causal),
        name=name,
    )


def _uniform_ints(lo: int, hi: int, n: int, gen: torch.Generator) -> List[int]:
    return [int(x) for x in torch.randint(lo, hi + 1, (n,), generator=gen)]


def zipf_lengths(n: int, s: float, lo: int, hi: int, seed: int) -> List[int]:
    """n lengths from a Zipf law on [lo, hi], P(len = k) proportional to k^-s: the
    heavy-tailed request mix the runtime scheduler is built to balance (greptalks
    summary, "Runtime Scheduler for Dynamic Problem Shapes")."""
    gen = _gen(seed)
    w = torch.arange(lo, hi + 1, dtype=torch.float64).pow(-float(s))
    return [lo + int(i) for i in torch.multinomial(w, n, replacement=True, generator=gen)]


def tiny_decode(seed: int = 1000, poison: bool = False) -> PagedBatch:
    """Tiny paged decode: batch 4, 8 q / 2 kv heads, head_dim 64, page 16, fp16,
    kv_len ~ U[1, 256], pages drawn from a randomly permuted 64-page pool."""
    gen = _gen(seed)
    kv_lens = _uniform_ints(1, 256, 4, gen)
    return make_paged_batch(qo_lens=[1] * 4, kv_lens=kv_lens, num_qo_heads=8, num_kv_heads=2,
                            head_dim=64, page_size=16, dtype=torch.float16, seed=seed + 1,
                            pool_pages=64, poison=poison, name="tiny_decode")


def llama3_decode(seed: int = 1001, batch: int = 64, poison: bool = False,
                  identity_pages: bool = False, page_size: int = 16) -> PagedBatch:
    """Llama-3-8B-shaped batch decode: 32 q / 8 kv heads, head_dim 128, page 16, bf16,
    kv_len ~ U[512, 4096], pool = exactly the pages used, randomly permuted."""
    gen = _gen(seed)
    kv_lens = _uniform_ints(512, 4096, batch, gen)
    return make_paged_batch(qo_lens=[1] * batch, kv_lens=kv_lens, num_qo_heads=32, num_kv_heads=8,
                            head_dim=128, page_size=page_size, dtype=torch.bfloat16, seed=seed + 1,
                            poison=poison, identity_pages=identity_pages, name="llama3_8b_decode")


def group8_decode(seed: int = 1008, batch: int = 64, poison: bool = False) -> PagedBatch:
    """Batch decode with a group of 8: 64 q / 8 kv heads (the GQA shape of 70B-class
    models), head_dim 128, page 16, bf16, kv_len ~ U[512, 4096] as in the
    Llama-3-8B-shaped batch, pool = exactly the pages used, randomly permuted."""
    gen = _gen(seed)
    kv_lens = _uniform_ints(512, 4096, batch, gen)
    return make_paged_batch(qo_lens=[1] * batch, kv_lens=kv_lens, num_qo_heads=64, num_kv_heads=8,
                            head_dim=128, page_size=16, dtype=torch.bfloat16, seed=seed + 1,
                            poison=poison, name="group8_decode")


def skewed_decode(seed: int = 1002, long_len: int = 131072, short_len: int = 1024,
                  n_short: int = 31, poison: bool = False) -> PagedBatch:
    """Skewed long-context decode: 31 requests of 1024 tokens and one of 131072,
    32 q / 8 kv heads, head_dim 128, page 16, bf16, random page permutation."""
    gen = _gen(seed)
    kv_lens = [short_len] * n_short + [long_len]
    order = torch.randperm(len(kv_lens), generator=gen).tolist()
    kv_lens = [kv_lens[i] for i in order]
    return make_paged_batch(qo_lens=[1] * len(kv_lens), kv_lens=kv_lens, num_qo_heads=32,
                            num_kv_heads=8, head_dim=128, page_size=16, dtype=torch.bfloat16,
                            seed=seed + 1, poison=poison, name="skewed_decode")


def ragged_prefill(seed: int = 1003, batch: int = 16, qo_lo: int = 128, qo_hi: int = 2048,
                   prefix_lo: int = 0, prefix_hi: int = 1024, poison: bool = False,
                   num_qo_heads: int = 32, num_kv_heads: int = 8, page_size: int = 16) -> PagedBatch:
    """Ragged causal batch prefill: qo_len ~ U[128, 2048], kv_len = qo_len + prefix with
    prefix ~ U[0, 1024], 32 q / 8 kv heads, head_dim 128, page 16, bf16."""
    gen = _gen(seed)
    qo_lens = _uniform_ints(qo_lo, qo_hi, batch, gen)
    prefix = _uniform_ints(prefix_lo, prefix_hi, batch, gen)
    kv_lens = [a + b for a, b in zip(qo_lens, prefix)]
    return make_paged_batch(qo_lens=qo_lens, kv_lens=kv_lens, num_qo_heads=num_qo_heads,
                            num_kv_heads=num_kv_heads, head_dim=128, page_size=page_size,
                            dtype=torch.bfloat16, seed=seed + 1, causal=True, poison=poison,
                            name="ragged_causal_prefill")


def cascade_decode(seed: int = 1004, batch: int = 64, prefix_len: int = 2048,
                   suffix_lo: int = 50, suffix_hi: int = 200, logits_cap: float = 30.0,
                   num_qo_heads: int = 32, num_kv_heads: int = 8, head_dim: int = 128,
                   page_size: int = 16, dtype: torch.dtype = torch.bfloat16,
                   poison: bool = False) -> CascadeBatch:
    """Shared-prefix (cascade) decode with logit soft-capping.

    ``batch`` requests share one ``prefix_len``-token prefix stored once in the pool;
    each has a private suffix of U[suffix_lo, suffix_hi] tokens.  The three views
    (full, prefix row block, suffix) index the same ``kv_data``.
    """
    gen = _gen(seed)
    suffix_lens = _uniform_ints(suffix_lo, suffix_hi, batch, gen)
    if prefix_len % page_size:
        raise ValueError("the shared prefix must fill whole pages")
    n_prefix = prefix_len // page_size
    n_suffix = [(s + page_size - 1) // page_size for s in suffix_lens]
    pool = n_prefix + sum(n_suffix)
    perm = torch.randperm(pool, generator=gen).to(torch.int32)
    prefix_pages = perm[:n_prefix]
    off = n_prefix
    suffix_pages = []
    for n in n_suffix:
        suffix_pages.append(perm[off:off + n])
        off += n
    q = _randn((batch, num_qo_heads, head_dim), gen, dtype)
    kv = _randn((pool, 2, num_kv_heads, page_size, head_dim), gen, dtype)
    suf_last = torch.tensor([s - (n - 1) * page_size for s, n in zip(suffix_lens, n_suffix)],
                            dtype=torch.int32)

    def indptr_of(counts):
        t = torch.zeros(len(counts) + 1, dtype=torch.int32)
        t[1:] = torch.cumsum(torch.tensor(counts, dtype=torch.int64), 0).to(torch.int32)
        return t

    full_indices = torch.cat([torch.cat([prefix_pages, sp]) for sp in suffix_pages])
    full_indptr = indptr_of([n_prefix + n for n in n_suffix])
    suf_indices = torch.cat(suffix_pages)
    suf_indptr = indptr_of(n_suffix)
    if poison:
        _poison_(kv, full_indices, full_indptr, suf_last, page_size)
    scale = 1.0 / math.sqrt(head_dim)
    common = dict(page_size=page_size, num_qo_heads=num_qo_heads, num_kv_heads=num_kv_heads,
                  head_dim=head_dim, dtype=dtype, kv_data=kv, sm_scale=scale, logits_cap=logits_cap)
    full = PagedBatch(q=q, qo_indptr=indptr_of([1] * batch), kv_indptr=full_indptr,
                      kv_indices=full_indices, kv_last_page_len=suf_last.clone(),
                      qo_lens=[1] * batch, kv_lens=[prefix_len + s for s in suffix_lens],
                      causal=False, name="cascade_full", **common)
    prefix = PagedBatch(q=q, qo_indptr=torch.tensor([0, batch], dtype=torch.int32),
                        kv_indptr=torch.tensor([0, n_prefix], dtype=torch.int32),
                        kv_indices=prefix_pages.clone(),
                        kv_last_page_len=torch.tensor([page_size], dtype=torch.int32),
                        qo_lens=[batch], kv_lens=[prefix_len], causal=False,
                        name="cascade_prefix", **common)
    suffix = PagedBatch(q=q, qo_indptr=indptr_of([1] * batch), kv_indptr=suf_indptr,
                        kv_indices=suf_indices, kv_last_page_len=suf_last.clone(),
                        qo_lens=[1] * batch, kv_lens=list(suffix_lens), causal=False,
                        name="cascade_suffix", **common)
    return CascadeBatch(full=full, prefix=prefix, suffix=suffix, prefix_len=prefix_len,
                        suffix_lens=list(suffix_lens))


def parallel_generation(seed: int = 1005, num_prompts: int = 8, samples: int = 8,
                        system_len: int = 1024, prompt_lo: int = 512, prompt_hi: int = 2048,
                        gen_lo: int = 50, gen_hi: int = 200, num_qo_heads: int = 32,
                        num_kv_heads: int = 8, head_dim: int = 128, page_size: int = 16,
                        dtype: torch.dtype = torch.bfloat16, logits_cap: float = 0.0,
                        poison: bool = False) -> MultiLevelBatch:
    """Parallel generation over a three-level prefix tree, one decode token per request
    (the parallel-generation scenario of the fdeinterviews summary, composable formats).

    Level 0: a ``system_len``-token system prompt shared by all
    ``num_prompts * samples`` requests.  Level 1: ``num_prompts`` user prompts of
    U[prompt_lo, prompt_hi] tokens (rounded down to whole pages), each shared by the
    ``samples`` requests generated from it.  Level 2: each request's own generated
    tokens, U[gen_lo, gen_hi].  Shared levels fill whole pages, so the full view is a
    plain page table; only a request's last (private) page is partial.
    """
    if system_len % page_size:
        raise ValueError("the shared system prompt must fill whole pages")
    if gen_lo < 1:
        raise ValueError("every request holds at least one generated token")
    gen = _gen(seed)
    batch = num_prompts * samples
    n_sys = system_len // page_size
    n_prompt = [max(1, x // page_size) for x in _uniform_ints(prompt_lo, prompt_hi, num_prompts, gen)]
    gen_lens = _uniform_ints(gen_lo, gen_hi, batch, gen)
    n_gen = [(g + page_size - 1) // page_size for g in gen_lens]
    pool = n_sys + sum(n_prompt) + sum(n_gen)
    perm = torch.randperm(pool, generator=gen).to(torch.int32)
    off = 0

    def take(n):
        nonlocal off
        t = perm[off:off + n]
        off += n
        return t

    sys_pages = take(n_sys)
    prompt_pages = [take(n) for n in n_prompt]
    gen_pages = [take(n) for n in n_gen]
    q = _randn((batch, num_qo_heads, head_dim), gen, dtype)
    kv = _randn((pool, 2, num_kv_heads, page_size, head_dim), gen, dtype)
    gen_last = torch.tensor([g - (n - 1) * page_size for g, n in zip(gen_lens, n_gen)], dtype=torch.int32)

    def indptr_of(counts):
        t = torch.zeros(len(counts) + 1, dtype=torch.int32)
        t[1:] = torch.cumsum(torch.tensor(counts, dtype=torch.int64), 0).to(torch.int32)
        return t

    owner = [r // samples for r in range(batch)]
    full_pages = [torch.cat([sys_pages, prompt_pages[owner[r]], gen_pages[r]]) for r in range(batch)]
    full_indices = torch.cat(full_pages)
    full_indptr = indptr_of([p.numel() for p in full_pages])
    if poison:
        _poison_(kv, full_indices, full_indptr, gen_last, page_size)
    common = dict(page_size=page_size, num_qo_heads=num_qo_heads, num_kv_heads=num_kv_heads,
                  head_dim=head_dim, dtype=dtype, kv_data=kv, sm_scale=1.0 / math.sqrt(head_dim),
                  logits_cap=logits_cap, causal=False)
    full = PagedBatch(q=q, qo_indptr=indptr_of([1] * batch), kv_indptr=full_indptr, kv_indices=full_indices,
                      kv_last_page_len=gen_last.clone(), qo_lens=[1] * batch,
                      kv_lens=[system_len + n_prompt[owner[r]] * page_size + gen_lens[r] for r in range(batch)],
                      name="parallel_generation_full", **common)
    system = PagedBatch(q=q, qo_indptr=torch.tensor([0, batch], dtype=torch.int32),
                        kv_indptr=torch.tensor([0, n_sys], dtype=torch.int32), kv_indices=sys_pages.clone(),
                        kv_last_page_len=torch.tensor([page_size], dtype=torch.int32), qo_lens=[batch],
                        kv_lens=[system_len], name="parallel_generation_system", **common)
    prompts = PagedBatch(q=q, qo_indptr=indptr_of([samples] * num_prompts), kv_indptr=indptr_of(n_prompt),
                         kv_indices=torch.cat(prompt_pages),
                         kv_last_page_len=torch.full((num_prompts,), page_size, dtype=torch.int32),
                         qo_lens=[samples] * num_prompts, kv_lens=[n * page_size for n in n_prompt],
                         name="parallel_generation_prompts", **common)
    own = PagedBatch(q=q, qo_indptr=indptr_of([1] * batch), kv_indptr=indptr_of(n_gen),
                     kv_indices=torch.cat(gen_pages), kv_last_page_len=gen_last.clone(), qo_lens=[1] * batch,
                     kv_lens=list(gen_lens), name="parallel_generation_own", **common)
    return MultiLevelBatch(full=full, levels=[system, prompts, own], level_names=["system", "prompt", "own"])


def new_kv_rows(b: PagedBatch, seed: int = 7) -> "tuple[torch.Tensor, torch.Tensor]":
    """K and V of the new tokens of a batch, one per query row: [total_q, Hkv, d] each,
    N(0, 1) in the batch's dtype.  With the batch's page table (which already counts
    them) and ``qo_indptr`` as the append row pointer, these are the inputs of the
    append stage: request b's qo_len new tokens are the last of its kv_len."""
    gen = _gen(seed)
    shape = (b.total_q, b.num_kv_heads, b.head_dim)
    return _randn(shape, gen, b.dtype), _randn(shape, gen, b.dtype)


def pack_mask(matrices: Sequence) -> torch.Tensor:
    """Pack per-request boolean masks [qo_len_b, kv_len_b] into the custom-mask format:
    row-major, requests back to back from bit 0, least significant bit first in each
    byte, zero-padded to whole 32-bit words.  Returns a uint8 tensor."""
    import numpy as np
    flat = [np.asarray(m, dtype=bool).reshape(-1) for m in matrices]
    bits = np.concatenate(flat) if flat else np.zeros(0, dtype=bool)
    packed = np.packbits(bits, bitorder="little")
    pad = (-packed.size) % 4
    if pad or packed.size == 0:
        packed = np.concatenate([packed, np.zeros(pad if packed.size else 4, dtype=np.uint8)])
    return torch.from_numpy(packed.copy())


@dataclasses.dataclass
class TreeBatch:
    """Tree verification for speculative decoding: each request's draft tree nodes are
    its query rows and its last keys; ``mask`` lets node i see the cached prefix and
    its own ancestors (and itself)."""

    batch: PagedBatch
    mask: torch.Tensor            # packed, see pack_mask
    parents: List[List[int]]      # parents[b][i] < i, -1 for the root
    prefix_lens: List[int]
    matrices: list                # the unpacked boolean masks, [qo_len, kv_len] each


def tree_verify(seed: int = 1006, batch: int = 16, prefix_lo: int = 512, prefix_hi: int = 4096,
                nodes: int = 64, num_qo_heads: int = 32, num_kv_heads: int = 8, head_dim: int = 128,
                page_size: int = 16, dtype: torch.dtype = torch.bfloat16, poison: bool = False) -> TreeBatch:
    """Speculative-decoding tree verification: ``batch`` requests, each with a cached
    prefix of U[prefix_lo, prefix_hi] tokens and a draft tree of ``nodes`` tokens whose
    parent pointers are drawn uniformly among the earlier nodes (node 0 is the root).
    The tree's tokens are the query rows and the request's last ``nodes`` keys."""
    import numpy as np
    gen = _gen(seed)
    prefix = _uniform_ints(prefix_lo, prefix_hi, batch, gen)
    parents, mats = [], []
    for b in range(batch):
        par = [-1] + [int(torch.randint(0, i, (1,), generator=gen)) for i in range(1, nodes)]
        m = np.zeros((nodes, prefix[b] + nodes), dtype=bool)
        m[:, :prefix[b]] = True
        for i in range(nodes):
            j = i
            while j >= 0:
                m[i, prefix[b] + j] = True
                j = par[j]
        parents.append(par)
        mats.append(m)
    pb = make_paged_batch(qo_lens=[nodes] * batch, kv_lens=[p + nodes for p in prefix], num_qo_heads=num_qo_heads,
                          num_kv_heads=num_kv_heads, head_dim=head_dim, page_size=page_size, dtype=dtype,
                          seed=seed + 1, causal=False, poison=poison, name="tree_verify")
    return TreeBatch(batch=pb, mask=pack_mask(mats), parents=parents, prefix_lens=prefix, matrices=mats)


def mixed_batch(seed: int = 1007, n_decode: int = 60, n_prefill: int = 4, decode_lo: int = 512,
                decode_hi: int = 4096, qo_lo: int = 256, qo_hi: int = 2048, prefix_lo: int = 0,
                prefix_hi: int = 1024, num_qo_heads: int = 32, num_kv_heads: int = 8, head_dim: int = 128,
                page_size: int = 16, dtype: torch.dtype = torch.bfloat16, poison: bool = False) -> PagedBatch:
    """One continuous-batching step: ``n_decode`` requests generating one token
    (kv_len ~ U[decode_lo, decode_hi]) and ``n_prefill`` requests taking a prompt chunk
    (qo_len ~ U[qo_lo, qo_hi] after a cached prefix ~ U[prefix_lo, prefix_hi]), in
    random order, causal, 32 q / 8 kv heads, head_dim 128, page 16, bf16."""
    gen = _gen(seed)
    dec = _uniform_ints(decode_lo, decode_hi, n_decode, gen)
    qo = _uniform_ints(qo_lo, qo_hi, n_prefill, gen)
    pre = _uniform_ints(prefix_lo, prefix_hi, n_prefill, gen)
    reqs = [(1, k) for k in dec] + [(q, q + p) for q, p in zip(qo, pre)]
    order = torch.randperm(len(reqs), generator=gen).tolist()
    reqs = [reqs[i] for i in order]
    return make_paged_batch(qo_lens=[r[0] for r in reqs], kv_lens=[r[1] for r in reqs], num_qo_heads=num_qo_heads,
                            num_kv_heads=num_kv_heads, head_dim=head_dim, page_size=page_size, dtype=dtype,
                            seed=seed + 1, causal=True, poison=poison, name="mixed_batch")


def sub_batch(b: PagedBatch, requests: Sequence[int], name: str = "") -> PagedBatch:
    """The listed requests of a batch as a batch of their own over the same pool
    (their query rows copied, page tables sliced; kv_data shared)."""
    reqs = list(requests)
    rows = [torch.arange(int(b.qo_indptr[r]), int(b.qo_indptr[r + 1])) for r in reqs]
    q = b.q[torch.cat(rows)] if rows else b.q[:0]
    pages = [b.kv_indices[int(b.kv_indptr[r]):int(b.kv_indptr[r + 1])] for r in reqs]

    def indptr_of(counts):
        t = torch.zeros(len(counts) + 1, dtype=torch.int32)
        if counts:
            t[1:] = torch.cumsum(torch.tensor(counts, dtype=torch.int64), 0).to(torch.int32)
        return t

    return dataclasses.replace(
        b, q=q, qo_indptr=indptr_of([b.qo_lens[r] for r in reqs]),
        kv_indptr=indptr_of([p.numel() for p in pages]),
        kv_indices=torch.cat(pages) if pages else b.kv_indices[:0],
        kv_last_page_len=b.kv_last_page_len[reqs] if reqs else b.kv_last_page_len[:0],
        qo_lens=[b.qo_lens[r] for r in reqs], kv_lens=[b.kv_lens[r] for r in reqs], name=name or b.name)


def levels_as_mixed(levels: Sequence[PagedBatch]) -> PagedBatch:
    """One mixed batch holding every level of a prefix tree (or both halves of a
    cascade): the levels' requests one after another, each level's query rows listed
    again (level l's rows are l*R .. l*R + R - 1 for R request rows), so every level's
    partial states land in their own output rows, ready for merge_state.  Multi-row
    nodes go to the prefill kernel and single-row ones to the decode kernel."""
    R = levels[0].total_q
    qo_lens, kv_lens, qo_parts, kv_ptr, idx, last = [], [], [0], [0], [], []
    for lv in levels:
        if lv.total_q != R:
            raise ValueError("every level must cover the same request rows")
        qo_lens += list(lv.qo_lens)
        kv_lens += list(lv.kv_lens)
        base_q, base_p = qo_parts[-1], kv_ptr[-1]
        qo_parts += [base_q + int(x) for x in lv.qo_indptr[1:]]
        kv_ptr += [base_p + int(x) for x in lv.kv_indptr[1:]]
        idx.append(lv.kv_indices)
        last.append(lv.kv_last_page_len)
    return dataclasses.replace(
        levels[-1], q=torch.cat([lv.q for lv in levels]), qo_indptr=torch.tensor(qo_parts, dtype=torch.int32),
        kv_indptr=torch.tensor(kv_ptr, dtype=torch.int32), kv_indices=torch.cat(idx),
        kv_last_page_len=torch.cat(last), qo_lens=qo_lens, kv_lens=kv_lens, causal=False, name="levels_mixed")


def cascade_as_mixed(prefix: PagedBatch, suffix: PagedBatch) -> PagedBatch:
    """Both halves of a cascade as one mixed batch: request 0 is the prefix row block
    (rows 0..B-1), requests 1..B the suffixes (rows B..2B-1); see levels_as_mixed."""
    return levels_as_mixed([prefix, suffix])


WORKLOADS = {
    "tiny_decode": tiny_decode,
    "llama3_8b_decode": llama3_decode,
    "skewed_decode": skewed_decode,
    "ragged_causal_prefill": ragged_prefill,
    "cascade_softcap_decode": cascade_decode,
    "parallel_generation": parallel_generation,
    "tree_verify": tree_verify,
    "mixed_batch": mixed_batch,
}
