"""GPU parity of batch decode (split-KV + merge) and merge_state against the fp64 oracle.

Every case runs through the C ABI (libpkvbsr.so) and compares element by
element with the oracle on the same seeded inputs.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_bsr_gb300 import api, runner, workloads as W
from gpu_util import LSE_TOL, TOL, assert_matches_oracle, kernel_nodes

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_bsr_gb300 import build
    build.build()
    oracle.build()
    api.load()
    torch.cuda.set_device(0)


def decode_vs_oracle(b, what="", plan_limits=None):
    db = runner.DeviceBatch.from_host(b)
    plan = runner.make_plan(b, api.PLAN_DECODE, **(plan_limits or {}))
    runner.plan_batch(plan, b)
    o, lse = runner.decode(db, plan)
    torch.cuda.synchronize()
    assert plan.device_error() == 0
    ref_o, ref_lse = oracle.attention_of(b)
    assert_matches_oracle(o, lse, ref_o, ref_lse, b.dtype, what)
    return plan, o, lse


# --------------------------------------------------------------------------- the workloads
def test_tiny_decode_fp16_d64():
    """Batch 4, 8/2 heads, d 64, page 16, fp16, 64-page permuted pool, poisoned."""
    decode_vs_oracle(W.tiny_decode(seed=1000, poison=True), "tiny")


@pytest.mark.slow
def test_llama3_8b_decode_full_size():
    """Batch 64, 32/8 heads, d 128, bf16, kv ~ U[512, 4096]: every output element."""
    plan, _, _ = decode_vs_oracle(W.llama3_decode(seed=1001, poison=True), "llama3")
    assert plan.info().num_merge > 0  # the plan split sequences at this size


@pytest.mark.slow
def test_skewed_decode_full_size():
    """31 x 1024 + 1 x 131072 tokens: the long request is split over most workers."""
    plan, _, _ = decode_vs_oracle(W.skewed_decode(seed=1002, poison=True), "skewed")
    info = plan.info()
    assert info.num_merge >= 8 and info.num_slots > 400


@pytest.mark.slow
def test_cascade_full_view_decode_softcap():
    """Shared 2048-token prefix + U[50, 200] suffix, logits soft-capped at 30 (non-cascade view)."""
    cb = W.cascade_decode(seed=1004, poison=True)
    decode_vs_oracle(cb.full, "cascade-full")


@pytest.mark.parametrize("kv_len,whole", [(16, True), (64, False), (128, False), (200, False)])
def test_plan_placements_of_short_lists(kv_len, whole):
    """64 requests x 8 kv heads of equal short lists: one-page lists are kept whole, one list
    per worker; four, eight and thirteen pages are split into runs spread over the CTAs and merged.
    Both placements give the oracle's result (poisoned pool, soft-cap on)."""
    b = W.make_paged_batch(qo_lens=[1] * 64, kv_lens=[kv_len] * 64, num_qo_heads=32, num_kv_heads=8,
                           head_dim=128, page_size=16, dtype=torch.bfloat16, seed=40 + kv_len, poison=True,
                           logits_cap=30.0)
    plan, _, _ = decode_vs_oracle(b, f"64 x {kv_len}")
    info = plan.info()
    assert (info.num_merge == 0) == whole
    if whole:
        assert info.active_workers == 64 * 8
    else:
        # the runs are spread one warp per CTA first: every CTA of the grid gets work
        ctas = {w // 8 for w in plan.work()[:, 0].tolist()}
        assert info.active_workers >= info.grid_ctas and len(ctas) == info.grid_ctas


# --------------------------------------------------------------------------- edge cases
@pytest.mark.parametrize("kv_lens", [[1, 15, 16, 17], [0, 3, 0], [1], [16], [33, 0, 257, 1000]])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_edge_lengths(kv_lens, dtype):
    b = W.make_paged_batch(qo_lens=[1] * len(kv_lens), kv_lens=kv_lens, num_qo_heads=8, num_kv_heads=2,
                           head_dim=128, page_size=16, dtype=dtype, seed=len(kv_lens) + sum(kv_lens),
                           poison=True, pool_pages=sum((n + 15) // 16 for n in kv_lens) + 3)
    decode_vs_oracle(b, f"edge {kv_lens}")


@pytest.mark.parametrize("group", [1, 2, 4, 8])
@pytest.mark.parametrize("head_dim", [64, 128])
@pytest.mark.parametrize("cap", [0.0, 30.0])
def test_group_sizes_head_dims_softcap(group, head_dim, cap):
    hkv = 2
    b = W.make_paged_batch(qo_lens=[1] * 5, kv_lens=[700, 1, 64, 129, 2500], num_qo_heads=hkv * group,
                           num_kv_heads=hkv, head_dim=head_dim, page_size=16, dtype=torch.bfloat16,
                           seed=group * 100 + head_dim, logits_cap=cap, poison=True)
    # a softer scale than 1/sqrt(d) keeps the capped logits spread out
    decode_vs_oracle(b, f"g{group} d{head_dim} cap{cap}")


@pytest.mark.parametrize("page_size", [1, 5, 8, 32, 64])
def test_page_sizes(page_size):
    b = W.make_paged_batch(qo_lens=[1] * 4, kv_lens=[1, 77, 300, 64], num_qo_heads=16, num_kv_heads=4,
                           head_dim=128, page_size=page_size, dtype=torch.float16, seed=page_size, poison=True)
    decode_vs_oracle(b, f"page {page_size}")


@pytest.mark.parametrize("group,head_dim,cap", [(1, 64, 0.0), (2, 128, 0.0), (4, 128, 30.0), (8, 128, 0.0),
                                                (8, 64, 30.0)])
def test_one_row_pages_take_tensor_gathers(group, head_dim, cap):
    """One-row pages (column-vector BSR) reach the tiles as four-row tensor gathers;
    lengths end inside a gather (1, 3), inside a tile (17) and at none (0)."""
    b = W.make_paged_batch(qo_lens=[1] * 6, kv_lens=[1, 3, 17, 0, 250, 1031], num_qo_heads=2 * group,
                           num_kv_heads=2, head_dim=head_dim, page_size=1, dtype=torch.bfloat16,
                           seed=group * 10 + head_dim, logits_cap=cap, poison=True)
    decode_vs_oracle(b, f"one-row pages g{group} d{head_dim} cap{cap}")


def test_one_row_pages_full_size():
    """The Llama-3-8B decode batch on one-row pages, split and merged."""
    decode_vs_oracle(W.llama3_decode(page_size=1, poison=True), "llama3 one-row pages")


@pytest.mark.parametrize("page_size", [16, 1])
def test_page_id_outside_the_pool_sets_the_error_bit(page_size):
    """A device page table that holds an id outside [0, num_pages) (the plan checked a
    host copy): the kernel reads no memory for it (bulk copies fall back to page 0,
    gathers to a row past the tensor), records the page-index error bit, and every
    request without the bad entry still gets its exact result."""
    b = W.make_paged_batch(qo_lens=[1] * 4, kv_lens=[40, 300, 77, 129], num_qo_heads=8, num_kv_heads=2,
                           head_dim=128, page_size=page_size, dtype=torch.bfloat16, seed=31 + page_size, poison=True)
    db = runner.DeviceBatch.from_host(b)
    plan = runner.make_plan(b, api.PLAN_DECODE)
    runner.plan_batch(plan, b)
    bad = int(b.kv_indptr[1])  # the first page of request 1
    db.kv_indices[bad] = b.num_pages + 7
    o, lse = runner.decode(db, plan)
    torch.cuda.synchronize()
    assert plan.device_error() & 1
    keep = [0, 2, 3]
    ref_o, ref_lse = oracle.attention_of(b)
    assert_matches_oracle(o[keep], lse[keep], ref_o[keep], ref_lse[keep], b.dtype, "other requests")


def test_request_split_by_key_range_merges_to_the_whole():
    """One long request split by key range as over three ranks (run here one after the
    other on one GPU): the decode kernel's partial states of the pieces, stacked as the
    all-gather would stack them, folded by merge_state on the device, equal the whole
    request's attention."""
    from paged_kv_cache_bsr_gb300 import shard
    b = W.make_paged_batch(qo_lens=[1], kv_lens=[30011], num_qo_heads=32, num_kv_heads=8, head_dim=128,
                           page_size=16, dtype=torch.bfloat16, seed=13, logits_cap=30.0, poison=True)
    kv = b.kv_data.cuda()
    os_, ls = [], []
    for piece in shard.split_sequence(b, 0, 3):
        o, lse = runner.decode(runner.DeviceBatch.from_host(piece, kv_data=kv))
        os_.append(o)
        ls.append(lse)
    o, lse = shard.merge_gathered(torch.stack(os_), torch.stack(ls))
    torch.cuda.synchronize()
    ref_o, ref_lse = oracle.attention_of(b)
    assert_matches_oracle(o, lse, ref_o, ref_lse, b.dtype, "key-range split merged")


def test_long_single_request_is_split_and_merged():
    b = W.make_paged_batch(qo_lens=[1], kv_lens=[60000], num_qo_heads=8, num_kv_heads=2, head_dim=128,
                           page_size=16, dtype=torch.bfloat16, seed=5, poison=True)
    plan, _, _ = decode_vs_oracle(b, "long")
    info = plan.info()
    assert info.num_merge == 2 and info.num_slots >= 2 * 100


def test_large_logits_stay_finite():
    """Scores of several hundred (q scaled up): the online softmax must not overflow."""
    b = W.make_paged_batch(qo_lens=[1] * 3, kv_lens=[500, 2000, 33], num_qo_heads=8, num_kv_heads=2,
                           head_dim=128, page_size=16, dtype=torch.bfloat16, seed=9, sm_scale=2.0)
    decode_vs_oracle(b, "large logits")


# --------------------------------------------------------------------------- invariants
def test_page_permutation_is_bit_exact():
    """Only the index arrays differ: the same logical KV through another physical layout."""
    b = W.llama3_decode(seed=77, batch=8)
    db = runner.DeviceBatch.from_host(b)
    plan = runner.make_plan(b, api.PLAN_DECODE)
    runner.plan_batch(plan, b)
    o1, l1 = runner.decode(db, plan)
    perm = torch.randperm(b.num_pages, generator=torch.Generator().manual_seed(3))
    kv2 = torch.empty_like(b.kv_data)
    kv2[perm] = b.kv_data
    b2 = W.PagedBatch(**{**b.__dict__, "kv_data": kv2, "kv_indices": perm[b.kv_indices.long()].to(torch.int32)})
    db2 = runner.DeviceBatch.from_host(b2)
    runner.plan_batch(plan, b2)
    o2, l2 = runner.decode(db2, plan)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_cuda_graph_replay_after_replanning():
    """Capture plan-independent run calls once; re-plan another batch into the same
    workspace and buffers; replaying the graph gives that batch's result."""
    hq, hkv, d, P = 16, 4, 128, 16
    pool = 800
    gen = torch.Generator().manual_seed(11)
    kv = torch.randn(pool, 2, hkv, P, d, generator=gen).to(torch.bfloat16)
    max_b, max_pages = 6, pool

    def batch_with(kv_lens, seed):
        g = torch.Generator().manual_seed(seed)
        perm = torch.randperm(pool, generator=g)
        ip, ix, last, _ = W.build_page_table(kv_lens, P, perm)
        q = torch.randn(len(kv_lens), hq, d, generator=g).to(torch.bfloat16)
        return W.PagedBatch(page_size=P, num_qo_heads=hq, num_kv_heads=hkv, head_dim=d, dtype=torch.bfloat16,
                            q=q, kv_data=kv, qo_indptr=torch.arange(len(kv_lens) + 1, dtype=torch.int32),
                            kv_indptr=ip, kv_indices=ix, kv_last_page_len=last, qo_lens=[1] * len(kv_lens),
                            kv_lens=list(kv_lens), sm_scale=1 / math.sqrt(d))

    a = batch_with([3000, 17, 900, 4000, 1, 64], 1)
    bb = batch_with([100, 5000, 2222, 1, 16, 3333], 2)
    plan = runner.make_plan(a, api.PLAN_DECODE, max_batch=max_b, max_kv_pages=max_pages)
    dev = "cuda"
    kv_d = kv.to(dev)
    q_buf = torch.empty(max_b, hq, d, dtype=torch.bfloat16, device=dev)
    o_buf = torch.empty_like(q_buf)
    lse_buf = torch.empty(max_b, hq, dtype=torch.float32, device=dev)
    ip_buf = torch.zeros(max_b + 1, dtype=torch.int32, device=dev)
    ix_buf = torch.zeros(max_pages, dtype=torch.int32, device=dev)
    last_buf = torch.zeros(max_b, dtype=torch.int32, device=dev)

    def load(b):
        q_buf.copy_(b.q)
        ip_buf.copy_(b.kv_indptr)
        ix_buf[: b.kv_indices.numel()].copy_(b.kv_indices)
        last_buf.copy_(b.kv_last_page_len)

    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        load(a)
        runner.plan_batch(plan, a, stream=s)
        plan.run(q_buf, kv_d, ix_buf, ip_buf, last_buf, o_buf, lse_buf, stream=s)  # warm-up outside capture
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        plan.run(q_buf, kv_d, ix_buf, ip_buf, last_buf, o_buf, lse_buf, stream=s)
    for b in (a, bb, a):
        with torch.cuda.stream(s):
            load(b)
            runner.plan_batch(plan, b, stream=s)
            g.replay()
        s.synchronize()
        ref_o, ref_lse = oracle.attention_of(b)
        assert_matches_oracle(o_buf, lse_buf, ref_o, ref_lse, torch.bfloat16, "graph replay")
    assert plan.device_error() == 0


# --------------------------------------------------------------------------- group 8 on the tensor cores
@pytest.mark.parametrize("dtype,cap", [(torch.bfloat16, 0.0), (torch.float16, 30.0)])
def test_group8_decode_runs_on_the_tensor_cores(dtype, cap):
    """64 q / 8 kv heads at head_dim 128: the decode plan's run launches the tcgen05
    prefill kernel with one query row per request (and its merge), not the CUDA-core
    decode kernel.  A 60000-token request is cut into key chunks whose partial states
    are merged; an empty request gives 0 and -inf; soft-capped and not."""
    b = W.make_paged_batch(qo_lens=[1] * 6, kv_lens=[60000, 1, 17, 0, 700, 4100], num_qo_heads=64,
                           num_kv_heads=8, head_dim=128, page_size=16, dtype=dtype, seed=88 + int(cap),
                           logits_cap=cap, poison=True)
    db = runner.DeviceBatch.from_host(b)
    plan = runner.make_plan(b, api.PLAN_DECODE)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        runner.plan_batch(plan, b, stream=s)
        o = torch.empty_like(db.q)
        lse = torch.empty(db.q.shape[:2], dtype=torch.float32, device="cuda")
    s.synchronize()

    def run():
        plan.run(db.q, db.kv_data, db.kv_indices, db.kv_indptr, db.kv_last_page_len, o, lse, stream=s)

    names = [n for n, _, _ in kernel_nodes(run, s)]
    assert len(names) == 2 and "prefill_kernel" in names[0] + names[1] and \
        any("prefill_merge" in n for n in names), names
    assert not any("decode_kernel" in n for n in names), names
    run()
    s.synchronize()
    assert plan.device_error() == 0
    assert plan.info().num_merge > 0  # the long request was cut into chunks
    ref_o, ref_lse = oracle.attention_of(b)
    assert_matches_oracle(o, lse, ref_o, ref_lse, dtype, f"group 8 cap {cap}")


@pytest.mark.slow
def test_group8_llama3_lengths_full_size():
    """64 q / 8 kv heads on the Llama-3-8B lengths (batch 64, kv ~ U[512, 4096]),
    through the tensor-core decode path: every output element."""
    ref = W.llama3_decode(seed=1001)
    b = W.make_paged_batch(qo_lens=[1] * 64, kv_lens=list(ref.kv_lens), num_qo_heads=64, num_kv_heads=8,
                           head_dim=128, page_size=16, dtype=torch.bfloat16, seed=1011, poison=True)
    decode_vs_oracle(b, "group 8 llama3 lengths")


# --------------------------------------------------------------------------- device-side checks
def test_device_checks_flag_inconsistent_device_arrays():
    b = W.make_paged_batch(qo_lens=[1] * 3, kv_lens=[40, 90, 7], num_qo_heads=8, num_kv_heads=2, head_dim=128,
                           page_size=16, dtype=torch.bfloat16, seed=2)
    db = runner.DeviceBatch.from_host(b)
    plan = runner.make_plan(b, api.PLAN_DECODE)
    runner.plan_batch(plan, b)
    bad_ip = db.kv_indptr.clone()
    bad_ip[1] += 1  # the device indptr no longer matches the plan
    o = torch.empty_like(db.q)
    plan.run(db.q, db.kv_data, db.kv_indices, bad_ip, db.kv_last_page_len, o)
    torch.cuda.synchronize()
    assert plan.device_error(clear=True) & 2
    assert plan.device_error() == 0
    bad_ix = db.kv_indices.clone()
    bad_ix[0] = b.num_pages + 5  # out of the pool: never dereferenced, flagged instead
    plan.run(db.q, db.kv_data, bad_ix, db.kv_indptr, db.kv_last_page_len, o)
    torch.cuda.synchronize()
    assert plan.device_error(clear=True) & 1


# --------------------------------------------------------------------------- merge_state
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
@pytest.mark.parametrize("head_dim", [64, 128])
def test_merge_state_matches_oracle(dtype, head_dim):
    n, h = 333, 8
    gen = torch.Generator().manual_seed(head_dim)
    o_a = torch.randn(n, h, head_dim, generator=gen).to(dtype)
    o_b = torch.randn(n, h, head_dim, generator=gen).to(dtype)
    l_a = (torch.randn(n, h, generator=gen) * 4).float()
    l_b = (torch.randn(n, h, generator=gen) * 4).float()
    l_a[0, :] = -math.inf          # an empty state: contributes nothing
    o_a[0, :] = float("nan")
    l_a[1, :] = -math.inf          # both empty
    l_b[1, :] = -math.inf
    ref_o, ref_l = oracle.merge_states([o_a.double().numpy(), o_b.double().numpy()],
                                       [l_a.double().numpy(), l_b.double().numpy()])
    d = lambda t: t.cuda()
    o_out = torch.empty(n, h, head_dim, dtype=dtype, device="cuda")
    l_out = torch.empty(n, h, dtype=torch.float32, device="cuda")
    api.merge_state(d(o_a), d(l_a), d(o_b), d(l_b), o_out, l_out)
    torch.cuda.synchronize()
    assert_matches_oracle(o_out, l_out, ref_o, ref_l, dtype, "merge_state")
    # in place: the output overwrites state a
    oa, la = d(o_a), d(l_a)
    api.merge_state(oa, la, d(o_b), d(l_b), oa, la)
    torch.cuda.synchronize()
    assert torch.equal(oa, o_out) and torch.equal(la, l_out)


@pytest.mark.parametrize("dtype,head_dim", [(torch.bfloat16, 128), (torch.float16, 64), (torch.float32, 128)])
@pytest.mark.parametrize("n_states", [1, 2, 3, 5])
def test_merge_states_matches_oracle(dtype, head_dim, n_states):
    """n states laid out one after another, merged in one call, against the oracle's
    n-way merge: rows where some states are empty (their o holds NaN and is not
    read), rows where every state is empty (0, -inf), and the merge written in place
    over the last state."""
    n, h = 257, 8
    gen = torch.Generator().manual_seed(head_dim + 10 * n_states)
    o = torch.randn(n_states * n, h, head_dim, generator=gen).to(dtype)
    lse = (torch.randn(n_states * n, h, generator=gen) * 4).float()
    lse[0, :] = -math.inf                # state 0 of row 0 empty
    o[0, :] = float("nan")
    for k in range(n_states):            # row 1 empty in every state
        lse[k * n + 1, :] = -math.inf
    if n_states > 2:
        lse[n + 2, 3] = -math.inf        # state 1 of row 2, head 3 empty
        o[n + 2, 3] = float("nan")
    ref_o, ref_l = oracle.merge_states([o[k * n:(k + 1) * n].double().numpy() for k in range(n_states)],
                                       [lse[k * n:(k + 1) * n].double().numpy() for k in range(n_states)])
    od, ld = o.cuda(), lse.cuda()
    o_out = torch.empty(n, h, head_dim, dtype=dtype, device="cuda")
    l_out = torch.empty(n, h, dtype=torch.float32, device="cuda")
    api.merge_states(od, ld, n_states, o_out, l_out)
    torch.cuda.synchronize()
    assert_matches_oracle(o_out, l_out, ref_o, ref_l, dtype, f"merge_states n={n_states}")
    last = slice((n_states - 1) * n, n_states * n)
    api.merge_states(od, ld, n_states, od[last], ld[last])  # in place over the last state
    torch.cuda.synchronize()
    assert torch.equal(od[last], o_out) and torch.equal(ld[last], l_out)


def test_split_decode_merged_with_merge_state_equals_unsplit():
    """FlashDecoding with the public merge: two halves of every page list, merged."""
    b = W.llama3_decode(seed=5, batch=6)
    counts = (b.kv_indptr[1:] - b.kv_indptr[:-1]).tolist()
    ip, ix, last = b.kv_indptr.tolist(), b.kv_indices.tolist(), b.kv_last_page_len.tolist()
    halves = []
    for part in (0, 1):
        nip, nix, nlast = [0], [], []
        for r, c in enumerate(counts):
            cut = c // 2
            pages = ix[ip[r]:ip[r + 1]]
            sel = pages[:cut] if part == 0 else pages[cut:]
            nix += sel
            nip.append(len(nix))
            nlast.append(b.page_size if part == 0 else last[r])
        t = lambda x: torch.tensor(x, dtype=torch.int32)
        halves.append(W.PagedBatch(**{**b.__dict__, "kv_indptr": t(nip), "kv_indices": t(nix),
                                      "kv_last_page_len": t(nlast)}))
    outs = []
    for hb in halves:
        db = runner.DeviceBatch.from_host(hb)
        outs.append(runner.decode(db))
    (o1, l1), (o2, l2) = outs
    api.merge_state(o1, l1, o2, l2, o1, l1)
    torch.cuda.synchronize()
    ref_o, ref_lse = oracle.attention_of(b)
    assert_matches_oracle(o1, l1, ref_o, ref_lse, torch.bfloat16, "split + merge_state")


@pytest.mark.parametrize("kind", ["decode", "prefill"])
def test_pipelined_plan_steps_without_sync(kind):
    """A pipelined plan re-planned every step with no host sync in between: each step's
    tables are copied on the plan's own stream while the previous step runs; every
    step's output must still match its own batch."""
    batches = []
    for i, kvs in enumerate(([40, 300, 17], [41, 301, 18, 900], [42, 5], [43, 302, 19, 901, 60])):
        qo = [1] * len(kvs) if kind == "decode" else [min(k, 37 + 11 * j) for j, k in enumerate(kvs)]
        batches.append(W.make_paged_batch(qo_lens=qo, kv_lens=kvs, num_qo_heads=8, num_kv_heads=2, head_dim=128,
                                          page_size=16, dtype=torch.bfloat16, seed=70 + i, causal=kind == "prefill",
                                          poison=True))
    max_b = max(b.batch for b in batches)
    max_q = max(b.total_q for b in batches)
    max_p = max(int(b.kv_indptr[-1]) for b in batches)
    k = api.PLAN_DECODE if kind == "decode" else api.PLAN_PREFILL
    plan = runner.make_plan(batches[0], k, pipelined=True, max_batch=max_b, max_total_q=max_q, max_kv_pages=max_p)
    dev = [runner.DeviceBatch.from_host(b) for b in batches]
    outs = []
    for b, d in zip(batches, dev):
        runner.plan_batch(plan, b)
        outs.append(runner.decode(d, plan) if kind == "decode" else runner.prefill(d, plan))
    torch.cuda.synchronize()
    assert plan.device_error() == 0
    for b, (o, lse) in zip(batches, outs):
        ref_o, ref_lse = oracle.attention_of(b)
        assert_matches_oracle(o, lse, ref_o, ref_lse, b.dtype, f"pipelined {kind}")
