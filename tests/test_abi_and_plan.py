"""CPU tests of the C ABI: exported symbols, argument validation, and the host
plan's decisions (every page covered once, equal chunks, slot and merge maps).

The plan is created with pkv_plan_create_host (no CUDA call), so these run
without a GPU.
"""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

from paged_kv_cache_bsr_gb300 import api, workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_bsr_gb300 import build
    build.build()
    return api.load()


def _declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(pkv_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_library_exports_every_declared_function(lib):
    declared = _declared_functions()
    assert len(declared) >= 14
    for name in declared:
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"
    assert set(api.EXPORTS) <= set(declared)


def test_status_strings(lib):
    for st in range(-6, 1):
        assert api.status_string(st) not in ("", "unknown status")
    assert api.status_string(-99) == "unknown status"


def test_public_header_is_plain_c(tmp_path):
    """include/pkv_bsr.h compiles as strict C99 and as C++ (a C ABI, no C++ types)."""
    import shutil
    import subprocess
    if not shutil.which("gcc"):
        pytest.skip("no gcc")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    src = tmp_path / "t.c"
    src.write_text('#include "pkv_bsr.h"\nint main(void) { pkv_params p; (void)p; '
                   'return (int)sizeof(pkv_plan_info) > 0 ? 0 : 1; }\n')
    inc = ["-I", os.path.join(root, "include")]
    cuda_inc = "/usr/local/cuda/include"
    if os.path.isdir(cuda_inc):
        inc += ["-I", cuda_inc]
    for cmd in (["gcc", "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror"],
                ["g++", "-std=c++17", "-Wall", "-Werror", "-x", "c++"]):
        r = subprocess.run(cmd + inc + ["-c", str(src), "-o", os.devnull], capture_output=True, text=True)
        assert r.returncode == 0, r.stderr


# --------------------------------------------------------------------------- helpers
def host_plan(b, kind, num_sms=152, **lim):
    params = api.make_params(b.num_qo_heads, b.num_kv_heads, b.head_dim, b.page_size, b.dtype, b.sm_scale,
                             b.logits_cap, b.causal)
    limits = api.Limits(lim.get("max_batch", max(b.batch, 1)), lim.get("max_total_q", max(b.total_q, 1)),
                        lim.get("max_kv_pages", max(int(b.kv_indptr[-1]), 1)))
    h = api.plan_create_host(kind, params, limits, num_sms)
    _, host_bytes = api.plan_workspace_bytes(h)
    ws = torch.empty(host_bytes + 64, dtype=torch.uint8)
    off = (-ws.data_ptr()) % 64
    return h, ws[off:off + host_bytes]


def compute(h, ws, b, **over):
    args = dict(batch=b.batch, qo=b.qo_indptr, ip=b.kv_indptr, ix=b.kv_indices, last=b.kv_last_page_len,
                num_pages=b.num_pages)
    args.update(over)
    api.plan_compute(h, args["batch"], args["qo"], args["ip"], args["ix"], args["last"], args["num_pages"], ws)


def table_batch(kv_lens, qo_lens=None, page_size=16, hq=32, hkv=8, d=128, causal=False):
    """A paged batch with tiny data: only the index arrays matter to the plan."""
    qo_lens = qo_lens or [1] * len(kv_lens)
    b = W.make_paged_batch(qo_lens=[1] * len(kv_lens), kv_lens=kv_lens, num_qo_heads=1, num_kv_heads=1,
                           head_dim=8, page_size=page_size, dtype=torch.bfloat16, seed=0, causal=causal)
    b.num_qo_heads, b.num_kv_heads, b.head_dim = hq, hkv, d
    b.qo_lens = list(qo_lens)
    qo = torch.zeros(len(qo_lens) + 1, dtype=torch.int32)
    qo[1:] = torch.cumsum(torch.tensor(qo_lens), 0)
    b.qo_indptr = qo
    b.q = torch.empty(int(qo[-1]), 1, 1)
    return b


# --------------------------------------------------------------------------- decode plan
def check_decode_plan(h, b, num_sms=152):
    info = api.plan_get_info(h)
    work = api.plan_get_work(h)
    P, hkv = b.page_size, b.num_kv_heads
    counts = (b.kv_indptr[1:] - b.kv_indptr[:-1]).tolist()
    covered = {}
    per_worker = {}
    slots = set()
    for w, bb, kvh, p0, n, last, slot, _ in work.tolist():
        per_worker[w] = per_worker.get(w, 0) + n
        for p in range(p0, p0 + n):
            key = (bb, kvh, p)
            assert key not in covered, f"page {key} covered twice"
            covered[key] = slot
        if n:
            assert last == (b.kv_last_page_len[bb].item() if p0 + n == counts[bb] else P)
        if slot >= 0:
            assert slot not in slots
            slots.add(slot)
    want = {(bb, kvh, p) for bb in range(b.batch) for kvh in range(hkv) for p in range(counts[bb])}
    assert set(covered) == want
    # workers appear in non-decreasing order and no run holds more than ceil(T / 8) pages
    ws_ = work[:, 0].tolist()
    assert ws_ == sorted(ws_)
    total = sum(counts) * hkv
    assert info.total_cost == total
    if total:
        # pages of one run have midpoints 8 apart inside a cost interval of length T
        assert info.max_cost <= -(-decode_cost_target(b, info.workers) // 8)
        assert max(per_worker.values()) == info.max_cost
    assert info.num_slots == len(slots)
    # an empty request still gets exactly one entry per kv head (it writes o = 0)
    for bb, n in enumerate(counts):
        if n == 0:
            assert sum(1 for r in work.tolist() if r[1] == bb) == hkv
    return info, work


def test_decode_plan_llama3_batch(lib):
    b = table_batch([int(x) for x in torch.randint(512, 4097, (64,), generator=torch.Generator().manual_seed(1))])
    h, ws = host_plan(b, api.PLAN_DECODE)
    compute(h, ws, b)
    info, work = check_decode_plan(h, b)
    assert info.active_workers <= info.workers == 152 * info.grid_ctas // 152 * (info.workers // info.grid_ctas)
    assert info.max_cost * info.active_workers >= info.total_cost
    api.plan_destroy(h)


def test_decode_plan_skewed_batch_splits_the_long_request(lib):
    b = table_batch([1024] * 31 + [131072])
    h, ws = host_plan(b, api.PLAN_DECODE)
    compute(h, ws, b)
    info, work = check_decode_plan(h, b)
    long_slots = [r for r in work.tolist() if r[1] == 31]
    assert len(long_slots) > 8 * 50  # the long request is spread over most workers
    assert info.num_merge >= 8
    api.plan_destroy(h)


@pytest.mark.parametrize("kv_lens,P", [([0, 5, 0, 17], 16), ([1, 15, 16, 17, 33], 16), ([7, 100, 3], 1),
                                       ([130, 64, 0], 64), ([0, 0], 16), ([1], 16)])
def test_decode_plan_edge_lengths(lib, kv_lens, P):
    b = table_batch(kv_lens, page_size=P, hq=8, hkv=2)
    h, ws = host_plan(b, api.PLAN_DECODE, num_sms=4)
    compute(h, ws, b)
    check_decode_plan(h, b, num_sms=4)
    api.plan_destroy(h)


def test_decode_plan_is_deterministic(lib):
    b = table_batch([300, 2000, 17, 4096, 1])
    h, ws = host_plan(b, api.PLAN_DECODE)
    compute(h, ws, b)
    w1 = api.plan_get_work(h).clone()
    bytes1 = ws.clone()
    compute(h, ws, b)
    assert torch.equal(w1, api.plan_get_work(h))
    assert torch.equal(bytes1, ws)
    api.plan_destroy(h)


# --------------------------------------------------------------------------- validation
def test_plan_rejects_malformed_index_arrays(lib):
    b = table_batch([40, 17, 3])
    h, ws = host_plan(b, api.PLAN_DECODE)
    ip = b.kv_indptr.tolist()
    bad_ip = torch.tensor([ip[0], ip[2], ip[1], ip[3]], dtype=torch.int32)
    cases = [
        dict(ip=bad_ip),                                                    # non-monotone indptr
        dict(ix=torch.where(torch.arange(b.kv_indices.numel()) == 0, b.num_pages, b.kv_indices)),  # id = pool size
        dict(ix=torch.where(torch.arange(b.kv_indices.numel()) == 1, -1, b.kv_indices)),          # negative id
        dict(last=torch.tensor([16, 0, 3], dtype=torch.int32)),             # last_page_len 0 with pages
        dict(last=torch.tensor([16, 17, 3], dtype=torch.int32)),            # last_page_len > page_size
        dict(ip=torch.cat([torch.tensor([1], dtype=torch.int32), b.kv_indptr[1:]])),  # indptr[0] != 0
    ]
    for over in cases:
        with pytest.raises(api.PkvError) as e:
            compute(h, ws, b, **over)
        assert e.value.status == -2, over
    with pytest.raises(api.PkvError) as e:                                  # more requests than the limits
        api.plan_compute(h, 4, None, torch.zeros(5, dtype=torch.int32), None, torch.zeros(4, dtype=torch.int32),
                         10, ws)
    assert e.value.status == -4
    with pytest.raises(api.PkvError) as e:                                  # host buffer too small
        api.plan_compute(h, b.batch, None, b.kv_indptr, b.kv_indices, b.kv_last_page_len, b.num_pages, ws[:64])
    assert e.value.status == -4
    api.plan_destroy(h)


def test_plan_rejects_an_indptr_whose_int32_difference_wraps(lib):
    """indptr [0, 2^31 - 1, -2^31] is not monotone, but its second difference taken in
    int32 wraps to +1: the plan must compare the entries, not their difference."""
    for kind in (api.PLAN_DECODE, api.PLAN_PREFILL):
        b = table_batch([1, 1], page_size=1)
        h, ws = host_plan(b, kind, max_kv_pages=4)
        ip = torch.tensor([0, (1 << 31) - 1, -(1 << 31)], dtype=torch.int32)
        qo = torch.tensor([0, 1, 2], dtype=torch.int32) if kind != api.PLAN_DECODE else None
        for ix in (torch.zeros(1, dtype=torch.int32), None):
            with pytest.raises(api.PkvError) as e:
                api.plan_compute(h, 2, qo, ip, ix, torch.tensor([1, 1], dtype=torch.int32), 1, ws)
            assert e.value.status == -2
        api.plan_destroy(h)


def test_plan_refuses_a_request_of_2_31_keys(lib):
    """Keys of one request are counted in int32: 2^27 page entries of 16 rows (a page id
    may repeat) make 2^31 keys, refused; one key fewer is planned."""
    b = table_batch([40])
    h, ws = host_plan(b, api.PLAN_DECODE, max_kv_pages=1 << 27)
    ip = torch.tensor([0, 1 << 27], dtype=torch.int32)
    with pytest.raises(api.PkvError) as e:
        api.plan_compute(h, 1, None, ip, None, torch.tensor([16], dtype=torch.int32), 10, ws)
    assert e.value.status == -4
    api.plan_compute(h, 1, None, ip, None, torch.tensor([15], dtype=torch.int32), 10, ws)
    assert api.plan_get_info(h).total_cost == (1 << 27) * b.num_kv_heads
    api.plan_destroy(h)


def test_plan_create_rejects_bad_params(lib):
    lim = api.Limits(4, 4, 100)
    for params, st in [
        (api.make_params(6, 4, 128, 16, torch.bfloat16, 0.1), -1),   # heads not a multiple
        (api.make_params(8, 2, 96, 16, torch.bfloat16, 0.1), -3),    # head_dim not built
        (api.make_params(8, 2, 128, 24, torch.bfloat16, 0.1), -3),   # page size neither <=16 nor 16k
        (api.make_params(8, 2, 128, 16, torch.float32, 0.1), -3),    # fp32 storage
        (api.make_params(48, 2, 128, 16, torch.bfloat16, 0.1), -3),  # group 24
        (api.make_params(8, 2, 128, 16, torch.bfloat16, 0.0), -1),   # scale 0
    ]:
        with pytest.raises(api.PkvError) as e:
            api.plan_create_host(api.PLAN_DECODE, params, lim, 152)
        assert e.value.status == st


def test_plan_create_refuses_limits_past_int32_tables(lib):
    """Table entries are counted in int32: limits that would need more are refused at
    create time (rather than wrapping the table sizes)."""
    big = (1 << 31) - 1
    dec = api.make_params(32, 8, 128, 16, torch.bfloat16, 0.1)
    with pytest.raises(api.PkvError) as e:                       # 300M requests x 8 kv heads
        api.plan_create_host(api.PLAN_DECODE, dec, api.Limits(300_000_000, 300_000_000, 1000), 152)
    assert e.value.status == -1
    wide = api.make_params(256, 256, 128, 16, torch.bfloat16, 0.1)
    for kind in (api.PLAN_PREFILL, api.PLAN_MIXED):              # 2^31 rows / 256 per tile x 256 kv heads
        with pytest.raises(api.PkvError) as e:
            api.plan_create_host(kind, wide, api.Limits(1, big, 1000), 152)
        assert e.value.status == -1
    # the largest row count with 8 kv heads still fits: 8.6 GB of tables, sized without wrapping
    h = api.plan_create_host(api.PLAN_PREFILL, api.make_params(8, 8, 128, 16, torch.bfloat16, 0.1),
                             api.Limits(1, big, 1000), 152)
    dev, host = api.plan_workspace_bytes(h)
    assert host >= 2 * 64 * 8 * (big // 256) and dev > host // 2
    api.plan_destroy(h)


def test_run_calls_refuse_host_only_plans(lib):
    b = table_batch([40])
    h, ws = host_plan(b, api.PLAN_DECODE)
    compute(h, ws, b)
    dummy = torch.empty(64, dtype=torch.uint8)
    with pytest.raises(api.PkvError):
        api.batch_decode_paged(h, dummy, dummy, dummy, dummy, dummy, dummy, None, dummy, stream=0)
    api.plan_destroy(h)


# --------------------------------------------------------------------------- prefill plan
def check_prefill_plan(h, b, num_sms=152, rows_per_tile=256):
    """Every (request, kv head, query position) gets exactly one tile family whose key
    chunks cover [0, causal limit of the family's last row) once, in 128-key blocks."""
    info = api.plan_get_info(h)
    work = api.plan_get_work(h).tolist()
    g = b.num_qo_heads // b.num_kv_heads
    mp_ = rows_per_tile // g
    fam = {}
    for w, bb, kvh, pos0, npos, kb, ke, slot in work:
        fam.setdefault((bb, kvh, pos0), []).append((kb, ke, slot, npos, w))
    for bb in range(b.batch):
        qo, kv = b.qo_lens[bb], b.kv_lens[bb]
        for kvh in range(b.num_kv_heads):
            for pos0 in range(0, qo, mp_):
                npos = min(mp_, qo - pos0)
                chunks = sorted(fam.pop((bb, kvh, pos0)))
                assert all(c[3] == npos for c in chunks)
                end = kv if not b.causal else max(0, min(kv, pos0 + npos + kv - qo))
                pos = 0
                for kb, ke, slot, _, _ in chunks:
                    assert kb == pos and kb % 128 == 0 and ke > kb or (kb == ke == 0 == end)
                    pos = ke
                assert pos == end
                if len(chunks) == 1:
                    assert chunks[0][2] == -1
                else:
                    slots = [c[2] for c in chunks]
                    assert min(slots) >= 0 and slots == list(range(slots[0], slots[0] + len(slots)))
    assert not fam, f"tiles for rows that do not exist: {list(fam)[:3]}"
    # workers appear in non-decreasing order; LPT keeps the loads within one tile of each other
    ws_ = [r[0] for r in work]
    assert ws_ == sorted(ws_)
    return info, work


def longest_first_prefill(b, C, rows_per_tile=256, keys=128):
    """The prefill plan's schedule restated plainly: query tiles per (request, kv head,
    rows_per_tile / G positions), their key ranges cut into near-equal chunks when longer
    than total / C blocks, item cost = blocks + 2, items longest first (ties: lower item)
    onto the least-loaded CTA (ties: lower CTA).  Returns the work rows in the plan's
    order (CTA by CTA, each CTA's items in the order assigned)."""
    import heapq
    g = b.num_qo_heads // b.num_kv_heads
    mp_ = rows_per_tile // g
    tiles, total = [], 0
    for bb in range(b.batch):
        qo, kv = b.qo_lens[bb], b.kv_lens[bb]
        for kvh in range(b.num_kv_heads):
            for pos0 in range(0, qo, mp_):
                npos = min(mp_, qo - pos0)
                end = max(0, min(kv, pos0 + npos + kv - qo)) if b.causal else kv
                tiles.append((bb, kvh, pos0, npos, end))
                total += max(1, -(-end // keys))
    chunk = max(-(-total // max(C, 1)), 1)
    items, slot = [], 0
    for bb, kvh, pos0, npos, end in tiles:
        nb = -(-end // keys)
        if nb <= chunk:
            items.append(((bb, kvh, pos0, npos, 0, end, -1), max(nb, 1) + 2))
        else:
            parts = -(-nb // chunk)
            for i in range(parts):
                lo, hi = i * nb // parts, (i + 1) * nb // parts
                items.append(((bb, kvh, pos0, npos, lo * keys, min(hi * keys, end), slot), hi - lo + 2))
                slot += 1
    order = sorted(range(len(items)), key=lambda i: -items[i][1])  # stable: ties keep item order
    ctas = min(C, len(items))
    heap = [(0, c) for c in range(ctas)]
    per = [[] for _ in range(ctas)]
    for i in order:
        load, c = heapq.heappop(heap)
        per[c].append(i)
        heapq.heappush(heap, (load + items[i][1], c))
    return [[c, *items[i][0]] for c in range(ctas) for i in per[c]]


@pytest.mark.parametrize("seed,batch,C,causal,page", [(1003, 16, 152, True, 16), (7, 5, 8, True, 16),
                                                      (9, 3, 152, False, 16), (11, 6, 20, True, 1),
                                                      (13, 1, 152, False, 16),
                                                      # CTA counts at the edges of 64-bit CTA sets
                                                      (21, 8, 64, True, 16), (23, 8, 65, True, 16),
                                                      (25, 4, 1, True, 16), (27, 10, 130, False, 8),
                                                      # pages of 1 and 4 rows: planned over the packed
                                                      # copy in 16-row pages, the same key ranges
                                                      (29, 6, 37, True, 1), (31, 5, 152, True, 4)])
def test_prefill_plan_is_the_longest_first_schedule(lib, seed, batch, C, causal, page):
    """The plan's work rows equal the plainly restated schedule, item by item and CTA by
    CTA (a faster implementation of the plan must not change what the GPU runs)."""
    b = W.ragged_prefill(seed=seed, batch=batch, page_size=page)
    if not causal:
        b = W.PagedBatch(**{**b.__dict__, "causal": False})
    if batch == 1:  # one long request: its key range is cut into chunks over the CTAs
        b = W.make_paged_batch(qo_lens=[300], kv_lens=[40000], num_qo_heads=32, num_kv_heads=8, head_dim=128,
                               page_size=16, dtype=torch.bfloat16, seed=seed)
    h, ws = host_plan(b, api.PLAN_PREFILL, num_sms=C)
    compute(h, ws, b)
    work = api.plan_get_work(h).tolist()
    assert work == longest_first_prefill(b, C)


def decode_cost_target(b, W):
    """The decode plan's cost per run T, in eighths of a page: a page costs 8 and each
    piece of a (request, kv head) page list 8 more; the whole cost counting one piece per
    list and one more per run boundary, over W runs (at least one piece and one page)."""
    lens = [int(b.kv_indptr[r + 1] - b.kv_indptr[r]) for r in range(b.batch)]
    total = sum(lens) * b.num_kv_heads
    return max(16, -(-(8 * total + 8 * (b.batch * b.num_kv_heads + W - 1)) // W))


def cost_runs_decode(b, W):
    """The decode plan restated plainly, page by page: the (request, kv head) page lists in
    order on a cost line, each page costing 8 and each piece of a list 8 before its first
    page.  A page belongs to run min(midpoint // T, W - 1); a piece starts at a list's first
    page and wherever a page (at the cost so far) falls in another run than the piece's.  A
    list of several pieces has a partial-state slot per piece.  Run r goes to warp r // C of
    CTA r % C (C = W // 8 CTAs of 8 warps), worker 8 * CTA + warp.  Returns the work rows
    [worker, request, kv head, first page, pages, last rows, slot, 0] in worker order."""
    P = b.page_size
    lens = [int(b.kv_indptr[r + 1] - b.kv_indptr[r]) for r in range(b.batch)]
    T = decode_cost_target(b, W)
    rows, slot, X = [], 0, 0
    for r in range(b.batch):
        n = lens[r]
        last = int(b.kv_last_page_len[r])
        for h in range(b.num_kv_heads):
            if n == 0:
                rows.append([min(X // T, W - 1), r, h, 0, 0, 0, -1, 0])
                continue
            pieces = []  # [run, first page, pages]
            for i in range(n):
                if not pieces or min((X + 4) // T, W - 1) != pieces[-1][0]:
                    X += 8  # the new piece's start
                    pieces.append([min((X + 4) // T, W - 1), i, 0])
                pieces[-1][2] += 1
                X += 8
            if len(pieces) == 1:
                rows.append([pieces[0][0], r, h, 0, n, last, -1, 0])
            else:
                for w, lo, cnt in pieces:
                    rows.append([w, r, h, lo, cnt, last if lo + cnt == n else P, slot, 0])
                    slot += 1
    C = W // 8
    for row in rows:
        row[0] = (row[0] % C) * 8 + row[0] // C
    return sorted(rows, key=lambda row: row[0])  # stable: a run keeps its order


@pytest.mark.parametrize("seed,batch,workers,page", [(1001, 64, 1216, 16), (3, 9, 40, 16), (5, 7, 1216, 1),
                                                       (8, 3, 8, 64)])
def test_decode_plan_is_the_equal_cost_split(lib, seed, batch, workers, page):
    """The decode plan's work rows equal the plainly restated equal-cost split, worker by
    worker (8 workers per SM)."""
    b = W.llama3_decode(seed=seed, batch=batch, page_size=page)
    h, ws = host_plan(b, api.PLAN_DECODE, num_sms=workers // 8)
    compute(h, ws, b)
    if fits_in_one_run(b, workers):
        check_whole_list_plan(h, b, workers)
    else:
        assert api.plan_get_work(h).tolist() == cost_runs_decode(b, workers)


def fits_in_one_run(b, W, tile_rows=16):
    """No (request, kv head) list longer than a run, and a worker for every list: the
    split plan then keeps each list whole, one per worker (the whole-list schedule)."""
    lens = [int(b.kv_indptr[r + 1] - b.kv_indptr[r]) for r in range(b.batch)]
    total = sum(lens) * b.num_kv_heads
    run = -(-total // W) if total else 1
    return b.batch * b.num_kv_heads <= W and max(lens, default=0) <= run


@pytest.mark.parametrize("kv_lens,sms,whole", [([16] * 64, 152, True), ([64] * 64, 152, False),
                                               ([128] * 64, 152, False), ([16] * 64, 4, False),
                                               ([16] * 100, 152, True)])
def test_decode_plan_keeps_short_lists_whole_when_workers_allow(lib, kv_lens, sms, whole):
    """64 x 8 lists of 1, 4 or 8 pages on 152 SMs (1216 workers: runs of 1, 2 and 4 pages), one
    page on 4 SMs (32 workers, fewer than the lists) and 100 x 8 one-page lists: whole lists
    exactly when none exceeds a run and every list has a worker."""
    b = table_batch(kv_lens)
    assert fits_in_one_run(b, sms * 8) == whole
    h, ws = host_plan(b, api.PLAN_DECODE, num_sms=sms)
    compute(h, ws, b)
    if whole:
        check_whole_list_plan(h, b, sms * 8)
    else:
        assert api.plan_get_work(h).tolist() == cost_runs_decode(b, sms * 8)
    api.plan_destroy(h)


def test_prefill_plan_ragged_causal(lib):
    b = W.ragged_prefill(seed=1003)
    h, ws = host_plan(b, api.PLAN_PREFILL)
    compute(h, ws, b)
    info, work = check_prefill_plan(h, b)
    costs = {}
    for w, bb, kvh, pos0, npos, kb, ke, slot in work:
        costs[w] = costs.get(w, 0) + -(-(ke - kb) // 128) + 2
    biggest = max(-(-(ke - kb) // 128) + 2 for _, _, _, _, _, kb, ke, _ in work)
    assert max(costs.values()) - min(costs.values()) <= biggest
    assert info.num_merge == 0  # thousands of tiles: no key range needs splitting
    api.plan_destroy(h)


def test_prefill_plan_splits_long_keys_of_few_tiles(lib):
    # the cascade prefix: one row block of 64 queries x 32 heads against 2048 shared keys
    cb = W.cascade_decode(seed=1004, num_qo_heads=32, num_kv_heads=8)
    b = cb.prefix
    h, ws = host_plan(b, api.PLAN_PREFILL)
    compute(h, ws, b)
    info, work = check_prefill_plan(h, b)
    assert info.num_merge == 8 and info.num_slots == len(work) and len(work) > 8 * 4
    api.plan_destroy(h)


@pytest.mark.parametrize("qo,kv,causal", [([5, 0, 300], [5, 9, 300], True), ([10, 3], [4, 3], True),
                                          ([257, 1], [1000, 1], False)])
def test_prefill_plan_edge_cases(lib, qo, kv, causal):
    b = W.make_paged_batch(qo_lens=qo, kv_lens=kv, num_qo_heads=8, num_kv_heads=2, head_dim=128, page_size=16,
                           dtype=torch.bfloat16, seed=1, causal=causal)
    h, ws = host_plan(b, api.PLAN_PREFILL, num_sms=8)
    compute(h, ws, b)
    check_prefill_plan(h, b)
    api.plan_destroy(h)


# --------------------------------------------------------------------------- mixed plans
def check_mixed_plan(h, b, num_sms=152):
    """Decode entries (listed first) cover each single-row request's pages once per kv
    head and read/write its own row; prefill tiles cover the other requests; the two
    halves use disjoint SM counts that add up to the GPU."""
    info = api.plan_get_info(h)
    work = api.plan_get_work(h).tolist()
    single = {i for i, q in enumerate(b.qo_lens) if q == 1}
    multi = {i for i, q in enumerate(b.qo_lens) if q > 1}
    n_dec = 0
    while n_dec < len(work) and work[n_dec][1] in single:
        n_dec += 1
    dec, pre = work[:n_dec], work[n_dec:]
    assert all(r[1] in multi for r in pre)
    assert {r[1] for r in dec} == single and {r[1] for r in pre} == multi
    # decode half: pages of each (request, kv head) covered exactly once
    seen = {}
    for w, bb, kvh, pb, npg, last, slot, _ in dec:
        seen.setdefault((bb, kvh), []).append((pb, npg))
        assert w < info.decode_ctas * 8
    for bb in single:
        n = int(b.kv_indptr[bb + 1] - b.kv_indptr[bb])
        for kvh in range(b.num_kv_heads):
            runs = sorted(seen.pop((bb, kvh)))
            pos = 0
            for pb, npg in runs:
                assert pb == pos
                pos += npg
            assert pos == n
    assert not seen
    # prefill half: every tile of a multi-row request, on the prefill CTAs only
    assert all(r[0] < info.prefill_ctas for r in pre)
    fam = {(r[1], r[2], r[3]) for r in pre}
    g = b.num_qo_heads // b.num_kv_heads
    mp = 256 // g
    for bb in multi:
        for kvh in range(b.num_kv_heads):
            for pos0 in range(0, b.qo_lens[bb], mp):
                assert (bb, kvh, pos0) in fam
    if single and multi:
        assert info.prefill_ctas >= 1 and info.decode_ctas >= 1
        assert info.prefill_ctas + info.decode_ctas == num_sms
    return info


def test_mixed_plan_routes_requests_by_row_count(lib):
    b = W.mixed_batch(seed=1007)
    h, ws = host_plan(b, api.PLAN_MIXED)
    compute(h, ws, b)
    info = check_mixed_plan(h, b)
    # the split follows the work: more prefill rows take more SMs
    b2 = W.mixed_batch(seed=1007, n_prefill=12)
    h2, ws2 = host_plan(b2, api.PLAN_MIXED)
    compute(h2, ws2, b2)
    info2 = check_mixed_plan(h2, b2)
    assert info2.prefill_ctas > info.prefill_ctas


@pytest.mark.parametrize("num_sms", [152, 10, 4, 2])
def test_mixed_split_gives_each_half_sms_and_is_even(lib, num_sms):
    """Both halves get SMs and together all of them; the prefill share is even when the
    GPU has room for it (an odd share would leave an SM pair with one CTA of each half)."""
    for seed, n_prefill in ((1007, 4), (1007, 12), (3, 1)):
        b = W.mixed_batch(seed=seed, n_prefill=n_prefill)
        h, ws = host_plan(b, api.PLAN_MIXED, num_sms=num_sms)
        compute(h, ws, b)
        info = check_mixed_plan(h, b, num_sms=num_sms)
        assert info.prefill_ctas >= 1 and info.decode_ctas >= 1
        assert info.prefill_ctas + info.decode_ctas == num_sms
        if num_sms >= 4:
            assert info.prefill_ctas % 2 == 0


def test_mixed_plan_needs_two_sms(lib):
    b = W.mixed_batch(seed=2, n_decode=2, n_prefill=1)
    with pytest.raises(api.PkvError):
        host_plan(b, api.PLAN_MIXED, num_sms=1)


@pytest.mark.parametrize("n_decode,n_prefill", [(0, 3), (5, 0), (0, 0)])
def test_mixed_plan_with_one_half_empty(lib, n_decode, n_prefill):
    b = W.mixed_batch(seed=5, n_decode=n_decode, n_prefill=n_prefill, qo_lo=20, qo_hi=300, decode_lo=1,
                      decode_hi=400)
    h, ws = host_plan(b, api.PLAN_MIXED)
    compute(h, ws, b)
    info = check_mixed_plan(h, b)
    assert (info.prefill_ctas > 0) == (n_prefill > 0)
    assert (info.decode_ctas > 0) == (n_decode > 0)


def test_mixed_plan_needs_qo_indptr(lib):
    b = W.mixed_batch(seed=6, n_decode=3, n_prefill=1)
    h, ws = host_plan(b, api.PLAN_MIXED)
    with pytest.raises(api.PkvError):
        compute(h, ws, b, qo=None)


@pytest.mark.parametrize("kind", [api.PLAN_PREFILL, api.PLAN_MIXED])
def test_replanning_after_other_batches_gives_a_fresh_plans_tables(lib, kind):
    """A plan keeps its working arrays from call to call: re-planning one plan object
    small -> big -> small gives each time the work and figures of a fresh plan of
    that batch (nothing left over from the previous call)."""
    big = W.mixed_batch(seed=1007, n_prefill=32)
    small = W.mixed_batch(seed=3, n_decode=5, n_prefill=3)
    lim = dict(max_batch=big.batch, max_total_q=big.total_q, max_kv_pages=int(big.kv_indptr[-1]))

    def fresh(b):
        h, ws = host_plan(b, kind, **lim)
        compute(h, ws, b)
        return api.plan_get_work(h), _info_tuple(api.plan_get_info(h))

    want = {id(b): fresh(b) for b in (small, big)}
    h, ws = host_plan(big, kind, **lim)
    for b in (small, big, small, big):
        compute(h, ws, b)
        work, info = api.plan_get_work(h), _info_tuple(api.plan_get_info(h))
        assert torch.equal(work, want[id(b)][0])
        assert info == want[id(b)][1]


def _info_tuple(info):
    return tuple(getattr(info, f) for f, _ in info._fields_)


# --------------------------------------------------------------------------- decode plan, split-KV off
def check_whole_list_plan(h, b, workers):
    """Every (request, kv head) page list whole on one worker, placed longest first on
    the least-loaded worker, ties to the lower rank (rank r = warp r // C of CTA r % C)
    (a plain restatement of that schedule); no slots, no merges."""
    info = api.plan_get_info(h)
    rows = api.plan_get_work(h).tolist()
    hkv = b.num_kv_heads
    counts = (b.kv_indptr[1:] - b.kv_indptr[:-1]).tolist()
    n_lists = b.batch * hkv
    ctas = workers // 8
    order = sorted(range(n_lists), key=lambda i: -counts[i // hkv])  # stable: ties keep list order
    loads = [0] * min(workers, n_lists)                               # by rank
    owner, seq = {}, {}
    for i in order:
        r = min(range(len(loads)), key=lambda j: (loads[j], j))
        w = (r % ctas) * 8 + r // ctas
        owner[(i // hkv, i % hkv)] = w
        seq.setdefault(w, []).append((i // hkv, i % hkv))
        loads[r] += counts[i // hkv]
    got = {}
    for w, bb, kvh, p0, n, last, slot, _ in rows:
        assert (bb, kvh) not in got
        got[(bb, kvh)] = w
        assert p0 == 0 and n == counts[bb] and slot == -1
        assert last == (int(b.kv_last_page_len[bb]) if n else 0)
    assert got == owner
    assert [r[0] for r in rows] == sorted(r[0] for r in rows)                 # grouped by worker
    assert [(r[1], r[2]) for r in rows] == [x for w in sorted(seq) for x in seq[w]]
    assert info.num_merge == 0 and info.num_slots == 0 and info.num_work == n_lists
    assert info.active_workers == len(loads)
    assert info.max_cost == max(loads, default=0) and info.total_cost == sum(counts) * hkv


def test_decode_plan_without_split_keeps_each_list_whole(lib):
    # the skewed long-context batch: 31 requests of 1024 tokens and one of 131072
    b = table_batch([1024] * 31 + [131072])
    h, ws = host_plan(b, api.PLAN_DECODE)
    api.plan_set_split_kv(h, False)
    compute(h, ws, b)
    check_whole_list_plan(h, b, 152 * 8)
    assert api.plan_get_info(h).max_cost == 8192          # the long request on one worker per kv head
    long_workers = [r[0] for r in api.plan_get_work(h).tolist() if r[1] == 31]
    assert len({w // 8 for w in long_workers}) == 8       # ... its 8 kv heads on 8 CTAs
    api.plan_set_split_kv(h, True)                        # back on: the split plan again
    compute(h, ws, b)
    check_decode_plan(h, b)
    assert api.plan_get_info(h).num_slots > 0
    api.plan_destroy(h)


def test_decode_plan_without_split_more_lists_than_workers(lib):
    rng = np.random.default_rng(7)
    kv = [int(x) for x in rng.integers(0, 900, size=11)] + [0, 5]   # an empty request, a short one
    b = table_batch(kv)
    h, ws = host_plan(b, api.PLAN_DECODE, num_sms=2)      # 16 workers for 13 x 8 lists
    api.plan_set_split_kv(h, False)
    compute(h, ws, b)
    check_whole_list_plan(h, b, 2 * 8)
    api.plan_destroy(h)


@pytest.mark.parametrize("kind", [api.PLAN_PREFILL, api.PLAN_MIXED])
def test_split_kv_switch_is_for_decode_plans(lib, kind):
    b = W.mixed_batch(seed=6, n_decode=3, n_prefill=1)
    h, ws = host_plan(b, kind)
    with pytest.raises(api.PkvError) as e:
        api.plan_set_split_kv(h, False)
    assert e.value.status == -1
    api.plan_destroy(h)


# --------------------------------------------------------------------------- argument checks of the run calls
def test_run_calls_refuse_bad_arguments_before_any_cuda_call(lib):
    """Each case fails a host-side check that comes before the first CUDA call (so no
    case can reach a kernel with these host pointers): the status the header states."""
    L = api.load()
    buf = torch.zeros(4096, dtype=torch.uint8)
    base = buf.data_ptr() + (-buf.data_ptr()) % 256
    p16, odd = ctypes.c_void_p(base), ctypes.c_void_p(base + 2)   # 256-aligned, and 2 bytes off
    INVALID, UNSUPPORTED = -1, -3
    # merge_state: sizes, dtype, pointers, alignment
    ms = L.pkv_merge_state
    assert ms(p16, p16, p16, p16, p16, p16, -1, 4, 64, api.PKV_BF16, None) == INVALID
    assert ms(p16, p16, p16, p16, p16, p16, 8, 0, 64, api.PKV_BF16, None) == INVALID
    assert ms(p16, p16, p16, p16, p16, p16, 8, 4, 0, api.PKV_BF16, None) == INVALID
    assert ms(p16, p16, p16, p16, p16, p16, 8, 4, 64, 7, None) == UNSUPPORTED
    assert ms(None, None, None, None, None, None, 0, 4, 64, api.PKV_BF16, None) == api.PKV_OK   # nothing to do
    assert ms(None, p16, p16, p16, p16, p16, 8, 4, 64, api.PKV_BF16, None) == INVALID
    assert ms(odd, p16, p16, p16, p16, p16, 8, 4, 64, api.PKV_BF16, None) == INVALID
    assert ms(p16, odd, p16, p16, p16, p16, 8, 4, 64, api.PKV_BF16, None) == INVALID
    # merge_states: counts, stride, sizes, dtype, pointers, alignment
    mn = L.pkv_merge_states
    assert mn(p16, p16, 0, 8, p16, p16, 8, 4, 64, api.PKV_BF16, None) == INVALID      # no state
    assert mn(p16, p16, 3, 7, p16, p16, 8, 4, 64, api.PKV_BF16, None) == INVALID      # states overlap
    assert mn(p16, p16, 3, 8, p16, p16, -1, 4, 64, api.PKV_BF16, None) == INVALID
    assert mn(p16, p16, 3, 8, p16, p16, 8, 0, 64, api.PKV_BF16, None) == INVALID
    assert mn(p16, p16, 3, 8, p16, p16, 8, 4, 64, 7, None) == UNSUPPORTED
    assert mn(None, None, 3, 0, None, None, 0, 4, 64, api.PKV_BF16, None) == api.PKV_OK  # nothing to do
    assert mn(None, p16, 3, 8, p16, p16, 8, 4, 64, api.PKV_BF16, None) == INVALID
    assert mn(odd, p16, 3, 8, p16, p16, 8, 4, 64, api.PKV_BF16, None) == INVALID
    assert mn(p16, p16, 3, 8, odd, p16, 8, 4, 64, api.PKV_BF16, None) == INVALID
    assert mn(p16, p16, 3, 1 << 62, p16, p16, 8, 4, 64, api.PKV_BF16, None) == INVALID  # offsets past int64
    # append: params, theta, head_dim, dtype, counts, pointers, alignment
    ap = L.pkv_append_paged_kv
    good = api.make_params(8, 2, 128, 16, torch.bfloat16, 0.1)

    def append(params, batch=2, nnz=5, theta=0.0, k=p16, q_in=None, q_out=None):
        return ap(ctypes.byref(params) if params is not None else None, batch, nnz, 10, p16, p16, p16, p16, k, p16,
                  p16, q_in, q_out, theta, None, None)
    assert append(None) == INVALID
    for theta in (-1.0, float("nan"), float("inf")):
        assert append(good, theta=theta) == INVALID
    assert append(api.make_params(8, 2, 96, 16, torch.bfloat16, 0.1)) == UNSUPPORTED
    assert append(api.make_params(8, 2, 128, 16, api.PKV_F32, 0.1)) == UNSUPPORTED
    assert append(good, nnz=0) == api.PKV_OK                                   # nothing to append
    assert append(good, batch=0) == INVALID                                    # tokens but no requests
    assert append(good, q_in=p16) == INVALID                                   # q_in without q_out
    assert append(good, k=odd) == INVALID
    # run calls: a plan of another kind, and a host-only plan of the right kind
    b = W.mixed_batch(seed=6, n_decode=3, n_prefill=1)
    plans = {k: host_plan(b, k) for k in (api.PLAN_DECODE, api.PLAN_PREFILL, api.PLAN_MIXED)}
    for k, (h, ws) in plans.items():
        compute(h, ws, b)
    ptrs = [p16] * 9
    dec = lambda h: L.pkv_batch_decode_paged(h, *ptrs[:7], p16, None)
    pre = lambda h: L.pkv_batch_prefill_paged(h, *ptrs[:8], p16, None)
    mix = lambda h: L.pkv_batch_mixed_paged(h, *ptrs[:8], p16, None)
    masked_no_mask = lambda h: L.pkv_batch_prefill_paged_masked(h, *ptrs[:6], None, 64, p16, p16, p16, None)
    for run, kind in ((dec, api.PLAN_DECODE), (pre, api.PLAN_PREFILL), (mix, api.PLAN_MIXED)):
        for k, (h, _) in plans.items():
            assert run(h) == INVALID, (kind, k)                    # other kinds, and host-only plans
    assert masked_no_mask(plans[api.PLAN_PREFILL][0]) == INVALID
    # setters and the error read-back
    h = plans[api.PLAN_DECODE][0]
    assert L.pkv_plan_set_timing_events(h, p16, None) == INVALID      # start without stop
    assert L.pkv_plan_set_pipelined(h, 1) == INVALID                  # host-only plan
    code = ctypes.c_int(0)
    assert L.pkv_get_device_error(None, p16, ctypes.byref(code), 0, None) == INVALID
    for h, _ in plans.values():
        api.plan_destroy(h)


def test_bench_mixed_batch_takes_the_measured_split(lib):
    """The bench's mixed batch (60 decodes + 4 prompt chunks) splits 72 prefill / 80 decode
    SMs of 152: the split its one-launch timings and profile were taken at."""
    b = W.mixed_batch(seed=1007)
    h, ws = host_plan(b, api.PLAN_MIXED)
    compute(h, ws, b)
    info = api.plan_get_info(h)
    assert (info.prefill_ctas, info.decode_ctas) == (72, 80)
    api.plan_destroy(h)


# --------------------------------------------------------------------------- Zipf-distributed lengths
@pytest.mark.parametrize("s", [1.1, 1.5])
def test_decode_plan_balances_zipf_request_lengths(lib, s):
    """Request lengths from a Zipf law (the skew the pages' scheduler is built for):
    every worker still streams at most ceil(T / 8) pages, T the equal cost per run (about
    total pages / workers, plus a page for each piece of a list it holds)."""
    kv = W.zipf_lengths(128, s, 16, 131072, seed=11)
    assert max(kv) > 20 * sorted(kv)[len(kv) // 2]                 # heavy-tailed
    b = table_batch(kv)
    h, ws = host_plan(b, api.PLAN_DECODE)
    compute(h, ws, b)
    info, _ = check_decode_plan(h, b)
    total = sum((n + 15) // 16 for n in kv) * b.num_kv_heads
    assert info.max_cost <= -(-decode_cost_target(b, info.workers) // 8)
    assert info.total_cost == total
    api.plan_destroy(h)


@pytest.mark.parametrize("s", [1.1, 1.5])
def test_prefill_plan_balances_zipf_prompt_lengths(lib, s):
    """Prompt lengths from a Zipf law: the busiest CTA carries at most the average load
    plus one work item (the list-scheduling bound), long tiles being cut into chunks."""
    qo = W.zipf_lengths(24, s, 16, 8192, seed=12)
    b = table_batch(qo, qo_lens=qo, causal=True)
    h, ws = host_plan(b, api.PLAN_PREFILL)
    compute(h, ws, b)
    info, work = check_prefill_plan(h, b)
    biggest = max(max(1, -(-(ke - kb) // 128)) + 2 for _, _, _, _, _, kb, ke, _ in work)
    assert info.max_cost <= -(-info.total_cost // info.active_workers) + biggest
    api.plan_destroy(h)


# --------------------------------------------------------------------------- group-8 decode on the tensor cores
def test_group8_decode_plans_hold_prefill_tiles_of_one_row(lib):
    """A decode plan with 8 query heads per kv head at head_dim 128 (pages of 8 rows or
    more) plans its batch as prefill tiles of one query row per request: every
    (request, kv head) key range is covered exactly once, on at most one CTA each
    unless the plan cut it into chunks (then with partial slots)."""
    rng = np.random.default_rng(11)
    kv = [int(x) for x in rng.integers(512, 4097, size=64)]
    b = table_batch(kv, hq=64, hkv=8)
    h, ws = host_plan(b, api.PLAN_DECODE)
    compute(h, ws, b)
    rows = api.plan_get_work(h).tolist()
    cover = {}
    for cta, req, kvh, pos0, npos, k0, k1, slot in rows:
        assert 0 <= cta < 152 and npos == 1 and pos0 == 0
        cover.setdefault((req, kvh), []).append((k0, k1, slot))
    assert sorted(cover) == [(r, k) for r in range(64) for k in range(8)]
    for (req, kvh), ranges in cover.items():
        ranges.sort()
        assert ranges[0][0] == 0 and ranges[-1][1] == kv[req]
        assert all(a[1] == c[0] for a, c in zip(ranges, ranges[1:]))
        assert (len(ranges) == 1) == (ranges[0][2] == -1)
    with pytest.raises(api.PkvError) as e:                 # the split switch is the CUDA-core schedule's
        api.plan_set_split_kv(h, False)
    assert e.value.status == -3
    api.plan_destroy(h)


@pytest.mark.parametrize("hd,P", [(64, 16), (128, 1), (128, 4)])
def test_group8_decode_keeps_the_decode_kernel_elsewhere(lib, hd, P):
    """head_dim 64 (the prefill kernel is head_dim 128 only) and pages of fewer than 8
    rows keep decode segments: one row per (worker, request, kv head, page run)."""
    b = table_batch([300, 17, 900], hq=64, hkv=8, d=hd, page_size=P)
    h, ws = host_plan(b, api.PLAN_DECODE)
    compute(h, ws, b)
    check_decode_plan(h, b)
    api.plan_set_split_kv(h, False)
    api.plan_destroy(h)


def test_group8_mixed_plan_sends_single_rows_to_the_prefill_half(lib):
    b = W.mixed_batch(seed=5, n_decode=9, n_prefill=2, num_qo_heads=64, num_kv_heads=8)
    h, ws = host_plan(b, api.PLAN_MIXED)
    compute(h, ws, b)
    info = api.plan_get_info(h)
    assert info.prefill_ctas == 152 and info.decode_ctas == 0
    api.plan_destroy(h)


# --------------------------------------------------------------------------- prefill on small pages: the packed copy
@pytest.mark.parametrize("P", [1, 2, 4])
def test_packed_prefill_workspace_holds_the_copy(lib, P):
    """A prefill plan on pages of fewer than 8 rows reserves, in its device workspace, a copy of
    its limits' keys in 16-row pages: ceil(max_kv_pages * P / 16) + max_batch pages of
    2 x Hkv x 16 x head_dim 16-bit values beyond what the same plan on 16-row pages needs."""
    hq, hkv, d = 32, 8, 128
    max_b, max_q, max_pages = 7, 4000, 3000
    def dev_bytes(page_size, kind=api.PLAN_PREFILL):
        params = api.make_params(hq, hkv, d, page_size, torch.bfloat16, d ** -0.5, 0.0, True)
        h = api.plan_create_host(kind, params, api.Limits(max_b, max_q, max_pages), 152)
        dev, _ = api.plan_workspace_bytes(h)
        api.plan_destroy(h)
        return dev
    packed_pages = -(-max_pages * P // 16) + max_b
    copy_bytes = packed_pages * 2 * hkv * 16 * d * 2
    assert dev_bytes(P) - dev_bytes(16) >= copy_bytes
    # decode plans and mixed plans read the caller's pages directly: no copy
    assert dev_bytes(P, api.PLAN_DECODE) == dev_bytes(16, api.PLAN_DECODE)
    assert dev_bytes(P, api.PLAN_MIXED) < dev_bytes(P) + dev_bytes(P, api.PLAN_DECODE)


def test_packed_prefill_refuses_limits_past_32_bit_rows(lib):
    """The packed copy's rows are counted in 32 bits: limits whose copy would pass 2^31 rows are
    refused at plan creation (PKV_ERR_INVALID_ARG), the same limits on 16-row pages are not."""
    params1 = api.make_params(32, 8, 128, 1, torch.bfloat16, 128 ** -0.5, 0.0, True)
    params16 = api.make_params(32, 8, 128, 16, torch.bfloat16, 128 ** -0.5, 0.0, True)
    lim = api.Limits(4, 1 << 20, 150_000_000)  # 150 M one-row pages: 9.4 M packed pages x 256 rows
    with pytest.raises(api.PkvError) as e:
        api.plan_create_host(api.PLAN_PREFILL, params1, lim, 152)
    assert e.value.status == -1
    h = api.plan_create_host(api.PLAN_PREFILL, params16, api.Limits(4, 1 << 20, 150_000_000 // 16), 152)
    api.plan_destroy(h)


# --------------------------------------------------------------------------- launch ordering
def _kernels(src):
    """(name, body) of every __global__ function in a CUDA source text."""
    out = []
    for m in re.finditer(r"__global__\s+void\s+(?:__launch_bounds__\([^)]*\)\s*)?(\w+)\s*\(", src):
        i = src.index("{", m.end())  # the body follows the parameter list
        depth, j = 0, i
        while True:
            depth += {"{": 1, "}": -1}.get(src[j], 0)
            if depth == 0:
                break
            j += 1
        out.append((m.group(1), src[i:j + 1]))
    return out


def test_dependent_kernels_wait_before_any_return():
    """Kernels launched as programmatic dependents are ordered only after the grid just
    before them; the chain stays ordered after every earlier kernel only if each of them
    waits (griddepcontrol.wait) before it can return.  Every kernel but the standalone
    prefill kernel is launched that way, and that one keeps an ordinary launch."""
    csrc = os.path.join(os.path.dirname(api.__file__), "csrc")
    seen = set()
    for f in sorted(os.listdir(csrc)):
        if not f.endswith((".cu", ".cuh")):
            continue
        src = open(os.path.join(csrc, f)).read()
        for name, body in _kernels(src):
            seen.add(name)
            if name == "prefill_kernel":
                assert "griddepcontrol" not in body
                continue
            w = body.find("griddepcontrol.wait")
            assert w >= 0, f"{f}: {name} never waits for the grid before it"
            r = body.find("return")
            assert r < 0 or r > w, f"{f}: {name} can return before griddepcontrol.wait"
    assert {"decode_kernel", "prefill_kernel", "mixed_kernel", "pack_pages_kernel", "append_rope_kernel",
            "decode_merge_kernel", "prefill_merge_kernel", "mixed_merge_kernel", "merge_state_kernel",
            "merge_states_kernel"} <= seen
    prefill_src = open(os.path.join(csrc, "prefill_kernel.cuh")).read()
    assert "kern<<<grid, kThreads, smem, s>>>(a, tq, tkv)" in prefill_src


@pytest.mark.parametrize("s,sms", [(1.1, 152), (1.5, 152), (1.1, 5), (1.5, 1)])
def test_decode_plan_is_the_equal_cost_split_on_zipf_lengths(lib, s, sms):
    """Heavy-tailed request lengths on grids of 8 to 1216 workers: the plan's work rows equal
    the page-by-page restatement of the equal-cost split exactly."""
    kv = W.zipf_lengths(96, s, 16, 65536, seed=21)
    b = table_batch(kv)
    h, ws = host_plan(b, api.PLAN_DECODE, num_sms=sms)
    compute(h, ws, b)
    check_decode_plan(h, b, num_sms=sms)
    if fits_in_one_run(b, sms * 8):
        check_whole_list_plan(h, b, sms * 8)
    else:
        assert api.plan_get_work(h).tolist() == cost_runs_decode(b, sms * 8)
    api.plan_destroy(h)
