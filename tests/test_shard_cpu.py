"""The multi-GPU forms of the path, on CPU: a batch partitioned by request over ranks
(no exchange), and one long request split by key range over two gloo ranks whose
partial states are all-gathered and merged (the one exchange step).  Each rank's
attention is computed by the fp64 oracle here; the exchange and the merge are the
parts under test."""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from paged_kv_cache_bsr_gb300 import shard, workloads as W  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_partition_covers_every_request_once_and_balances():
    rng = np.random.default_rng(3)
    uniform = [int(c) for c in rng.integers(1, 500, size=37)]
    zipf = W.zipf_lengths(200, 1.1, 16, 131072, seed=5)       # a heavy-tailed request mix
    for costs in (uniform, zipf):
        for world in (1, 2, 3, 8):
            parts = shard.partition_requests(costs, world)
            assert sorted(r for p in parts for r in p) == list(range(len(costs)))
            loads = [sum(costs[r] for r in p) for p in parts]
            # longest first: no rank ends more than one request's cost above another
            assert max(loads) - min(loads) <= max(costs)
    # longest first: 5 -> rank 0, 4 -> rank 1, 2 -> rank 1 (4 < 5), 1 -> rank 0: loads 6 and 6
    assert shard.partition_requests([5, 1, 4, 2], 2) == [[0, 1], [2, 3]]
    with pytest.raises(ValueError):
        shard.partition_requests([1], 0)


def test_split_sequence_pieces_tile_the_key_range():
    b = W.make_paged_batch(qo_lens=[1, 1], kv_lens=[37, 1000], num_qo_heads=4, num_kv_heads=2, head_dim=16,
                           page_size=16, dtype=torch.float16, seed=2)
    for world in (1, 2, 3, 7, 80):
        pieces = shard.split_sequence(b, 1, world)
        assert len(pieces) == world
        assert sum(p.kv_lens[0] for p in pieces) == 1000
        assert torch.equal(torch.cat([p.kv_indices for p in pieces]), b.kv_indices[int(b.kv_indptr[1]):])
    causal = W.make_paged_batch(qo_lens=[5], kv_lens=[40], num_qo_heads=4, num_kv_heads=2, head_dim=16,
                                page_size=16, dtype=torch.float16, seed=2, causal=True)
    with pytest.raises(ValueError):
        shard.split_sequence(causal, 0, 2)


def _split_rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import oracle
    from paged_kv_cache_bsr_gb300 import shard as S, workloads as Wk
    b = Wk.make_paged_batch(qo_lens=[1], kv_lens=[20011], num_qo_heads=8, num_kv_heads=2, head_dim=64,
                            page_size=16, dtype=torch.bfloat16, seed=11, logits_cap=30.0)
    piece = S.split_sequence(b, 0, world)[rank]
    o, lse = oracle.attention_of(piece)                       # this rank's partial state (fp64)
    os_, ls = S.allgather_states(torch.from_numpy(o), torch.from_numpy(lse))
    mo, ml = oracle.merge_states(list(os_.numpy()), list(ls.numpy()))
    ref_o, ref_lse = oracle.attention_of(b)
    out[rank] = (float(np.abs(mo - ref_o).max()), float(np.abs(ml - ref_lse).max()), tuple(os_.shape))
    dist.destroy_process_group()


def test_two_ranks_split_one_long_request_and_merge():
    world = 2
    out = mp.get_context("spawn").Manager().dict()
    mp.spawn(_split_rank, args=(world, _free_port(), out), nprocs=world, join=True)
    for rank in range(world):
        do, dl, shape = out[rank]
        assert shape[0] == world
        assert do < 1e-12 and dl < 1e-12


def _partition_rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import oracle
    from paged_kv_cache_bsr_gb300 import shard as S, workloads as Wk
    b = Wk.llama3_decode(seed=21, batch=6)
    mine = S.partition_requests(S.request_costs(b), world)[rank]
    sub = Wk.sub_batch(b, mine)
    o, lse = oracle.attention_of(sub)                         # no exchange: these rows are this rank's
    ref_o, ref_lse = oracle.attention_of(b, rows=mine)
    out[rank] = (mine, float(np.abs(o - ref_o).max()), float(np.abs(lse - ref_lse).max()))
    dist.destroy_process_group()


def test_two_ranks_partition_requests_without_exchange():
    world = 2
    out = mp.get_context("spawn").Manager().dict()
    mp.spawn(_partition_rank, args=(world, _free_port(), out), nprocs=world, join=True)
    assert sorted(out[0][0] + out[1][0]) == list(range(6))
    for rank in range(world):
        assert out[rank][1] == 0.0 and out[rank][2] == 0.0
