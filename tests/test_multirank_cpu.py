"""The N > 1 path of bench.py on CPU: two gloo ranks, each with its own batch (weak
scaling), combined into one whole-job figure with no data-path collective."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from paged_kv_cache_bsr_gb300 import workloads as W
    # each rank draws its own batch of the bench workload (smaller here) from its own seed
    b = W.llama3_decode(seed=bench.rank_seed(rank), batch=4)
    ms = 0.10 * (rank + 1)  # the ranks' step times differ; the job takes the slowest
    ms_max, total = bench.combine_over_ranks(ms, b.kv_bytes())
    out[rank] = (ms_max, total, b.kv_bytes(), float(b.kv_lens[0]))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_combine_to_whole_job_figures():
    world = 2
    out = mp.get_context("spawn").Manager().dict()
    mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
    r0, r1 = out[0], out[1]
    assert r0[0] == r1[0] == pytest.approx(0.2)               # max over ranks
    assert r0[1] == r1[1] == r0[2] + r1[2]                     # bytes of every rank
    assert r0[3] != r1[3]                                       # each rank has its own batch
    value = r0[1] / (r0[0] * 1e-3) / 1e9                        # bench's whole-job GB/s
    assert value == pytest.approx((r0[2] + r1[2]) / 0.2e-3 / 1e9)
