"""The multi-GPU form of the benchmark is independent replicas (one per rank, no collective on
the data path): each rank trains on its own token stream and the job's time is the slowest
rank's. These run the same helpers bench.py uses on two gloo ranks on the CPU."""
import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from decoder_only_transformer_05_b300 import synthetic as S  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w, r, _ = bench.dist_setup()
    assert (w, r) == (world, rank)
    wl = dict(S.WORKLOADS["char-bf16"])
    ids = bench.rank_token_batches(wl, rank, 3)
    elapsed = 10.0 + 5.0 * rank             # this replica's time
    worst = bench.max_over_ranks(elapsed, "cpu")
    out.put((rank, ids, worst))
    dist.barrier()
    dist.destroy_process_group()


def test_two_replicas_on_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict()
    for _ in range(2):
        r, ids, worst = q.get(timeout=120)
        got[r] = (ids, worst)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # every rank sees the slowest replica's time
    assert got[0][1] == got[1][1] == 15.0
    # the replicas train on different, reproducible streams
    ids0, ids1 = got[0][0], got[1][0]
    assert ids0.shape == ids1.shape == (3, 64, 257)
    assert not np.array_equal(ids0, ids1)
    wl = dict(S.WORKLOADS["char-bf16"])
    assert np.array_equal(ids1, bench.rank_token_batches(wl, 1, 3))


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(3.5, "cpu") == 3.5


def test_job_throughput_counts_every_replica():
    # 2 replicas x 3 steps x (12 x 1024 tokens x 40 micro-batches) in 1.5 s
    assert bench.job_tokens_per_s(2, 3, 12, 1024, 40, 1.5) == pytest.approx(
        2 * 3 * 12 * 1024 * 40 / 1.5)
