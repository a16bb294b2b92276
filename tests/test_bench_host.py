"""Host-side logic of bench.py: the FLOP counts it uses and the whole-job
aggregation over ranks (world size 2 over gloo on the CPU)."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from block_sparse_masked_mask_gb300 import workloads as W
from conftest import ROOT

sys.path.insert(0, ROOT)
import bench  # noqa: E402


@pytest.mark.parametrize("c", [1, 2, 3, 4, 5])
def test_unmasked_pair_table_matches_oracle(c):
    w = W.make_workload(c, tensors=False)
    assert bench.UNMASKED_PAIRS[c] == oracle.unmasked_pairs(w.kind, w.cu_seqlens, w.meta())


def test_aggregate_is_whole_job_throughput():
    assert bench.aggregate_throughput(1e12, 1, 1.0) == pytest.approx(1.0)
    assert bench.aggregate_throughput(1e12, 4, 0.5) == pytest.approx(8.0)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    # each rank "measured" a different time; the job's time is the slowest
    t = bench.reduce_max(0.010 * (rank + 1), ws)
    v = bench.aggregate_throughput(2e12, ws, t)
    bench.barrier(ws)
    q.put((rank, t, v))
    dist.destroy_process_group()


def test_reduce_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [pytest.approx(0.02)] * 2
    assert [r[2] for r in res] == [pytest.approx(2e12 * 2 / 0.02 / 1e12)] * 2
