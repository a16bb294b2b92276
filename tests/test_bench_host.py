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


@pytest.mark.parametrize("c", [1, 2, 3, 4, 5, 6, 7, 8])
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


def test_profiled_traffic_only_for_the_profiled_kernel_source(tmp_path, monkeypatch):
    """The roofline's DRAM traffic comes from the committed ncu summary, scaled by
    heads, and is dropped (None) once the kernel source differs from the one
    that was captured."""
    import hashlib
    fields = {}
    for line in open(bench.TRAFFIC_PROFILE):
        if ":" in line and not line.startswith(("|", "#", " ", "*")):
            k, _, v = line.partition(":")
            fields[k.strip()] = v.strip()
    src = tmp_path / "kernel.cu"
    src.write_bytes(b"// some other kernel\n")
    monkeypatch.setattr(bench, "FWD_SOURCE", str(src))
    assert bench.profiled_traffic(5, 32) == (None, None)
    # a source whose hash matches the capture: traffic scales with the head count
    monkeypatch.setattr(hashlib, "sha256", lambda b: type("H", (), {
        "hexdigest": lambda self: fields["source_sha256"]})())
    t, note = bench.profiled_traffic(5, 32)
    assert t == int(fields["traffic_bytes_per_launch_h8"]) * 32 / int(fields["heads"])
    assert "scaled" in note
    assert bench.profiled_traffic(3, 32) == (None, None)
