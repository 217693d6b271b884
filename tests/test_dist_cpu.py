"""Multi-rank host logic of the benchmark on CPU (gloo, world size 2).

Each rank serves an independent batch (data-parallel attention), so the only
cross-rank work is reducing the timing: bytes are summed, seconds take the
maximum, and the whole-job throughput is total bytes over the slowest rank."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    from decode_attention_mfa_gb300 import dist as mdist
    r, w, lr = mdist.init("gloo")
    assert (r, w, lr) == (rank, world, rank)
    mdist.barrier()
    mx = mdist.reduce_scalar(1.0 + rank, "max")
    sm = mdist.reduce_scalar(10.0 * (rank + 1), "sum")
    total_bytes, max_s = mdist.aggregate(bytes_done=100.0 * (rank + 1), seconds=0.5 + rank)
    many_b, many_s = mdist.aggregate_many([1.0 + rank, 2.0], [0.25 * (rank + 1), 3.0 - rank])
    out[rank] = (mx, sm, total_bytes, max_s, tuple(many_b), tuple(many_s))
    mdist.finalize()


def test_two_rank_timing_reduction():
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(2):
        assert out[r] == (2.0, 30.0, 300.0, 1.5, (3.0, 4.0), (0.5, 3.0))


def test_single_process_is_identity(monkeypatch):
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    from decode_attention_mfa_gb300 import dist as mdist
    assert mdist.init() == (0, 1, 0)
    assert mdist.aggregate(5.0, 2.0) == (5.0, 2.0)
    assert mdist.aggregate_many([5.0, 6.0], [2.0, 1.0]) == ([5.0, 6.0], [2.0, 1.0])
