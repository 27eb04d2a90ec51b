"""bench.py's multi-rank bookkeeping on CPU: two gloo ranks, one replica each (no data-path
collective); the reported rate is the units of all ranks over the slowest rank's time, and
the reference arm runs on rank 0 only."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE="2",
                      LOCAL_RANK=str(rank))
    import bench
    import torch.distributed as dist
    r, ws, local = bench.dist_setup(2, backend="gloo")
    assert (r, ws, local) == (rank, 2, rank)
    secs = [2.0, 4.0][rank]          # rank 1 is the slow one
    bench.barrier(ws)
    out[rank] = (bench.max_over_ranks(secs, ws), bench.whole_job_rate(100, secs, ws))
    # the reference arm works on rank 0 only; other ranks return without work
    if rank == 1:
        class A:
            pass
        assert bench.run_reference(A()) is None
    dist.destroy_process_group()


def test_two_gloo_ranks_aggregate():
    mp_ctx = mp.get_context("spawn")
    with mp_ctx.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()
        procs = [mp_ctx.Process(target=_rank, args=(r, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
        assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
        for r in range(2):
            mx, rate = out[r]
            assert mx == 4.0
            assert rate == pytest.approx(2 * 100 / 4.0)
