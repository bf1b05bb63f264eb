"""The bench's multi-rank host logic with two gloo ranks on the CPU (one
process per rank, as torchrun would start them): the rank environment, the
max-over-ranks timed region, the whole-job aggregate, and the reference arm
doing its work on rank 0 only."""
import io
import os
import socket
import contextlib

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, q):
    import torch.distributed as dist
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(ws), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        got_ws, got_rank, got_local = bench.dist_env()
        slowest = bench.max_over_ranks(1.0 + rank, got_ws)        # rank r "took" 1 + r seconds
        value = bench.job_throughput(10.0, got_ws, slowest)      # 10 units a rank
        # the reference arm prints its line on rank 0 only
        class A:
            workload, steps, warmup = "2b", 1, 0
        out = io.StringIO()
        with contextlib.redirect_stdout(out):
            if rank != 0:
                bench.run_reference(A())
        q.put((rank, got_ws, got_rank, got_local, slowest, value, out.getvalue()))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ws, got_rank, local, slowest, value, printed in res:
        assert (ws, got_rank, local) == (2, rank, rank)
        assert slowest == 2.0                                  # the slower rank's time, on every rank
        assert value == pytest.approx(10.0 * 2 / 2.0)          # both ranks' units over the slowest time
        if rank == 1:
            assert printed == ""                               # non-zero ranks of the reference arm exit silently


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.job_throughput(7.0, 1, 2.0) == 3.5
