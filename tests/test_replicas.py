"""The N > 1 benchmark path on CPU: two gloo ranks run bench.py's cross-rank logic
(max-over-ranks timing, whole-job throughput).  The decode path shards as independent
replicas -- no collective on the data path -- so this is the only multi-rank logic."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench

    dist, r, w, local = bench.dist_setup()
    assert (r, w, local) == (rank, world, rank)
    # each replica reports its own step timings; the job takes the slowest
    mine = [10.0 + rank, 20.0 - rank]
    got = bench.max_over_ranks(dist, mine)
    value = bench.job_throughput(w, 1_000_000, 5, got[0])
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, got, value))


def test_two_gloo_ranks_max_timing_and_job_value():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, value in out:
        assert got == [11.0, 20.0]  # max over ranks, element-wise
        # 2 ranks x 1 MB x 5 steps in 11 ms
        assert value == pytest.approx(2 * 1e6 * 5 / 11e-3 / 1e9)


def test_single_process_needs_no_group():
    import bench

    assert bench.max_over_ranks(None, [3, 4]) == [3.0, 4.0]
    assert bench.job_throughput(1, 2_000_000_000, 1, 1000.0) == pytest.approx(2.0)
