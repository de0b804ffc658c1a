"""The bench's multi-rank logic on CPU: two gloo ranks (world size 2, 127.0.0.1), each with
its own time; the job time must be the slowest rank's, the job throughput the sum of the
ranks' work over that time, and the environment must be read the torchrun way."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        w, r, local = bench.dist_env()
        t = bench.max_over_ranks(1.0 + 2.5 * rank, dist, "cpu")        # rank 1 is the slow one
        tput = bench.job_throughput(w, 1e12, t)
        dist.barrier()
        out.put((rank, w, r, local, t, tput))
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    out = ctx.SimpleQueue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(90)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = sorted(out.get() for _ in range(2))
    for rank, w, r, local, t, tput in got:
        assert (w, r, local) == (2, rank, rank)
        assert t == 3.5                       # the max over ranks
        assert abs(tput - 2 * 1e12 / 3.5 / 1e12) < 1e-12


def test_single_process_needs_no_group():
    import bench
    assert bench.max_over_ranks(4.25, None, "cpu") == 4.25
    assert bench.job_throughput(1, 2e12, 0.5) == 4.0
