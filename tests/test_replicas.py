"""The replicas-only multi-GPU path of bench.py, host side, on CPU: two gloo ranks agree
on the step count and take the slowest rank's times (no GPU, no data-path collective)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        steps = bench.max_over_ranks([50 + 7 * rank], world)
        times = bench.max_over_ranks([1.5 - rank, 2.0 + rank], world)
        dist.barrier()
        out.put((rank, steps, times))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_maximum():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == [(0, [57.0], [1.5, 3.0]), (1, [57.0], [1.5, 3.0])]


def test_single_rank_is_the_identity():
    import bench
    assert bench.max_over_ranks([3, 4.5], 1) == [3.0, 4.5]


if __name__ == "__main__":
    pytest.main([__file__])
