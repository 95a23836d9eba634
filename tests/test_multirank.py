"""Host logic of the multi-GPU bench path (independent replicas), run as two
gloo ranks on CPU: each rank reports its own step time, all agree on the
slowest, and the whole-job value counts every rank's tokens."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = bench.max_over_ranks(1.0 + rank * 0.5, world)
    v = bench.whole_job_tokens_per_s(16, world, ms)
    out.put((rank, ms, v))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(2))
    assert [r[1] for r in res] == [1.5, 1.5]
    assert all(abs(r[2] - 2 * 16 / 1.5e-3) < 1e-6 for r in res)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(2.5, 1) == 2.5
    assert bench.whole_job_tokens_per_s(16, 1, 2.0) == 8000.0
