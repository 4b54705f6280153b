"""The multi-process path of the benchmark on CPU: two ranks over gloo
(127.0.0.1). Ranks hold shares (KV heads) of one pool, with no data-path
collective; the only exchange is the maximum of the per-rank step times,
so the job's rate is set by its slowest rank."""

import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import sys

    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    phases = ["compress", "attend", "decompress"]
    # rank r is slower in a different phase than its peer
    ph = {"compress": 1.0 + rank, "attend": 2.0 - rank, "decompress": 0.5 + 0.25 * rank}
    step, got = bench.max_over_ranks(sum(ph.values()), ph, phases)
    out[rank] = (step, got["compress"], got["attend"], got["decompress"])
    ws, r, _ = bench._dist()
    out[10 + rank] = (ws, r)
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_rank():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank_main, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
        res = dict(out)
    # per-rank sums: rank 0 = 1 + 2 + 0.5 = 3.5, rank 1 = 2 + 1 + 0.75 = 3.75
    for rank in (0, 1):
        step, c, a, d = res[rank]
        assert step == pytest.approx(3.75)
        assert (c, a, d) == pytest.approx((2.0, 2.0, 0.75))
        assert res[10 + rank] == (2, rank)


def test_single_process_is_unchanged():
    import sys

    sys.path.insert(0, ROOT)
    import bench

    step, got = bench.max_over_ranks(1.5, {"a": 1.0, "b": 0.5}, ["a", "b"])
    assert step == 1.5 and got == {"a": 1.0, "b": 0.5}
