"""bench.py's multi-rank helpers on CPU: two gloo ranks agree on the slowest
time (the maximum over ranks), and the reference arm only runs on rank 0."""
import multiprocessing as mp
import os
import socket

import pytest


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import torch.distributed as td

    import bench
    td.init_process_group("gloo", rank=rank, world_size=world)
    m = bench.max_over_ranks(1.5 + rank, world)
    bench.barrier(world)
    q.put((rank, m))
    td.destroy_process_group()


def test_max_over_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    res = dict(q.get(timeout=120) for _ in ps)
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == {0: 2.5, 1: 2.5}


def test_reference_arm_only_on_rank_zero(capsys):
    import bench
    args = bench.parse_args(["--impl", "reference", "--steps", "1", "--warmup", "0"])
    bench.run_reference(args, rank=1, world=2)
    assert capsys.readouterr().out == ""
