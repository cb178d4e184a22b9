"""The N > 1 path of bench.py is N independent replicas ("replicas only": the hot path has no
exchange step). Its host logic - process group set-up, the barriers around the timed
region, the max over ranks of the timed duration and the reference arm's rank-0-only rule -
runs here as two gloo ranks on the CPU."""

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
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    import bench
    import torch.distributed as dist
    r, local, w = bench.dist_setup()
    assert (r, local, w) == (rank, rank, world) and dist.get_backend() == "gloo"
    bench.barrier(w)
    t = bench.max_over_ranks(1.5 + rank, w)    # each rank's own timed seconds
    bench.barrier(w)
    rc = None
    if rank != 0:
        rc = bench.reference_main(bench.parse_args(["--impl", "reference", "--steps", "1", "--warmup", "0"]))
    out.put((rank, t, rc))
    dist.destroy_process_group()


def test_two_replicas_share_the_max_duration():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [t for _, t, _ in res] == [2.5, 2.5]      # both ranks report the slowest rank's time
    assert res[1][2] == 0                             # the reference arm: ranks > 0 exit 0 at once
