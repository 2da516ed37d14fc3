"""The N > 1 path of bench.py (replicas, one process per GPU) on CPU: two gloo
ranks set up the process group the way bench.py does, meet at its barrier and
agree on the max over ranks of their timings."""
import multiprocessing as mp
import os
import socket
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    r, w, _, pg = bench.dist_setup(None)
    bench.barrier(pg)
    m = bench.max_over_ranks(pg, 10.0 * (r + 1))
    out.put((r, w, m, dist.get_backend()))
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_max():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [x[0] for x in res] == [0, 1]
    assert all(x[1] == 2 and x[2] == 20.0 and x[3] == "gloo" for x in res)
