"""The replica path of bench.py (one independent drafter per rank, no data-path
collective): ranks agree on the max-over-ranks time used for the whole-job
rate.  Two gloo ranks on the CPU."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
mp = pytest.importorskip("torch.multiprocessing")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    r, w, _ = bench.dist_setup(world)
    t = bench.reduce_max(10.0 * (rank + 1), w, "cpu")
    bench.barrier(w)
    out.put((r, w, t))
    torch.distributed.destroy_process_group()


def test_two_gloo_ranks_agree_on_max_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == [(0, 2, 20.0), (1, 2, 20.0)]
