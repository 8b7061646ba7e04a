"""The bench's multi-rank logic on the CPU: two gloo ranks (world_size 2, 127.0.0.1) agree on
the maximum of their timings, pass the barrier, and only rank 0 runs the reference arm."""
import contextlib
import io
import os
import socket
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    m = bench.dist_max(1.5 * (rank + 1))
    bench.dist_barrier()
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        if rank != 0:
            bench.run_reference(type("A", (), {"steps": 1, "warmup": 3})(), rank, world)
    q.put((rank, m, buf.getvalue()))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_max_and_barrier():
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
    assert [r[1] for r in res] == [3.0, 3.0]
    assert res[1][2] == ""  # rank 1 prints nothing for the reference arm
