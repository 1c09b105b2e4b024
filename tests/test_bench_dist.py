"""The multi-rank plumbing of bench.py on CPU: two gloo ranks, as torchrun would start them.

Checks that timings reduce to the slowest rank, work sums over ranks, barriers pass, and
the reference arm runs on rank 0 only (the other rank exits without work)."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import bench
    r, w = bench.dist_init("gloo")
    bench.barrier()
    out = {
        "rank": r, "world": w,
        "max": bench.max_over_ranks(1.5 if r == 1 else 0.5),
        "sum": bench.sum_over_ranks(10.0 * (r + 1)),
    }
    args = bench.parse_args(["--impl", "reference", "--steps", "2", "--warmup", "3"])
    if r != 0:
        rr, line = bench.reference_arm(args)
        out["ref_line"] = line
    bench.barrier()
    import torch.distributed as dist
    dist.destroy_process_group()
    q.put(out)


def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    res.sort(key=lambda d: d["rank"])
    for d in res:
        assert d["world"] == 2
        assert d["max"] == 1.5
        assert d["sum"] == 30.0
    assert res[1]["ref_line"] is None
