"""Multi-rank host logic of bench.py on CPU (two gloo ranks): the step time is the maximum over
ranks, and the reference arm prints from rank 0 only."""
import io
import os
import contextlib

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import sys
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    got = bench.reduce_max(1.5 + rank * 2.0, "cpu")
    w, r, lr = bench.dist_env()
    out = io.StringIO()
    args = type("A", (), dict(steps=1, warmup=3, ref_tokens=1, cpu_tokens=1))()
    if r != 0:
        with contextlib.redirect_stdout(out):
            bench.run_reference(args)           # ranks other than 0 do no work and print nothing
    q.put((rank, got, (w, r, lr), out.getvalue()))
    dist.destroy_process_group()


def test_two_rank_max_and_rank0_only_printing():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + (os.getpid() % 1000)
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [3.5, 3.5]
    assert [r[2] for r in res] == [(2, 0, 0), (2, 1, 1)]
    assert res[1][3] == ""
