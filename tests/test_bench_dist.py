"""The multi-rank bench path on CPU: two gloo ranks started the way torchrun
starts them (RANK / WORLD_SIZE / MASTER_* in the environment) agree on the
max-over-ranks step time, pass the timing barriers, and only rank 0 runs the
reference arm."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update({"RANK": str(rank), "LOCAL_RANK": str(rank), "WORLD_SIZE": str(world),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    w, r, local = bench.dist_setup()
    try:
        bench.barrier(w)
        elapsed = 10.0 * (r + 1)                  # rank-specific "step time"
        got = bench.max_over_ranks(elapsed, w, "cpu")
        bench.barrier(w)

        class Args:
            workload, steps, warmup = "tiny_256", 1, 1
        ret = bench.run_reference(Args, w, r) if r != 0 else None
        q.put((r, w, got, ret))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_and_skip_reference_on_other_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
    for p in procs:
        if p.is_alive():
            p.kill()
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = sorted(q.get(timeout=10) for _ in range(2))
    assert [r[0] for r in res] == [0, 1]
    assert all(r[1] == 2 for r in res)
    assert all(r[2] == 20.0 for r in res)       # max over ranks on every rank
    assert res[1][3] == 0                       # rank 1: reference arm exits 0 without work


def test_single_process_defaults():
    sys.path.insert(0, ROOT)
    import bench
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        assert k not in os.environ or os.environ[k] in ("0", "1")
    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5
