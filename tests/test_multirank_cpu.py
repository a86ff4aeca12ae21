"""The N > 1 host logic of bench.py on CPU: two gloo ranks.

With several GPUs each rank runs an independent replica of the step; the
reported time is the slowest rank's (an all-reduce-max) and `value` sums the
work of all ranks over that time.  No GPU and no NCCL: gloo on 127.0.0.1.
"""
import importlib.util
import os
import socket

import pytest
import torch.multiprocessing as tmp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out_q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        b = _bench()
        w, r, _ = b.dist_setup()
        b.barrier(w)
        t_max = b.max_over_ranks(times[r], w)
        out_q.put((r, w, t_max))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    ctx = tmp.get_context("spawn")
    q = ctx.Queue()
    times = [3.25, 4.5]
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, times, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r for r, _, _ in res] == [0, 1]
    assert all(w == 2 for _, w, _ in res)
    assert all(t == max(times) for _, _, t in res)


def test_single_rank_is_identity():
    b = _bench()
    assert b.max_over_ranks(1.5, 1) == 1.5
    assert b.dist_setup()[0] == int(os.environ.get("WORLD_SIZE", "1"))
