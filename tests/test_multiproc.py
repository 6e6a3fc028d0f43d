"""Multi-process host logic on CPU (gloo, world size 2).

With more than one GPU the benchmark runs independent replicas: each rank
processes its own batch and the job's time is the maximum over ranks.  These
tests cover that reduction, and failure detection on the host: a rank that
never joins makes the other rank's next collective fail after a short
process-group timeout instead of hanging."""
import datetime
import multiprocessing as mp
import os
import socket
import sys
import traceback

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _max_worker(rank, world, port, q):
    try:
        sys.path.insert(0, ROOT)
        import torch
        import torch.distributed as dist
        import bench
        dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world,
                                timeout=datetime.timedelta(seconds=60))
        out = bench.max_over_ranks([10.0 + rank, 5.0 - rank], torch.device("cpu"))
        dist.destroy_process_group()
        q.put((rank, out))
    except Exception:
        q.put((rank, traceback.format_exc()))


def _put_and_exit(q, item):
    q.put(item)
    q.close()
    q.join_thread()      # flush before the abrupt exit
    os._exit(0)


def _absent_worker(rank, world, port, q):
    try:
        import torch
        import torch.distributed as dist
        dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world,
                                timeout=datetime.timedelta(seconds=3))
        if rank == 1:
            _put_and_exit(q, (rank, "left"))   # leaves between steps, nothing in flight
        try:
            t = torch.ones(1)
            dist.all_reduce(t)   # the partner never joins
            msg = "completed"
        except Exception as e:   # the collective must fail, not hang
            msg = f"error:{type(e).__name__}"
        _put_and_exit(q, (rank, msg))
    except Exception:
        q.put((rank, traceback.format_exc()))


def _run(target, world=2, timeout=120):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=target, args=(r, world, port, q)) for r in range(world)]
    for p in ps:
        p.start()
    res = dict(q.get(timeout=timeout) for _ in range(world))
    for p in ps:
        p.join(timeout=30)
        if p.is_alive():
            p.kill()
    return res


def test_max_over_ranks_gloo():
    res = _run(_max_worker)
    for r in range(2):
        assert res[r] == [11.0, 5.0], res[r]


def test_absent_rank_is_detected_not_hung():
    res = _run(_absent_worker)
    assert res[1] == "left"
    assert res[0].startswith("error:"), res[0]
