"""The multi-rank path of bench.py on CPU: two ranks over gloo (127.0.0.1).

The work is replicated (every rank runs the whole workload on its own GPU,
no collective on the data path), so what the ranks share is the timing:
a barrier around the timed region, the slowest rank's time, and the
whole-job rate computed from it.  These are the bench's own functions, run
here without a GPU.
"""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, seconds, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        import bench
        w, r, local = bench._dist()
        bench._barrier(w)
        slowest = bench._max_over_ranks(seconds[rank], w, torch.device("cpu"))
        rate = bench._whole_job_rate(10.0, 4, w, slowest)
        bench._barrier(w)
        q.put((rank, w, r, local, slowest, rate))
    finally:
        dist.destroy_process_group()


def test_two_replicas_share_the_slowest_time_and_the_whole_job_rate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    seconds = [1.5, 2.5]
    procs = [ctx.Process(target=_worker, args=(r, 2, port, seconds, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        res = sorted(q.get(timeout=120) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert all(p.exitcode == 0 for p in procs)
    for rank, (r_rank, w, r, local, slowest, rate) in enumerate(res):
        assert (r_rank, w, r, local) == (rank, 2, rank, rank)
        assert slowest == 2.5                          # every rank reports the slowest rank's time
        assert rate == pytest.approx(10.0 * 4 * 2 / 2.5)   # work of both ranks over that time


def test_single_process_needs_no_process_group():
    import bench
    assert bench._dist()[0] == int(os.environ.get("WORLD_SIZE", "1"))
    assert bench._max_over_ranks(3.0, 1, torch.device("cpu")) == 3.0
    assert bench._whole_job_rate(10.0, 4, 1, 2.0) == 20.0
