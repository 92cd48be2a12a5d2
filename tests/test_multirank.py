"""The multi-rank side of bench.py on CPU (gloo, world size 2): replicas
verify their own batches, the timed region is the slowest rank's, and the
whole-job rate counts every rank's rounds.  No GPU."""
import os
import queue
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        ms = (12.5, 20.0)[rank]  # this rank's timed region
        total = bench.max_over_ranks(ms, world, torch.device("cpu"))
        rate = bench.whole_job_rate(10, total, world)
        seeds = [bench.synth.large(s + 16 * rank, B=1).uniforms[0, :4].tolist()
                 for s in range(2)]
        out.put((rank, total, rate, seeds))
    finally:
        dist.destroy_process_group()


def test_two_ranks_slowest_time_and_whole_job_rate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q))
             for r in range(2)]
    for p in procs:
        p.start()
    try:
        res = sorted(q.get(timeout=180) for _ in range(2))
    except queue.Empty:
        raise AssertionError("a rank did not report")
    finally:
        for p in procs:
            p.join(60)
    assert [p.exitcode for p in procs] == [0, 0]
    for rank, total, rate, _ in res:
        assert total == 20.0
        assert abs(rate - 2 * 10 / 0.020) < 1e-9
    assert res[0][3] != res[1][3]  # each rank draws its own batches


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(7.0, 1, torch.device("cpu")) == 7.0
    assert bench.whole_job_rate(5, 10.0, 1) == 500.0
