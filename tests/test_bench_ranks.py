"""bench.py's multi-rank host logic on CPU: two gloo ranks (spawned processes,
rendezvous on 127.0.0.1) reduce their step times to the slowest one, and the
whole-job value aggregates the replicas."""
import multiprocessing as mp
import os
import socket

from datagen import configs as C


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        q.put((rank, bench.max_over_ranks(2.0 + rank, world)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_report_the_slowest_step():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == {0: 3.0, 1: 3.0}


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(1.25, 1) == 1.25


def test_whole_job_value_aggregates_replicas():
    import bench
    # decode: two replicas each finish one token per 0.128 ms -> 64 us per token for the job
    assert abs(bench.metric_value(C.DECODE, 0.128, 2) - 64.0) < 1e-9
    assert abs(bench.metric_value(C.DECODE, 0.128, 1) - 128.0) < 1e-9
    # prefill: tokens per second of all replicas
    assert abs(bench.metric_value(C.PREFILL, 5.0, 2) - 2 * 4096 / 5e-3) < 1e-6
