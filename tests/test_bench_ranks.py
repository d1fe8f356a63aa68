"""The benchmark's multi-process plumbing on CPU (gloo, two ranks): every
rank times its own replica of the layer and the reported step time is the
maximum over ranks; the reference arm runs on rank 0 only."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        got = bench.max_over_ranks(10.0 + 7.5 * rank)
        ws, r, local = bench.dist_env()
        q.put((rank, got, ws, r, local))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_step_time_is_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(2))
    assert [r[1] for r in res] == [17.5, 17.5]
    assert [(r[2], r[3], r[4]) for r in res] == [(2, 0, 0), (2, 1, 1)]


def test_single_process_max_is_identity():
    import bench
    assert bench.max_over_ranks(3.25) == 3.25


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class A:
        config, T, steps, warmup, gpus = 1, 8, 1, 3, 2
    assert bench.run_reference(A) is None
    assert capsys.readouterr().out == ""
