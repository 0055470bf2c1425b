"""The multi-process path of bench.py on CPU (gloo, world size 2, 127.0.0.1): every rank runs an
independent replica, the job's time is the slowest rank's, throughput counts all ranks' tokens,
and the reference arm prints on rank 0 only.  No GPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        local = [12.5, 17.25][rank]
        ms = bench.max_over_ranks(local)
        q.put((rank, ms, bench.replica_throughput(16384, 10, world, ms)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput_with_gloo():
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
    assert [r[1] for r in res] == [17.25, 17.25]           # both ranks see the slowest time
    assert res[0][2] == res[1][2] == pytest.approx(16384 * 10 * 2 / 0.01725)


def test_single_rank_is_identity():
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.replica_throughput(100, 4, 1, 2.0) == pytest.approx(200000.0)


def test_reference_arm_prints_on_rank_zero_only(monkeypatch):
    import argparse
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = argparse.Namespace(seed=0, ref_tokens=4, warmup=0, steps=1)
    assert bench.run_reference(args, bench.moe_inputs.CONFIGS["tiny"]) is None
