"""The N>1 host logic of bench.py on CPU ranks (gloo, world size 2): per-rank
inputs differ (weak scaling, one independent batch per rank), timings reduce
to the slowest rank, and the job's rate counts every rank's bytes."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import torch.distributed as dist

    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        inp = bench.make_inputs(rank, n_move=64)
        digest = int(np.bitwise_xor.reduce(inp["slots"])) ^ int(inp["g"].block_table[0, 0])
        ms = bench.reduce_max([10.0 + 5 * rank, 1.0 * (2 - rank)])
        val = bench.whole_job_gbps(1_000_000_000, world, ms[0])
        q.put((rank, digest, ms, val))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=300) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, d0, ms0, v0), (r1, d1, ms1, v1) = out
    assert d0 != d1, "ranks must draw independent batches"
    assert ms0 == ms1 == [15.0, 2.0], "timings reduce to the slowest rank on every rank"
    assert v0 == v1 == pytest.approx(2 * 1.0 / 15e-3)


def test_reference_arm_other_ranks_exit_quietly(capsys, monkeypatch):
    import argparse

    import bench

    monkeypatch.setenv("RANK", "1")
    bench.run_reference(argparse.Namespace(steps=1, warmup=0))
    assert capsys.readouterr().out == ""
