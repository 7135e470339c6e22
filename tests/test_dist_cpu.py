"""The N>1 host logic of bench.py on CPU: two gloo ranks, barrier, the
max-over-ranks timing reduction, independent per-rank head sets, and the
reference arm running on rank 0 only."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import plx_synth


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "WORLD_SIZE": str(world),
                       "RANK": str(rank), "LOCAL_RANK": str(rank)})
    w, r = bench.dist_init("gloo")
    assert (w, r) == (world, rank)
    bench.barrier(world)
    t = bench.max_over_ranks(10.0 + rank, world)
    seed = bench.rank_seed(3, rank)
    inp = plx_synth.generate(1, 1, 8, 4, "bf16", seed=seed)
    gathered = [None] * world
    dist.all_gather_object(gathered, inp["q"].tobytes())
    q.put((rank, t, len(set(gathered))))
    bench.barrier(world)
    dist.destroy_process_group()


def test_two_gloo_ranks_barrier_and_max_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    assert [r[1] for r in res] == [11.0, 11.0]   # every rank sees the max over ranks
    assert all(r[2] == world for r in res)        # every rank drew its own inputs


def test_reference_arm_runs_on_rank_zero_only(capsys):
    class A:
        workload, steps, warmup = "c4", 1, 3
    bench.run_reference(A, world=2, rank=1)
    assert capsys.readouterr().out == ""


def test_single_process_helpers_are_identity():
    assert bench.max_over_ranks(3.5, 1) == 3.5
    bench.barrier(1)
    assert bench.rank_seed(3, 0) == 3 and bench.rank_seed(3, 1) != 3


def test_clock_summary_flags_reasons():
    rows = [["0", "1900", "2032", "900", "0x4", "Not Active", "Not Active", "Not Active", "Active"],
            ["0", "1950", "2032", "950", "0x4", "Not Active", "Not Active", "Not Active", "Not Active"]]
    s = bench.summarize_clocks(rows)
    assert s["sm_mhz"] == 1925 and s["sm_max_mhz"] == 2032 and s["reasons"] == ["sw_power_cap"]
