"""Batch sharding with the dP all-reduce, on CPU with two gloo ranks.

Each rank takes its contiguous slice of the batch, computes the gradients of
that slice with the oracle (fp64), and sums its partial dP_h with the other
rank through parallax_local_linear_fwd_b300.shard.allreduce_dP.  The summed
dP must equal the full-batch oracle's, and dq, dk, dv of each slice must equal
the full-batch ones on those rows: the layer's batches are independent except
for dP_h, which sums over the batch.
"""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import plx_synth
from parallax_local_linear_fwd_b300.shard import allreduce_dP, shard_range


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs():
    inp = plx_synth.generate(5, 2, 9, 4, "bf16", seed=31, p_std=0.3, backward=True)
    f = {n: plx_synth.widen(inp[n]) for n in ("q", "k", "v", "dout")}
    f["P"] = inp["P"].astype(np.float64)
    return f


def _worker(rank, world, port, q):
    import oracle
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    dist.init_process_group("gloo", rank=rank, world_size=world)
    f = _inputs()
    lo, hi = shard_range(f["q"].shape[0], rank, world)
    sl = {n: f[n][lo:hi] for n in ("q", "k", "v", "dout")}
    dq, dk, dv, dP = oracle.backward(sl["q"], sl["k"], sl["v"], f["P"], sl["dout"], nthreads=1)
    dP_t = torch.from_numpy(dP.copy())
    allreduce_dP(dP_t)
    q.put((rank, lo, hi, dq, dk, dv, dP_t.numpy()))
    dist.barrier()
    dist.destroy_process_group()


def test_batch_shards_with_dP_allreduce_match_the_full_batch():
    import oracle
    oracle.build()
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted((q.get(timeout=120) for _ in range(world)), key=lambda r: r[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    f = _inputs()
    rdq, rdk, rdv, rdP = oracle.backward(f["q"], f["k"], f["v"], f["P"], f["dout"], nthreads=1)
    covered = []
    for rank, lo, hi, dq, dk, dv, dP in res:
        covered += list(range(lo, hi))
        np.testing.assert_allclose(dq, rdq[lo:hi], rtol=0, atol=1e-12)
        np.testing.assert_allclose(dk, rdk[lo:hi], rtol=0, atol=1e-12)
        np.testing.assert_allclose(dv, rdv[lo:hi], rtol=0, atol=1e-12)
        # every rank holds the full-batch projector gradient after the sum
        np.testing.assert_allclose(dP, rdP, rtol=1e-12, atol=1e-12)
    assert covered == list(range(f["q"].shape[0]))
    # without the exchange a rank's dP is only its own slice's share
    lo, hi = res[0][1], res[0][2]
    part = oracle.backward(f["q"][lo:hi], f["k"][lo:hi], f["v"][lo:hi], f["P"], f["dout"][lo:hi], nthreads=1)[3]
    assert np.abs(part - rdP).max() > 1e-3


def test_shard_range_partitions_every_item_once():
    for n in (0, 1, 5, 8, 17):
        for world in (1, 2, 3, 8):
            ranges = [shard_range(n, r, world) for r in range(world)]
            items = [i for lo, hi in ranges for i in range(lo, hi)]
            assert items == list(range(n))
            sizes = [hi - lo for lo, hi in ranges]
            assert max(sizes) - min(sizes) <= 1


def test_allreduce_is_identity_without_a_process_group():
    x = torch.arange(8, dtype=torch.float32).view(2, 2, 2)
    assert torch.equal(allreduce_dP(x.clone()), x)
