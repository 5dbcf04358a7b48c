"""Data-parallel sharding of one batch, world size 2 over gloo (CPU only).

Each rank runs the float64 oracle on its shard; the fp32-gradient exchange is an all-reduce (sum) of the
pool-shaped dA/dB.  The reassembled outputs must equal the single-process oracle.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
import workloads
from lora_co_serving_gb300 import shard


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _small():
    return workloads.config5(K=40, N=48, n_adapters=10, n_decode=30, prefill_tokens=60, len_lo=5, len_hi=30,
                             train_len=12)


def _worker(rank, world, port, affine, outdir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    wl = _small()
    # affine: each adapter on one rank; round-robin: the two fine-tuning segments land on different ranks,
    # so their adapter's gradient is the sum over ranks
    shards = shard.shard_segments(wl.segs, world, affine=affine)
    d = shards[rank]
    rows = d["rows"]
    x, dY = wl.x[rows], wl.dY[rows]
    y = oracle.forward(x, wl.Wt, wl.A, wl.B, wl.a_off, wl.b_off, wl.rank, wl.scale, d["segs"])
    _, dA, dB = oracle.backward(x, wl.Wt, wl.A, wl.B, wl.a_off, wl.b_off, wl.rank, wl.scale, d["segs"], dY,
                                want_dx=False)
    gA = torch.from_numpy(dA)
    gB = torch.from_numpy(dB)
    dist.all_reduce(gA)
    dist.all_reduce(gB)
    ys = [None] * world
    dist.all_gather_object(ys, y)
    if rank == 0:
        yg = shard.gather_rows(shards, ys, wl.T)
        np.save(os.path.join(outdir, "y.npy"), yg)
        np.save(os.path.join(outdir, "dA.npy"), gA.numpy())
        np.save(os.path.join(outdir, "dB.npy"), gB.numpy())
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("affine", [True, False])
def test_two_rank_shard_matches_single(tmp_path, affine):
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, affine, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    wl = _small()
    y = oracle.forward_wl(wl)
    _, dA, dB = oracle.backward_wl(wl, want_dx=False)
    assert np.allclose(np.load(tmp_path / "y.npy"), y, rtol=1e-12, atol=1e-12)
    assert np.allclose(np.load(tmp_path / "dA.npy"), dA, rtol=1e-12, atol=1e-12)
    assert np.allclose(np.load(tmp_path / "dB.npy"), dB, rtol=1e-12, atol=1e-12)


def test_affine_placement_keeps_adapters_whole():
    wl = workloads.config5(K=16, N=16)
    shards = shard.shard_segments(wl.segs, 4, affine=True)
    owner = {}
    for r, d in enumerate(shards):
        for st, ln, a, tr in d["segs"].tolist():
            if a >= 0:
                assert owner.setdefault(a, r) == r
    assert sum(d["rows"].shape[0] for d in shards) == wl.T
    loads = [d["rows"].shape[0] for d in shards]
    assert max(loads) - min(loads) <= 1024 + 64   # within one large segment of balance
    allrows = np.sort(np.concatenate([d["rows"] for d in shards]))
    assert np.array_equal(allrows, np.arange(wl.T))
