"""GPU: a batch split into data-parallel shards, each shard run through the CUDA library on its own rows.

The layer shards by segment (tokens are independent in the forward); the only exchange is the sum of the fp32
dA/dB of a fine-tuning adapter whose segments land on different ranks ("Data-Driven Optimization of GPU
efficiency for Distributed LLM-Adapter Serving", adapter placement and request routing).  One GPU stands in for
the ranks by running the shards one after another; the host sums their gradient pools (the all-reduce) and puts
the rows of y and dX back in global order.  The result must match the float64 oracle of the whole batch, and the
single-call result of the whole batch on the GPU.
"""
import numpy as np
import pytest

import oracle
import workloads
from gpu_util import Dev, compare, to_np, train_blocks
from lora_co_serving_gb300 import shard

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    import lora_co_serving_gb300 as lm
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lm.build()
    lm.library()


def batch():
    return workloads.config5(K=512, N=768, n_adapters=24, n_decode=150, prefill_tokens=500, len_lo=30, len_hi=250,
                             train_len=100)


@pytest.mark.parametrize("world,affine", [(2, False), (3, True)])
def test_shards_reassemble_to_the_whole_batch(world, affine):
    import torch
    wl = batch()
    shards = shard.shard_segments(wl.segs, world, affine=affine)
    if not affine:
        # round-robin placement sends the two fine-tuning segments to different ranks: their adapter's gradient
        # is a sum over ranks
        owners = [r for r, d in enumerate(shards) for s in d["segs"].tolist() if s[3]]
        assert len(set(owners)) == 2
    ys, dxs = [], []
    dA = np.zeros(wl.A.shape, np.float32)
    dB = np.zeros(wl.B.shape, np.float32)
    for d in shards:
        rows = d["rows"]
        sub = workloads.Workload(**{**wl.__dict__, "T": int(rows.shape[0]), "x": wl.x[rows], "dY": wl.dY[rows],
                                    "segs": d["segs"]})
        dev = Dev(sub)
        y = dev.forward()
        gX, gA, gB = dev.backward()
        torch.cuda.synchronize()
        ys.append(to_np(y))
        dxs.append(to_np(gX))
        dA += gA.cpu().numpy()
        dB += gB.cpu().numpy()
    y = shard.gather_rows(shards, ys, wl.T)
    dX = shard.gather_rows(shards, dxs, wl.T)

    ry = oracle.forward_wl(wl)
    rX, rA, rB = oracle.backward_wl(wl)
    trows = wl.train_rows()
    ia, ib = train_blocks(wl)
    compare(y, ry, "y (sharded)")
    compare(dX[trows], rX, "dX (sharded)")
    compare(dA[ia], rA[ia], "dA (sharded, summed over ranks)")
    compare(dB[ib], rB[ib], "dB (sharded, summed over ranks)")

    whole = Dev(wl)
    y1 = to_np(whole.forward())
    gX1, gA1, gB1 = whole.backward()
    torch.cuda.synchronize()
    compare(y, y1, "y (sharded vs one call)")
    compare(dX[trows], to_np(gX1)[trows], "dX (sharded vs one call)")
    compare(dA[ia], gA1.cpu().numpy()[ia], "dA (sharded vs one call)")
    compare(dB[ib], gB1.cpu().numpy()[ib], "dB (sharded vs one call)")
