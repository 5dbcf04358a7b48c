"""GPU parity of a decoder layer's LoRA projections chained on one stream.

The layer of Llama 3-8B (the model of "DeltaServe: Host-Agnostic Co-Serving of Inference and Fine-Tuning for
LLMs", section 4.1, whose fine-tuning adapter sits on the attention projections) at reduced width: q|k|v as one
sliced call, o, gate|up as one sliced call, down.  Attention and the MLP activation stay outside the library, so
each projection reads its own seeded input.  The forward runs q|k|v -> o -> gate|up -> down and the backward the
reverse, all enqueued back to back on one stream with ONE workspace sized for the largest call and no host
synchronisation in between; every output is compared with the float64 oracle, and with the same chain run with a
fresh workspace per call (bitwise: a call must not depend on what an earlier call left in the workspace).
"""
import numpy as np
import pytest

import oracle
import workloads
from oracle import sliced as osl
from gpu_util import Dev, compare, to_np

pytestmark = pytest.mark.gpu

ORDER = ["qkv", "o", "gate_up", "down"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    import lora_co_serving_gb300 as lm
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lm.build()
    lm.library()


def layer():
    return workloads.llama_layer(hidden=512, kv=256, inter=768, n_adapters=24, n_decode=120, prefill_tokens=400,
                                 len_lo=30, len_hi=200, train_len=96)


def ws_bytes(d, wl):
    import lora_co_serving_gb300 as lm
    if wl.bounds is not None:
        return lm.sliced_workspace_size(wl.T, wl.K, wl.N, lm.BF16, d.pool, wl.bounds, wl.segs)
    return lm.workspace_size(wl.T, wl.K, wl.N, lm.BF16, d.pool, wl.segs)


def chain(L, devs, shared):
    """Forward over the four projections, then the backward in reverse order; returns {name: (y, dX, dA, dB)}."""
    import torch
    import lora_co_serving_gb300 as lm
    ws = None
    if shared:
        need = max(ws_bytes(devs[n], L[n]) for n in ORDER)
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    out = {}
    for n in ORDER:
        d, wl = devs[n], L[n]
        if wl.bounds is not None:
            y = lm.sliced_forward(d.x, d.Wt, d.pool, wl.bounds, d.segs, workspace=ws)
        else:
            y = lm.forward(d.x, d.Wt, d.pool, d.segs, workspace=ws)
        out[n] = [y]
    for n in reversed(ORDER):
        d, wl = devs[n], L[n]
        if wl.bounds is not None:
            g = lm.sliced_backward(d.x, d.Wt, d.pool, wl.bounds, d.segs, d.dY, recompute=True, workspace=ws)
        else:
            g = lm.backward(d.x, d.Wt, d.pool, d.segs, d.dY, recompute=True, workspace=ws)
        out[n] += list(g)
    torch.cuda.synchronize()
    return out


def train_blocks(wl):
    a = int(wl.meta["train_adapter"])
    S = wl.n_slices
    ia = np.arange(wl.a_off[a], wl.a_off[a] + S * wl.rank[a] * wl.K)
    ib = np.arange(wl.b_off[a], wl.b_off[a] + wl.rank[a] * wl.N)
    return ia, ib


def test_layer_chain_matches_oracle_and_is_workspace_independent():
    import torch
    L = layer()
    devs = {n: Dev(L[n]) for n in ORDER}
    got = chain(L, devs, shared=True)
    for n in ORDER:
        wl = L[n]
        y, dX, dA, dB = got[n]
        if wl.bounds is not None:
            ry = osl.forward_wl(wl)
            rX, rA, rB = osl.backward_wl(wl)
        else:
            ry = oracle.forward_wl(wl)
            rX, rA, rB = oracle.backward_wl(wl)
        compare(to_np(y), ry, n + ": y")
        compare(to_np(dX)[wl.train_rows()], rX, n + ": dX")
        ia, ib = train_blocks(wl)
        compare(to_np(dA)[ia], rA[ia], n + ": dA")
        compare(to_np(dB)[ib], rB[ib], n + ": dB")
    again = chain(L, devs, shared=False)
    for n in ORDER:
        for a, b in zip(got[n], again[n]):
            assert torch.equal(a, b), n + ": shared-workspace chain differs from per-call workspaces"


def test_layer_full_size_sampled():
    """The benchmark's layer (Llama-3-8B shapes, 8192-token co-serving batch, 320 adapters), every projection
    computed in full on the GPU and checked on sampled rows and columns: a sliced projection slice by slice through
    the plain oracle (each slice is a plain LoRA layer on the shared input), its dX as the sum over slices."""
    import gc
    import torch
    import lora_co_serving_gb300 as lm
    from test_gpu_fullsize import sample_rows
    L = workloads.llama_layer()
    rng = np.random.default_rng(3)
    for n in ORDER:
        wl = L[n]
        d = Dev(wl)
        if wl.bounds is not None:
            y = lm.sliced_forward(d.x, d.Wt, d.pool, wl.bounds, d.segs)
            dX, dA, dB = lm.sliced_backward(d.x, d.Wt, d.pool, wl.bounds, d.segs, d.dY, recompute=True)
        else:
            y = lm.forward(d.x, d.Wt, d.pool, d.segs)
            dX, dA, dB = lm.backward(d.x, d.Wt, d.pool, d.segs, d.dY, recompute=True)
        torch.cuda.synchronize()
        y, dX, dA, dB = to_np(y), to_np(dX), to_np(dA), to_np(dB)
        del d
        gc.collect()
        torch.cuda.empty_cache()
        rows = sample_rows(wl, cap=16)
        trows = wl.train_rows()
        pick = trows[np.unique(np.concatenate([[0, trows.shape[0] - 1], rng.integers(0, trows.shape[0], 6)]))]
        a = int(wl.meta["train_adapter"])
        r = int(wl.rank[a])
        ca = np.unique(np.concatenate([[0, wl.K - 1], rng.integers(0, wl.K, 24)]))
        parts = [workloads.slice_of(wl, i) for i in range(wl.n_slices)] if wl.bounds is not None else [wl]
        bounds = wl.bounds if wl.bounds is not None else np.array([0, wl.N])
        rX = 0.0
        for i, sw in enumerate(parts):
            c0, c1 = int(bounds[i]), int(bounds[i + 1])
            compare(y[rows, c0:c1], oracle.forward_wl(sw, rows=rows), "%s slice %d: y (sampled rows)" % (n, i))
            cb = np.unique(np.concatenate([[0, sw.N - 1], rng.integers(0, sw.N, 24)]))
            sX, sA, sB = oracle.backward_wl(sw, dx_rows=pick, cols_b=cb, cols_a=ca)
            rX = rX + sX
            gB = dB.reshape(-1, wl.N)[int(wl.b_off[a]) // wl.N:int(wl.b_off[a]) // wl.N + r, c0:c1][:, cb]
            eB = sB[sw.b_off[a]:sw.b_off[a] + r * sw.N].reshape(r, sw.N)[:, cb]
            compare(gB, eB, "%s slice %d: dB (sampled columns)" % (n, i))
            row0 = int(wl.a_off[a]) // wl.K + i * r
            gA = dA.reshape(-1, wl.K)[row0:row0 + r][:, ca]
            eA = sA[sw.a_off[a]:sw.a_off[a] + r * wl.K].reshape(r, wl.K)[:, ca]
            compare(gA, eA, "%s slice %d: dA (sampled columns)" % (n, i))
        compare(dX[pick], rX, "%s: dX (sampled rows, summed over slices)" % n)
