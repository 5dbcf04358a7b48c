"""Parity at the full workload sizes, in the launch configuration the benchmark times.

The GPU computes every output; the float64 oracle computes a sample of them one by one (rows of y and dX, columns
of dA and dB), chosen to touch every segment kind and every adapter of the fine-tuning set.  Same tolerance as the
small cases, applied to the sampled values.
"""
import gc

import numpy as np
import pytest

import oracle
import workloads
from gpu_util import Dev, compare, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    import lora_co_serving_gb300 as lm
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lm.build()


def sample_rows(wl, per_seg=2, cap=64, seed=0):
    """Rows covering segments of every kind: first and last row of a spread of segments, plus random rows."""
    rng = np.random.default_rng(seed)
    segs = sorted(wl.segs.tolist())
    idx = np.unique(np.linspace(0, len(segs) - 1, min(len(segs), cap // per_seg)).astype(int))
    rows = []
    for i in idx:
        st, ln, a, tr = segs[i]
        rows += [st, st + ln - 1][:per_seg]
    rows = np.unique(np.array(rows + list(rng.integers(0, wl.T, 8))))
    return rows


def free():
    import torch
    gc.collect()
    torch.cuda.empty_cache()


def test_config2_decode_full():
    wl = workloads.config2()
    d = Dev(wl)
    y = to_np(d.forward())
    compare(y, oracle.forward_wl(wl), "y (all 256 rows)")
    del d
    free()


def test_config3_mixed_forward_full():
    wl = workloads.config3()
    d = Dev(wl)
    y, xs = d.forward(save_xa=True)
    rows = sample_rows(wl)
    ref, u = oracle.forward_wl(wl, rows=rows, want_u=True)
    compare(to_np(y)[rows], ref, "y (sampled rows)")
    # saved xA of the sampled fine-tuning rows
    xs = to_np(xs)
    off, got, exp = 0, [], []
    for st, ln, a, tr in sorted(wl.segs.tolist()):
        if not tr:
            continue
        r = int(wl.rank[a])
        for i, t in enumerate(rows):
            if st <= t < st + ln:
                got.append(xs[off + (t - st) * r: off + (t - st + 1) * r])
                exp.append(u[i, :r])
        off += ln * r
    assert got
    compare(np.concatenate(got), np.concatenate(exp), "xa_save (sampled rows)")
    del d
    free()


def check_backward_sampled(wl, dX, dA, dB, n_rows=24, n_cols=64):
    rng = np.random.default_rng(1)
    trows = wl.train_rows()
    pick = np.unique(np.concatenate([[0, trows.shape[0] - 1], rng.integers(0, trows.shape[0], n_rows)]))
    cb = np.unique(np.concatenate([[0, wl.N - 1], rng.integers(0, wl.N, n_cols)]))
    ca = np.unique(np.concatenate([[0, wl.K - 1], rng.integers(0, wl.K, n_cols)]))
    rX, rA, rB = oracle.backward_wl(wl, dx_rows=trows[pick], cols_b=cb, cols_a=ca)
    compare(to_np(dX)[trows[pick]], rX, "dX (sampled rows)")
    dA, dB = to_np(dA), to_np(dB)
    for a in sorted(set(int(s[2]) for s in wl.segs.tolist() if s[3])):
        r = int(wl.rank[a])
        gB = dB[wl.b_off[a]:wl.b_off[a] + r * wl.N].reshape(r, wl.N)[:, cb]
        eB = rB[wl.b_off[a]:wl.b_off[a] + r * wl.N].reshape(r, wl.N)[:, cb]
        gA = dA[wl.a_off[a]:wl.a_off[a] + r * wl.K].reshape(r, wl.K)[:, ca]
        eA = rA[wl.a_off[a]:wl.a_off[a] + r * wl.K].reshape(r, wl.K)[:, ca]
        compare(gB, eB, "dB (sampled columns, adapter %d)" % a)
        compare(gA, eA, "dA (sampled columns, adapter %d)" % a)


@pytest.mark.parametrize("r", [16, 64])
def test_config4_backward_full(r):
    wl = workloads.config4(r=r)
    d = Dev(wl)
    dX, dA, dB = d.backward()
    check_backward_sampled(wl, dX, dA, dB)
    del d
    free()


def test_config5_forward_backward_full():
    wl = workloads.config5()
    d = Dev(wl)
    y = d.forward()
    dX, dA, dB = d.backward()
    y = to_np(y)
    rows = sample_rows(wl, cap=48)
    compare(y[rows], oracle.forward_wl(wl, rows=rows), "y (sampled rows)")
    check_backward_sampled(wl, dX, dA, dB, n_rows=12, n_cols=48)
    del d
    free()
