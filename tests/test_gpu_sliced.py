"""GPU parity of sliced (fused) projections: q|k|v and gate|up run as one layer over the concatenated weight.

Each slice is an ordinary LoRA linear layer on the shared input (its own down factor, the up factor's columns of
the slice), so besides the float64 oracle of ``oracle/sliced.py`` every slice of a sliced call is checked
BITWISE against a plain call of that slice alone: the sliced plan keeps each row's shrink and expand summation
order, so fusing the slices must not change a single bit of y, dA or dB.
"""
import numpy as np
import pytest

import workloads
from oracle import sliced as osl
from gpu_util import Dev, compare, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    import lora_co_serving_gb300 as lm
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lm.build()
    lm.library()


def mixed(bounds, K=512, seed=21, n_adapters=24, ranks=(8, 16, 32, 64), n_decode=150, prefill=500, train_len=100,
          n_train=2):
    """A co-serving batch (Zipf decode, prefill, fine-tuning) on a sliced layer."""
    base = workloads.config5(K=64, N=64, n_adapters=n_adapters, n_decode=n_decode, prefill_tokens=prefill, len_lo=30,
                             len_hi=250, train_len=train_len, n_train=n_train, ranks=ranks)
    wl = workloads.sliced(seed, base.T, K, bounds, base.segs, base.rank)
    wl.meta["train_adapter"] = base.meta["train_adapter"]
    return wl


def sliced_train_blocks(wl):
    ads = sorted(set(int(s[2]) for s in wl.segs.tolist() if s[3]))
    S = wl.n_slices
    ia = np.concatenate([np.arange(wl.a_off[a], wl.a_off[a] + S * wl.rank[a] * wl.K) for a in ads])
    ib = np.concatenate([np.arange(wl.b_off[a], wl.b_off[a] + wl.rank[a] * wl.N) for a in ads])
    return ia, ib


def run_forward(wl, save=False):
    import lora_co_serving_gb300 as lm
    d = Dev(wl)
    out = lm.sliced_forward(d.x, d.Wt, d.pool, wl.bounds, d.segs, save_xa=save)
    return d, out


def check_forward(wl):
    import torch
    d, (y, xs) = run_forward(wl, save=True)
    torch.cuda.synchronize()
    ref, u = osl.forward_wl(wl, want_u=True)
    compare(to_np(y), ref, "y")
    # saved xA: per fine-tuning segment (increasing start) a [len, S*r] block, slice i in columns [i r, (i+1) r)
    exp = []
    S = wl.n_slices
    for st, ln, a, tr in sorted(wl.segs.tolist()):
        if tr and ln > 0:
            r = int(wl.rank[a])
            blk = np.concatenate([u[st:st + ln, 128 * i:128 * i + r] for i in range(S)], axis=1)
            exp.append(blk.reshape(-1))
    if exp:
        exp = np.concatenate(exp)
        compare(to_np(xs)[:exp.shape[0]], exp, "xa_save")
    return d, y, xs


def check_backward(wl, d, xs=None):
    import torch
    import lora_co_serving_gb300 as lm
    dX, dA, dB = lm.sliced_backward(d.x, d.Wt, d.pool, wl.bounds, d.segs, d.dY, xa_saved=xs,
                                    recompute=xs is None)
    torch.cuda.synchronize()
    rX, rA, rB = osl.backward_wl(wl)
    rows = wl.train_rows()
    compare(to_np(dX)[rows], rX, "dX")
    ia, ib = sliced_train_blocks(wl)
    compare(to_np(dA)[ia], rA[ia], "dA")
    compare(to_np(dB)[ib], rB[ib], "dB")
    mA = np.ones(dA.numel(), bool)
    mA[ia] = False
    mB = np.ones(dB.numel(), bool)
    mB[ib] = False
    assert np.all(to_np(dA)[mA] == 0) and np.all(to_np(dB)[mB] == 0)
    return dX, dA, dB


QKV = [0, 512, 768, 1024]          # q 512, k 256, v 256 (the 4:1:1 of a grouped-query attention layer)


def test_sliced_qkv_forward_and_backward():
    wl = mixed(QKV)
    d, y, xs = check_forward(wl)
    check_backward(wl, d)              # recompute xA
    check_backward(wl, d, xs)          # from the saved xA


def test_sliced_slices_equal_plain_calls_bitwise():
    import torch
    import lora_co_serving_gb300 as lm
    wl = mixed(QKV, seed=22)
    d, y = run_forward(wl)
    dX, dA, dB = lm.sliced_backward(d.x, d.Wt, d.pool, wl.bounds, d.segs, d.dY, recompute=True)
    torch.cuda.synchronize()
    ya = y.cpu()
    A_s = dA.cpu().numpy()
    B_s = dB.cpu().numpy().reshape(-1, wl.N)
    for i in range(wl.n_slices):
        c0, c1 = int(wl.bounds[i]), int(wl.bounds[i + 1])
        sw = workloads.slice_of(wl, i)
        ds = Dev(sw)
        yi = ds.forward()
        _, gA, gB = ds.backward(recompute=True)
        torch.cuda.synchronize()
        assert torch.equal(ya[:, c0:c1], yi.cpu()), "slice %d: y differs from the plain call" % i
        gA = gA.cpu().numpy()
        gB = gB.cpu().numpy()
        for a in range(wl.n_adapters):
            r = int(wl.rank[a])
            row = int(wl.a_off[a])
            got = A_s[row + i * r * wl.K:row + (i + 1) * r * wl.K]
            assert np.array_equal(got, gA[sw.a_off[a]:sw.a_off[a] + r * wl.K]), ("slice dA", i, a)
            brow = int(wl.b_off[a]) // wl.N
            assert np.array_equal(B_s[brow:brow + r, c0:c1],
                                  gB[sw.b_off[a]:sw.b_off[a] + r * (c1 - c0)].reshape(r, c1 - c0)), ("slice dB", i, a)


def test_sliced_one_slice_is_the_plain_layer():
    import torch
    import lora_co_serving_gb300 as lm
    wl = mixed([0, 768], seed=23)
    d = Dev(wl)
    y1 = lm.sliced_forward(d.x, d.Wt, d.pool, wl.bounds, d.segs)
    y0 = lm.forward(d.x, d.Wt, d.pool, d.segs)
    g1 = lm.sliced_backward(d.x, d.Wt, d.pool, wl.bounds, d.segs, d.dY, recompute=True)
    g0 = lm.backward(d.x, d.Wt, d.pool, d.segs, d.dY, recompute=True)
    torch.cuda.synchronize()
    assert torch.equal(y0, y1)
    for a, b in zip(g0, g1):
        assert torch.equal(a, b)


@pytest.mark.parametrize("bounds,r", [([0, 512, 1024], 128), ([0, 256, 512, 768, 1024], 128), ([0, 256, 456], 24)])
def test_sliced_gate_up_and_wide_ranks(bounds, r):
    # gate|up (2 slices) and 4 slices at rank 128: the fine-tuning adapter's stacked down factors have 256 and 512
    # rows (two dA passes); a ragged last slice of 200 columns
    base = workloads.config4(K=384, N=64, n_samples=2, sample_len=180, r=r, four_adapters=True)
    segs = base.segs.tolist() + [(base.T + i, 1, i % 2, 0) for i in range(40)]
    wl = workloads.sliced(31, base.T + 40, 384, bounds, segs, [r, r // 2 + 8])
    d, y, xs = check_forward(wl)
    check_backward(wl, d)
    check_backward(wl, d, xs)


def test_sliced_split_gradients():
    """Gradient items of a three-slice layer split three ways along the tokens (pinned on the host), splits
    crossing segment boundaries, one adapter's 384 stacked rank rows over two dA items: dX, dA (every slice's
    down factor), dB against the sliced oracle."""
    from gpu_util import grad_split_table
    wl = grad_split_table(sliced=True)
    check_backward(wl, Dev(wl))


def random_sliced(seed):
    """A seeded random call on a sliced layer: 2..4 slices (all but the last a multiple of 256 wide, the last any
    multiple of 8), K up to 520, 1..12 adapters of ranks 1..128, decode, prefill, fine-tuning and base-only segments
    listed in shuffled order."""
    rng = np.random.default_rng(7100 + seed)
    S = int(rng.integers(2, 5))
    widths = [256 * int(rng.integers(1, 3)) for _ in range(S - 1)] + [8 * int(rng.integers(1, 33))]
    bounds = np.concatenate([[0], np.cumsum(widths)]).astype(np.int32)
    K = 8 * int(rng.integers(1, 66))
    n_ad = int(rng.integers(1, 13))
    rank = [int(rng.integers(1, 129)) for _ in range(n_ad)]
    segs, t, n_train = [], 0, 0
    for _ in range(int(rng.integers(1, 25))):
        kind = int(rng.integers(0, 4))
        if kind == 0:
            for _ in range(int(rng.integers(1, 20))):
                segs.append((t, 1, int(rng.integers(-1, n_ad)), 0))
                t += 1
        elif kind == 1:
            ln = int(rng.integers(2, 260))
            segs.append((t, ln, int(rng.integers(-1, n_ad)), 0))
            t += ln
        elif n_train < 8:
            ln = int(rng.integers(1, 200))
            segs.append((t, ln, int(rng.integers(0, n_ad)), 1))
            t += ln
            n_train += 1
    order = rng.permutation(len(segs))
    return workloads.sliced(7300 + seed, t, K, bounds, [segs[i] for i in order], rank), n_train


@pytest.mark.parametrize("seed", range(8))
def test_sliced_random_tables(seed):
    wl, n_train = random_sliced(seed)
    d, y, xs = check_forward(wl)
    if n_train:
        check_backward(wl, d)          # recompute xA
        check_backward(wl, d, xs)      # from the saved xA
