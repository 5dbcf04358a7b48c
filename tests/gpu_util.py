"""Helpers for the GPU tests: upload a seeded workload, call the library, compare with the oracle."""
import numpy as np

import lora_co_serving_gb300 as lm
import workloads

# Tolerance of the layer (bf16 inputs, fp32 accumulation): per output tensor
MAX_ERR = 2e-2      # max |err| <= MAX_ERR * max |ref|
FRO_ERR = 5e-3      # ||err||_F <= FRO_ERR * ||ref||_F


def to_dev(a, dtype):
    import torch
    if dtype == "bf16":
        bits = workloads.bf16_bits(a)
        return torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def to_np(t):
    import torch
    return t.detach().float().cpu().numpy().astype(np.float64)


class Dev:
    """A workload on the device."""

    def __init__(self, wl):
        import torch
        self.wl = wl
        self.x = to_dev(wl.x, wl.dtype)
        self.Wt = to_dev(wl.Wt, wl.dtype)
        self.A = to_dev(wl.A, wl.dtype)
        self.B = to_dev(wl.B, wl.dtype)
        self.dY = to_dev(wl.dY, wl.dtype) if wl.dY is not None else None
        self.pool = lm.Pool(self.A, self.B, wl.a_off, wl.b_off, wl.rank, wl.scale)
        self.segs = wl.segs

    def forward(self, **kw):
        return lm.forward(self.x, self.Wt, self.pool, self.segs, **kw)

    def backward(self, **kw):
        return lm.backward(self.x, self.Wt, self.pool, self.segs, self.dY, **kw)


def compare(got, ref, name, max_err=MAX_ERR, fro_err=FRO_ERR):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), name + ": non-finite values"
    d = got - ref
    mref = np.abs(ref).max() if ref.size else 0.0
    mx = np.abs(d).max() if d.size else 0.0
    fro = np.linalg.norm(d) / max(np.linalg.norm(ref), 1e-300)
    assert mx <= max_err * max(mref, 1e-30), "%s: max|err| %.3g > %.3g * max|ref| %.3g" % (name, mx, max_err, mref)
    assert fro <= fro_err, "%s: relative Frobenius error %.3g > %.3g" % (name, fro, fro_err)
    return mx / max(mref, 1e-30), fro


def train_blocks(wl):
    """Pool index ranges of the A and B blocks of adapters with fine-tuning segments."""
    ads = sorted(set(int(s[2]) for s in wl.segs.tolist() if s[3]))
    ia = np.concatenate([np.arange(wl.a_off[a], wl.a_off[a] + wl.rank[a] * wl.K) for a in ads])
    ib = np.concatenate([np.arange(wl.b_off[a], wl.b_off[a] + wl.rank[a] * wl.N) for a in ads])
    return ia, ib


SPLIT_BOUNDS = [0, 256, 512, 640]      # the sliced variant: three slices (256, 256, 128 columns)


def grad_split_table(seed=4242, K=320, N=384, sliced=False):
    """A backward whose gradient items are few enough for the planner to split their token ranges three ways:
    adapter 0 (rank 24) fine-tunes on three segments of 700, 333 and 1100 tokens (35 token blocks, so that splits
    cross segment boundaries), adapter 1 (rank 40) on one of 1600 tokens (25 blocks); decode, prefill and
    base-only rows of other adapters sit between them.  12 gradient items (dB: 3 column tiles, dA: 3 row tiles per
    adapter) -> 36 split items.  sliced: the same table on a sliced layer of K = 256 and the three slices of
    SPLIT_BOUNDS, adapter 0 of rank 128 so that its three stacked down factors (384 rank rows) span two dA items
    per row tile (dB: 5 column tiles over the slices; dA: 2 row tiles x 2 rank ranges for adapter 0, x 1 for
    adapter 1) -> 16 items, 48 split items."""
    spans = [(700, 0, 1), (5, 2, 0), (333, 0, 1), (90, 3, 0), (1, 4, 0), (1600, 1, 1), (40, -1, 0), (1100, 0, 1),
             (1, 5, 0)]
    segs, t = [], 0
    for ln, a, tr in spans:
        segs.append((t, ln, a, tr))
        t += ln
    rank = [24, 40, 8, 16, 64, 128]
    if sliced:
        rank[0] = 128
        return workloads.sliced(seed, t, 256, np.asarray(SPLIT_BOUNDS, np.int32), segs, rank)
    return workloads.custom(seed, t, K, N, segs, rank)


# A fine-tuning table whose backward dY B^T shrink passes are cut into 8 pieces instead of the default 4: 32 tiles
# of 64 k-blocks (N = 4096), whose 160 default items would leave a last wave of 8 on 152 CTAs.
RESPLIT_SMALL = dict(T=4096, K=256, N=4096, segs=[(i * 512, 512, i % 2, 1) for i in range(8)], rank=[16, 40])


def random_table(seed):
    """A seeded random call: K and N up to 520 (multiples of 8 for bf16, any size for f32), 1..20 adapters of
    ranks 1..128 (a few absent from the table), decode tokens, prefill segments of 2..300 tokens, fine-tuning
    segments of 1..260 tokens (at most 12), some base-only tokens, the table listed in shuffled order."""
    rng = np.random.default_rng(9000 + seed)
    dtype = "f32" if seed % 4 == 3 else "bf16"
    if dtype == "bf16":
        K, N = 8 * int(rng.integers(1, 66)), 8 * int(rng.integers(1, 66))
    else:
        K, N = int(rng.integers(1, 300)), int(rng.integers(1, 300))
    n_ad = int(rng.integers(1, 21))
    rank = [int(rng.integers(1, 129)) for _ in range(n_ad)]
    segs, t, n_train = [], 0, 0
    for _ in range(int(rng.integers(1, 40))):
        kind = int(rng.integers(0, 4))
        if kind == 0:                                 # decode tokens (some base-only)
            for _ in range(int(rng.integers(1, 30))):
                segs.append((t, 1, int(rng.integers(-1, n_ad)), 0))
                t += 1
        elif kind == 1:
            ln = int(rng.integers(2, 301))
            segs.append((t, ln, int(rng.integers(-1, n_ad)), 0))
            t += ln
        elif n_train < 12:
            ln = int(rng.integers(1, 261))
            segs.append((t, ln, int(rng.integers(0, n_ad)), 1))
            t += ln
            n_train += 1
    order = rng.permutation(len(segs))
    return workloads.custom(5000 + seed, t, K, N, [segs[i] for i in order], rank, dtype=dtype), n_train
