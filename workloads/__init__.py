"""Seeded synthetic inputs for the mixed-batch multi-adapter LoRA layer.

This module only draws inputs: segment tables, adapter ranks and pool
offsets, and the values of x, W, A, B and dY.  It holds none of the layer's
arithmetic, and it is the one module that both the CUDA path's tests and the
float64 oracle read.

Every array is float32 holding values that are exact in the workload's
element type: for bf16 workloads each draw is rounded to bf16 (round to
nearest even) before anything else sees it, so the oracle and the GPU read
the same numbers.  ``bf16_bits`` turns such an array into the raw 16-bit
patterns the GPU gets.

The shapes follow the pages' workloads (Llama-3-8B q_proj 4096x4096 and MLP
up 4096x14336, Mistral-Small-24B-like 5120x5120, Llama-70B-like MLP
8192x28672; LoRA rank 16 with alpha 32, ranks 8..128, pools of up to 320
adapters, fine-tuning sequences of 1024 tokens).  The pages' own traces and
datasets are not used; these draws stand in for them.

Generation order per workload (one PCG64 stream, seed 1000 + config number):
segment table -> ranks -> W -> A -> B -> x -> dY.
"""
from dataclasses import dataclass, field
from typing import Optional

import numpy as np

__all__ = ["Workload", "config", "custom", "bf16_round", "bf16_bits", "CONFIGS"]


def bf16_round(a):
    """Round float32 values to the nearest bf16 (ties to even); returns float32."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) & np.uint32(0xFFFF0000)
    return r.view(np.float32)


def bf16_bits(a):
    """Raw bf16 bit patterns (uint16) of float32 values that are already bf16-exact."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    return (a.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


@dataclass
class Workload:
    name: str
    T: int
    K: int
    N: int
    dtype: str                     # "bf16" or "f32"
    segs: np.ndarray               # [n, 4] int32: start, len, adapter_id, is_train
    rank: np.ndarray               # [P] int32
    scale: np.ndarray              # [P] float32
    a_off: np.ndarray              # [P] int64, element offset of adapter a's [r,K] block in A
    b_off: np.ndarray              # [P] int64, element offset of adapter a's [r,N] block in B
    x: np.ndarray                  # [T, K] float32
    Wt: np.ndarray                 # [N, K] float32 (W stored transposed, nn.Linear layout)
    A: np.ndarray                  # flat float32, sum_a r_a*K
    B: np.ndarray                  # flat float32, sum_a r_a*N
    dY: Optional[np.ndarray]       # [T, N] float32 or None
    forward: bool = True
    backward: bool = False
    xa_mode: str = "recompute"     # "save" (forward keeps xA) or "recompute"
    meta: dict = field(default_factory=dict)
    bounds: Optional[np.ndarray] = None   # sliced layers: [S+1] int32 output-column bounds of the slices

    @property
    def n_slices(self):
        return 1 if self.bounds is None else int(self.bounds.shape[0]) - 1

    @property
    def n_adapters(self):
        return int(self.rank.shape[0])

    def train_rows(self):
        """Training-token rows in increasing segment-start order."""
        tr = sorted([tuple(s) for s in self.segs.tolist() if s[3] and s[1] > 0])
        return np.concatenate([np.arange(s[0], s[0] + s[1]) for s in tr]) if tr else np.zeros(0, np.int64)


def _normal(rng, shape, std, dtype):
    v = rng.standard_normal(size=shape, dtype=np.float32)
    v *= np.float32(std)
    return bf16_round(v) if dtype == "bf16" else v


def _uniform(rng, shape, bound, dtype):
    v = rng.random(size=shape, dtype=np.float32)
    v *= np.float32(2.0 * bound)
    v -= np.float32(bound)
    return bf16_round(v) if dtype == "bf16" else v


def _pool_offsets(rank, K, N, n_slices=1):
    """Adapters back to back: adapter a holds n_slices * r_a rows of K in A and r_a rows of N in B."""
    rank = np.asarray(rank, dtype=np.int64)
    a_off = np.zeros(rank.shape[0], np.int64)
    b_off = np.zeros(rank.shape[0], np.int64)
    if rank.shape[0]:
        a_off[1:] = np.cumsum(n_slices * rank[:-1] * K)
        b_off[1:] = np.cumsum(rank[:-1] * N)
    return a_off, b_off


def _fill(name, rng, T, K, N, dtype, segs, rank, scale, *, want_dy, w_var=None, a_bound=None, b_var=0.02,
          bounds=None, **kw):
    """Draw W, A, B, x, dY in that order and assemble the workload."""
    rank = np.asarray(rank, dtype=np.int32)
    S = 1 if bounds is None else len(bounds) - 1
    a_off, b_off = _pool_offsets(rank, K, N, S)
    w_std = np.sqrt(1.0 / K if w_var is None else w_var)
    a_bound = 1.0 / np.sqrt(K) if a_bound is None else a_bound
    Wt = _normal(rng, (N, K), w_std, dtype)
    A = _uniform(rng, (S * int(rank.sum()) * K,), a_bound, dtype)
    B = _normal(rng, (int(rank.sum()) * N,), np.sqrt(b_var), dtype)
    x = _normal(rng, (T, K), 1.0, dtype)
    dY = _normal(rng, (T, N), 1.0, dtype) if want_dy else None
    return Workload(name=name, T=T, K=K, N=N, dtype=dtype, segs=np.asarray(segs, np.int32).reshape(-1, 4),
                    rank=rank, scale=np.asarray(scale, np.float32), a_off=a_off, b_off=b_off, x=x, Wt=Wt, A=A,
                    B=B, dY=dY, bounds=None if bounds is None else np.asarray(bounds, np.int32), **kw)


def _draw_lengths(rng, total, lo, hi):
    """Segment lengths U{lo..hi} until their sum reaches ``total``; the last one takes the remainder."""
    lens = []
    left = total
    while left > 0:
        ln = int(rng.integers(lo, hi + 1))
        ln = min(ln, left)
        lens.append(ln)
        left -= ln
    return lens


def _zipf_ids(rng, n, n_adapters, s):
    """n adapter ids with P(popularity rank i) ~ i^-s; popularity order is a seeded permutation of the ids."""
    order = rng.permutation(n_adapters)
    p = np.arange(1, n_adapters + 1, dtype=np.float64) ** (-s)
    p /= p.sum()
    ranks = rng.choice(n_adapters, size=n, p=p)
    return order[ranks]


# --------------------------------------------------------------------------------------------------------------
# The five workload shapes.  ``scale`` shrinks the token count and the layer width for parity tests that the
# oracle must finish in seconds; the structure (segment kinds, rank mix, value distributions) is kept.


def config1(seed=1001):
    """Tiny fp32 layer: 256->256, 64 tokens in 4 segments of 16, 4 rank-8 adapters (scale 2), segment 3 trains."""
    rng = np.random.Generator(np.random.PCG64(seed))
    perm = rng.permutation(4)
    segs = [(16 * i, 16, int(perm[i]), 1 if i == 3 else 0) for i in range(4)]
    rank = [8] * 4
    return _fill("tiny_256x256_T64_fp32", rng, 64, 256, 256, "f32", segs, rank, [2.0] * 4, want_dy=True,
                 forward=True, backward=True, xa_mode="recompute")


def config2(seed=1002, T=256, K=4096, N=4096, n_adapters=64):
    """Decode batch: T single-token segments over n_adapters adapters, ranks U{8,16,32,64}, scale 2, forward only."""
    rng = np.random.Generator(np.random.PCG64(seed))
    ids = rng.integers(0, n_adapters, size=T)
    segs = [(t, 1, int(ids[t]), 0) for t in range(T)]
    rank = rng.choice(np.array([8, 16, 32, 64]), size=n_adapters)
    return _fill("decode_%dx%d_T%d_P%d" % (K, N, T, n_adapters), rng, T, K, N, "bf16", segs, rank,
                 [2.0] * n_adapters, want_dy=False, forward=True, backward=False)


def config3(seed=1003, K=4096, N=14336, prefill_tokens=6144, train_len=1024, n_train=2, len_lo=128, len_hi=1024,
            n_inf=16, r=16):
    """Prefill segments over n_inf rank-16 adapters plus fine-tuning segments on a reserved 17th adapter (xA saved)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    lens = _draw_lengths(rng, prefill_tokens, len_lo, len_hi)
    ids = rng.integers(0, n_inf, size=len(lens))
    segs, t = [], 0
    for ln, a in zip(lens, ids):
        segs.append((t, ln, int(a), 0))
        t += ln
    for _ in range(n_train):
        segs.append((t, train_len, n_inf, 1))
        t += train_len
    rank = [r] * (n_inf + 1)
    return _fill("mixed_%dx%d_T%d" % (K, N, t), rng, t, K, N, "bf16", segs, rank, [2.0] * (n_inf + 1),
                 want_dy=True, forward=True, backward=False, xa_mode="save")


def config4(seed=1004, K=5120, N=5120, n_samples=4, sample_len=1024, r=16, four_adapters=False):
    """Fine-tuning backward: n_samples segments of sample_len on one rank-r adapter (or one adapter each); xA recomputed."""
    rng = np.random.Generator(np.random.PCG64(seed))
    n_ad = n_samples if four_adapters else 1
    segs = [(i * sample_len, sample_len, (i if four_adapters else 0), 1) for i in range(n_samples)]
    rank = [r] * n_ad
    T = n_samples * sample_len
    return _fill("ftbwd_%dx%d_T%d_r%d%s" % (K, N, T, r, "_4ad" if four_adapters else ""), rng, T, K, N, "bf16",
                 segs, rank, [2.0] * n_ad, want_dy=True, forward=False, backward=True, xa_mode="recompute")


def config5(seed=1005, K=8192, N=28672, n_adapters=320, n_decode=2048, prefill_tokens=4096, len_lo=64, len_hi=1024,
            n_train=2, train_len=1024, zipf_s=1.1, ranks=(8, 16, 32, 64, 128)):
    """Large heterogeneous co-serving batch: Zipf decode + prefill + fine-tuning, forward and backward in one step."""
    rng = np.random.Generator(np.random.PCG64(seed))
    dec = _zipf_ids(rng, n_decode, n_adapters, zipf_s)
    lens = _draw_lengths(rng, prefill_tokens, len_lo, len_hi)
    pre_ids = rng.integers(0, n_adapters, size=len(lens))
    train_ad = int(rng.integers(0, n_adapters))
    segs, t = [], 0
    for a in dec:
        segs.append((t, 1, int(a), 0))
        t += 1
    for ln, a in zip(lens, pre_ids):
        segs.append((t, ln, int(a), 0))
        t += ln
    for _ in range(n_train):
        segs.append((t, train_len, train_ad, 1))
        t += train_len
    rank = rng.choice(np.array(ranks), size=n_adapters)
    return _fill("cosrv_%dx%d_T%d_P%d" % (K, N, t, n_adapters), rng, t, K, N, "bf16", segs, rank,
                 [2.0] * n_adapters, want_dy=True, forward=True, backward=True, xa_mode="recompute",
                 meta={"n_decode": n_decode, "train_adapter": train_ad})


def custom(seed, T, K, N, segs, rank, scale=None, dtype="bf16", want_dy=True, **kw):
    """A workload with a given segment table and rank list; values drawn as in the configs."""
    rng = np.random.Generator(np.random.PCG64(seed))
    rank = list(rank)
    scale = [2.0] * len(rank) if scale is None else scale
    return _fill("custom_%dx%d_T%d" % (K, N, T), rng, T, K, N, dtype, segs, rank, scale, want_dy=want_dy, **kw)


def sliced(seed, T, K, bounds, segs, rank, scale=None, dtype="bf16", want_dy=True, **kw):
    """A fused projection of several slices (e.g. q|k|v over one input): output columns [bounds[i], bounds[i+1])
    form slice i.  Adapter a holds one [r_a, K] down factor per slice, stacked in slice order in A, and one
    [r_a, N] up factor in B whose columns of slice i are that slice's up factor."""
    rng = np.random.Generator(np.random.PCG64(seed))
    rank = list(rank)
    scale = [2.0] * len(rank) if scale is None else scale
    N = int(bounds[-1])
    return _fill("sliced_%dx%d_S%d_T%d" % (K, N, len(bounds) - 1, T), rng, T, K, N, dtype, segs, rank, scale,
                 want_dy=want_dy, bounds=bounds, **kw)


def llama_layer(seed=1006, hidden=4096, kv=1024, inter=14336, n_adapters=320, n_decode=2048, prefill_tokens=4096,
                len_lo=64, len_hi=1024, n_train=2, train_len=1024, zipf_s=1.1, ranks=(8, 16, 32), train_rank=16):
    """The LoRA projections of one Llama-3-8B decoder layer on a co-serving batch.

    Shapes: q|k|v fused (hidden -> hidden + 2 kv, three slices), o (hidden -> hidden), gate|up fused
    (hidden -> 2 inter, two slices), down (inter -> hidden).  Every projection has its own adapter pool; the
    segment table and the adapters' ranks are shared (one adapter = one rank on every projection).  The
    batch: Zipf(zipf_s) decode tokens over the pool, prefill segments of U{len_lo..len_hi} tokens, and
    n_train fine-tuning sequences on a reserved adapter of rank train_rank (scale 2, the pages' r = 16,
    alpha = 32).  Inference adapters draw their rank from ``ranks``.  Generation order: table -> ranks ->
    then each projection in the order qkv, o, gate_up, down (W, A, B, x, dY each)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    n_inf = n_adapters - 1
    dec = _zipf_ids(rng, n_decode, n_inf, zipf_s)
    lens = _draw_lengths(rng, prefill_tokens, len_lo, len_hi)
    pre_ids = rng.integers(0, n_inf, size=len(lens))
    segs, t = [], 0
    for a in dec:
        segs.append((t, 1, int(a), 0))
        t += 1
    for ln, a in zip(lens, pre_ids):
        segs.append((t, ln, int(a), 0))
        t += ln
    for _ in range(n_train):
        segs.append((t, train_len, n_inf, 1))
        t += train_len
    rank = np.concatenate([rng.choice(np.array(ranks), size=n_inf), [train_rank]]).astype(np.int32)
    scale = [2.0] * n_adapters
    shapes = [("qkv", hidden, [0, hidden, hidden + kv, hidden + 2 * kv]), ("o", hidden, [0, hidden]),
              ("gate_up", hidden, [0, inter, 2 * inter]), ("down", inter, [0, hidden])]
    out = {}
    for name, K, bounds in shapes:
        N = bounds[-1]
        b = bounds if len(bounds) > 2 else None
        wl = _fill("llama_layer_%s_%dx%d_T%d" % (name, K, N, t), rng, t, K, N, "bf16", segs, rank, scale,
                   want_dy=True, forward=True, backward=True, xa_mode="recompute", bounds=b,
                   meta={"n_decode": n_decode, "train_adapter": n_inf, "projection": name})
        out[name] = wl
    return out


def slice_of(wl, i):
    """Slice i of a sliced workload as a plain workload: that slice's weight rows, down factors and up-factor
    columns, with the same segment table and inputs (plain indexing of the drawn arrays)."""
    import dataclasses
    c0, c1 = int(wl.bounds[i]), int(wl.bounds[i + 1])
    Ni = c1 - c0
    A2 = wl.A.reshape(-1, wl.K)
    B2 = wl.B.reshape(-1, wl.N)
    As, Bs, ao, bo = [], [], [], []
    at_a = at_b = 0
    for a in range(wl.n_adapters):
        r = int(wl.rank[a])
        row = int(wl.a_off[a]) // wl.K
        As.append(A2[row + i * r:row + (i + 1) * r])
        brow = int(wl.b_off[a]) // wl.N
        Bs.append(B2[brow:brow + r, c0:c1])
        ao.append(at_a)
        bo.append(at_b)
        at_a += r * wl.K
        at_b += r * Ni
    return dataclasses.replace(wl, N=Ni, Wt=np.ascontiguousarray(wl.Wt[c0:c1]),
                               A=np.ascontiguousarray(np.concatenate(As).reshape(-1)),
                               B=np.ascontiguousarray(np.concatenate(Bs).reshape(-1)),
                               a_off=np.asarray(ao, np.int64), b_off=np.asarray(bo, np.int64),
                               dY=None if wl.dY is None else np.ascontiguousarray(wl.dY[:, c0:c1]), bounds=None)


CONFIGS = {1: config1, 2: config2, 3: config3, 4: config4, 5: config5}


def config(i, **kw):
    """The i-th workload (1..5) at its full size, or with keyword overrides for reduced sizes."""
    return CONFIGS[i](**kw)
