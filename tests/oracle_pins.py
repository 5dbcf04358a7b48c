"""Pins of the float64 oracle against facts other than itself.

Each ``pin_*`` function raises AssertionError when the oracle (``lib``: a
loaded oracle library, None = the real one) disagrees with
  - the pure-Python brute force through the merged weight W + s*A*B,
  - central finite differences of the loss sum(dY * y) (exact here: y is
    linear in each of x, A and B separately),
  - closed forms (zero B, integer routing patterns, trainable-parameter counts),
  - invariances (segment order, adapter-pool order).
``test_oracle_pins.py`` runs them on the real oracle; ``test_oracle_mutants.py``
plants mistakes in copies of the oracle source and checks that some pin fails.
"""
import numpy as np

import oracle
from oracle import brute
from oracle import sliced
import workloads


def _tiny(seed, T=None, K=None, N=None, n_ad=None):
    rng = np.random.default_rng(seed)
    T = T or int(rng.integers(3, 9))
    K = K or int(rng.integers(4, 13))
    N = N or int(rng.integers(4, 13))
    n_ad = n_ad or int(rng.integers(1, 4))
    rank = [int(rng.integers(1, 5)) for _ in range(n_ad)]
    # random cut of [0,T) into segments, random adapters (some -1), some training
    cuts = sorted(set([0, T] + list(rng.integers(1, T, size=int(rng.integers(0, 4))))))
    segs = []
    for i in range(len(cuts) - 1):
        a = int(rng.integers(-1, n_ad))
        tr = 1 if (a >= 0 and rng.random() < 0.6) else 0
        segs.append((cuts[i], cuts[i + 1] - cuts[i], a, tr))
    if not any(s[3] for s in segs):
        st, ln, _, _ = segs[0]
        segs[0] = (st, ln, 0, 1)
    order = rng.permutation(len(segs))
    segs = [segs[i] for i in order]
    scale = [float(rng.choice([0.5, 1.0, 2.0, 3.0])) for _ in range(n_ad)]
    return workloads.custom(seed + 77, T, K, N, segs, rank, scale=scale, dtype="f32")


def _rel(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    d = np.abs(a - b).max() if a.size else 0.0
    return d / max(1e-300, np.abs(b).max() if b.size else 1.0)


def pin_brute_forward(lib=None, seeds=range(8)):
    for s in seeds:
        wl = _tiny(s)
        y = oracle.forward_wl(wl, lib=lib)
        yb = brute.forward(wl.T, wl.K, wl.N, wl.x.reshape(-1), wl.Wt.reshape(-1), wl.A, wl.B, wl.a_off, wl.b_off,
                           wl.rank, wl.scale, wl.segs.tolist())
        assert _rel(y, yb) <= 1e-12, ("brute forward", s, _rel(y, yb))


def pin_brute_backward(lib=None, seeds=range(8)):
    for s in seeds:
        wl = _tiny(s + 100)
        dX, dA, dB = oracle.backward_wl(wl, lib=lib)
        bX, bA, bB = brute.backward(wl.T, wl.K, wl.N, wl.x.reshape(-1), wl.Wt.reshape(-1), wl.A, wl.B, wl.a_off,
                                    wl.b_off, wl.rank, wl.scale, wl.segs.tolist(), wl.dY.reshape(-1))
        assert _rel(dX, np.array(bX).reshape(dX.shape)) <= 1e-12, ("brute dX", s)
        assert _rel(dA, bA) <= 1e-12, ("brute dA", s)
        assert _rel(dB, bB) <= 1e-12, ("brute dB", s)


def pin_merged_weight_config1(lib=None):
    """Config-1 size: y_t = x_t (W + s A^T B) per token's adapter, with numpy float64 matmul as the witness."""
    wl = workloads.config1()
    y = oracle.forward_wl(wl, lib=lib)
    x = wl.x.astype(np.float64)
    for st, ln, a, _ in wl.segs.tolist():
        W = wl.Wt.astype(np.float64).T.copy()
        if a >= 0:
            r = int(wl.rank[a])
            Aa = wl.A[wl.a_off[a]:wl.a_off[a] + r * wl.K].astype(np.float64).reshape(r, wl.K)
            Ba = wl.B[wl.b_off[a]:wl.b_off[a] + r * wl.N].astype(np.float64).reshape(r, wl.N)
            W = W + float(wl.scale[a]) * (Aa.T @ Ba)
        ref = x[st:st + ln] @ W
        assert _rel(y[st:st + ln], ref) <= 1e-12, ("merged weight", st)


def pin_zero_B(lib=None):
    """B = 0: y = x W (numpy witness) and dA = 0 exactly; dB = s * u^T dY."""
    wl = workloads.config1()
    wl.B[:] = 0.0
    y, u = oracle.forward_wl(wl, want_u=True, lib=lib)
    ref = wl.x.astype(np.float64) @ wl.Wt.astype(np.float64).T
    assert _rel(y, ref) <= 1e-13, "zero-B forward"
    dX, dA, dB = oracle.backward_wl(wl, lib=lib)
    assert np.all(dA == 0.0), "zero-B dA must be exactly zero"
    rows = wl.train_rows()
    refX = wl.dY[rows].astype(np.float64) @ wl.Wt.astype(np.float64)
    assert _rel(dX, refX) <= 1e-13, "zero-B dX"
    for st, ln, a, tr in wl.segs.tolist():
        if tr:
            r = int(wl.rank[a])
            g = float(wl.scale[a]) * (u[st:st + ln, :r].T @ wl.dY[st:st + ln].astype(np.float64))
            got = dB[wl.b_off[a]:wl.b_off[a] + r * wl.N].reshape(r, wl.N)
            assert _rel(got, g) <= 1e-12, "zero-B dB"


def _loss(wl, rows, lib):
    y = oracle.forward_wl(wl, rows=rows, lib=lib)
    return float((y * wl.dY[rows].astype(np.float64)).sum())


def pin_finite_differences(lib=None, n_dx=48, wl=None, every=True):
    """Central differences of L = sum over training rows of dY*y.

    L is linear in each single entry of x, A and B, so the difference quotient over the float32 steps
    actually taken (about +-1) equals the derivative up to float64 roundoff.
    """
    wl = wl or workloads.config1()
    rows = wl.train_rows()
    dX, dA, dB = oracle.backward_wl(wl, lib=lib)
    rng = np.random.default_rng(5)
    train_ads = sorted(set(int(s[2]) for s in wl.segs.tolist() if s[3]))
    for a in train_ads:
        r = int(wl.rank[a])
        idxA = np.arange(wl.a_off[a], wl.a_off[a] + r * wl.K)
        idxB = np.arange(wl.b_off[a], wl.b_off[a] + r * wl.N)
        if not every:
            idxA = rng.choice(idxA, 64, replace=False)
            idxB = rng.choice(idxB, 64, replace=False)
        for arr, idx, grad, name in ((wl.A, idxA, dA, "dA"), (wl.B, idxB, dB, "dB")):
            for i in idx:
                old = arr[i]
                arr[i] = old + np.float32(1.0)
                hp = float(arr[i]) - float(old)      # the step actually taken in float32
                lp = _loss(wl, rows, lib)
                arr[i] = old - np.float32(1.0)
                hm = float(old) - float(arr[i])
                lm = _loss(wl, rows, lib)
                arr[i] = old
                fd = (lp - lm) / (hp + hm)
                assert abs(fd - grad[i]) <= 1e-9 * max(1.0, abs(grad[i])), (name, int(i), fd, grad[i])
    for q in range(n_dx):
        p = int(rng.integers(0, rows.shape[0]))
        t = int(rows[p])
        k = int(rng.integers(0, wl.K))
        old = wl.x[t, k]
        wl.x[t, k] = old + np.float32(1.0)
        hp = float(wl.x[t, k]) - float(old)
        lp = _loss(wl, np.array([t]), lib)
        wl.x[t, k] = old - np.float32(1.0)
        hm = float(old) - float(wl.x[t, k])
        lm = _loss(wl, np.array([t]), lib)
        wl.x[t, k] = old
        fd = (lp - lm) / (hp + hm)
        assert abs(fd - dX[p, k]) <= 1e-9 * max(1.0, abs(dX[p, k])), ("dX", t, k, fd, dX[p, k])


def pin_segment_order(lib=None):
    wl = workloads.config5(K=64, N=96, n_adapters=12, n_decode=24, prefill_tokens=80, len_lo=4, len_hi=40,
                           train_len=20)
    y0 = oracle.forward_wl(wl, lib=lib)
    g0 = oracle.backward_wl(wl, lib=lib)
    rng = np.random.default_rng(3)
    wl.segs = wl.segs[rng.permutation(wl.segs.shape[0])]
    y1 = oracle.forward_wl(wl, lib=lib)
    g1 = oracle.backward_wl(wl, lib=lib)
    assert np.array_equal(y0, y1), "segment order changed y"
    for a, b in zip(g0, g1):
        assert np.array_equal(a, b), "segment order changed a gradient"


def permute_pool(wl, perm):
    """Reorder the adapter pool: new adapter i is old adapter perm[i]; ids in the table are remapped."""
    inv = np.empty_like(perm)
    inv[perm] = np.arange(perm.shape[0])
    rank = wl.rank[perm]
    scale = wl.scale[perm]
    A = np.concatenate([wl.A[wl.a_off[p]:wl.a_off[p] + wl.rank[p] * wl.K] for p in perm])
    B = np.concatenate([wl.B[wl.b_off[p]:wl.b_off[p] + wl.rank[p] * wl.N] for p in perm])
    a_off = np.concatenate([[0], np.cumsum(rank[:-1].astype(np.int64) * wl.K)]).astype(np.int64)
    b_off = np.concatenate([[0], np.cumsum(rank[:-1].astype(np.int64) * wl.N)]).astype(np.int64)
    segs = wl.segs.copy()
    m = segs[:, 2] >= 0
    segs[m, 2] = inv[segs[m, 2]]
    return rank, scale, A, B, a_off, b_off, segs


def pin_pool_order(lib=None):
    wl = workloads.config5(K=64, N=96, n_adapters=12, n_decode=24, prefill_tokens=80, len_lo=4, len_hi=40,
                           train_len=20)
    y0 = oracle.forward_wl(wl, lib=lib)
    dX0, dA0, dB0 = oracle.backward_wl(wl, lib=lib)
    perm = np.random.default_rng(9).permutation(wl.n_adapters)
    rank, scale, A, B, a_off, b_off, segs = permute_pool(wl, perm)
    y1 = oracle.forward(wl.x, wl.Wt, A, B, a_off, b_off, rank, scale, segs, lib=lib)
    dX1, dA1, dB1 = oracle.backward(wl.x, wl.Wt, A, B, a_off, b_off, rank, scale, segs, wl.dY, lib=lib)
    assert np.array_equal(y0, y1), "pool order changed y"
    assert np.array_equal(dX0, dX1), "pool order changed dX"
    for i, p in enumerate(perm):
        r = wl.rank[p]
        assert np.array_equal(dA1[a_off[i]:a_off[i] + r * wl.K], dA0[wl.a_off[p]:wl.a_off[p] + r * wl.K]), "dA perm"
        assert np.array_equal(dB1[b_off[i]:b_off[i] + r * wl.N], dB0[wl.b_off[p]:wl.b_off[p] + r * wl.N]), "dB perm"


def routing_pattern(wl):
    """W = 0, A_a = e_0 (u[t,0] = x[t,0]), B_a[0,n] = a+1+(n%3), s = 1, integer x: y[t,n] = x[t,0]*B_a[0,n]."""
    wl.Wt[:] = 0.0
    wl.A[:] = 0.0
    wl.B[:] = 0.0
    for a in range(wl.n_adapters):
        wl.A[wl.a_off[a]] = 1.0
        wl.B[wl.b_off[a]:wl.b_off[a] + wl.N] = (a % 61) + 1 + (np.arange(wl.N) % 3)
    wl.scale[:] = 1.0
    rng = np.random.default_rng(11)
    wl.x[:] = rng.integers(-3, 4, size=wl.x.shape).astype(np.float32)
    return wl


def routing_expected(wl):
    y = np.zeros((wl.T, wl.N), np.float64)
    for st, ln, a, _ in wl.segs.tolist():
        if a >= 0:
            y[st:st + ln] = wl.x[st:st + ln, :1].astype(np.float64) * wl.B[wl.b_off[a]:wl.b_off[a] + wl.N]
    return y


def pin_routing(lib=None):
    wl = routing_pattern(workloads.config2(T=96, K=32, N=40, n_adapters=10))
    y = oracle.forward_wl(wl, lib=lib)
    assert np.array_equal(y, routing_expected(wl)), "routing pattern"


def pin_trainable_count(lib=None):
    """Backward writes exactly the r(K+N) entries of each training adapter and nothing else."""
    wl = workloads.config5(K=40, N=56, n_adapters=9, n_decode=10, prefill_tokens=30, len_lo=4, len_hi=20,
                           train_len=12)
    sentinel_A = np.full(wl.A.shape[0], 12345.0)
    sentinel_B = np.full(wl.B.shape[0], 12345.0)
    _, dA, dB = oracle.backward_wl(wl, dA_init=sentinel_A, dB_init=sentinel_B, lib=lib)
    train_ads = sorted(set(int(s[2]) for s in wl.segs.tolist() if s[3]))
    written = int((dA != 12345.0).sum() + (dB != 12345.0).sum())
    expect = sum(int(wl.rank[a]) * (wl.K + wl.N) for a in train_ads)
    assert written == expect, ("trainable entries", written, expect)


def pin_accumulate(lib=None):
    wl = workloads.config1()
    _, dA, dB = oracle.backward_wl(wl, lib=lib)
    initA = np.random.default_rng(1).standard_normal(wl.A.shape[0])
    initB = np.random.default_rng(2).standard_normal(wl.B.shape[0])
    _, aA, aB = oracle.backward_wl(wl, accumulate=True, dA_init=initA, dB_init=initB, lib=lib)
    train_ads = sorted(set(int(s[2]) for s in wl.segs.tolist() if s[3]))
    mA = np.zeros(wl.A.shape[0], bool)
    mB = np.zeros(wl.B.shape[0], bool)
    for a in train_ads:
        mA[wl.a_off[a]:wl.a_off[a] + wl.rank[a] * wl.K] = True
        mB[wl.b_off[a]:wl.b_off[a] + wl.rank[a] * wl.N] = True
    assert np.allclose(aA[mA], initA[mA] + dA[mA], rtol=1e-13, atol=1e-13), "accumulate dA"
    assert np.allclose(aB[mB], initB[mB] + dB[mB], rtol=1e-13, atol=1e-13), "accumulate dB"
    assert np.array_equal(aA[~mA], initA[~mA]) and np.array_equal(aB[~mB], initB[~mB]), "untouched blocks"


def pin_sampled_columns(lib=None):
    """Column-restricted gradients and row-restricted outputs equal the matching slices of the full ones."""
    wl = workloads.config5(K=48, N=72, n_adapters=9, n_decode=12, prefill_tokens=40, len_lo=4, len_hi=20,
                           train_len=16)
    y = oracle.forward_wl(wl, lib=lib)
    rows = np.array([0, 5, wl.T - 1, 17])
    assert np.array_equal(oracle.forward_wl(wl, rows=rows, lib=lib), y[rows]), "row-sampled forward"
    dX, dA, dB = oracle.backward_wl(wl, lib=lib)
    cb = np.array([0, 3, wl.N - 1])
    ca = np.array([1, wl.K - 2])
    _, sA, sB = oracle.backward_wl(wl, want_dx=False, cols_b=cb, cols_a=ca, lib=lib)
    a = int(wl.meta["train_adapter"])
    r = int(wl.rank[a])
    fB = dB[wl.b_off[a]:wl.b_off[a] + r * wl.N].reshape(r, wl.N)
    gB = sB[wl.b_off[a]:wl.b_off[a] + r * wl.N].reshape(r, wl.N)
    fA = dA[wl.a_off[a]:wl.a_off[a] + r * wl.K].reshape(r, wl.K)
    gA = sA[wl.a_off[a]:wl.a_off[a] + r * wl.K].reshape(r, wl.K)
    assert np.array_equal(gB[:, cb], fB[:, cb]) and np.array_equal(gA[:, ca], fA[:, ca]), "column-sampled grads"
    others = np.setdiff1d(np.arange(wl.N), cb)
    assert np.all(gB[:, others] == 0.0), "unsampled columns untouched"
    trows = wl.train_rows()
    pick = np.array([2, 20])
    sX, _, _ = oracle.backward_wl(wl, dx_rows=trows[pick], want_grads=False, lib=lib)
    assert np.array_equal(sX, dX[pick]), "row-sampled dX"


def _saved_case():
    """Three fine-tuning segments on two adapters of different ranks, given out of start order, plus inference
    segments: the saved-activation layout then has blocks of different widths at nonzero offsets."""
    segs = [(30, 7, 1, 1), (0, 9, 0, 1), (9, 5, -1, 0), (14, 6, 2, 0), (20, 10, 0, 1)]
    return workloads.custom(4242, 37, 12, 10, segs, [3, 5, 2], scale=[2.0, 0.5, 1.0], dtype="f32")


def pin_saved_u_exact(lib=None):
    """Captured xA equal to what the backward would recompute: every gradient bit for bit the recompute's."""
    wl = _saved_case()
    _, u = oracle.forward_wl(wl, want_u=True, lib=lib)
    us = oracle.saved_u(wl, u)
    g0 = oracle.backward_wl(wl, lib=lib)
    g1 = oracle.backward_wl(wl, u_saved=us, lib=lib)
    for a, b, n in zip(g0, g1, ("dX", "dA", "dB")):
        assert np.array_equal(a, b), "saved exact u changed " + n


def pin_saved_u_onehot(lib=None):
    """Captured xA that is zero except u[t, j] = 1 (t the p-th row of the q-th fine-tuning segment in start order):
    dB_a = s_a e_j dY[t] exactly (a the segment's adapter), every other dB entry 0; dA and dX do not read u."""
    wl = _saved_case()
    g0 = oracle.backward_wl(wl, lib=lib)
    train = sorted(q for q in wl.segs.tolist() if q[3])
    n_u = sum(ln * int(wl.rank[a]) for _, ln, a, _ in train)
    off = 0
    picks = []
    for st, ln, a, _ in train:
        r = int(wl.rank[a])
        picks += [(off + p * r + j, st + p, a, j) for p, j in ((0, 0), (ln - 1, r - 1), (ln // 2, r // 2))]
        off += ln * r
    for idx, t, a, j in picks:
        us = np.zeros(n_u, np.float64)
        us[idx] = 1.0
        dX, dA, dB = oracle.backward_wl(wl, u_saved=us, lib=lib)
        assert np.array_equal(dX, g0[0]) and np.array_equal(dA, g0[1]), "dX / dA read the saved u"
        exp = np.zeros_like(dB)
        b0 = int(wl.b_off[a]) + j * wl.N
        exp[b0:b0 + wl.N] = float(wl.scale[a]) * wl.dY[t].astype(np.float64)
        assert np.array_equal(dB, exp), ("one-hot saved u", idx, t, a, j)


def pin_saved_u_double(lib=None):
    """Doubling the captured xA doubles dB exactly (dB is linear in u; scaling by 2 is exact)."""
    wl = _saved_case()
    us = np.random.default_rng(17).standard_normal(
        sum(ln * int(wl.rank[a]) for _, ln, a, tr in wl.segs.tolist() if tr))
    _, _, dB1 = oracle.backward_wl(wl, u_saved=us, lib=lib)
    _, _, dB2 = oracle.backward_wl(wl, u_saved=2.0 * us, lib=lib)
    assert np.array_equal(dB2, 2.0 * dB1), "dB not linear in the saved u"


def _tiny_sliced(seed):
    """A tiny fp32 sliced projection: 2-3 slices of random widths, 1-3 adapters of rank 1-3."""
    rng = np.random.default_rng(seed)
    S = int(rng.integers(2, 4))
    bounds = np.concatenate([[0], np.cumsum([int(rng.integers(2, 7)) for _ in range(S)])])
    T = int(rng.integers(3, 8))
    K = int(rng.integers(4, 10))
    n_ad = int(rng.integers(1, 4))
    rank = [int(rng.integers(1, 4)) for _ in range(n_ad)]
    cuts = sorted(set([0, T] + list(rng.integers(1, T, size=int(rng.integers(0, 3))))))
    segs = []
    for i in range(len(cuts) - 1):
        a = int(rng.integers(-1, n_ad))
        segs.append((cuts[i], cuts[i + 1] - cuts[i], a, 1 if (a >= 0 and rng.random() < 0.6) else 0))
    if not any(q[3] for q in segs):
        segs[0] = (segs[0][0], segs[0][1], 0, 1)
    scale = [float(rng.choice([0.5, 1.0, 2.0])) for _ in range(n_ad)]
    return workloads.sliced(seed + 91, T, K, bounds, segs, rank, scale=scale, dtype="f32")


def _block_diagonal(wl):
    """The sliced pool restated as a plain pool of rank S*r_a: the same stacked A, and an up factor with slice i's
    columns in rows [i r_a, (i+1) r_a) and zeros elsewhere (so x A_cat B_cat = sum over slices, each on its own
    columns)."""
    S = wl.n_slices
    rank = wl.rank.astype(np.int64) * S
    blocks, b_off, at = [], [], 0
    for a in range(wl.n_adapters):
        r = int(wl.rank[a])
        brow = int(wl.b_off[a]) // wl.N
        Bc = np.zeros((S * r, wl.N), np.float32)
        for i in range(S):
            c0, c1 = int(wl.bounds[i]), int(wl.bounds[i + 1])
            Bc[i * r:(i + 1) * r, c0:c1] = wl.B.reshape(-1, wl.N)[brow:brow + r, c0:c1]
        blocks.append(Bc.reshape(-1))
        b_off.append(at)
        at += S * r * wl.N
    return rank.astype(np.int32), np.concatenate(blocks), np.asarray(b_off, np.int64)


def pin_sliced_block_diagonal(lib=None, seeds=range(6)):
    """A sliced projection equals one LoRA layer of rank S*r with a block-diagonal up factor."""
    for sd in seeds:
        wl = _tiny_sliced(sd)
        rank_c, B_c, b_off_c = _block_diagonal(wl)
        y = sliced.forward_wl(wl, lib=lib)
        yc = oracle.forward(wl.x, wl.Wt, wl.A, B_c, wl.a_off, b_off_c, rank_c, wl.scale, wl.segs, lib=lib)
        assert _rel(y, yc) <= 1e-12, ("sliced forward vs block diagonal", sd)
        dX, dA, dB = sliced.backward_wl(wl, lib=lib)
        cX, cA, cB = oracle.backward(wl.x, wl.Wt, wl.A, B_c, wl.a_off, b_off_c, rank_c, wl.scale, wl.segs, wl.dY,
                                     lib=lib)
        assert _rel(dX, cX) <= 1e-12, ("sliced dX", sd)
        assert _rel(dA, cA) <= 1e-12, ("sliced dA", sd)
        for a in range(wl.n_adapters):
            r = int(wl.rank[a])
            got = dB.reshape(-1, wl.N)[int(wl.b_off[a]) // wl.N:int(wl.b_off[a]) // wl.N + r]
            full = cB[b_off_c[a]:b_off_c[a] + wl.n_slices * r * wl.N].reshape(wl.n_slices * r, wl.N)
            for i in range(wl.n_slices):
                c0, c1 = int(wl.bounds[i]), int(wl.bounds[i + 1])
                assert _rel(got[:, c0:c1], full[i * r:(i + 1) * r, c0:c1]) <= 1e-12 or \
                    (np.abs(full[i * r:(i + 1) * r, c0:c1]).max() == 0 and np.abs(got[:, c0:c1]).max() == 0), \
                    ("sliced dB", sd, a, i)


def pin_sliced_merged_weight(lib=None, seeds=range(6)):
    """Per output column n of slice i, the token's merged weight is W[:, n] + s A_{a,i}^T B_a[:, n]."""
    for sd in seeds:
        wl = _tiny_sliced(sd + 50)
        y = sliced.forward_wl(wl, lib=lib)
        x = wl.x.astype(np.float64)
        A2 = wl.A.reshape(-1, wl.K).astype(np.float64)
        B2 = wl.B.reshape(-1, wl.N).astype(np.float64)
        for st, ln, a, _ in wl.segs.tolist():
            W = wl.Wt.astype(np.float64).T.copy()
            if a >= 0:
                r = int(wl.rank[a])
                arow = int(wl.a_off[a]) // wl.K
                brow = int(wl.b_off[a]) // wl.N
                for n in range(wl.N):
                    i = int(np.searchsorted(wl.bounds, n, side="right")) - 1
                    for k in range(wl.K):
                        W[k, n] += float(wl.scale[a]) * sum(A2[arow + i * r + j, k] * B2[brow + j, n]
                                                            for j in range(r))
            ref = x[st:st + ln] @ W
            assert _rel(y[st:st + ln], ref) <= 1e-12, ("sliced merged weight", sd, st)


def pin_sliced_finite_differences(lib=None, seeds=range(3)):
    """Central differences of L = sum over training rows of dY*y for the sliced layer (exact: L is linear in every
    single entry of x, A and B)."""
    for sd in seeds:
        wl = _tiny_sliced(sd + 200)
        rows = wl.train_rows()
        dX, dA, dB = sliced.backward_wl(wl, lib=lib)

        def loss():
            y = sliced.forward_wl(wl, lib=lib)
            return float((y[rows] * wl.dY[rows].astype(np.float64)).sum())

        def fd(arr, idx):
            old = arr[idx]
            arr[idx] = old + np.float32(1.0)
            hp = float(arr[idx]) - float(old)
            lp = loss()
            arr[idx] = old - np.float32(1.0)
            hm = float(old) - float(arr[idx])
            lm = loss()
            arr[idx] = old
            return (lp - lm) / (hp + hm)

        for i in range(wl.A.shape[0]):
            g = fd(wl.A, i)
            assert abs(g - dA[i]) <= 1e-9 * max(1.0, abs(dA[i])), ("sliced dA fd", sd, i, g, dA[i])
        for i in range(wl.B.shape[0]):
            g = fd(wl.B, i)
            assert abs(g - dB[i]) <= 1e-9 * max(1.0, abs(dB[i])), ("sliced dB fd", sd, i, g, dB[i])
        for p in range(rows.shape[0]):
            for k in range(wl.K):
                g = fd(wl.x, (int(rows[p]), k))
                assert abs(g - dX[p, k]) <= 1e-9 * max(1.0, abs(dX[p, k])), ("sliced dX fd", sd, p, k)


def pin_sliced_one_slice(lib=None):
    """One slice covering every column is the plain layer."""
    wl = workloads.config5(K=48, N=64, n_adapters=7, n_decode=10, prefill_tokens=30, len_lo=4, len_hi=20,
                           train_len=12)
    b = np.array([0, wl.N], np.int32)
    y = sliced.forward(wl.x, wl.Wt, wl.A, wl.B, wl.a_off, wl.b_off, wl.rank, wl.scale, wl.segs, b, lib=lib)
    assert np.array_equal(y, oracle.forward_wl(wl, lib=lib)), "one-slice forward"
    g = sliced.backward(wl.x, wl.Wt, wl.A, wl.B, wl.a_off, wl.b_off, wl.rank, wl.scale, wl.segs, b, wl.dY, lib=lib)
    for u, v in zip(g, oracle.backward_wl(wl, lib=lib)):
        assert np.array_equal(u, v), "one-slice backward"


def sliced_saved_u(wl, u):
    """The sliced saved-activation layout (per training segment in increasing start order, a [len, S r_a] block,
    slice i in columns [i r_a, (i+1) r_a)) of sliced.forward(..., want_u=True)'s per-row values (slice i's xA in
    columns [128 i, 128 i + r_a))."""
    out = []
    for st, ln, a, tr in sorted(wl.segs.tolist()):
        if tr and ln > 0:
            r = int(wl.rank[a])
            out.append(np.concatenate([u[st:st + ln, 128 * i:128 * i + r] for i in range(wl.n_slices)], axis=1)
                       .reshape(-1))
    return np.concatenate(out)


def pin_sliced_saved_u(lib=None, seeds=range(3)):
    """Sliced layer: captured xA equal to the recompute gives the recompute's gradients bit for bit, and a one-hot
    captured xA in slice i reaches only slice i's columns of dB (= s e_j dY[t] there)."""
    for sd in seeds:
        wl = _tiny_sliced(sd + 300)
        _, u = sliced.forward_wl(wl, want_u=True, lib=lib)
        us = sliced_saved_u(wl, u)
        g0 = sliced.backward_wl(wl, lib=lib)
        g1 = sliced.backward_wl(wl, u_saved=us, lib=lib)
        for a, b in zip(g0, g1):
            assert np.array_equal(a, b), ("sliced saved exact u", sd)
        st, ln, a, _ = sorted(q for q in wl.segs.tolist() if q[3])[0]
        r = int(wl.rank[a])
        for i in range(wl.n_slices):
            oh = np.zeros_like(us)
            p, j = ln - 1, r - 1
            oh[p * wl.n_slices * r + i * r + j] = 1.0
            _, _, dB = sliced.backward_wl(wl, u_saved=oh, lib=lib)
            exp = np.zeros(wl.B.shape[0], np.float64).reshape(-1, wl.N)
            c0, c1 = int(wl.bounds[i]), int(wl.bounds[i + 1])
            exp[int(wl.b_off[a]) // wl.N + j, c0:c1] = float(wl.scale[a]) * wl.dY[st + p, c0:c1]
            assert np.array_equal(dB, exp.reshape(-1)), ("sliced one-hot saved u", sd, i)


ALL_PINS = [pin_brute_forward, pin_brute_backward, pin_merged_weight_config1, pin_zero_B, pin_finite_differences,
            pin_segment_order, pin_pool_order, pin_routing, pin_trainable_count, pin_accumulate,
            pin_sampled_columns, pin_sliced_block_diagonal, pin_sliced_merged_weight, pin_sliced_finite_differences,
            pin_sliced_one_slice, pin_saved_u_exact, pin_saved_u_onehot, pin_saved_u_double, pin_sliced_saved_u]
