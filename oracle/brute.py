"""Pure-Python brute force through the merged weight (test infrastructure only).

For tiny inputs (a handful of tokens, K and N up to a few dozen) this states
the layer a second way, independent of ``oracle.c``: it builds each adapter's
merged weight W_eff = W + s*A*B ("DeltaServe: Host-Agnostic Co-Serving of
Inference and Fine-Tuning for LLMs" section 2.2; "MOLT ..." section 2.1, with
the page's column form h = (W + BA) x written for row vectors) and multiplies
each token by the merged weight of its own adapter.

Backward through the merged weight: with y_t = x_t W_eff(a), the gradient of
the loss sum_t <dY_t, y_t> gives
    dX_t        = dY_t W_eff(a)^T
    G_a         = sum over a's training tokens of x_t^T dY_t      ([K, N])
    dA_a[j, k]  = s * sum_n G_a[k, n] * B_a[j, n]
    dB_a[j, n]  = s * sum_k A_a[j, k] * G_a[k, n]
which is a different route to the same numbers than the per-token formulas in
``oracle.c`` (no u = xA, no v = dY B^T).

Plain nested Python loops over Python floats (IEEE double).
"""


def _seg_of(segs, t):
    for i, (st, ln, a, tr) in enumerate(segs):
        if st <= t < st + ln:
            return i
    raise ValueError("token %d in no segment" % t)


def merged_weight(Wt, A, B, a_off, b_off, rank, scale, a, K, N):
    """W_eff[k][n] for adapter a (a = -1: W alone)."""
    W = [[float(Wt[n * K + k]) for n in range(N)] for k in range(K)]
    if a < 0:
        return W
    r = int(rank[a])
    s = float(scale[a])
    for k in range(K):
        for n in range(N):
            d = 0.0
            for j in range(r):
                d += float(A[a_off[a] + j * K + k]) * float(B[b_off[a] + j * N + n])
            W[k][n] += s * d
    return W


def forward(T, K, N, x, Wt, A, B, a_off, b_off, rank, scale, segs):
    """y as a list of T lists of N floats.  Arrays are flat sequences."""
    segs = [tuple(int(v) for v in s) for s in segs]
    cache = {}
    y = []
    for t in range(T):
        a = segs[_seg_of(segs, t)][2]
        if a not in cache:
            cache[a] = merged_weight(Wt, A, B, a_off, b_off, rank, scale, a, K, N)
        W = cache[a]
        y.append([sum(float(x[t * K + k]) * W[k][n] for k in range(K)) for n in range(N)])
    return y


def backward(T, K, N, x, Wt, A, B, a_off, b_off, rank, scale, segs, dY):
    """(dX rows of training tokens in increasing start order, dA, dB as flat lists)."""
    segs = [tuple(int(v) for v in s) for s in segs]
    train = sorted([s for s in segs if s[3] and s[1] > 0], key=lambda s: s[0])
    dX = []
    dA = [0.0] * len(A)
    dB = [0.0] * len(B)
    G = {}
    for (st, ln, a, _) in train:
        W = merged_weight(Wt, A, B, a_off, b_off, rank, scale, a, K, N)
        Ga = G.setdefault(a, [[0.0] * N for _ in range(K)])
        for t in range(st, st + ln):
            dX.append([sum(float(dY[t * N + n]) * W[k][n] for n in range(N)) for k in range(K)])
            for k in range(K):
                xv = float(x[t * K + k])
                for n in range(N):
                    Ga[k][n] += xv * float(dY[t * N + n])
    for a, Ga in G.items():
        r = int(rank[a])
        s = float(scale[a])
        for j in range(r):
            for k in range(K):
                dA[a_off[a] + j * K + k] = s * sum(Ga[k][n] * float(B[b_off[a] + j * N + n]) for n in range(N))
            for n in range(N):
                dB[b_off[a] + j * N + n] = s * sum(float(A[a_off[a] + j * K + k]) * Ga[k][n] for k in range(K))
    return dX, dA, dB
