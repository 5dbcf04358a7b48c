"""Float64 oracle of a sliced (fused) projection -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this module.

A decoder layer applies one adapter to several projections of the same input:
the fine-tuning adapter of "DeltaServe: Host-Agnostic Co-Serving of Inference
and Fine-Tuning for LLMs" (section 4.1, Fine-tuning Workload) sits on every
attention projection of Llama 3-8B, whose q, k and v projections all read the
layer's normalised hidden state.  A *sliced* projection runs such projections
as one layer over the concatenated weight: output columns [b_i, b_{i+1}) form
slice i, and every slice is an ordinary LoRA linear layer of its own (section
2.2 of the same page) on the shared input x:

    y[:, b_i:b_{i+1}] = x W_i + s_a (x A_{a,i}) B_{a,i}

Pool layout: adapter a's block in A stacks its S down factors, slice i's
[r_a, K] factor at rows [i r_a, (i+1) r_a); its block in B is [r_a, N], and the
columns [b_i, b_{i+1}) of it are slice i's up factor.

Backward: the loss sum <dY, y> reaches x through every slice, so dX is the sum
over slices of each slice's dX (chain rule for a shared input); the gradients
of A_{a,i} and B_{a,i} are those of slice i alone.

Every slice is computed by the float64 oracle of ``oracle.c`` on that slice's
weight columns and factors, gathered here with plain numpy indexing.
Pinned by ``tests/oracle_pins.py`` (block-diagonal rank-S r statement, merged
weight brute force per slice, exact finite differences).
"""
import numpy as np

from . import backward as _backward
from . import forward as _forward


def _slice_pool(A, B, a_off, b_off, rank, K, N, bounds, i):
    """Compact pool (A_i, B_i, a_off_i, b_off_i) of slice i."""
    c0, c1 = int(bounds[i]), int(bounds[i + 1])
    Ni = c1 - c0
    Ab, Bb, ao, bo = [], [], [], []
    at_a = at_b = 0
    for a in range(len(rank)):
        r = int(rank[a])
        base = int(a_off[a]) // K
        Ab.append(np.asarray(A, np.float32).reshape(-1, K)[base + i * r:base + (i + 1) * r])
        brow = int(b_off[a]) // N
        Bb.append(np.asarray(B, np.float32).reshape(-1, N)[brow:brow + r, c0:c1])
        ao.append(at_a)
        bo.append(at_b)
        at_a += r * K
        at_b += r * Ni
    Ai = np.concatenate(Ab).reshape(-1) if Ab else np.zeros(0, np.float32)
    Bi = np.concatenate(Bb).reshape(-1) if Bb else np.zeros(0, np.float32)
    return Ai, Bi, np.asarray(ao, np.int64), np.asarray(bo, np.int64)


def forward(x, Wt, A, B, a_off, b_off, rank, scale, segs, bounds, want_u=False, lib=None):
    """y [T, N] in float64; with want_u also xA [T, S*128]: slice i's xA in columns [128 i, 128 i + r_a)."""
    x = np.asarray(x, np.float32)
    Wt = np.asarray(Wt, np.float32)
    T, K = x.shape
    N = Wt.shape[0]
    S = len(bounds) - 1
    y = np.zeros((T, N), np.float64)
    u = np.zeros((T, 128 * S), np.float64) if want_u else None
    for i in range(S):
        c0, c1 = int(bounds[i]), int(bounds[i + 1])
        Ai, Bi, ao, bo = _slice_pool(A, B, a_off, b_off, rank, K, N, bounds, i)
        res = _forward(x, Wt[c0:c1], Ai, Bi, ao, bo, rank, scale, segs, want_u=want_u, lib=lib)
        if want_u:
            y[:, c0:c1], u[:, 128 * i:128 * (i + 1)] = res
        else:
            y[:, c0:c1] = res
    return (y, u) if want_u else y


def _slice_saved(u_saved, segs, rank, S, i):
    """Slice i's captured xA in the plain saved-activation layout ([len, r_a] per training segment, increasing
    start) out of the sliced layout ([len, S r_a] per segment, slice i in columns [i r_a, (i+1) r_a))."""
    u = np.asarray(u_saved, np.float64).reshape(-1)
    out, off = [], 0
    for st, ln, a, tr in sorted(np.asarray(segs).reshape(-1, 4).tolist()):
        if tr and ln > 0:
            r = int(rank[a])
            blk = u[off:off + ln * S * r].reshape(ln, S * r)
            out.append(blk[:, i * r:(i + 1) * r].reshape(-1))
            off += ln * S * r
    return np.concatenate(out) if out else np.zeros(0, np.float64)


def backward(x, Wt, A, B, a_off, b_off, rank, scale, segs, bounds, dY, u_saved=None, lib=None):
    """(dX over the training rows in increasing start order, dA pool-shaped like A, dB pool-shaped like B).
    ``u_saved``: captured xA in the sliced saved-activation layout (each slice's dB then uses its columns of it,
    DeltaServe section 3.2, "Backward subprocess"); None = recompute."""
    x = np.asarray(x, np.float32)
    Wt = np.asarray(Wt, np.float32)
    dY = np.asarray(dY, np.float32)
    T, K = x.shape
    N = Wt.shape[0]
    S = len(bounds) - 1
    dX = None
    dA = np.zeros(np.asarray(A).size, np.float64)
    dB = np.zeros(np.asarray(B).size, np.float64).reshape(-1, N) if N else np.zeros((0, 0))
    for i in range(S):
        c0, c1 = int(bounds[i]), int(bounds[i + 1])
        Ai, Bi, ao, bo = _slice_pool(A, B, a_off, b_off, rank, K, N, bounds, i)
        ui = None if u_saved is None else _slice_saved(u_saved, segs, rank, S, i)
        dXi, dAi, dBi = _backward(x, Wt[c0:c1], Ai, Bi, ao, bo, rank, scale, segs, dY[:, c0:c1], u_saved=ui,
                                  lib=lib)
        dX = dXi if dX is None else dX + dXi
        for a in range(len(rank)):
            r = int(rank[a])
            base = int(a_off[a])
            dA[base + i * r * K:base + (i + 1) * r * K] = dAi[ao[a]:ao[a] + r * K]
            brow = int(b_off[a]) // N
            dB[brow:brow + r, c0:c1] = dBi[bo[a]:bo[a] + r * (c1 - c0)].reshape(r, c1 - c0)
    return dX, dA, dB.reshape(-1)


def forward_wl(wl, want_u=False, lib=None):
    return forward(wl.x, wl.Wt, wl.A, wl.B, wl.a_off, wl.b_off, wl.rank, wl.scale, wl.segs, wl.bounds,
                   want_u=want_u, lib=lib)


def backward_wl(wl, u_saved=None, lib=None):
    return backward(wl.x, wl.Wt, wl.A, wl.B, wl.a_off, wl.b_off, wl.rank, wl.scale, wl.segs, wl.bounds, wl.dY,
                    u_saved=u_saved, lib=lib)
