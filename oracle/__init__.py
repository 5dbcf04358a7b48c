"""Float64 CPU oracle for the mixed-batch multi-adapter LoRA layer.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  It shares no
code with the CUDA library (``lora_co_serving_gb300``) and never imports it.

``oracle.c`` holds the definition (LoRA linear layer: "DeltaServe:
Host-Agnostic Co-Serving of Inference and Fine-Tuning for LLMs" section 2.2,
"MOLT: A Fine-Grained GPU Memory Sharing System for LLM Serving with
Opportunistic Fine-Tuning" section 2.1; mixed batches of inference and
fine-tuning entries: DeltaServe section 3.2).  ``brute.py`` is a second,
pure-Python statement through the merged weight W + s*A*B used to pin it.

Parity status: every function here is pinned by the tests in
``tests/test_oracle_pins.py`` (brute force, finite differences, closed forms,
invariants, mutation checks).
"""
import ctypes
import os

import numpy as np

from . import build as _build

_LIB = None


def _lib():
    global _LIB
    if _LIB is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        I32 = ctypes.c_int32
        lib.oracle_forward.argtypes = [I64, I64, I64, P, P, P, P, P, P, P, P, I32, P, I32, P, I64, P, P]
        lib.oracle_forward.restype = ctypes.c_int
        lib.oracle_backward.argtypes = [I64, I64, I64, P, P, P, P, P, P, P, P, I32, P, I32, P, P, I64, P, P,
                                        P, ctypes.c_int, P, I64, P, I64, P]
        lib.oracle_backward.restype = ctypes.c_int
        _LIB = lib
    return _LIB


def load_library(path):
    """Load an oracle built from another source (used by the mutation pins)."""
    global _LIB
    old = _LIB
    _LIB = None
    lib = ctypes.CDLL(path)
    _LIB = old
    P = ctypes.c_void_p
    I64 = ctypes.c_int64
    I32 = ctypes.c_int32
    lib.oracle_forward.argtypes = [I64, I64, I64, P, P, P, P, P, P, P, P, I32, P, I32, P, I64, P, P]
    lib.oracle_forward.restype = ctypes.c_int
    lib.oracle_backward.argtypes = [I64, I64, I64, P, P, P, P, P, P, P, P, I32, P, I32, P, P, I64, P, P,
                                    P, ctypes.c_int, P, I64, P, I64, P]
    lib.oracle_backward.restype = ctypes.c_int
    return lib


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def _ptr(a):
    return None if a is None else a.ctypes.data


class _Args:
    def __init__(self, x, Wt, A, B, a_off, b_off, rank, scale, segs):
        self.x = _f32(x)
        self.Wt = _f32(Wt)
        self.A = _f32(A).reshape(-1)
        self.B = _f32(B).reshape(-1)
        self.a_off = np.ascontiguousarray(a_off, dtype=np.int64)
        self.b_off = np.ascontiguousarray(b_off, dtype=np.int64)
        self.rank = np.ascontiguousarray(rank, dtype=np.int32)
        self.scale = np.ascontiguousarray(scale, dtype=np.float64)
        self.segs = np.ascontiguousarray(np.asarray(segs, dtype=np.int32).reshape(-1, 4))
        self.T, self.K = self.x.shape
        self.N = self.Wt.shape[0]


def forward(x, Wt, A, B, a_off, b_off, rank, scale, segs, rows=None, want_u=False, lib=None):
    """y (float64, [n_rows or T, N]) and optionally u = xA ([.., 128], zero padded)."""
    g = _Args(x, Wt, A, B, a_off, b_off, rank, scale, segs)
    rows_a = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    n = g.T if rows_a is None else rows_a.shape[0]
    y = np.zeros((n, g.N), dtype=np.float64)
    u = np.zeros((n, 128), dtype=np.float64) if want_u else None
    rc = (lib or _lib()).oracle_forward(g.T, g.K, g.N, _ptr(g.x), _ptr(g.Wt), _ptr(g.A), _ptr(g.B), _ptr(g.a_off),
                                        _ptr(g.b_off), _ptr(g.rank), _ptr(g.scale), len(g.rank), _ptr(g.segs),
                                        g.segs.shape[0], _ptr(rows_a), n, _ptr(y), _ptr(u))
    if rc != 0:
        raise ValueError("oracle_forward: malformed segment table or adapter id")
    return (y, u) if want_u else y


def backward(x, Wt, A, B, a_off, b_off, rank, scale, segs, dY, dx_rows=None, want_dx=True, want_grads=True,
             accumulate=False, dA_init=None, dB_init=None, cols_b=None, cols_a=None, u_saved=None, lib=None):
    """(dX, dA, dB) in float64.

    dX holds the rows listed in ``dx_rows`` (default: every training token in
    increasing segment-start order).  dA/dB are pool-shaped; adapters without
    training segments keep ``dA_init``/``dB_init`` (zeros by default).
    ``cols_b`` / ``cols_a`` restrict dB to the listed columns n and dA to the
    listed columns k (other entries keep their initial values).
    ``u_saved``: captured shrink activations xA in the saved-activation layout
    (per training segment in increasing start order, a [len, r_a] block); dB
    then uses them instead of recomputing xA (DeltaServe section 3.2,
    "Backward subprocess"; MOLT section 4.3).  None = recompute.
    """
    g = _Args(x, Wt, A, B, a_off, b_off, rank, scale, segs)
    dYa = _f32(dY)
    rows_a = None if dx_rows is None else np.ascontiguousarray(dx_rows, dtype=np.int64)
    cb = None if cols_b is None else np.ascontiguousarray(cols_b, dtype=np.int64)
    ca = None if cols_a is None else np.ascontiguousarray(cols_a, dtype=np.int64)
    if want_dx:
        if rows_a is None:
            tr = g.segs[g.segs[:, 3] != 0]
            n = int(tr[:, 1].sum())
        else:
            n = rows_a.shape[0]
        dX = np.zeros((n, g.K), dtype=np.float64)
    else:
        dX = None
    us = None if u_saved is None else np.ascontiguousarray(u_saved, dtype=np.float64).reshape(-1)
    if us is not None:
        tr = g.segs[(g.segs[:, 3] != 0) & (g.segs[:, 1] > 0)]
        need = int(sum(int(ln) * int(g.rank[a]) for _, ln, a, _ in tr.tolist()))
        if us.shape[0] < need:
            raise ValueError("u_saved holds %d values, the training segments need %d" % (us.shape[0], need))
    dA = dB = None
    if want_grads:
        dA = np.zeros(g.A.shape[0], np.float64) if dA_init is None else np.array(dA_init, np.float64).reshape(-1)
        dB = np.zeros(g.B.shape[0], np.float64) if dB_init is None else np.array(dB_init, np.float64).reshape(-1)
    rc = (lib or _lib()).oracle_backward(g.T, g.K, g.N, _ptr(g.x), _ptr(g.Wt), _ptr(g.A), _ptr(g.B), _ptr(g.a_off),
                                         _ptr(g.b_off), _ptr(g.rank), _ptr(g.scale), len(g.rank), _ptr(g.segs),
                                         g.segs.shape[0], _ptr(dYa), _ptr(rows_a),
                                         0 if rows_a is None else rows_a.shape[0], _ptr(dX), _ptr(dA), _ptr(dB),
                                         1 if accumulate else 0, _ptr(cb), 0 if cb is None else cb.shape[0],
                                         _ptr(ca), 0 if ca is None else ca.shape[0], _ptr(us))
    if rc != 0:
        raise ValueError("oracle_backward: malformed segment table")
    return dX, dA, dB


def forward_wl(wl, rows=None, want_u=False, lib=None):
    """forward() on a workload object (attributes x, Wt, A, B, a_off, b_off, rank, scale, segs)."""
    return forward(wl.x, wl.Wt, wl.A, wl.B, wl.a_off, wl.b_off, wl.rank, wl.scale, wl.segs, rows=rows,
                   want_u=want_u, lib=lib)


def backward_wl(wl, dx_rows=None, want_dx=True, want_grads=True, accumulate=False, dA_init=None, dB_init=None,
                cols_b=None, cols_a=None, u_saved=None, lib=None):
    return backward(wl.x, wl.Wt, wl.A, wl.B, wl.a_off, wl.b_off, wl.rank, wl.scale, wl.segs, wl.dY,
                    dx_rows=dx_rows, want_dx=want_dx, want_grads=want_grads, accumulate=accumulate,
                    dA_init=dA_init, dB_init=dB_init, cols_b=cols_b, cols_a=cols_a, u_saved=u_saved, lib=lib)


def saved_u(wl, u):
    """The saved-activation layout (per training segment in increasing start order, a [len, r_a] block, flat) of
    per-row shrink values ``u`` [T, >= r] (e.g. forward(..., want_u=True)'s second result)."""
    out = []
    for st, ln, a, tr in sorted(np.asarray(wl.segs).tolist()):
        if tr and ln > 0:
            out.append(np.asarray(u, np.float64)[st:st + ln, :int(wl.rank[a])].reshape(-1))
    return np.concatenate(out) if out else np.zeros(0, np.float64)
