"""Python binding of the mixed-batch multi-adapter LoRA layer library (``liblora_mixed.so``).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  PyTorch supplies device memory and streams.  The entry points mirror
``include/lora_mixed.h``:

    forward(x, Wt, pool, segs, ...)         -> y   (and the saved xA when asked)
    backward(x, Wt, pool, segs, dY, ...)    -> dX, dA, dB
    sliced_forward / sliced_backward        -> the same for a fused projection of several slices
                                               (q|k|v, gate|up) over one input

``segs`` is an int32 array (or list) of rows {start, len, adapter_id, is_train};
``Pool`` holds the stacked adapter factors (A blocks [r_a, K], B blocks [r_a, N])
on the device plus their host-side offsets, ranks and scales.

If the compiled library is missing, calls raise ``LibraryNotBuilt``: there is no
fallback path.
"""
import ctypes
import os

import numpy as np

from . import _build

__all__ = ["Pool", "forward", "backward", "sliced_forward", "sliced_backward", "sliced_workspace_size",
           "sliced_xa_size", "workspace_size", "xa_size", "workspace_status", "plan_describe",
           "LoraError", "LibraryNotBuilt", "library", "build", "SAVE_XA", "RECOMPUTE_XA", "ACCUMULATE_GRAD",
           "DEBUG_CHECKS", "plan_check", "static_status", "set_wait_limit"]

SAVE_XA = 1
RECOMPUTE_XA = 2
ACCUMULATE_GRAD = 4
DEBUG_CHECKS = 8
BF16 = 0
F32 = 1

ERRORS = {0: "LORA_OK", -1: "LORA_ERR_INVALID_ARG", -2: "LORA_ERR_SEGMENTS", -3: "LORA_ERR_ADAPTER",
          -4: "LORA_ERR_TRAIN_BASE", -5: "LORA_ERR_ALIGNMENT", -6: "LORA_ERR_WORKSPACE", -7: "LORA_ERR_DTYPE",
          -8: "LORA_ERR_CUDA", -9: "LORA_ERR_RANK", -10: "LORA_ERR_LIMIT", -11: "LORA_ERR_TIMEOUT",
          -12: "LORA_ERR_BOUNDS"}

EXPORTED = ["lora_workspace_size", "lora_xa_size", "lora_mixed_forward", "lora_mixed_backward", "lora_last_error",
            "lora_workspace_status", "lora_plan_describe", "lora_set_trace_events", "lora_mixed_forward_static",
            "lora_selftest_wait_timeout", "lora_adamw_step", "lora_mixed_backward_flagged",
            "lora_sliced_workspace_size", "lora_sliced_xa_size", "lora_sliced_forward", "lora_sliced_backward",
            "lora_latency_terms", "lora_latency_features", "lora_latency_fit", "lora_latency_predict",
            "lora_static_status", "lora_plan_check", "lora_set_wait_limit"]


class LoraError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__("%s (%d): %s" % (ERRORS.get(code, "?"), code, msg))
        self.code = code


class LibraryNotBuilt(ImportError):
    pass


class _Segment(ctypes.Structure):
    _fields_ = [("start", ctypes.c_int32), ("len", ctypes.c_int32), ("adapter_id", ctypes.c_int32),
                ("is_train", ctypes.c_int32)]


class _Pool(ctypes.Structure):
    _fields_ = [("A", ctypes.c_void_p), ("B", ctypes.c_void_p), ("a_off", ctypes.c_void_p),
                ("b_off", ctypes.c_void_p), ("rank", ctypes.c_void_p), ("scale", ctypes.c_void_p),
                ("n_adapters", ctypes.c_int32)]


class _Slices(ctypes.Structure):
    _fields_ = [("n_slices", ctypes.c_int32), ("col_bounds", ctypes.c_void_p)]


_LIB = None


def build(force=False):
    """Compile the CUDA library for sm_103a (in-tree) and return its path."""
    return _build.build(force=force)


def library(path=None):
    """The loaded ``liblora_mixed.so`` (ctypes); raises LibraryNotBuilt if it has not been built."""
    global _LIB
    if _LIB is not None and path is None:
        return _LIB
    p = path or _build.LIB
    if not os.path.exists(p):
        raise LibraryNotBuilt("liblora_mixed.so is not built; run lora_co_serving_gb300.build()")
    lib = ctypes.CDLL(p)
    P, I32, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    lib.lora_workspace_size.argtypes = [I32, I32, I32, ctypes.c_int, P, P, I32]
    lib.lora_workspace_size.restype = SZ
    lib.lora_xa_size.argtypes = [ctypes.c_int, P, P, I32]
    lib.lora_xa_size.restype = SZ
    lib.lora_mixed_forward.argtypes = [I32, I32, I32, ctypes.c_int, P, P, P, P, I32, P, P, ctypes.c_uint32, P, SZ, P]
    lib.lora_mixed_forward.restype = ctypes.c_int
    lib.lora_mixed_backward.argtypes = [I32, I32, I32, ctypes.c_int, P, P, P, P, I32, P, P, P, P, P, ctypes.c_uint32,
                                        P, SZ, P]
    lib.lora_mixed_backward.restype = ctypes.c_int
    lib.lora_last_error.argtypes = []
    lib.lora_last_error.restype = ctypes.c_char_p
    lib.lora_workspace_status.argtypes = [P, P]
    lib.lora_workspace_status.restype = ctypes.c_int
    lib.lora_plan_describe.argtypes = [I32, I32, I32, P, P, I32, P, P, P, I32]
    lib.lora_plan_describe.restype = ctypes.c_int
    lib.lora_set_trace_events.argtypes = [P]
    lib.lora_set_trace_events.restype = ctypes.c_int
    lib.lora_mixed_forward_static.argtypes = [I32, I32, I32, ctypes.c_int, P, P, P, P, I32, P, P, ctypes.c_uint32, P]
    lib.lora_mixed_forward_static.restype = ctypes.c_int
    lib.lora_plan_check.argtypes = [I32, I32, I32, P, P, P, I32, I32]
    lib.lora_plan_check.restype = ctypes.c_int
    lib.lora_static_status.argtypes = [P]
    lib.lora_static_status.restype = ctypes.c_int
    lib.lora_set_wait_limit.argtypes = [ctypes.c_uint64]
    lib.lora_set_wait_limit.restype = ctypes.c_int
    lib.lora_selftest_wait_timeout.argtypes = [P, SZ, P]
    lib.lora_selftest_wait_timeout.restype = ctypes.c_int
    lib.lora_adamw_step.argtypes = [ctypes.c_int, P, I32, I32, P, P, P, P, P, P, P, P, P, P, P, I32, P, P]
    lib.lora_adamw_step.restype = ctypes.c_int
    lib.lora_mixed_backward_flagged.argtypes = [I32, I32, I32, ctypes.c_int, P, P, P, P, I32, P, P, P, P, P, P,
                                                ctypes.c_uint32, P, SZ, P]
    lib.lora_mixed_backward_flagged.restype = ctypes.c_int
    lib.lora_sliced_workspace_size.argtypes = [I32, I32, I32, ctypes.c_int, P, P, P, I32]
    lib.lora_sliced_workspace_size.restype = SZ
    lib.lora_sliced_xa_size.argtypes = [ctypes.c_int, P, P, P, I32]
    lib.lora_sliced_xa_size.restype = SZ
    lib.lora_sliced_forward.argtypes = [I32, I32, I32, ctypes.c_int, P, P, P, P, P, I32, P, P, ctypes.c_uint32, P, SZ,
                                        P]
    lib.lora_sliced_forward.restype = ctypes.c_int
    lib.lora_sliced_backward.argtypes = [I32, I32, I32, ctypes.c_int, P, P, P, P, P, I32, P, P, P, P, P,
                                         ctypes.c_uint32, P, SZ, P]
    lib.lora_sliced_backward.restype = ctypes.c_int
    lib.lora_latency_terms.argtypes = [I32]
    lib.lora_latency_terms.restype = I32
    lib.lora_latency_features.argtypes = [I32, P, I32, ctypes.c_double, P]
    lib.lora_latency_features.restype = ctypes.c_int
    lib.lora_latency_fit.argtypes = [I32, P, P, I32, P]
    lib.lora_latency_fit.restype = ctypes.c_int
    lib.lora_latency_predict.argtypes = [I32, P, P]
    lib.lora_latency_predict.restype = ctypes.c_double
    if path is None:
        _LIB = lib
    return lib


def _check(rc):
    if rc != 0:
        raise LoraError(rc, library().lora_last_error().decode())


def _ptr(t):
    """Raw address of a torch tensor / numpy array (None -> NULL)."""
    if t is None:
        return None
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    return t.data_ptr()


def _dtype_code(t):
    import torch
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError("unsupported dtype %s (bf16 or float32)" % t.dtype)


def _stream_ptr(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def segments(segs):
    """Segment table as a contiguous int32 [n, 4] numpy array."""
    a = np.ascontiguousarray(np.asarray(segs, dtype=np.int32).reshape(-1, 4))
    return a


class AdamW(ctypes.Structure):
    """lora_adamw_t: AdamW hyperparameters (step is 1-based)."""
    _fields_ = [("lr", ctypes.c_float), ("beta1", ctypes.c_float), ("beta2", ctypes.c_float),
                ("eps", ctypes.c_float), ("weight_decay", ctypes.c_float), ("step", ctypes.c_int32)]


def adamw_step(pool, K, N, dA, dB, mA, vA, mB, vB, adapters, step, lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8,
               weight_decay=0.01, A_master=None, B_master=None, stream=None):
    """AdamW on the listed adapters' blocks of pool.A / pool.B (and fp32 masters if given), in place."""
    code = _dtype_code(pool.A)
    ids = np.ascontiguousarray(adapters, dtype=np.int32)
    hp = AdamW(lr, beta1, beta2, eps, weight_decay, step)
    _check(library().lora_adamw_step(code, pool.cptr(), K, N, _ptr(pool.A), _ptr(pool.B), _ptr(A_master),
                                     _ptr(B_master), _ptr(dA), _ptr(dB), _ptr(mA), _ptr(vA), _ptr(mB), _ptr(vB),
                                     _ptr(ids), ids.shape[0], ctypes.addressof(hp), _stream_ptr(stream)))


class Pool:
    """Stacked adapter pool: A (concatenated [r_a, K] blocks) and B (concatenated [r_a, N] blocks) on the device,
    with host arrays of element offsets, ranks and scales."""

    def __init__(self, A, B, a_off, b_off, rank, scale):
        self.A = A
        self.B = B
        self.a_off = np.ascontiguousarray(a_off, dtype=np.int64)
        self.b_off = np.ascontiguousarray(b_off, dtype=np.int64)
        self.rank = np.ascontiguousarray(rank, dtype=np.int32)
        self.scale = np.ascontiguousarray(scale, dtype=np.float32)
        n = self.rank.shape[0]
        self._c = _Pool(_ptr(A), _ptr(B), _ptr(self.a_off), _ptr(self.b_off), _ptr(self.rank), _ptr(self.scale), n)

    @property
    def n_adapters(self):
        return int(self.rank.shape[0])

    def cptr(self):
        return ctypes.addressof(self._c)


def workspace_size(T, K, N, dtype_code, pool, segs):
    s = segments(segs)
    n = library().lora_workspace_size(T, K, N, dtype_code, pool.cptr(), _ptr(s), s.shape[0])
    if n == 0:
        raise LoraError(-1, library().lora_last_error().decode())
    return int(n)


def xa_size(dtype_code, pool, segs):
    s = segments(segs)
    return int(library().lora_xa_size(dtype_code, pool.cptr(), _ptr(s), s.shape[0]))


def _workspace(T, K, N, code, pool, s, workspace, device):
    """The caller's workspace, or a new one of the size this call needs (the library checks a given one)."""
    import torch
    if workspace is None:
        workspace = torch.empty(workspace_size(T, K, N, code, pool, s), dtype=torch.uint8, device=device)
    return workspace


def forward(x, Wt, pool, segs, y=None, xa_save=None, save_xa=False, workspace=None, stream=None, debug=False,
            check_status=False):
    """y [T, N] = x W + per-segment LoRA; returns y, or (y, xa_save) when save_xa is set.

    debug: LORA_DEBUG_CHECKS (host plan check, in-kernel bounds checks on every store).  check_status: wait for the
    call and raise LoraError if a kernel reported a problem in the workspace status word (a bounded wait that gave
    up, or a debug bounds check)."""
    import torch
    T, K = x.shape
    N = Wt.shape[0]
    code = _dtype_code(x)
    s = segments(segs)
    if y is None:
        y = torch.empty((T, N), dtype=x.dtype, device=x.device)
    if save_xa and xa_save is None:
        n = xa_size(code, pool, s) // x.element_size()
        xa_save = torch.empty(max(n, 1), dtype=x.dtype, device=x.device)
    ws = _workspace(T, K, N, code, pool, s, workspace, x.device)
    flags = (SAVE_XA if save_xa else 0) | (DEBUG_CHECKS if debug else 0)
    _check(library().lora_mixed_forward(T, K, N, code, _ptr(x), _ptr(Wt), pool.cptr(), _ptr(s), s.shape[0], _ptr(y),
                                        _ptr(xa_save), flags, _ptr(ws), ws.numel(), _stream_ptr(stream)))
    if check_status:
        workspace_status(ws, stream)
    return (y, xa_save) if save_xa else y


def forward_static(x, Wt, pool, segs, y=None, xa_save=None, save_xa=False, stream=None):
    """forward() with the library's fixed device scratch instead of a caller workspace (allocates nothing in
    the library; see lora_mixed_forward_static).  Returns y, or (y, xa_save) when save_xa is set."""
    import torch
    T, K = x.shape
    N = Wt.shape[0]
    code = _dtype_code(x)
    s = segments(segs)
    if y is None:
        y = torch.empty((T, N), dtype=x.dtype, device=x.device)
    if save_xa and xa_save is None:
        n = xa_size(code, pool, s) // x.element_size()
        xa_save = torch.empty(max(n, 1), dtype=x.dtype, device=x.device)
    flags = SAVE_XA if save_xa else 0
    _check(library().lora_mixed_forward_static(T, K, N, code, _ptr(x), _ptr(Wt), pool.cptr(), _ptr(s), s.shape[0],
                                               _ptr(y), _ptr(xa_save), flags, _stream_ptr(stream)))
    return (y, xa_save) if save_xa else y


def set_wait_limit(seconds):
    """Limit of every bounded wait in the library's kernels on the current device (1 ms to 60 s; default 1 s)."""
    _check(library().lora_set_wait_limit(int(round(seconds * 1e9))))


def static_status(stream=None):
    """Raise LoraError if a kernel of the last lora_mixed_forward_static call on this device gave up a wait."""
    _check(library().lora_static_status(_stream_ptr(stream)))


def backward(x, Wt, pool, segs, dY, xa_saved=None, dX=None, dA=None, dB=None, want_dx=True, want_grads=True,
             recompute=False, accumulate=False, workspace=None, stream=None, debug=False, check_status=False):
    """LoRA backward of the fine-tuning segments; returns (dX, dA, dB) (dA/dB float32, pool-shaped).
    debug / check_status: as in forward()."""
    import torch
    T, K = x.shape
    N = Wt.shape[0]
    code = _dtype_code(x)
    s = segments(segs)
    if want_dx and dX is None:
        dX = torch.zeros((T, K), dtype=x.dtype, device=x.device)
    if want_grads and dA is None:
        dA = torch.zeros(pool.A.numel(), dtype=torch.float32, device=x.device)
    if want_grads and dB is None:
        dB = torch.zeros(pool.B.numel(), dtype=torch.float32, device=x.device)
    ws = _workspace(T, K, N, code, pool, s, workspace, x.device)
    flags = (RECOMPUTE_XA if recompute else 0) | (ACCUMULATE_GRAD if accumulate else 0) | (DEBUG_CHECKS if debug else 0)
    _check(library().lora_mixed_backward(T, K, N, code, _ptr(x), _ptr(Wt), pool.cptr(), _ptr(s), s.shape[0],
                                         _ptr(dY), _ptr(xa_saved), _ptr(dX) if want_dx else None,
                                         _ptr(dA) if want_grads else None, _ptr(dB) if want_grads else None, flags,
                                         _ptr(ws), ws.numel(), _stream_ptr(stream)))
    if check_status:
        workspace_status(ws, stream)
    return dX, dA, dB


def backward_flagged(x, Wt, pool, segs, dY, xa_saved, xa_valid, dX=None, dA=None, dB=None, accumulate=False,
                     workspace=None, stream=None):
    """backward() with a device flag table choosing, per fine-tuning segment (increasing start order), the saved
    xA (nonzero) or a recompute (zero)."""
    import torch
    T, K = x.shape
    N = Wt.shape[0]
    code = _dtype_code(x)
    s = segments(segs)
    if dX is None:
        dX = torch.zeros((T, K), dtype=x.dtype, device=x.device)
    if dA is None:
        dA = torch.zeros(pool.A.numel(), dtype=torch.float32, device=x.device)
    if dB is None:
        dB = torch.zeros(pool.B.numel(), dtype=torch.float32, device=x.device)
    ws = _workspace(T, K, N, code, pool, s, workspace, x.device)
    flags = ACCUMULATE_GRAD if accumulate else 0
    _check(library().lora_mixed_backward_flagged(T, K, N, code, _ptr(x), _ptr(Wt), pool.cptr(), _ptr(s), s.shape[0],
                                                 _ptr(dY), _ptr(xa_saved), _ptr(xa_valid), _ptr(dX), _ptr(dA),
                                                 _ptr(dB), flags, _ptr(ws), ws.numel(), _stream_ptr(stream)))
    return dX, dA, dB


def workspace_status(workspace, stream=None):
    """Raise LoraError if a kernel of the last call on this workspace gave up a bounded wait."""
    _check(library().lora_workspace_status(_ptr(workspace), _stream_ptr(stream)))


def set_trace_events(events):
    """Record 8 torch.cuda.Event objects around the four launch groups of later calls (None: off)."""
    if events is None:
        _check(library().lora_set_trace_events(None))
        return
    assert len(events) == 8
    arr = (ctypes.c_void_p * 8)(*[e.cuda_event for e in events])
    _check(library().lora_set_trace_events(ctypes.cast(arr, ctypes.c_void_p)))


def plan_check(T, K, N, pool, segs, backward=False, bounds=None):
    """Host check of the bf16 plan of this table (LORA_DEBUG_CHECKS' host half); raises LoraError on a violation."""
    s = segments(segs)
    sl = None if bounds is None else _slices(bounds)
    _check(library().lora_plan_check(T, K, N, pool.cptr(), None if sl is None else sl.cptr(), _ptr(s), s.shape[0],
                                     1 if backward else 0))


def plan_describe(T, K, N, pool, segs, cap=None):
    """(rows [n_tiles, 128], info [n_tiles, 4]) of the forward tile plan; info = gathered, adapters, LoRA cols, x row."""
    s = segments(segs)
    cap = cap or (T // 128 + 2 * s.shape[0] + 8)
    rows = np.zeros((cap, 128), np.int32)
    info = np.zeros((cap, 4), np.int32)
    nt = ctypes.c_int32(0)
    _check(library().lora_plan_describe(T, K, N, pool.cptr(), _ptr(s), s.shape[0], ctypes.addressof(nt), _ptr(rows),
                                        _ptr(info), cap))
    return rows[:nt.value], info[:nt.value]


class Slices:
    """Output-column bounds of a sliced (fused) projection: slice i = columns [bounds[i], bounds[i+1])."""

    def __init__(self, bounds):
        self.bounds = np.ascontiguousarray(bounds, dtype=np.int32)
        self._c = _Slices(self.bounds.shape[0] - 1, _ptr(self.bounds))

    @property
    def n_slices(self):
        return int(self.bounds.shape[0]) - 1

    def cptr(self):
        return ctypes.addressof(self._c)


def _slices(bounds):
    return bounds if isinstance(bounds, Slices) else Slices(bounds)


def sliced_workspace_size(T, K, N, dtype_code, pool, bounds, segs):
    s = segments(segs)
    sl = _slices(bounds)
    n = library().lora_sliced_workspace_size(T, K, N, dtype_code, pool.cptr(), sl.cptr(), _ptr(s), s.shape[0])
    if n == 0:
        raise LoraError(-1, library().lora_last_error().decode())
    return int(n)


def sliced_xa_size(dtype_code, pool, bounds, segs):
    s = segments(segs)
    return int(library().lora_sliced_xa_size(dtype_code, pool.cptr(), _slices(bounds).cptr(), _ptr(s), s.shape[0]))


def sliced_forward(x, Wt, pool, bounds, segs, y=None, xa_save=None, save_xa=False, workspace=None, stream=None):
    """Forward of a sliced projection (Wt [N, K] = the slices' weights stacked; pool laid out per
    lora_sliced_forward).  Returns y, or (y, xa_save) when save_xa is set."""
    import torch
    T, K = x.shape
    N = Wt.shape[0]
    code = _dtype_code(x)
    s = segments(segs)
    sl = _slices(bounds)
    if y is None:
        y = torch.empty((T, N), dtype=x.dtype, device=x.device)
    if save_xa and xa_save is None:
        n = sliced_xa_size(code, pool, sl, s) // x.element_size()
        xa_save = torch.empty(max(n, 1), dtype=x.dtype, device=x.device)
    if workspace is None:
        workspace = torch.empty(sliced_workspace_size(T, K, N, code, pool, sl, s), dtype=torch.uint8, device=x.device)
    flags = SAVE_XA if save_xa else 0
    _check(library().lora_sliced_forward(T, K, N, code, _ptr(x), _ptr(Wt), pool.cptr(), sl.cptr(), _ptr(s),
                                         s.shape[0], _ptr(y), _ptr(xa_save), flags, _ptr(workspace),
                                         workspace.numel(), _stream_ptr(stream)))
    return (y, xa_save) if save_xa else y


def sliced_backward(x, Wt, pool, bounds, segs, dY, xa_saved=None, dX=None, dA=None, dB=None, want_dx=True,
                    want_grads=True, recompute=False, accumulate=False, workspace=None, stream=None):
    """LoRA backward of a sliced projection; dX sums every slice's contribution.  Returns (dX, dA, dB)."""
    import torch
    T, K = x.shape
    N = Wt.shape[0]
    code = _dtype_code(x)
    s = segments(segs)
    sl = _slices(bounds)
    if want_dx and dX is None:
        dX = torch.zeros((T, K), dtype=x.dtype, device=x.device)
    if want_grads and dA is None:
        dA = torch.zeros(pool.A.numel(), dtype=torch.float32, device=x.device)
    if want_grads and dB is None:
        dB = torch.zeros(pool.B.numel(), dtype=torch.float32, device=x.device)
    if workspace is None:
        workspace = torch.empty(sliced_workspace_size(T, K, N, code, pool, sl, s), dtype=torch.uint8, device=x.device)
    flags = (RECOMPUTE_XA if recompute else 0) | (ACCUMULATE_GRAD if accumulate else 0)
    _check(library().lora_sliced_backward(T, K, N, code, _ptr(x), _ptr(Wt), pool.cptr(), sl.cptr(), _ptr(s),
                                          s.shape[0], _ptr(dY), _ptr(xa_saved), _ptr(dX) if want_dx else None,
                                          _ptr(dA) if want_grads else None, _ptr(dB) if want_grads else None, flags,
                                          _ptr(workspace), workspace.numel(), _stream_ptr(stream)))
    return dX, dA, dB


# ----------------------------------------------------------------------------------------------- latency model
EQ_I = 1
EQ_II = 2


def latency_features(model, segs, kv_size=0.0):
    """Feature vector of one step (Eq. I: {sum (n_i+B_d)^2, T_in+B_d, T_ft, K, 1}; Eq. II: {B_d, K, 1})."""
    s = segments(segs)
    p = library().lora_latency_terms(model)
    out = np.zeros(p, np.float64)
    _check(library().lora_latency_features(model, _ptr(s), s.shape[0], float(kv_size), _ptr(out)))
    return out


def latency_fit(model, feats, times):
    """Least-squares coefficients of the model over measured steps (feats [n, terms], times [n])."""
    f = np.ascontiguousarray(feats, dtype=np.float64)
    t = np.ascontiguousarray(times, dtype=np.float64)
    p = library().lora_latency_terms(model)
    coef = np.zeros(p, np.float64)
    _check(library().lora_latency_fit(model, _ptr(f), _ptr(t), t.shape[0], _ptr(coef)))
    return coef


def latency_predict(model, coef, feat):
    c = np.ascontiguousarray(coef, dtype=np.float64)
    f = np.ascontiguousarray(feat, dtype=np.float64)
    return float(library().lora_latency_predict(model, _ptr(c), _ptr(f)))
