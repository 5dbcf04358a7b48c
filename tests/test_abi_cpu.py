"""The C-ABI library on the CPU: it loads, exports what include/ declares, and validates on the host.

No GPU is touched: every call here fails validation (or the workspace check)
before anything is launched.
"""
import ctypes
import os
import re

import numpy as np
import pytest

import lora_co_serving_gb300 as lm
import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    lm.build()
    return lm.library()


def declared_functions():
    names = []
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            text = open(os.path.join(ROOT, "include", f)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^[A-Za-z_][\w \*]*?\b(lora_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert "lora_mixed_forward" in names and "lora_mixed_backward" in names
    for n in names:
        assert hasattr(lib, n), "missing export " + n
    assert sorted(lm.EXPORTED) == names


class FakePool:
    """Host arrays plus fake (never dereferenced) device addresses."""

    def __init__(self, rank, K, N, A=0x10000000, B=0x20000000):
        self.rank = np.asarray(rank, np.int32)
        self.a_off = np.concatenate([[0], np.cumsum(self.rank[:-1].astype(np.int64) * K)]).astype(np.int64)
        self.b_off = np.concatenate([[0], np.cumsum(self.rank[:-1].astype(np.int64) * N)]).astype(np.int64)
        self.scale = np.full(len(rank), 2.0, np.float32)
        self._c = lm._Pool(A, B, self.a_off.ctypes.data, self.b_off.ctypes.data, self.rank.ctypes.data,
                           self.scale.ctypes.data, len(rank))

    def cptr(self):
        return ctypes.addressof(self._c)


def call_fwd(lib, T, K, N, pool, segs, dt=0, x=0x30000000, W=0x40000000, y=0x50000000, ws=None, wsb=0, flags=0,
             xa=None):
    s = lm.segments(segs)
    return lib.lora_mixed_forward(T, K, N, dt, x, W, pool.cptr(), s.ctypes.data, s.shape[0], y, xa, flags, ws, wsb,
                                  None)


def call_bwd(lib, T, K, N, pool, segs, ws=None, wsb=0, dX=0x60000000, dA=0x70000000, dB=0x80000000, dY=0x90000000):
    s = lm.segments(segs)
    return lib.lora_mixed_backward(T, K, N, 0, 0x30000000, 0x40000000, pool.cptr(), s.ctypes.data, s.shape[0], dY,
                                   None, dX, dA, dB, 0, ws, wsb, None)


def test_validation_codes(lib):
    K, N = 64, 64
    pool = FakePool([8, 16], K, N)
    ok = [(0, 10, 0, 0), (10, 6, 1, 1)]
    # a valid table gets as far as the workspace check
    assert call_fwd(lib, 16, K, N, pool, ok) == -6
    assert call_bwd(lib, 16, K, N, pool, ok) == -6
    assert call_fwd(lib, 16, K, N, pool, [(0, 10, 0, 0), (9, 7, 1, 0)]) == -2        # overlap
    assert call_fwd(lib, 16, K, N, pool, [(0, 9, 0, 0), (10, 6, 1, 0)]) == -2        # gap
    assert call_fwd(lib, 17, K, N, pool, ok) == -2                                   # does not cover T
    assert call_fwd(lib, 16, K, N, pool, [(0, 10, 2, 0), (10, 6, 1, 0)]) == -3       # id out of range
    assert call_fwd(lib, 16, K, N, pool, [(0, 10, -2, 0), (10, 6, 1, 0)]) == -3
    assert call_fwd(lib, 16, K, N, pool, [(0, 10, -1, 1), (10, 6, 1, 0)]) == -4      # training on base
    assert call_fwd(lib, 16, 60, N, FakePool([8, 16], 60, N), ok) == -5              # K not multiple of 8
    assert call_fwd(lib, 16, K, N, pool, ok, x=0x30000002) == -5                     # misaligned x
    assert call_fwd(lib, 16, K, N, pool, ok, dt=7) == -7
    assert call_fwd(lib, 16, K, N, FakePool([8, 129], K, N), ok) == -9               # rank > 128
    assert call_fwd(lib, 16, K, N, FakePool([8, 0], K, N), ok) == -9
    assert call_fwd(lib, 16, K, N, pool, ok, flags=1 << 10) == -1                    # unknown flag
    assert call_fwd(lib, 16, K, N, pool, ok, flags=1) == -1                          # save without buffer
    assert call_fwd(lib, -1, K, N, pool, ok) == -1
    msg = lib.lora_last_error().decode()
    assert "T must be" in msg
    # workspace: misaligned and too small
    assert call_fwd(lib, 16, K, N, pool, ok, ws=0xA0000010, wsb=1 << 30) == -6
    assert "256-byte" in lib.lora_last_error().decode()
    assert call_fwd(lib, 16, K, N, pool, ok, ws=0xA0000000, wsb=16) == -6
    assert "too small" in lib.lora_last_error().decode()
    # more than 48 training segments
    many = [(i, 1, 0, 1) for i in range(49)]
    assert call_bwd(lib, 49, K, N, pool, many) == -10
    # pool offsets must be row aligned
    bad = FakePool([8, 16], K, N)
    bad.a_off[1] = 5
    assert call_fwd(lib, 16, K, N, bad, ok) == -3


def test_sizes(lib):
    K, N = 64, 96
    pool = FakePool([8, 16, 32], K, N)
    segs = [(0, 5, 0, 1), (5, 3, 2, 0), (8, 7, 1, 1), (15, 0, 2, 1)]
    s = lm.segments(segs)
    assert lib.lora_xa_size(0, pool.cptr(), s.ctypes.data, 4) == 2 * (5 * 8 + 7 * 16)
    assert lib.lora_xa_size(1, pool.cptr(), s.ctypes.data, 4) == 4 * (5 * 8 + 7 * 16)
    ws = lib.lora_workspace_size(15, K, N, 0, pool.cptr(), s.ctypes.data, 4)
    assert ws > 0 and ws % 256 == 0
    assert lib.lora_workspace_size(16, K, N, 0, pool.cptr(), s.ctypes.data, 4) == 0   # invalid: gap at the end
    # the saved-activation size is the page's activation-capture cost per token at rank r, bf16 (r*2 bytes per token
    # and layer; the DeltaServe example N_L*d*p is the same product for the residual stream)
    one = lm.segments([(0, 1, 1, 1)])
    assert lib.lora_xa_size(0, pool.cptr(), one.ctypes.data, 1) == 16 * 2


def _plan(wl):
    pool = FakePool(wl.rank, wl.K, wl.N)
    rows, info = lm.plan_describe(wl.T, wl.K, wl.N, pool, wl.segs)
    return rows, info


@pytest.mark.parametrize("cfg", [2, 3, 5])
def test_plan_covers_every_token_once(lib, cfg):
    wl = workloads.config(cfg, K=64, N=64) if cfg != 2 else workloads.config2(K=64, N=64)
    rows, info = _plan(wl)
    got = rows[rows >= 0]
    assert np.array_equal(np.sort(got), np.arange(wl.T)), "every token exactly once"
    seg_of = np.empty(wl.T, np.int64)
    for i, (st, ln, a, tr) in enumerate(wl.segs.tolist()):
        seg_of[st:st + ln] = i
    assert rows.shape[0] % 2 == 0, "tiles come in pairs"
    for ti in range(rows.shape[0]):
        r = rows[ti]
        v = r[r >= 0]
        pr = rows[ti - ti % 2: ti - ti % 2 + 2]      # the tile pair shares one adapter list
        pv = pr[pr >= 0]
        ads = sorted(set(int(wl.segs[seg_of[t], 2]) for t in pv) - {-1})
        assert info[ti, 1] == len(ads)
        assert info[ti, 2] == sum((int(wl.rank[a]) + 15) // 16 * 16 for a in ads)
        if info[ti, 0] == 0:   # window tile: rows are x rows [row0, row0+128) or -1
            base = info[ti, 3]
            for i, t in enumerate(r):
                assert t == -1 or t == base + i
        else:                  # gathered: decode rows sorted by adapter
            keys = [(int(wl.segs[seg_of[t], 2]), int(t)) for t in v]
            assert keys == sorted(keys)
            assert all(wl.segs[seg_of[t], 1] < 16 and not wl.segs[seg_of[t], 3] for t in v)


def test_plan_segment_order_does_not_matter(lib):
    wl = workloads.config5(K=64, N=64, n_adapters=40, n_decode=300, prefill_tokens=700, len_lo=20, len_hi=300,
                           train_len=100)
    r0, i0 = _plan(wl)
    rng = np.random.default_rng(0)
    wl.segs = wl.segs[rng.permutation(wl.segs.shape[0])]
    r1, i1 = _plan(wl)
    assert np.array_equal(r0, r1) and np.array_equal(i0, i1)


def call_sliced_fwd(lib, T, K, N, pool, bounds, segs, dt=0, ws=None, wsb=0):
    s = lm.segments(segs)
    sl = lm.Slices(bounds)
    return lib.lora_sliced_forward(T, K, N, dt, 0x30000000, 0x40000000, pool.cptr(), sl.cptr(), s.ctypes.data,
                                   s.shape[0], 0x50000000, None, 0, ws, wsb, None)


def test_sliced_validation(lib):
    K, N = 256, 1024
    pool = FakePool([8, 16], K, N)
    segs = [(0, 10, 0, 0), (10, 6, 1, 1)]
    # bounds must start at 0, end at N, increase, and have interior bounds on 256-column tiles
    assert call_sliced_fwd(lib, 16, K, N, pool, [0, 512, 1000], segs) == -1
    assert call_sliced_fwd(lib, 16, K, N, pool, [8, 512, 1024], segs) == -1
    assert call_sliced_fwd(lib, 16, K, N, pool, [0, 520, 1024], segs) == -1
    assert call_sliced_fwd(lib, 16, K, N, pool, [0, 512, 512, 1024], segs) == -1
    assert call_sliced_fwd(lib, 16, K, N, pool, [0, 256, 512, 768, 896, 1024], segs) == -1   # 5 slices
    # float32 layers take one slice only
    assert call_sliced_fwd(lib, 16, K, N, pool, [0, 512, 1024], segs, dt=1) == -7
    # a NULL slices argument is rejected by the sliced entry point
    s = lm.segments(segs)
    assert lib.lora_sliced_forward(16, K, N, 0, 0x30000000, 0x40000000, pool.cptr(), None, s.ctypes.data, 2,
                                   0x50000000, None, 0, None, 0, None) == -1
    # valid slices, missing workspace: the workspace check is the first failure
    assert call_sliced_fwd(lib, 16, K, N, pool, [0, 512, 768, 1024], segs) == -6


def test_sliced_sizes(lib):
    K, N = 256, 1024
    pool = FakePool([8, 16], K, N)
    segs = lm.segments([(0, 10, 0, 0), (10, 6, 1, 1), (16, 20, 0, 1)])
    for S, b in ((1, [0, 1024]), (3, [0, 512, 768, 1024]), (4, [0, 256, 512, 768, 1024])):
        sl = lm.Slices(b)
        xa = lib.lora_sliced_xa_size(0, pool.cptr(), sl.cptr(), segs.ctypes.data, segs.shape[0])
        assert xa == 2 * S * (6 * 16 + 20 * 8)
        ws = lib.lora_sliced_workspace_size(36, K, N, 0, pool.cptr(), sl.cptr(), segs.ctypes.data, segs.shape[0])
        assert ws > 0
    sl1 = lm.Slices([0, 1024])
    one = lib.lora_sliced_workspace_size(36, K, N, 0, pool.cptr(), sl1.cptr(), segs.ctypes.data, 3)
    assert one == lib.lora_workspace_size(36, K, N, 0, pool.cptr(), segs.ctypes.data, 3)


def test_wait_limit_range(lib):
    """lora_set_wait_limit refuses limits outside 1 ms .. 60 s on the host, before any CUDA call."""
    for ns in (0, 999_999, 60_000_000_001, 2**63):
        assert lib.lora_set_wait_limit(ns) == -1, ns
        assert "between 1 ms and 60 s" in lib.lora_last_error().decode()
