"""Per-segment save/recompute chosen on the device (lora_mixed_backward_flagged).

The flag table plays the role of an activation-slot state table whose entries the host flips between calls: a
segment flagged "saved" must be read from xa_saved, a segment flagged zero must be recomputed even if xa_saved
holds garbage for it.
"""
import numpy as np
import pytest

import oracle
import workloads
from gpu_util import Dev, compare, to_np, train_blocks

pytestmark = pytest.mark.gpu


def _segments_xa_ranges(wl):
    """Element ranges of each fine-tuning segment's block in xa_save (increasing start order)."""
    out, off = [], 0
    for st, ln, a, tr in sorted(wl.segs.tolist()):
        if tr and ln > 0:
            out.append((off, off + ln * int(wl.rank[a])))
            off += ln * int(wl.rank[a])
    return out


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_flag_table_picks_saved_or_recomputed_per_segment(dtype):
    import torch
    import lora_co_serving_gb300 as lm
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lm.build()
    if dtype == "bf16":
        wl = workloads.config4(K=384, N=512, n_samples=4, sample_len=90, r=32, four_adapters=True)
    else:
        wl = workloads.custom(3, 96, 64, 80, [(0, 30, 0, 1), (30, 20, 1, 0), (50, 46, 1, 1)], [8, 16], dtype="f32")
    d = Dev(wl)
    _, xs = d.forward(save_xa=True)
    ranges = _segments_xa_ranges(wl)
    n = len(ranges)
    rX, rA, rB = oracle.backward_wl(wl)
    ia, ib = train_blocks(wl)
    for pattern in ([1] * n, [0] * n, [i % 2 for i in range(n)], [1 - i % 2 for i in range(n)]):
        flags = torch.tensor(pattern, dtype=torch.int32, device="cuda")
        bad = xs.clone()
        for (lo, hi), f in zip(ranges, pattern):
            if not f:
                bad[lo:hi] = float("nan")           # must not be read: the segment is recomputed
        dX, dA, dB = lm.backward_flagged(d.x, d.Wt, d.pool, wl.segs, d.dY, bad, flags)
        torch.cuda.synchronize()
        rows = wl.train_rows()
        compare(to_np(dX)[rows], rX, "dX %s" % pattern)
        compare(to_np(dA)[ia], rA[ia], "dA %s" % pattern)
        compare(to_np(dB)[ib], rB[ib], "dB %s" % pattern)


def test_flagged_all_saved_equals_plain_saved_bitwise():
    import torch
    import lora_co_serving_gb300 as lm
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    wl = workloads.config3(K=256, N=512, prefill_tokens=600, train_len=150, len_lo=64, len_hi=300)
    d = Dev(wl)
    _, xs = d.forward(save_xa=True)
    n = sum(1 for s in wl.segs.tolist() if s[3])
    g_saved = d.backward(xa_saved=xs)
    g_flag = lm.backward_flagged(d.x, d.Wt, d.pool, wl.segs, d.dY, xs, torch.ones(n, dtype=torch.int32, device="cuda"))
    g_rec = d.backward(recompute=True)
    g_flag0 = lm.backward_flagged(d.x, d.Wt, d.pool, wl.segs, d.dY, xs, torch.zeros(n, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    for a, b in zip(g_saved, g_flag):
        assert torch.equal(a, b)
    for a, b in zip(g_rec, g_flag0):
        assert torch.equal(a, b)
