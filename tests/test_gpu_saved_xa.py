"""The backward reads the captured xA it is handed (GPU).

DeltaServe section 3.2 ("Backward subprocess") computes the LoRA gradients from the activations captured during
the mixed forward and recomputes only what was not captured; MOLT section 4.3 reads a checkpointed activation
back when its slot is still backed and recomputes it otherwise.  A captured xA equal to the recompute cannot tell
reading from recomputing, so these tests hand the backward a captured activation that differs from the recompute
(an independent seeded draw of the same size and scale) and compare
  - dB, the one gradient that reads xA, with the oracle evaluated on that same captured activation,
  - dX and dA (which read dY B^T, never xA) with the plain oracle.
Each test first checks that the substituted-activation oracle's dB is far outside the tolerance of the
recompute's, so a kernel that ignored the captured activation (or the flag table choosing it) fails.
"""
import numpy as np
import pytest

import oracle
import workloads
from gpu_util import MAX_ERR, Dev, compare, random_table, to_dev, to_np, train_blocks

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    import lora_co_serving_gb300 as lm
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lm.build()


def _blocks(wl, width=1):
    """Element ranges of the fine-tuning segments' blocks in the saved-activation layout (increasing start)."""
    out, off = [], 0
    for st, ln, a, tr in sorted(wl.segs.tolist()):
        if tr and ln > 0:
            n = ln * width * int(wl.rank[a])
            out.append((off, off + n))
            off += n
    return out


def _substitute(wl, n, seed):
    """An independent captured activation: seeded N(0, 0.6^2) values (about the spread of x A here), exact in
    the workload's element type."""
    v = np.random.default_rng(seed).standard_normal(n).astype(np.float32) * np.float32(0.6)
    return workloads.bf16_round(v) if wl.dtype == "bf16" else v


def _far_apart(sub_dB, rec_dB, ib):
    """The two oracles' dB differ by far more than the tolerance: a kernel that recomputed would fail."""
    ref = sub_dB[ib]
    err = np.abs(rec_dB[ib] - ref).max() / np.abs(ref).max()
    assert err > 10 * MAX_ERR, "substitute too close to the recompute (%.3g)" % err


CASES = {
    "ftbwd_4adapters": lambda: workloads.config4(K=384, N=512, n_samples=4, sample_len=90, r=32, four_adapters=True),
    "mixed_fwd_save": lambda: workloads.config3(K=256, N=512, prefill_tokens=600, train_len=150, len_lo=64,
                                                len_hi=300),
    "cosrv": lambda: workloads.config5(K=384, N=640, n_adapters=30, n_decode=200, prefill_tokens=600, len_lo=40,
                                       len_hi=300, train_len=120),
    "f32": lambda: workloads.custom(3, 96, 64, 80, [(0, 30, 0, 1), (30, 20, 1, 0), (50, 46, 1, 1)], [8, 16],
                                    dtype="f32"),
}


@pytest.mark.parametrize("case", list(CASES))
def test_backward_reads_saved_xa(case):
    import torch
    wl = CASES[case]()
    d = Dev(wl)
    n = sum(hi - lo for lo, hi in _blocks(wl))
    sub = _substitute(wl, n, 31)
    rX, rA, rB = oracle.backward_wl(wl)
    _, _, sB = oracle.backward_wl(wl, want_dx=False, u_saved=sub)
    ia, ib = train_blocks(wl)
    _far_apart(sB, rB, ib)
    dX, dA, dB = d.backward(xa_saved=to_dev(sub, wl.dtype))
    torch.cuda.synchronize()
    compare(to_np(dB)[ib], sB[ib], "dB from the captured xA")
    compare(to_np(dA)[ia], rA[ia], "dA")
    compare(to_np(dX)[wl.train_rows()], rX, "dX")
    # LORA_RECOMPUTE_XA overrides a given captured activation
    _, _, dB2 = d.backward(xa_saved=to_dev(sub, wl.dtype), recompute=True)
    torch.cuda.synchronize()
    compare(to_np(dB2)[ib], rB[ib], "dB recomputed despite xa_saved")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_flag_table_reads_saved_where_flagged(dtype):
    """Flagged segments take the (substituted) captured xA, unflagged ones recompute it; their blocks of the
    captured buffer hold NaN, which must never be read."""
    import torch
    import lora_co_serving_gb300 as lm
    if dtype == "bf16":
        wl = workloads.config4(K=384, N=512, n_samples=4, sample_len=90, r=32, four_adapters=True)
    else:
        wl = workloads.custom(5, 120, 64, 80, [(0, 30, 0, 1), (30, 20, 1, 0), (50, 40, 1, 1), (90, 30, 0, 1)],
                              [8, 16], dtype="f32")
    d = Dev(wl)
    blocks = _blocks(wl)
    n = blocks[-1][1]
    sub = _substitute(wl, n, 47)
    _, u = oracle.forward_wl(wl, want_u=True)
    exact = oracle.saved_u(wl, u)
    rX, rA, rB = oracle.backward_wl(wl)
    ia, ib = train_blocks(wl)
    k = len(blocks)
    for pattern in ([1] * k, [i % 2 for i in range(k)], [1 - i % 2 for i in range(k)], [0] * k):
        ours = np.full(n, np.nan, np.float32)
        ref_u = exact.copy()
        for (lo, hi), f in zip(blocks, pattern):
            if f:
                ours[lo:hi] = sub[lo:hi]
                ref_u[lo:hi] = sub[lo:hi]
        _, _, sB = oracle.backward_wl(wl, want_dx=False, u_saved=ref_u)
        if any(pattern):
            _far_apart(sB, rB, ib)
        flags = torch.tensor(pattern, dtype=torch.int32, device="cuda")
        dX, dA, dB = lm.backward_flagged(d.x, d.Wt, d.pool, wl.segs, d.dY, to_dev(ours, wl.dtype), flags)
        torch.cuda.synchronize()
        compare(to_np(dB)[ib], sB[ib], "dB %s" % pattern)
        compare(to_np(dA)[ia], rA[ia], "dA %s" % pattern)
        compare(to_np(dX)[wl.train_rows()], rX, "dX %s" % pattern)


def test_sliced_backward_reads_saved_xa():
    import torch
    import lora_co_serving_gb300 as lm
    from oracle import sliced
    wl = workloads.sliced(12, 400, 256, [0, 512, 768, 1024], [(0, 150, 2, 0), (150, 130, 1, 1), (280, 120, 0, 1)],
                          [16, 8, 32])
    d = Dev(wl)
    S = wl.n_slices
    n = sum(hi - lo for lo, hi in _blocks(wl, S))
    sub = _substitute(wl, n, 53)
    rX, rA, rB = sliced.backward_wl(wl)
    _, _, sB = sliced.backward_wl(wl, u_saved=sub)
    ads = sorted(set(int(q[2]) for q in wl.segs.tolist() if q[3]))
    ia = np.concatenate([np.arange(wl.a_off[a], wl.a_off[a] + S * wl.rank[a] * wl.K) for a in ads])
    ib = np.concatenate([np.arange(wl.b_off[a], wl.b_off[a] + wl.rank[a] * wl.N) for a in ads])
    _far_apart(sB, rB, ib)
    dX, dA, dB = lm.sliced_backward(d.x, d.Wt, d.pool, wl.bounds, d.segs, d.dY, xa_saved=to_dev(sub, "bf16"))
    torch.cuda.synchronize()
    compare(to_np(dB)[ib], sB[ib], "sliced dB from the captured xA")
    compare(to_np(dA)[ia], rA[ia], "sliced dA")
    compare(to_np(dX)[wl.train_rows()], rX, "sliced dX")


@pytest.mark.parametrize("seed", [0, 1, 3, 4, 7, 11])
def test_flag_table_random_tables(seed):
    """The flag table on seeded random calls (ragged shapes, bf16 and f32, up to 12 fine-tuning segments on ranks
    1..128): a random subset of segments flagged saved, given a substituted captured xA; the others recompute and
    their captured blocks hold NaN.  dB against the oracle on the same mix of captured and exact activations."""
    import torch
    import lora_co_serving_gb300 as lm
    wl, n_train = random_table(seed)
    assert n_train > 0
    d = Dev(wl)
    blocks = _blocks(wl)
    n = blocks[-1][1]
    sub = _substitute(wl, n, 60 + seed)
    _, u = oracle.forward_wl(wl, want_u=True)
    exact = oracle.saved_u(wl, u)
    rX, rA, _ = oracle.backward_wl(wl)
    ia, ib = train_blocks(wl)
    pattern = [int(v) for v in np.random.default_rng(900 + seed).integers(0, 2, len(blocks))]
    ours = np.full(n, np.nan, np.float32)
    ref_u = exact.copy()
    for (lo, hi), f in zip(blocks, pattern):
        if f:
            ours[lo:hi] = sub[lo:hi]
            ref_u[lo:hi] = sub[lo:hi]
    _, _, sB = oracle.backward_wl(wl, want_dx=False, u_saved=ref_u)
    flags = torch.tensor(pattern, dtype=torch.int32, device="cuda")
    dX, dA, dB = lm.backward_flagged(d.x, d.Wt, d.pool, wl.segs, d.dY, to_dev(ours, wl.dtype), flags)
    torch.cuda.synchronize()
    compare(to_np(dB)[ib], sB[ib], "dB %s" % pattern)
    compare(to_np(dA)[ia], rA[ia], "dA %s" % pattern)
    compare(to_np(dX)[wl.train_rows()], rX, "dX %s" % pattern)
