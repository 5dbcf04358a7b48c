"""GPU parity: the CUDA library against the float64 oracle on the same seeded inputs.

Every comparison uses the layer's tolerance (max |err| <= 2e-2 * max |ref|, relative Frobenius
error <= 5e-3, per output tensor); routing and indexing checks are bit-exact (test_gpu_invariants.py).
"""
import numpy as np
import pytest

import oracle
import workloads
from gpu_util import RESPLIT_SMALL, Dev, compare, grad_split_table, random_table, to_np, train_blocks

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    import lora_co_serving_gb300 as lm
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lm.build()
    lm.library()


def check_forward(wl, save=False):
    import lora_co_serving_gb300 as lm
    d = Dev(wl)
    ref, u = oracle.forward_wl(wl, want_u=True)
    if save:
        y, xs = d.forward(save_xa=True)
    else:
        y = d.forward()
    import torch
    torch.cuda.synchronize()
    compare(to_np(y), ref, "y")
    if save:
        exp = []
        for st, ln, a, tr in sorted(wl.segs.tolist()):
            if tr and ln > 0:
                exp.append(u[st:st + ln, :wl.rank[a]].reshape(-1))
        exp = np.concatenate(exp)
        compare(to_np(xs)[:exp.shape[0]], exp, "xa_save")
    return d, y


def check_backward(wl, d=None, xa_saved=None, recompute=True):
    import torch
    d = d or Dev(wl)
    dX, dA, dB = d.backward(xa_saved=xa_saved, recompute=recompute)
    torch.cuda.synchronize()
    rX, rA, rB = oracle.backward_wl(wl)
    rows = wl.train_rows()
    compare(to_np(dX)[rows], rX, "dX")
    ia, ib = train_blocks(wl)
    compare(to_np(dA)[ia], rA[ia], "dA")
    compare(to_np(dB)[ib], rB[ib], "dB")
    # entries outside the fine-tuning adapters' blocks and dX rows outside fine-tuning segments stay zero
    mA = np.ones(dA.numel(), bool)
    mA[ia] = False
    mB = np.ones(dB.numel(), bool)
    mB[ib] = False
    assert np.all(to_np(dA)[mA] == 0) and np.all(to_np(dB)[mB] == 0)
    other = np.setdiff1d(np.arange(wl.T), rows)
    assert np.all(to_np(dX)[other] == 0)


def test_f32_config1():
    wl = workloads.config1()
    d, _ = check_forward(wl, save=True)
    check_backward(wl, d)


def test_bf16_base_only():
    wl = workloads.custom(7, 256, 256, 512, [(0, 256, -1, 0)], [16])
    check_forward(wl)


def test_bf16_single_adapter_ragged():
    # ragged T (3 tiles, last partial), ragged N (last 256-column tile half full), K not a multiple of 64
    wl = workloads.custom(8, 300, 328, 384, [(0, 300, 0, 0)], [16])
    check_forward(wl)


def test_bf16_adapters_and_base_mixed():
    segs = [(0, 100, 2, 0), (100, 60, -1, 0), (160, 90, 0, 0), (250, 50, 1, 0), (300, 33, 2, 0)]
    wl = workloads.custom(9, 333, 256, 512, segs, [8, 24, 128])
    check_forward(wl)


def test_bf16_decode_small():
    wl = workloads.config2(T=256, K=512, N=512, n_adapters=64)
    check_forward(wl)


def unsplit_with_decode_pairs(wl):
    """True when the forward main pass is not split along K (at least 96 output tiles) and has gathered decode
    pairs: every output tile is then one item that runs all its LoRA K-steps and writes y directly (no reduce)."""
    import lora_co_serving_gb300 as lm
    d = Dev(wl)
    _, info = lm.plan_describe(wl.T, wl.K, wl.N, d.pool, d.segs)
    return (info.shape[0] // 2) * -(-wl.N // 256) >= 96 and int(info[:, 0].sum()) > 0


@pytest.mark.parametrize("N", [8192, 7432])
def test_bf16_decode_pairs_unsplit_wide(N):
    # 32 or 30 (the last one 8 columns wide) output tiles per pair: the unsplit main pass of the large calls, with
    # gathered decode pairs (many adapters per pair, ranks up to 128) and prefill windows, at an oracle-sized K
    wl = workloads.config5(K=256, N=N, n_adapters=40, n_decode=300, prefill_tokens=500, len_lo=30, len_hi=250,
                           train_len=100, ranks=(8, 16, 24, 64, 128))
    assert unsplit_with_decode_pairs(wl)
    d, _ = check_forward(wl)
    check_backward(wl, d)


EDGE = {
    # one decode token; the smallest K and N the layer accepts (multiples of 8)
    "one_token": (1, 64, 64, [(0, 1, 0, 0)], [8]),
    "one_token_k8_n8": (1, 8, 8, [(0, 1, 1, 0)], [4, 16]),
    # a handful of tokens: decode, a 2-token prefill, a 1-token fine-tuning segment, a base-only token
    "few_mixed": (5, 136, 72, [(0, 1, 0, 0), (1, 2, 1, 0), (3, 1, 2, 1), (4, 1, -1, 0)], [8, 32, 16]),
    # one 129-token fine-tuning segment (a tile and one row), ranks at the ends of the range
    "train_129_rank128": (129, 200, 264, [(0, 129, 1, 1)], [1, 128]),
    # decode rows of 40 adapters of rank 1..128 around a 300-token prefill and a 20-token fine-tuning segment
    "decode_mixed_ranks": (360, 256, 256, [(t, 1, t % 40, 0) for t in range(40)] + [(40, 300, 7, 0), (340, 20, 3, 1)],
                           [1 + (a * 37) % 128 for a in range(40)]),
}


@pytest.mark.parametrize("case", sorted(EDGE))
def test_bf16_edge_shapes(case):
    T, K, N, segs, ranks = EDGE[case]
    wl = workloads.custom(31, T, K, N, segs, ranks)
    d, _ = check_forward(wl)
    if any(s[3] for s in segs):
        check_backward(wl, d)


def test_bf16_odd_ranks():
    segs = [(0, 40, 0, 0), (40, 1, 1, 0), (41, 1, 2, 0), (42, 86, 3, 0), (128, 3, 4, 0), (131, 61, 1, 0)]
    wl = workloads.custom(10, 192, 256, 256, segs, [1, 4, 13, 100, 127])
    check_forward(wl)


def test_bf16_mixed_small_forward_backward():
    wl = workloads.config5(K=512, N=768, n_adapters=24, n_decode=150, prefill_tokens=500, len_lo=30, len_hi=250,
                           train_len=100)
    d, _ = check_forward(wl)
    check_backward(wl, d)


def test_bf16_config3_small_save_then_backward_from_saved():
    wl = workloads.config3(K=512, N=1024, prefill_tokens=1000, train_len=200, len_lo=64, len_hi=400)
    d, _ = check_forward(wl, save=True)
    _, xs = d.forward(save_xa=True)
    check_backward(wl, d, xa_saved=xs, recompute=False)
    check_backward(wl, d, xa_saved=xs, recompute=True)


@pytest.mark.parametrize("r,four", [(16, False), (64, False), (16, True), (64, True)])
def test_bf16_config4_small(r, four):
    wl = workloads.config4(K=640, N=640, n_samples=4, sample_len=160, r=r, four_adapters=four)
    check_backward(wl)


def test_bf16_backward_accumulate():
    import torch
    wl = workloads.config4(K=256, N=384, n_samples=3, sample_len=70, r=32, four_adapters=True)
    d = Dev(wl)
    _, dA, dB = d.backward()
    dA0 = torch.randn_like(dA)
    dB0 = torch.randn_like(dB)
    _, aA, aB = d.backward(dA=dA0.clone(), dB=dB0.clone(), accumulate=True)
    torch.cuda.synchronize()
    ia, ib = train_blocks(wl)
    compare(to_np(aA)[ia], to_np(dA0)[ia] + to_np(dA)[ia], "dA accumulate", max_err=1e-5, fro_err=1e-6)
    compare(to_np(aB)[ib], to_np(dB0)[ib] + to_np(dB)[ib], "dB accumulate", max_err=1e-5, fro_err=1e-6)


def test_bf16_split_gradients():
    """Gradient items split three ways along the tokens (the table's planning is pinned on the CPU), with splits
    that cross segment boundaries: dX, dA, dB against the oracle, then accumulated onto random gradients."""
    import torch
    wl = grad_split_table()
    d = Dev(wl)
    check_backward(wl, d)
    _, dA, dB = d.backward()
    dA0 = torch.randn_like(dA)
    dB0 = torch.randn_like(dB)
    _, aA, aB = d.backward(dA=dA0.clone(), dB=dB0.clone(), accumulate=True)
    torch.cuda.synchronize()
    ia, ib = train_blocks(wl)
    compare(to_np(aA)[ia], to_np(dA0)[ia] + to_np(dA)[ia], "dA accumulate", max_err=1e-5, fro_err=1e-6)
    compare(to_np(aB)[ib], to_np(dB0)[ib] + to_np(dB)[ib], "dB accumulate", max_err=1e-5, fro_err=1e-6)
    mA = np.ones(dA.numel(), bool)
    mA[ia] = False
    assert np.array_equal(to_np(aA)[mA], to_np(dA0)[mA])


def test_bf16_backward_shrink_resplit():
    """A fine-tuning batch whose dY B^T shrink passes the planner cuts into 8 pieces instead of the default 4 (32
    tiles of 64 k-blocks: the default's 160 items leave a last wave of 8 on 152 CTAs; the count is pinned on the
    CPU): dX on sampled rows, dA and dB whole, against the oracle."""
    c = RESPLIT_SMALL
    wl = workloads.custom(77, c["T"], c["K"], c["N"], c["segs"], c["rank"])
    d = Dev(wl)
    dX, dA, dB = d.backward()
    import torch
    torch.cuda.synchronize()
    rows = wl.train_rows()[np.random.default_rng(5).choice(wl.T, 96, replace=False)]
    rows = np.unique(np.concatenate([rows, [0, wl.T - 1]]))
    rX, rA, rB = oracle.backward_wl(wl, dx_rows=rows)
    compare(to_np(dX)[rows], rX, "dX (sampled rows)")
    ia, ib = train_blocks(wl)
    compare(to_np(dA)[ia], rA[ia], "dA")
    compare(to_np(dB)[ib], rB[ib], "dB")


def test_bf16_backward_small_batch_split_k():
    # one 200-token fine-tuning segment on a 1024x1024 layer: 4 output tiles of dX, so the dX loop over N is
    # split four ways and the last split of each tile reduces the partials
    wl = workloads.config4(K=1024, N=1024, n_samples=1, sample_len=200, r=64)
    check_backward(wl)
    # and again with a second segment on another adapter, so two tile pairs share the launch
    wl2 = workloads.config4(K=1024, N=1024, n_samples=2, sample_len=150, r=32, four_adapters=True)
    check_backward(wl2)


def test_max_fine_tuning_segments():
    """The documented maximum of 48 fine-tuning segments in one call: ragged lengths down to one token on six
    adapters of ranks 1..128 (several segments per adapter, summed in start order), between decode tokens and
    prefill segments; forward with xA saved, backward from the saved xA and recomputed."""
    rng = np.random.default_rng(48)
    rank = [1, 7, 16, 33, 64, 128]
    segs, t, n_train = [], 0, 0
    while n_train < 48:
        kind = rng.integers(0, 4)
        if kind == 0:
            segs.append((t, 1, int(rng.integers(-1, 6)), 0))
            t += 1
        elif kind == 1:
            ln = int(rng.integers(20, 90))
            segs.append((t, ln, int(rng.integers(0, 6)), 0))
            t += ln
        else:
            ln = int(rng.choice([1, 2, 5, 17, 40, 64, 129]))
            segs.append((t, ln, int(rng.integers(0, 6)), 1))
            t += ln
            n_train += 1
    order = rng.permutation(len(segs))
    wl = workloads.custom(48, t, 200, 264, [segs[i] for i in order], rank)
    assert sum(1 for q in wl.segs.tolist() if q[3]) == 48
    d, _ = check_forward(wl, save=True)
    _, xs = d.forward(save_xa=True)
    check_backward(wl, d, xa_saved=xs, recompute=False)
    check_backward(wl, d)


@pytest.mark.parametrize("seed", range(16))
def test_random_tables(seed):
    wl, n_train = random_table(seed)
    d, _ = check_forward(wl, save=n_train > 0)
    if n_train:
        check_backward(wl, d)
