"""Bit-exact routing and invariance properties of the CUDA path (GPU).

  - zero-B adapters give y bitwise equal to the base projection (adapter -1) for the same rows, and dA == 0;
  - the order of the segment table does not change a single bit of y, dX, dA, dB;
  - permuting the adapter pool (ids remapped) does not change a bit of y or dX, and permutes dA/dB blocks;
  - an integer routing pattern (W = 0, A = e_0, integer B, s = 1) reproduces the adapter of every token exactly;
  - all of the above also on the full co-serving segment table (2048 decode rows: the tensor-core gathered shrink);
  - repeated calls are bitwise identical (no atomics in any reduction);
  - a single base-only segment matches torch.matmul as a second witness.
"""
import numpy as np
import pytest

import oracle_pins as P
import workloads
from gpu_util import Dev, compare, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    import lora_co_serving_gb300 as lm
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lm.build()


def mixed_small(seed=1005, N=640):
    return workloads.config5(seed=seed, K=384, N=N, n_adapters=30, n_decode=200, prefill_tokens=600, len_lo=40,
                             len_hi=300, train_len=120)


def cosrv_full_table(N):
    """The full co-serving segment table (2048 Zipf(1.1) decode tokens over 320 adapters of ranks 8..128, 4096
    prefill tokens, 2 x 1024 fine-tuning tokens) at a reduced layer width: its 2048 gathered decode rows exceed the
    CUDA-core decode-shrink limit (1024 rows), so they take the tensor-core shrink of gathered tiles."""
    return workloads.config5(K=256, N=N)


# N = 640: the forward main pass is split along K (few output tiles, chunk-aligned LoRA splits, a reduce launch);
# N = 7680: unsplit (every output tile one item that writes y).  "full_*": the full co-serving table, split (512)
# and unsplit (1024) main pass.
WIDTHS = [640, 7680, "full_512", "full_1024"]


def table(N):
    if isinstance(N, str):
        return cosrv_full_table(int(N.split("_")[1]))
    return mixed_small(N=N)


def bits(t):
    import torch
    return t.detach().contiguous().view(torch.int16 if t.dtype == torch.bfloat16 else torch.int32).cpu().numpy()


@pytest.mark.parametrize("N", WIDTHS)
def test_zero_B_is_base_bitwise(N):
    wl = table(N)
    zero = [a for a in range(wl.n_adapters) if a % 3 == 0]
    for a in zero:
        wl.B[wl.b_off[a]:wl.b_off[a] + wl.rank[a] * wl.N] = 0.0
    y1 = Dev(wl).forward()
    base = wl.segs.copy()
    for i in range(base.shape[0]):
        if base[i, 2] in zero and not base[i, 3]:
            base[i, 2] = -1
    wl2 = workloads.Workload(**{**wl.__dict__, "segs": base})
    y2 = Dev(wl2).forward()
    rows = np.concatenate([np.arange(s, s + l) for s, l, a, t in wl.segs.tolist() if a in zero and not t])
    assert rows.size > 0
    assert np.array_equal(bits(y1)[rows], bits(y2)[rows])
    # dA = s x^T (dY B^T) vanishes exactly when the training adapter's B is zero
    a = int(wl.meta["train_adapter"])
    wl.B[wl.b_off[a]:wl.b_off[a] + wl.rank[a] * wl.N] = 0.0
    _, dA, _ = Dev(wl).backward()
    assert np.all(to_np(dA) == 0.0)


@pytest.mark.parametrize("N", WIDTHS)
def test_segment_order_bitwise(N):
    wl = table(N)
    d = Dev(wl)
    y0 = bits(d.forward())
    g0 = [bits(t) for t in d.backward()]
    perm = np.random.default_rng(4).permutation(wl.segs.shape[0])
    d.segs = wl.segs[perm]
    y1 = bits(d.forward())
    g1 = [bits(t) for t in d.backward()]
    assert np.array_equal(y0, y1)
    for a, b in zip(g0, g1):
        assert np.array_equal(a, b)


@pytest.mark.parametrize("N", WIDTHS)
def test_pool_order_bitwise(N):
    wl = table(N)
    d = Dev(wl)
    y0 = bits(d.forward())
    dX0, dA0, dB0 = [bits(t) for t in d.backward()]
    perm = np.random.default_rng(8).permutation(wl.n_adapters)
    rank, scale, A, B, a_off, b_off, segs = P.permute_pool(wl, perm)
    wl2 = workloads.Workload(**{**wl.__dict__, "rank": rank, "scale": scale, "A": A, "B": B, "a_off": a_off,
                                "b_off": b_off, "segs": segs})
    d2 = Dev(wl2)
    y1 = bits(d2.forward())
    dX1, dA1, dB1 = [bits(t) for t in d2.backward()]
    assert np.array_equal(y0, y1)
    assert np.array_equal(dX0, dX1)
    for i, p in enumerate(perm):
        r = wl.rank[p]
        assert np.array_equal(dA1[a_off[i]:a_off[i] + r * wl.K], dA0[wl.a_off[p]:wl.a_off[p] + r * wl.K])
        assert np.array_equal(dB1[b_off[i]:b_off[i] + r * wl.N], dB0[wl.b_off[p]:wl.b_off[p] + r * wl.N])


@pytest.mark.parametrize("which", ["decode", "cosrv", "cosrv_wide", "cosrv_full_512", "cosrv_full_1024"])
def test_routing_integer_pattern_exact(which):
    if which == "decode":
        wl = workloads.config2(T=256, K=256, N=512, n_adapters=64)
    elif which.startswith("cosrv_full"):
        wl = cosrv_full_table(int(which.split("_")[-1]))
    else:
        wl = workloads.config5(K=256, N=512 if which == "cosrv" else 6144, n_adapters=64, n_decode=512,
                               prefill_tokens=700, len_lo=20, len_hi=200, train_len=150)
    wl = P.routing_pattern(wl)
    y = to_np(Dev(wl).forward())
    assert np.array_equal(y, P.routing_expected(wl))


@pytest.mark.parametrize("N", [512, 1024])
def test_full_table_matches_oracle(N):
    """Every row and every fine-tuning gradient of the full co-serving table against the oracle (the tensor-core
    shrink of the 2048 gathered decode rows included), at a reduced layer width."""
    import torch
    import oracle
    from gpu_util import train_blocks
    wl = cosrv_full_table(N)
    d = Dev(wl)
    y = d.forward()
    dX, dA, dB = d.backward()
    torch.cuda.synchronize()
    compare(to_np(y), oracle.forward_wl(wl), "y")
    rX, rA, rB = oracle.backward_wl(wl)
    ia, ib = train_blocks(wl)
    compare(to_np(dX)[wl.train_rows()], rX, "dX")
    compare(to_np(dA)[ia], rA[ia], "dA")
    compare(to_np(dB)[ib], rB[ib], "dB")


def test_repeatable_bitwise():
    wl = mixed_small(seed=77)
    d = Dev(wl)
    a = [bits(d.forward())] + [bits(t) for t in d.backward()]
    b = [bits(d.forward())] + [bits(t) for t in d.backward()]
    for u, v in zip(a, b):
        assert np.array_equal(u, v)


def test_base_only_matches_torch_matmul():
    import torch
    wl = workloads.custom(3, 640, 512, 768, [(0, 640, -1, 0)], [16])
    d = Dev(wl)
    y = d.forward()
    ref = d.x.float() @ d.Wt.float().t()
    torch.cuda.synchronize()
    compare(to_np(y), to_np(ref), "y vs torch.matmul")


def test_status_word_clear():
    import torch
    import lora_co_serving_gb300 as lm
    wl = mixed_small(seed=5)
    d = Dev(wl)
    ws = torch.empty(lm.workspace_size(wl.T, wl.K, wl.N, 0, d.pool, wl.segs), dtype=torch.uint8, device="cuda")
    d.forward(workspace=ws)
    lm.workspace_status(ws)
    d.backward(workspace=ws)
    lm.workspace_status(ws)


def test_empty_batch_is_a_no_op():
    import torch
    import lora_co_serving_gb300 as lm
    wl = workloads.custom(1, 0, 64, 64, [], [8])
    d = Dev(wl)
    y = d.forward()
    assert y.shape == (0, 64)
    dX, dA, dB = d.backward()
    torch.cuda.synchronize()
    assert np.all(to_np(dA) == 0)


def test_launch_parameters_follow_each_call():
    """Launch parameters kept from a call are reused only when a call repeats its pointers: alternating outputs and
    inputs on one workspace and plan give each call its own result, and a call with the same pointers sees new
    contents.  Scaling x by a power of two scales y exactly (every rounding step scales with it)."""
    import torch
    import lora_co_serving_gb300 as lm
    wl = mixed_small(seed=91)
    d = Dev(wl)
    ws = torch.empty(lm.workspace_size(wl.T, wl.K, wl.N, 0, d.pool, wl.segs), dtype=torch.uint8, device="cuda")
    yA = torch.empty((wl.T, wl.N), dtype=torch.bfloat16, device="cuda")
    yB = torch.empty_like(yA)
    x2 = d.x * 0.5
    lm.forward(d.x, d.Wt, d.pool, wl.segs, y=yA, workspace=ws)
    ref = yA.clone()
    lm.forward(x2, d.Wt, d.pool, wl.segs, y=yB, workspace=ws)
    assert torch.equal(yB, ref * 0.5)
    lm.forward(d.x, d.Wt, d.pool, wl.segs, y=yA, workspace=ws)
    assert torch.equal(yA, ref)
    d.x.mul_(2.0)                                # same pointers, new contents
    lm.forward(d.x, d.Wt, d.pool, wl.segs, y=yA, workspace=ws)
    assert torch.equal(yA, ref * 2.0)
    # the backward likewise: dX and dA scale with dY, dB with x
    gA = [t.clone() for t in lm.backward(d.x, d.Wt, d.pool, wl.segs, d.dY, workspace=ws)]
    gB = lm.backward(d.x, d.Wt, d.pool, wl.segs, d.dY * 0.25, workspace=ws)
    for a, b in zip(gA, gB):
        assert torch.equal(b, a * 0.25)
