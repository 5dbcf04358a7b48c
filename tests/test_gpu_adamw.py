"""GPU parity of lora_adamw_step against the float64 AdamW oracle."""
import numpy as np
import pytest

import oracle
import workloads
from gpu_util import Dev, compare, to_dev, to_np, train_blocks
from oracle import adamw as oadamw

pytestmark = pytest.mark.gpu
HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
# the ABI takes the hyperparameters as float32: the oracle gets exactly those values
HP32 = {k: float(np.float32(v)) for k, v in HP.items()}


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    import lora_co_serving_gb300 as lm
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lm.build()


def _states(n, seed):
    rng = np.random.default_rng(seed)
    g = rng.standard_normal(n).astype(np.float32)
    m = (0.1 * rng.standard_normal(n)).astype(np.float32)
    v = (0.01 * rng.random(n)).astype(np.float32)
    return g, m, v


def _dev32(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


@pytest.mark.parametrize("with_master", [True, False])
def test_adamw_bf16_pool(with_master):
    import torch
    import lora_co_serving_gb300 as lm
    wl = workloads.config4(K=264, N=392, n_samples=3, sample_len=40, r=24, four_adapters=True)
    d = Dev(wl)
    ads = [0, 2]
    gA, mA, vA = _states(wl.A.size, 1)
    gB, mB, vB = _states(wl.B.size, 2)
    masterA = wl.A.copy()
    masterB = wl.B.copy()
    tgA, tmA, tvA, tgB, tmB, tvB = (_dev32(a) for a in (gA, mA, vA, gB, mB, vB))
    A0, B0 = d.A.clone(), d.B.clone()
    tMA, tMB = (_dev32(masterA), _dev32(masterB)) if with_master else (None, None)
    lm.adamw_step(d.pool, wl.K, wl.N, tgA, tgB, tmA, tvA, tmB, tvB, ads, step=3, A_master=tMA, B_master=tMB, **HP)
    torch.cuda.synchronize()
    eA, emA, evA = oadamw.adamw_pool(masterA, gA, mA, vA, wl.a_off, wl.rank, wl.K, ads, step=3, **HP32)
    eB, emB, evB = oadamw.adamw_pool(masterB, gB, mB, vB, wl.b_off, wl.rank, wl.N, ads, step=3, **HP32)
    compare(to_np(tmA), emA, "mA", 1e-5, 1e-6)
    compare(to_np(tvA), evA, "vA", 1e-5, 1e-6)
    compare(to_np(tmB), emB, "mB", 1e-5, 1e-6)
    compare(to_np(tvB), evB, "vB", 1e-5, 1e-6)
    sel_a = np.zeros(wl.A.size, bool)
    sel_b = np.zeros(wl.B.size, bool)
    for a in ads:
        sel_a[wl.a_off[a]:wl.a_off[a] + wl.rank[a] * wl.K] = True
        sel_b[wl.b_off[a]:wl.b_off[a] + wl.rank[a] * wl.N] = True
    if with_master:
        compare(to_np(tMA), eA, "A master", 1e-5, 1e-6)
        compare(to_np(tMB), eB, "B master", 1e-5, 1e-6)
        # the bf16 pool holds the updated masters rounded to bf16, bit for bit
        assert torch.equal(d.A, tMA.to(torch.bfloat16)) or np.array_equal(
            to_np(d.A)[sel_a], workloads.bf16_round(to_np(tMA).astype(np.float32))[sel_a])
    # bf16 pool within one bf16 rounding of the float64 result
    got = to_np(d.A)[sel_a]
    assert np.all(np.abs(got - eA[sel_a]) <= 2 ** -8 * np.abs(eA[sel_a]) + 1e-12)
    # untouched entries are unchanged, bit for bit
    assert torch.equal(d.A[torch.from_numpy(~sel_a).cuda()], A0[torch.from_numpy(~sel_a).cuda()])
    assert torch.equal(d.B[torch.from_numpy(~sel_b).cuda()], B0[torch.from_numpy(~sel_b).cuda()])
    assert np.array_equal(to_np(tmA)[~sel_a], mA[~sel_a].astype(np.float64))


def test_adamw_f32_pool_after_backward():
    """A whole fine-tuning step of the tiny fp32 layer: backward, then AdamW on the trained adapter."""
    import torch
    import lora_co_serving_gb300 as lm
    wl = workloads.config1()
    d = Dev(wl)
    _, dA, dB = d.backward()
    ads = sorted(set(int(s[3] and s[2]) for s in wl.segs.tolist() if s[3]))
    zA, zB = torch.zeros_like(dA), torch.zeros_like(dB)
    mA, vA, mB, vB = zA.clone(), zA.clone(), zB.clone(), zB.clone()
    lm.adamw_step(d.pool, wl.K, wl.N, dA, dB, mA, vA, mB, vB, ads, step=1, **HP)
    torch.cuda.synchronize()
    _, rA, rB = oracle.backward_wl(wl)
    eA, _, _ = oadamw.adamw_pool(wl.A, rA, np.zeros(wl.A.size), np.zeros(wl.A.size), wl.a_off, wl.rank, wl.K, ads,
                                 step=1, **HP32)
    eB, _, _ = oadamw.adamw_pool(wl.B, rB, np.zeros(wl.B.size), np.zeros(wl.B.size), wl.b_off, wl.rank, wl.N, ads,
                                 step=1, **HP32)
    ia, ib = train_blocks(wl)
    # first step: the update is lr * g/(|g|+eps) ~ lr * sign(g); compare the update itself
    compare(to_np(d.A)[ia] - wl.A[ia], eA[ia] - wl.A[ia], "A update", 2e-2, 5e-3)
    compare(to_np(d.B)[ib] - wl.B[ib], eB[ib] - wl.B[ib], "B update", 2e-2, 5e-3)
