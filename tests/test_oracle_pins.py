"""The float64 oracle against its pins (CPU only)."""
import json
import os

import numpy as np
import pytest

import oracle_pins as P
import workloads

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin()


def test_golden_page_sizes():
    g = json.load(open(os.path.join(HERE, "golden", "page_sizes.json")))
    act = g["activation_bytes_per_token"]
    assert act["N_L"] * act["d"] * act["p"] == act["bytes"]
    assert abs(act["bytes"] / 2 ** 20 - act["approx_MB"]) < 1e-12
    # trainable parameters r(d+k): the pool laid out by the generator holds exactly that many entries per adapter
    for c in g["lora_trainable_params"]["cases"]:
        assert c["r"] * (c["d"] + c["k"]) == c["params"]
        wl = workloads.custom(1, 4, c["k"] // 64, c["d"] // 64, [(0, 4, 0, 1)], [c["r"]], dtype="f32")
        assert wl.A.size + wl.B.size == c["params"] // 64
    s = g["lora_alpha_scale"]
    assert s["alpha"] / s["r"] == s["scale"]
    assert workloads.config1().scale[0] == s["scale"]


def test_oracle_rejects_bad_table():
    import oracle
    wl = workloads.config1()
    segs = wl.segs.copy()
    segs[0, 2] = 99
    with pytest.raises(ValueError):
        oracle.forward(wl.x, wl.Wt, wl.A, wl.B, wl.a_off, wl.b_off, wl.rank, wl.scale, segs)
    segs = wl.segs.copy()
    segs[0, 1] = 5  # leaves tokens 5..15 uncovered
    with pytest.raises(ValueError):
        oracle.forward(wl.x, wl.Wt, wl.A, wl.B, wl.a_off, wl.b_off, wl.rank, wl.scale, segs)


def test_workload_structure():
    wl = workloads.config3(K=64, N=64)
    segs = wl.segs
    assert segs[:, 1].sum() == wl.T == 8192
    pre = segs[segs[:, 3] == 0]
    assert pre[:, 1].sum() == 6144 and pre[:-1, 1].min() >= 128 and pre[:, 1].max() <= 1024
    tr = segs[segs[:, 3] == 1]
    assert tr.shape[0] == 2 and np.all(tr[:, 1] == 1024) and np.all(tr[:, 2] == 16)
    wl5 = workloads.config5(K=64, N=64)
    s5 = wl5.segs
    assert s5[:, 1].sum() == 8192
    assert (s5[:, 1] == 1).sum() >= 2048
    assert sorted(set(wl5.rank.tolist())) <= [8, 16, 32, 64, 128]
    # bf16 exactness of every drawn value
    for a in (wl5.x, wl5.Wt, wl5.A, wl5.B, wl5.dY):
        assert np.array_equal(workloads.bf16_round(a), a)
