"""The step-latency model (Eq. I and II of "DeltaServe: Host-Agnostic Co-Serving of Inference and Fine-Tuning for
LLMs", section 3.3) on the CPU: features of a segment table, the least-squares fit against numpy's lstsq, exact
recovery of known coefficients, and the error paths."""
import numpy as np
import pytest

import lora_co_serving_gb300 as lm


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lm.build()
    lm.library()


def test_features_of_a_mixed_table():
    # prefill prompts of 100 and 300 tokens, five decode requests, two fine-tuning sequences of 64, one empty
    segs = [(0, 100, 3, 0), (100, 1, 0, 0), (101, 1, 1, 0), (102, 300, 2, 0), (402, 1, 0, 0), (403, 1, 5, 0),
            (404, 1, -1, 0), (405, 64, 7, 1), (469, 64, 7, 1), (533, 0, 2, 0)]
    f = lm.latency_features(lm.EQ_I, segs, kv_size=12345.0)
    assert f.tolist() == [(100 + 5) ** 2 + (300 + 5) ** 2, 400 + 5, 128, 12345.0, 1.0]
    g = lm.latency_features(lm.EQ_II, segs, kv_size=7.0)
    assert g.tolist() == [5.0, 7.0, 1.0]


def random_tables(rng, n):
    tabs = []
    for _ in range(n):
        segs, t = [], 0
        for _ in range(int(rng.integers(0, 300))):
            segs.append((t, 1, 0, 0))
            t += 1
        for _ in range(int(rng.integers(0, 6))):
            ln = int(rng.integers(16, 1024))
            segs.append((t, ln, 1, 0))
            t += ln
        for _ in range(int(rng.integers(0, 3))):
            ln = int(rng.integers(64, 1024))
            segs.append((t, ln, 2, 1))
            t += ln
        if not segs:
            segs.append((0, 1, 0, 0))
        tabs.append(segs)
    return tabs


def test_fit_recovers_known_coefficients_exactly():
    rng = np.random.default_rng(4)
    true = np.array([2.5e-9, 3.1e-4, 7.7e-4, 0.0, 0.12])     # alpha, beta, gamma, eps (no key-value cache), c
    F = np.array([lm.latency_features(lm.EQ_I, s) for s in random_tables(rng, 40)])
    t = F @ true
    c = lm.latency_fit(lm.EQ_I, F, t)
    assert c[3] == 0.0                                       # an all-zero feature is left out
    assert np.allclose(c, true, rtol=1e-9, atol=0.0)
    for f in F[:5]:
        assert abs(lm.latency_predict(lm.EQ_I, c, f) - float(f @ true)) <= 1e-9 * float(f @ true)


def test_fit_matches_numpy_lstsq_on_noisy_times():
    rng = np.random.default_rng(5)
    F = np.array([lm.latency_features(lm.EQ_I, s, kv_size=float(rng.integers(0, 10 ** 6))) for s in
                  random_tables(rng, 60)])
    t = F @ np.array([1e-9, 2e-4, 5e-4, 3e-7, 0.05]) * (1 + 0.05 * rng.standard_normal(60))
    c = lm.latency_fit(lm.EQ_I, F, t)
    ref = np.linalg.lstsq(F, t, rcond=None)[0]
    assert np.allclose(c, ref, rtol=1e-7, atol=1e-15)
    G = np.array([lm.latency_features(lm.EQ_II, s, kv_size=float(rng.integers(0, 10 ** 6))) for s in
                  random_tables(rng, 30)])
    u = G @ np.array([4e-4, 2e-7, 0.03]) + 0.001 * rng.standard_normal(30)
    assert np.allclose(lm.latency_fit(lm.EQ_II, G, u), np.linalg.lstsq(G, u, rcond=None)[0], rtol=1e-7, atol=1e-15)


def test_fit_errors():
    F = np.array([[1.0, 2.0, 2.0, 0.0, 1.0], [4.0, 3.0, 3.0, 0.0, 1.0], [9.0, 5.0, 5.0, 0.0, 1.0],
                  [2.0, 7.0, 7.0, 0.0, 1.0]])
    with pytest.raises(lm.LoraError) as e:                    # T_in + B_d and T_ft always equal: no unique fit
        lm.latency_fit(lm.EQ_I, F, np.ones(4))
    assert e.value.code == -10
    with pytest.raises(lm.LoraError) as e:                    # fewer steps than terms
        lm.latency_fit(lm.EQ_I, F[:2], np.ones(2))
    assert e.value.code == -1
    with pytest.raises(lm.LoraError):
        lm.latency_features(3, [(0, 1, 0, 0)])
