"""Pins of the float64 AdamW oracle (CPU only)."""
import math

import numpy as np
import pytest

from oracle import adamw

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)


def test_matches_torch_adamw_float64():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(0)
    theta0 = rng.standard_normal(257)
    p = torch.nn.Parameter(torch.tensor(theta0, dtype=torch.float64))
    opt = torch.optim.AdamW([p], lr=HP["lr"], betas=(HP["beta1"], HP["beta2"]), eps=HP["eps"],
                            weight_decay=HP["weight_decay"])
    theta, m, v = theta0.copy(), np.zeros(257), np.zeros(257)
    for step in range(1, 6):
        g = rng.standard_normal(257) * (step + 0.5)
        p.grad = torch.tensor(g, dtype=torch.float64)
        opt.step()
        theta, m, v = adamw.adamw_step(theta, g, m, v, step=step, **HP)
        assert np.allclose(theta, p.detach().numpy(), rtol=1e-13, atol=1e-15)


def test_first_step_closed_form():
    # from zero moments, step 1: m_hat = g, v_hat = g^2, so the update is lr * g / (|g| + eps) after decay
    g = np.array([3.0, -0.5, 1e-3, 0.0])
    theta = np.array([1.0, 2.0, -1.0, 0.5])
    out, m, v = adamw.adamw_step(theta, g, np.zeros(4), np.zeros(4), step=1, **HP)
    expect = theta * (1 - HP["lr"] * HP["weight_decay"]) - HP["lr"] * g / (np.abs(g) + HP["eps"])
    assert np.allclose(out, expect, rtol=1e-12, atol=0)
    assert np.allclose(m, (1 - HP["beta1"]) * g) and np.allclose(v, (1 - HP["beta2"]) * g * g)


def test_zero_gradient_only_decays():
    theta = np.linspace(-1, 1, 11)
    out, m, v = adamw.adamw_step(theta, np.zeros(11), np.zeros(11), np.zeros(11), step=3, **HP)
    assert np.array_equal(out, theta * (1 - HP["lr"] * HP["weight_decay"]))
    assert not m.any() and not v.any()


def test_pool_blocks_only():
    ranks = np.array([2, 3, 1])
    width = 5
    offs = np.array([0, 10, 25])
    theta = np.arange(30, dtype=np.float64)
    g = np.ones(30)
    out, m, v = adamw.adamw_pool(theta, g, np.zeros(30), np.zeros(30), offs, ranks, width, [1], step=1, **HP)
    changed = np.nonzero(out != theta)[0]
    assert changed.min() == 10 and changed.max() == 24 and changed.size == 15
