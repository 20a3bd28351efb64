"""Pins for the oracle's AdaRMSNorm and its conditioning (CPU only).

"Reflex: Real-Time VLA Control through Streaming Inference", §III Eq. (2) and
§V "Key implementation".  Checks: zero MLP reduces Eq. (2) to plain RMSNorm
(compared with PyTorch's own fp64 rms_norm), the constant-vector closed form,
the tiny-input regime where eps dominates, scale invariance, the gamma MLP
against torch.nn modules in fp64, and closed-form embedding values.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import adarms as R
from partitioned_kv_cache_gb300 import workload as W


def _randn(seed, *shape, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def test_zero_mlp_is_plain_rmsnorm():
    x = _randn(1, 7, 64, scale=3.0)
    g = R.gamma_mlp(np.ones(32), np.zeros((16, 32)), np.zeros(16), np.zeros((64, 16)), np.zeros(64))
    np.testing.assert_array_equal(g, np.ones(64))
    y = R.ada_rms_norm(x, g, 1e-6)
    ref = F.rms_norm(torch.from_numpy(x), (64,), eps=1e-6).numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-13, atol=0)


def test_rmsnorm_with_gain_matches_torch():
    x = _randn(2, 5, 128)
    gamma = 1.0 + _randn(3, 128, scale=0.1)
    ref = F.rms_norm(torch.from_numpy(x), (128,), weight=torch.from_numpy(gamma), eps=1e-6).numpy()
    np.testing.assert_allclose(R.ada_rms_norm(x, gamma, 1e-6), ref, rtol=1e-13, atol=0)


@pytest.mark.parametrize("a", [3.0, -0.25, 1e-3, 1e-6, 1e3])
def test_constant_vector_closed_form(a):
    d, eps = 32, 1e-6
    gamma = 1.0 + _randn(4, d, scale=0.05)
    y = R.ada_rms_norm(np.full((1, d), a), gamma, eps)
    np.testing.assert_allclose(y[0], a / math.sqrt(a * a + eps) * gamma, rtol=1e-14, atol=0)


def test_scale_invariance_when_mean_square_dominates_eps():
    x = _randn(5, 4, 256)
    gamma = 1.0 + _randn(6, 256, scale=0.1)
    y1 = R.ada_rms_norm(x, gamma, 1e-6)
    y2 = R.ada_rms_norm(x * 37.0, gamma, 1e-6)
    np.testing.assert_allclose(y1, y2, rtol=1e-6, atol=0)


def test_gamma_mlp_matches_torch_modules():
    wl = W.WORKLOADS["c2"]
    W1, b1, W2, b2 = (W.bf16_bits_to_f64(a) for a in W.mlp_weights(wl, 0, 0, 0))
    c = R.conditioning(0.7, W.robot_state(wl, 0, 3), wl.emb_dim)
    mlp = torch.nn.Sequential(torch.nn.Linear(wl.cond_dim, wl.hidden), torch.nn.SiLU(),
                              torch.nn.Linear(wl.hidden, wl.d_model)).double()
    with torch.no_grad():
        mlp[0].weight.copy_(torch.from_numpy(W1))
        mlp[0].bias.copy_(torch.from_numpy(b1))
        mlp[2].weight.copy_(torch.from_numpy(W2))
        mlp[2].bias.copy_(torch.from_numpy(b2))
        ref = 1.0 + mlp(torch.from_numpy(c)).numpy()
    np.testing.assert_allclose(R.gamma_mlp(c, W1, b1, W2, b2), ref, rtol=0, atol=1e-13)


def test_sinusoidal_embedding_closed_forms():
    e0 = R.sinusoidal_embedding(0.0, 16)
    np.testing.assert_array_equal(e0, np.r_[np.zeros(8), np.ones(8)])
    t = 0.37
    e = R.sinusoidal_embedding(t, 16)
    assert e[0] == pytest.approx(math.sin(t), abs=1e-15)          # lowest index: w = 1
    assert e[8] == pytest.approx(math.cos(t), abs=1e-15)
    assert e[7] == pytest.approx(math.sin(t * 10000.0 ** (-7 / 8)), abs=1e-15)
    np.testing.assert_allclose(e[:8] ** 2 + e[8:] ** 2, 1.0, rtol=0, atol=1e-15)
    c = R.conditioning(t, np.arange(4.0), 16)
    np.testing.assert_array_equal(c[16:], np.arange(4.0))


def test_magnitude_sweep_is_finite_and_bounded():
    """Eq. (2) keeps the output at unit RMS times gamma across 1e-6..1e3 inputs
    except where eps dominates (then y ~ x / sqrt(eps))."""
    x = W.bf16_bits_to_f64(W.magnitude_sweep(64, 1024, 0))
    gamma = np.ones(1024)
    y = R.ada_rms_norm(x, gamma, 1e-6)
    assert np.all(np.isfinite(y))
    ms = np.mean(x * x, axis=1)
    rms_y = np.sqrt(np.mean(y * y, axis=1))
    np.testing.assert_allclose(rms_y, np.sqrt(ms / (ms + 1e-6)), rtol=1e-12)
