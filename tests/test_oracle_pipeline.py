"""Pins for the oracle's stream composition (CPU only)."""
import numpy as np

from oracle import attention as A
from oracle.pipeline import OracleStream
from partitioned_kv_cache_gb300 import workload as W


def test_stream_window_follows_fifo_and_rows_are_independent():
    wl = W.WORKLOADS["c1"]
    st = OracleStream(wl, seed=3)
    for t in range(5):
        st.push(t)
        assert st.window_ticks() == list(range(max(0, t + 1 - wl.N), t + 1))
    full = st.attend(4, 1, 0)
    part = st.attend(4, 1, 0, tokens=[2, 5])
    np.testing.assert_allclose(part, full[[2, 5]], rtol=0, atol=1e-14)


def test_stream_attention_equals_torch_over_explicit_window():
    """The composed tick attends over exactly pin + last N frames + dyn."""
    import torch
    import torch.nn.functional as F
    wl = W.WORKLOADS["c1"]
    st = OracleStream(wl, seed=5)
    for t in range(3):
        st.push(t)
    f = W.bf16_bits_to_f64
    q, kd, vd = (f(a) for a in W.suffix_qkv(wl, 5, 2, 0, 0))
    pk, pv = (f(a) for a in W.pinned_kv(wl, 5))
    frames = [tuple(f(a) for a in W.frame_kv(wl, 5, t)) for t in (1, 2)]
    K = np.concatenate([pk[0]] + [fr[0][0] for fr in frames] + [kd])
    V = np.concatenate([pv[0]] + [fr[1][0] for fr in frames] + [vd])
    qt = torch.from_numpy(q).permute(1, 0, 2)
    kt = torch.from_numpy(K).permute(1, 0, 2).expand(wl.Hq, -1, -1)
    vt = torch.from_numpy(V).permute(1, 0, 2).expand(wl.Hq, -1, -1)
    ref = F.scaled_dot_product_attention(qt, kt, vt).permute(1, 0, 2).numpy()
    np.testing.assert_allclose(st.attend(2, 0, 0), ref, rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# The stream's AdaRMSNorm composition ("Reflex ...", §III Eq. (2) and "Model
# components"; §V AdaRMSNorm forward), pinned to PyTorch modules built here
# from the seeded draws named by explicit (tick, step, layer, site) indices.
# ---------------------------------------------------------------------------
import dataclasses
import math

import pytest


def _torch_gamma(wl, seed, tick, step, layer, site):
    """gamma = 1 + Linear -> SiLU -> Linear of c = [sin(t w), cos(t w), state],
    w_j = 10000^(-j / (E/2)), with torch.nn modules in float64."""
    import torch
    f = W.bf16_bits_to_f64
    W1, b1, W2, b2 = (torch.from_numpy(f(a)) for a in W.mlp_weights(wl, seed, layer, site))
    t = float(W.timesteps(wl)[step])
    half = wl.emb_dim // 2
    emb = [math.sin(t * 10000.0 ** (-j / half)) for j in range(half)] + \
          [math.cos(t * 10000.0 ** (-j / half)) for j in range(half)]
    c = torch.tensor(emb + [float(s) for s in W.robot_state(wl, seed, tick)], dtype=torch.float64)
    mlp = torch.nn.Sequential(torch.nn.Linear(wl.cond_dim, wl.hidden), torch.nn.SiLU(),
                              torch.nn.Linear(wl.hidden, wl.d_model)).double()
    with torch.no_grad():
        mlp[0].weight.copy_(W1)
        mlp[0].bias.copy_(b1)
        mlp[2].weight.copy_(W2)
        mlp[2].bias.copy_(b2)
        return 1.0 + mlp(c)


def _torch_norm(wl, seed, tick, step, layer, site):
    import torch
    import torch.nn.functional as F
    x = torch.from_numpy(W.bf16_bits_to_f64(W.norm_input(wl, seed, tick, step, layer, site)))
    return F.rms_norm(x, (wl.d_model,), weight=_torch_gamma(wl, seed, tick, step, layer, site),
                      eps=wl.eps).numpy()


def _torch_attention(wl, seed, window_ticks, tick, step, layer):
    import torch
    import torch.nn.functional as F
    f = W.bf16_bits_to_f64
    q, kd, vd = (f(a) for a in W.suffix_qkv(wl, seed, tick, step, layer))
    pk, pv = (f(a) for a in W.pinned_kv(wl, seed))
    frames = [tuple(f(a) for a in W.frame_kv(wl, seed, t)) for t in window_ticks]
    K = np.concatenate([pk[layer]] + [fr[0][layer] for fr in frames] + [kd])
    V = np.concatenate([pv[layer]] + [fr[1][layer] for fr in frames] + [vd])
    qt = torch.from_numpy(q).permute(1, 0, 2)
    kt = torch.from_numpy(np.repeat(K, wl.G, axis=1)).permute(1, 0, 2)
    vt = torch.from_numpy(np.repeat(V, wl.G, axis=1)).permute(1, 0, 2)
    return F.scaled_dot_product_attention(qt, kt, vt).permute(1, 0, 2).numpy()


@pytest.fixture(scope="module")
def wl2():
    """c1's shapes with two layers, so that layer and site indices are both
    exercised; every (layer, site) has its own weight draw."""
    return dataclasses.replace(W.WORKLOADS["c1"], L=2)


def test_stream_gamma_matches_torch_mlp_per_site_layer_step_and_tick(wl2):
    st = OracleStream(wl2, seed=8)
    seen = []
    for tick in (0, 2):
        for step in range(wl2.steps):
            for layer in range(wl2.L):
                for site in (0, 1):
                    ref = _torch_gamma(wl2, 8, tick, step, layer, site).numpy()
                    np.testing.assert_allclose(st.gamma(tick, step, layer, site), ref, rtol=0, atol=1e-13)
                    seen.append(ref)
    # Every index changes gamma by far more than the tolerance, so a swapped
    # site, layer, step or tick would fail above.
    seen = np.stack(seen)
    gaps = [np.abs(a - b).max() for i, a in enumerate(seen) for b in seen[i + 1:]]
    assert min(gaps) > 1e-5


def test_stream_norm_matches_torch_rms_norm(wl2):
    st = OracleStream(wl2, seed=9)
    for step in range(wl2.steps):
        for layer in range(wl2.L):
            for site in (0, 1):
                ref = _torch_norm(wl2, 9, 1, step, layer, site)
                np.testing.assert_allclose(st.norm(1, step, layer, site), ref, rtol=1e-12, atol=1e-14)


def test_stream_tick_outputs_in_order_for_every_step_and_layer(wl2):
    """tick(T) pushes frame T, then for every (step, layer) returns (the
    pre-attention norm, the attention output over pin + last N frames + the
    step's dynamic keys, the pre-MLP norm), each equal to the torch
    reference built from that (tick, step, layer)."""
    st = OracleStream(wl2, seed=10)
    for T in range(4):
        out = st.tick(T)
        window = list(range(max(0, T + 1 - wl2.N), T + 1))
        assert st.window_ticks() == window
        assert sorted(out) == [(k, l) for k in range(wl2.steps) for l in range(wl2.L)]
        for (k, l), (y0, o, y1) in out.items():
            np.testing.assert_allclose(y0, _torch_norm(wl2, 10, T, k, l, 0), rtol=1e-12, atol=1e-14)
            np.testing.assert_allclose(o, _torch_attention(wl2, 10, window, T, k, l), rtol=0, atol=1e-12)
            np.testing.assert_allclose(y1, _torch_norm(wl2, 10, T, k, l, 1), rtol=1e-12, atol=1e-14)
