"""AdaRMSNorm and its gamma MLP on the GPU against the fp64 oracle.

"Reflex: Real-Time VLA Control through Streaming Inference", §III Eq. (2),
"Model components" (MLP), §V forward (FP32 mean of squares).  Bar: relative
error <= 1e-2 elementwise and no NaN/Inf for inputs spanning 1e-6..1e3.
"""
import numpy as np
import pytest

from oracle import adarms as OA
from partitioned_kv_cache_gb300 import workload as W
from tests._util import check_norm, dev, ensure_built, host64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rx():
    ensure_built()
    from partitioned_kv_cache_gb300 import rx as m
    return m


@pytest.mark.parametrize("name,n_sets", [("c1", 2), ("c2", 3)])
def test_gamma_matches_oracle(rx, name, n_sets):
    import torch
    wl = W.WORKLOADS[name]
    seed, tick = 9, 2
    ws = [W.mlp_weights(wl, seed, i // 2, i % 2) for i in range(n_sets)]
    W1, b1, W2, b2 = (dev(np.stack([w[j] for w in ws])) for j in range(4))
    t = torch.from_numpy(W.timesteps(wl)).cuda()
    st = W.robot_state(wl, seed, tick)
    state = torch.from_numpy(np.repeat(st[None], wl.steps, axis=0)).cuda()
    gamma = rx.ada_gamma(t, state, W1, b1, W2, b2, wl.emb_dim).cpu().numpy()
    for i in range(n_sets):
        w64 = [W.bf16_bits_to_f64(a) for a in ws[i]]
        for k, tk in enumerate(W.timesteps(wl)):
            ref = OA.gamma_mlp(OA.conditioning(float(tk), st, wl.emb_dim), *w64)
            np.testing.assert_allclose(gamma[i, k], ref, rtol=0, atol=2e-5)


# Up to one CTA (8 rows) per SM the kernel prefetches its rows into L2 before
# the dependency wait; the last two sizes are larger than that on GB300.
@pytest.mark.parametrize("rows,d", [(51, 1024), (8, 128), (3, 4096), (5, 8), (1, 2048), (300, 1000),
                                    (2000, 1024), (1300, 40)])
def test_norm_matches_oracle_across_magnitudes(rx, rows, d):
    import torch
    x = W.magnitude_sweep(rows, d, seed=rows * d)
    gamma = (1.0 + 0.1 * np.random.default_rng(d).standard_normal(d)).astype(np.float32)
    y = rx.adarmsnorm(dev(x), torch.from_numpy(gamma).cuda(), 1e-6)
    ref = OA.ada_rms_norm(W.bf16_bits_to_f64(x), gamma.astype(np.float64), 1e-6)
    check_norm(host64(y), ref)


def test_norm_of_suffix_activations_with_mlp_gamma(rx):
    import torch
    wl = W.WORKLOADS["c2"]
    x = W.norm_input(wl, 1, 0, 0, 0, 0)
    w = W.mlp_weights(wl, 1, 0, 0)
    st = W.robot_state(wl, 1, 0)
    g = rx.ada_gamma(torch.tensor([1.0], device="cuda"), torch.from_numpy(st[None]).cuda(),
                     *(dev(a)[None] for a in w), wl.emb_dim)[0, 0]
    y = rx.adarmsnorm(dev(x), g, wl.eps)
    ref_g = OA.gamma_mlp(OA.conditioning(1.0, st, wl.emb_dim), *(W.bf16_bits_to_f64(a) for a in w))
    check_norm(host64(y), OA.ada_rms_norm(W.bf16_bits_to_f64(x), ref_g, wl.eps))


def test_zero_rows_is_a_noop(rx):
    import torch
    x = torch.zeros((0, 64), dtype=torch.bfloat16, device="cuda")
    g = torch.ones(64, device="cuda")
    assert rx.adarmsnorm(x, g, 1e-6).shape == (0, 64)


@pytest.mark.parametrize("d,hidden,emb,state_dim,n_cond,wscale", [
    (1000, 80, 16, 16, 16, 1.0),     # ragged 128-row tile, hidden not a multiple of 64, 16 vectors
    (136, 2048, 6, 5, 1, 1.0),       # widest hidden; conditioning width 11 (not a multiple of 8)
    (8, 16, 2, 0, 5, 1.0),           # smallest shapes, no state
    (256, 512, 16, 16, 10, 50.0),    # weights ~N(0, 1): gamma - 1 of order 100
    (512, 256, 16, 16, 3, 1.0),      # 4 row tiles: a cluster of 4 sharing 4 blocks of the first layer
    (384, 192, 16, 16, 7, 1.0),      # 3 row tiles: no cluster, every CTA computes all 3 blocks
])
def test_gamma_shapes_and_scales(rx, d, hidden, emb, state_dim, n_cond, wscale):
    """Eq. (2)'s gamma MLP over the edge shapes of the kernel.  Bound: the
    error of an fp32 evaluation with the hidden activation carried to 2^-16
    of itself (two bf16 parts: the second holds the first's rounding error,
    itself rounded within 2^-8), 4e-5 x sum_j |W2_ij h_j| + |b2_i| per
    element."""
    import torch
    wl = W.Workload("gamma-shape", L=1, Hq=1, Hkv=1, D=64, P=0, N=1, F=1, S=1, steps=n_cond,
                    ticks=1, d_model=d, emb_dim=emb, state_dim=state_dim, hidden=hidden)
    seed = 31
    ws = []
    for site in range(2):
        w = W.mlp_weights(wl, seed, 0, site)
        if wscale != 1.0:
            w = tuple(W.to_bf16_bits((W.bf16_bits_to_f64(a) * wscale).astype(np.float32)) for a in w)
        ws.append(w)
    W1, b1, W2, b2 = (dev(np.stack([w[j] for w in ws])) for j in range(4))
    t = torch.from_numpy(W.timesteps(wl)).cuda()
    st = W.robot_state(wl, seed, 0)
    state = torch.from_numpy(np.repeat(st[None], n_cond, axis=0).reshape(n_cond, state_dim)).cuda()
    gamma = rx.ada_gamma(t, state, W1, b1, W2, b2, emb).cpu().numpy()
    assert np.all(np.isfinite(gamma))
    for s_i, w in enumerate(ws):
        w64 = [W.bf16_bits_to_f64(a) for a in w]
        for k, tk in enumerate(W.timesteps(wl)):
            c = OA.conditioning(float(tk), st, emb)
            ref = OA.gamma_mlp(c, *w64)
            h = OA.silu(w64[0] @ c + w64[1])
            bound = 4e-5 * (np.abs(w64[2]) @ np.abs(h) + np.abs(w64[3])) + 1e-7
            err = np.abs(gamma[s_i, k] - ref)
            assert np.all(err <= bound), "set %d vector %d: worst err/bound %.2f" % (
                s_i, k, float(np.max(err / bound)))
