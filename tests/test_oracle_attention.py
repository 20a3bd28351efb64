"""Pins for the oracle's partitioned attention (CPU only).

Each check ties ``oracle.attention`` to something other than itself: pure
Python brute force, PyTorch's own fp64 scaled-dot-product attention (an
independent library routine), Proposition A.1 of "Reflex: Real-Time VLA
Control through Streaming Inference" (§III, region split == full batch),
permutation invariance, and closed-form special cases.
"""
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import attention as A
from partitioned_kv_cache_gb300 import workload as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _randn(seed, *shape, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def _sdpa(q, K, V):
    """torch fp64 SDPA with explicit GQA expansion (kv head of q head h = h // G)."""
    S, Hq, D = q.shape
    T, Hkv, _ = K.shape
    G = Hq // Hkv
    qt = torch.from_numpy(q).permute(1, 0, 2)                           # [Hq][S][D]
    kt = torch.from_numpy(K).permute(1, 0, 2).repeat_interleave(G, 0)   # [Hq][T][D]
    vt = torch.from_numpy(V).permute(1, 0, 2).repeat_interleave(G, 0)
    o = F.scaled_dot_product_attention(qt, kt, vt)                      # scale 1/sqrt(D)
    return o.permute(1, 0, 2).numpy()


@pytest.mark.parametrize("S,Hq,Hkv,D,T", [(3, 2, 1, 8, 7), (2, 4, 2, 4, 5), (1, 1, 1, 3, 1)])
def test_brute_force_matches(S, Hq, Hkv, D, T):
    q = _randn(1, S, Hq, D)
    K = _randn(2, T, Hkv, D)
    V = _randn(3, T, Hkv, D)
    bf = np.array(A.brute_force_attention(q.tolist(), K.tolist(), V.tolist()))
    np.testing.assert_allclose(A.full_attention(q, K, V), bf, rtol=0, atol=1e-12)


@pytest.mark.parametrize("S,Hq,Hkv,D,T", [(8, 2, 1, 64, 56), (51, 8, 1, 256, 300),
                                          (5, 8, 2, 32, 40), (4, 3, 3, 16, 9)])
def test_matches_torch_sdpa(S, Hq, Hkv, D, T):
    q = _randn(4, S, Hq, D)
    K = _randn(5, T, Hkv, D)
    V = _randn(6, T, Hkv, D)
    np.testing.assert_allclose(A.full_attention(q, K, V), _sdpa(q, K, V), rtol=0, atol=1e-12)


def test_proposition_a1_region_split_equals_full_batch():
    """Table 4 prints MSE 0.00 between partitioned and full recompute."""
    golden = dict(l.split() for l in open(os.path.join(GOLDEN, "reflex_table4_table5.txt"))
                  if l.strip() and not l.startswith("#"))
    q = _randn(7, 6, 4, 32)
    regions = [(_randn(10 + i, t, 1, 32, scale=s), _randn(20 + i, t, 1, 32))
               for i, (t, s) in enumerate([(5, 1.0), (16, 20.0), (16, 1.0), (0, 1.0), (6, 3.0)])]
    ks = [r[0] for r in regions]
    vs = [r[1] for r in regions]
    full = A.partitioned_attention(q, ks, vs)
    split = A.region_split_attention(q, ks, vs)
    np.testing.assert_allclose(split, full, rtol=0, atol=1e-12)
    assert float(np.mean((split - full) ** 2)) < 0.005 + float(golden["partitioned_vs_full_mse"])


def test_frame_order_does_not_change_the_output():
    """Softmax is invariant to permuting its logit set (Proposition A.1 proof),
    so a ring read in physical slot order equals the logical FIFO order."""
    q = _randn(8, 5, 2, 16)
    pin = (_randn(30, 3, 1, 16), _randn(31, 3, 1, 16))
    frames = [(_randn(40 + i, 4, 1, 16), _randn(50 + i, 4, 1, 16)) for i in range(4)]
    dyn = (_randn(60, 5, 1, 16), _randn(61, 5, 1, 16))
    logical = [pin] + frames + [dyn]
    physical = [pin] + frames[2:] + frames[:2] + [dyn]     # wrapped ring, head = 2
    o1 = A.partitioned_attention(q, [r[0] for r in logical], [r[1] for r in logical])
    o2 = A.partitioned_attention(q, [r[0] for r in physical], [r[1] for r in physical])
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)


def test_softmax_rows_sum_to_one():
    q = _randn(9, 7, 4, 32, scale=3.0)
    K = _randn(10, 50, 2, 32, scale=5.0)
    a = A.attention_weights(q, K)
    assert np.all(a >= 0)
    np.testing.assert_allclose(a.sum(axis=-1), 1.0, rtol=0, atol=1e-12)


def test_single_key_returns_its_value():
    q = _randn(11, 3, 2, 8)
    K = _randn(12, 1, 1, 8)
    V = _randn(13, 1, 1, 8)
    o = A.full_attention(q, K, V)
    np.testing.assert_allclose(o, np.broadcast_to(V[0, 0], o.shape), rtol=0, atol=1e-15)


def test_identical_keys_average_the_values():
    q = _randn(14, 3, 2, 8)
    K = np.broadcast_to(_randn(15, 1, 1, 8), (6, 1, 8)).copy()
    V = _randn(16, 6, 1, 8)
    o = A.full_attention(q, K, V)
    np.testing.assert_allclose(o, np.broadcast_to(V[:, 0].mean(axis=0), o.shape), rtol=0, atol=1e-14)


def test_empty_window_attends_pinned_and_dynamic_only():
    """Before any frame is pushed the window holds nothing; zero-filled slots of
    the preallocated store are not keys."""
    q = _randn(17, 4, 2, 8)
    pin = (_randn(18, 3, 1, 8), _randn(19, 3, 1, 8))
    dyn = (_randn(20, 4, 1, 8), _randn(21, 4, 1, 8))
    empty = (np.zeros((0, 1, 8)), np.zeros((0, 1, 8)))
    o = A.partitioned_attention(q, [pin[0], empty[0], dyn[0]], [pin[1], empty[1], dyn[1]])
    ref = _sdpa(q, np.concatenate([pin[0], dyn[0]]), np.concatenate([pin[1], dyn[1]]))
    np.testing.assert_allclose(o, ref, rtol=0, atol=1e-12)
    # attending zero slots instead would differ: exp(0)-weighted zero values
    zeros = (np.zeros((16, 1, 8)), np.zeros((16, 1, 8)))
    o0 = A.partitioned_attention(q, [pin[0], zeros[0], dyn[0]], [pin[1], zeros[1], dyn[1]])
    assert np.max(np.abs(o0 - o)) > 1e-3


def test_shared_cache_requests_see_only_their_own_tail():
    """OxyGen §"Core method": a stream's appended KV never enters another view."""
    shared_k = [_randn(22, 5, 1, 8), _randn(23, 8, 1, 8)]
    shared_v = [_randn(24, 5, 1, 8), _randn(25, 8, 1, 8)]
    reqs = [(_randn(26 + i, 1 + i, 2, 8), _randn(40 + i, i, 1, 8), _randn(50 + i, i, 1, 8))
            for i in range(3)]
    outs = A.shared_cache_attention(shared_k, shared_v, reqs)
    for (q, kp, vp), o in zip(reqs, outs):
        ref = _sdpa(q, np.concatenate(shared_k + [kp]), np.concatenate(shared_v + [vp]))
        np.testing.assert_allclose(o, ref, rtol=0, atol=1e-12)


def test_workload_bf16_inputs_are_exact():
    """The generator's bf16 values round-trip exactly through torch.bfloat16."""
    wl = W.WORKLOADS["c1"]
    q, k, v = W.suffix_qkv(wl, 0, 0, 0, 0)
    f = W.bf16_bits_to_f64(q)
    t = torch.from_numpy(f.astype(np.float32)).to(torch.bfloat16)
    assert np.array_equal(t.view(torch.int16).numpy().view(np.uint16), q)


def test_c4_outliers_present():
    wl = W.WORKLOADS["c4"]
    k, _ = W.frame_kv(wl, 0, 0)
    a = np.abs(W.bf16_bits_to_f64(k))
    frac = float(np.mean(a > 8.0))
    assert 0.004 < frac < 0.012


def test_block_causal_reduces_to_eq1_and_matches_masked_sdpa():
    """n_state = 0 (and n_state = S) is plain Eq. 1; otherwise it equals torch
    SDPA with the explicit boolean mask, and a brute-force masked loop."""
    q = _randn(40, 6, 2, 8)
    regions = [(_randn(41, 5, 1, 8), _randn(42, 5, 1, 8)), (_randn(43, 7, 1, 8), _randn(44, 7, 1, 8)),
               (_randn(45, 6, 1, 8), _randn(46, 6, 1, 8))]
    ks, vs = [r[0] for r in regions], [r[1] for r in regions]
    full = A.partitioned_attention(q, ks, vs)
    np.testing.assert_allclose(A.block_causal_attention(q, ks, vs, 0), full, rtol=0, atol=1e-15)
    np.testing.assert_allclose(A.block_causal_attention(q, ks, vs, 6), full, rtol=0, atol=1e-15)
    n_state = 2
    got = A.block_causal_attention(q, ks, vs, n_state)
    K, V = np.concatenate(ks), np.concatenate(vs)
    T, cached = K.shape[0], 12
    allowed = np.ones((6, T), dtype=bool)
    allowed[:n_state, cached + n_state:] = False
    qt = torch.from_numpy(q).permute(1, 0, 2)
    kt = torch.from_numpy(K).permute(1, 0, 2).expand(2, -1, -1)
    vt = torch.from_numpy(V).permute(1, 0, 2).expand(2, -1, -1)
    ref = F.scaled_dot_product_attention(qt, kt, vt, attn_mask=torch.from_numpy(allowed)).permute(1, 0, 2).numpy()
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)
    # brute force on the state rows: drop the masked keys explicitly
    keep = [j for j in range(T) if allowed[0, j]]
    bf = np.array(A.brute_force_attention(q[:n_state].tolist(), K[keep].tolist(), V[keep].tolist()))
    np.testing.assert_allclose(got[:n_state], bf, rtol=0, atol=1e-12)
    assert np.max(np.abs(got[:n_state] - full[:n_state])) > 1e-3
