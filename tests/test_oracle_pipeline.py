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
