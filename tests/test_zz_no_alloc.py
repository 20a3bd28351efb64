"""The allocation-free attention entry point (rx_attend_regions_static).

It serves callers that cannot allocate device memory -- a real-time control
loop that must never stall on cudaMalloc, an embedded runtime with a fixed
memory budget, a plugin inside a framework that owns the allocator -- by
running the same attention kernels with their scratch in a fixed array
inside the library.  This file checks, through the C ABI, that two calls in a
row give the same results as the allocating path (rx_attend_suffix on an
rx_cache holding the same regions), within the attention tolerance the other
tests use.  It is named so that pytest collects it last.
"""
import numpy as np
import pytest

from partitioned_kv_cache_gb300 import workload as W
from tests._util import ATT_MAX, ATT_MEAN, dev, ensure_built, host64

pytestmark = pytest.mark.gpu


def test_static_entry_matches_cache_path_on_two_calls():
    import torch
    ensure_built()
    from partitioned_kv_cache_gb300 import rx
    wl = W.WORKLOADS["c2"]
    seed = 21
    pk, pv = W.pinned_kv(wl, seed)
    cache = rx.Cache(wl.L, wl.Hq, wl.Hkv, wl.D, wl.P, wl.N, wl.F, wl.S)
    cache.pin_prefix(dev(pk), dev(pv))
    frames = [W.frame_kv(wl, seed, t) for t in range(wl.N)]
    for fk, fv in frames:
        cache.push_frame(dev(fk), dev(fv))
    # The same window as one contiguous run of N*F tokens (order is free).
    k_win = dev(np.concatenate([f[0][0] for f in frames]))
    v_win = dev(np.concatenate([f[1][0] for f in frames]))
    out = torch.empty((wl.S, wl.Hq, wl.D), dtype=torch.bfloat16, device="cuda")
    for call in range(2):
        q, kd, vd = (dev(a) for a in W.suffix_qkv(wl, seed, 0, call, 0))
        want = host64(cache.attend_suffix(0, q, kd, vd))
        rx.attend_regions_static(q, dev(pk[0]), dev(pv[0]), k_win, v_win, kd, vd, out)
        got = host64(out)
        err = np.abs(got - want)
        assert np.all(np.isfinite(got))
        assert err.max() <= ATT_MAX and err.mean() <= ATT_MEAN, (call, err.max(), err.mean())
    cache.close()


def test_static_entry_rejects_too_many_query_rows():
    import torch
    ensure_built()
    from partitioned_kv_cache_gb300 import rx
    S, Hq, D = 15500, 1, 256         # 15616 padded rows x (2*256 + 32) B > 8 MiB
    q = torch.zeros((S, Hq, D), dtype=torch.bfloat16, device="cuda")
    kd = torch.zeros((4, 1, D), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(rx.RxError) as e:
        rx.attend_regions_static(q, None, None, None, None, kd, kd, torch.empty_like(q))
    assert e.value.status == -3
