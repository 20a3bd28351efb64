"""Ring append on the GPU: the window after T pushes is exactly the last N
frames in order, bit-exact ("Reflex: Real-Time VLA Control through Streaming
Inference", §III "System architecture": FIFO of N observations, enqueue newest
/ evict oldest; §V add_new_prefix() returns the eviction count)."""
import numpy as np
import pytest

from oracle.ring import FrameWindow
from tests._util import ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rx():
    ensure_built()
    from partitioned_kv_cache_gb300 import rx as m
    return m


def _frame(torch, L, F, Hkv, D, fid):
    # K holds the frame id, V the layer index + 1: small integers, exact in bf16.
    k = torch.full((L, F, Hkv, D), float(fid), dtype=torch.bfloat16, device="cuda")
    v = torch.arange(1, L + 1, dtype=torch.float32, device="cuda").view(L, 1, 1, 1)
    v = v.expand(L, F, Hkv, D).to(torch.bfloat16).contiguous()
    return k, v


@pytest.mark.parametrize("L,Hkv,D,N,F", [(2, 1, 64, 3, 16), (1, 1, 256, 4, 256), (3, 2, 128, 1, 8),
                                         (18, 1, 256, 8, 256)])
def test_window_after_every_push_is_bit_exact(rx, L, Hkv, D, N, F):
    import torch
    cache = rx.Cache(L, 2 * Hkv, Hkv, D, 16, N, F, 8)
    ref = FrameWindow(N)
    assert cache.get_state() == (0, 0, 0)
    assert cache.debug_window() == []
    for T in range(1, 3 * N + 2):
        k, v = _frame(torch, L, F, Hkv, D, T - 1)
        ev = cache.push_frame(k, v)
        assert ev == ref.push(T - 1)
        head, valid, pushes = cache.get_state()
        assert (head, valid, pushes) == (T % N, min(T, N), T)
        for layer in sorted({0, L - 1}):
            kw, vw = cache.export_window(layer)
            ids = kw.view(valid, F * Hkv * D).float()
            want = torch.tensor(ref.window(), dtype=torch.float32, device="cuda")
            assert torch.equal(ids, want[:, None].expand_as(ids)), (T, layer)
            assert torch.equal(vw.float(), torch.full_like(vw.float(), layer + 1))
    assert cache.check_device_error() == 0
    cache.close()


def test_push_leaves_pinned_region_and_other_slots_untouched(rx):
    import torch
    L, Hkv, D, N, F = 2, 1, 64, 4, 16
    cache = rx.Cache(L, 2, Hkv, D, 16, N, F, 8)
    for T in range(2):
        cache.push_frame(*_frame(torch, L, F, Hkv, D, 7 + T))
    kw, _ = cache.export_window(1)
    assert kw.view(2, -1).float().amax(dim=1).tolist() == [7.0, 8.0]
    cache.close()


def test_push_rejects_misaligned_frames(rx):
    import torch
    cache = rx.Cache(1, 2, 1, 64, 16, 2, 16, 8)
    k = torch.zeros(16 * 64 + 1, dtype=torch.bfloat16, device="cuda")
    km = k[1:].view(1, 16, 1, 64)    # the right shape, 2 bytes off a 16-byte boundary
    with pytest.raises(rx.RxError):
        cache.push_frame(km, km)
    cache.close()
