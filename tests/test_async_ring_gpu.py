"""Concurrent producer / consumer ring (a spare frame slot, rx_push_frame_async).

"Reflex: Real-Time VLA Control through Streaming Inference", §III "System
architecture": Thread A encodes frames into the ring buffer while Thread B
reads the latest tokens and denoises.  Here the push runs on its own stream;
every attention on the consumer stream must see a whole window (the one after
the previous push or after the current one), never a torn mix.
"""
import numpy as np
import pytest

from oracle import attention as OA
from oracle.pipeline import OracleStream
from partitioned_kv_cache_gb300 import workload as W
from tests._util import ATT_MAX, ATT_MEAN, check_attention, dev, ensure_built, host64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rx():
    ensure_built()
    from partitioned_kv_cache_gb300 import rx as m
    return m


def _cache(rx, wl, seed):
    cache = rx.Cache(wl.L, wl.Hq, wl.Hkv, wl.D, wl.P, wl.N, wl.F, wl.S, spare_slot=1)
    pk, pv = W.pinned_kv(wl, seed)
    cache.pin_prefix(dev(pk), dev(pv))
    return cache


def test_spare_slot_ring_on_one_stream(rx):
    """With N + 1 physical slots the window is still the last N frames."""
    wl = W.WORKLOADS["c2"]
    seed = 51
    cache = _cache(rx, wl, seed)
    ost = OracleStream(wl, seed)
    f = W.bf16_bits_to_f64
    for t in range(2 * wl.N + 3):
        fk, fv = W.frame_kv(wl, seed, t)
        ev = cache.push_frame(dev(fk), dev(fv))
        assert ev == ost.push(t)
        kw, _ = cache.export_window(0)
        want = np.concatenate([fr[1][0] for fr in ost.window.window()])
        np.testing.assert_array_equal(host64(kw), want)
        q, kd, vd = W.suffix_qkv(wl, seed, t, 0, 0)
        got = host64(cache.attend_suffix(0, dev(q), dev(kd), dev(vd)))
        ks, vs = ost.regions(0, f(kd), f(vd))
        check_attention(got, OA.partitioned_attention(f(q), ks, vs))
    cache.close()


def test_spare_slot_ring_at_the_long_history_size(rx):
    """c4's window of 32 frames with a spare slot (33 physical slots, two
    layers): once the ring is full, the slot a push is about to overwrite is
    left out of the window, and with each push that gap moves to another of
    the 27 key splits.  Every checked call must see exactly the last N
    frames.  The ×20 outlier keys make the output scale max|ref|, and both
    bounds are taken relative to it."""
    import dataclasses
    wl = dataclasses.replace(W.WORKLOADS["c4"], L=2)
    seed = 54
    cache = _cache(rx, wl, seed)
    ost = OracleStream(wl, seed)
    f = W.bf16_bits_to_f64
    check_at = {wl.N - 1, wl.N, wl.N + 1, wl.N + 9, wl.N + 17, wl.N + 26, 2 * wl.N + 1}
    for t in range(2 * wl.N + 2):
        fk, fv = W.frame_kv(wl, seed, t)
        assert cache.push_frame(dev(fk), dev(fv)) == ost.push(t)
        if t not in check_at:
            continue
        q, kd, vd = W.suffix_qkv(wl, seed, t, 0, 1)
        got = host64(cache.attend_suffix(1, dev(q), dev(kd), dev(vd)))
        ks, vs = ost.regions(1, f(kd), f(vd))
        ref = OA.partitioned_attention(f(q), ks, vs)
        scale = max(1.0, float(np.abs(ref).max())) if wl.outlier_frac > 0 else 1.0
        check_attention(got, ref, scale)
    assert cache.check_device_error() == 0
    cache.close()


def test_concurrent_pushes_never_tear_the_window(rx):
    import torch
    wl = W.WORKLOADS["c2"]
    seed = 52
    cache = _cache(rx, wl, seed)
    ost = OracleStream(wl, seed)
    f = W.bf16_bits_to_f64
    for t in range(wl.N):
        fk, fv = W.frame_kv(wl, seed, t)
        cache.push_frame(dev(fk), dev(fv))
        ost.push(t)
    torch.cuda.synchronize()
    prod, cons = torch.cuda.Stream(), torch.cuda.Stream()
    q, kd, vd = W.suffix_qkv(wl, seed, 0, 0, 0)
    qd, kdd, vdd = dev(q), dev(kd), dev(vd)
    frames = [tuple(dev(a) for a in W.frame_kv(wl, seed, t)) for t in range(wl.N, wl.N + 6)]
    outs = []   # (push index after which the call was enqueued, output)
    for i, (fk, fv) in enumerate(frames):
        cache.push_frame_async(fk, fv, prod, cons)
        with torch.cuda.stream(cons):
            for _ in range(3):
                outs.append((i, cache.attend_suffix(0, qd, kdd, vdd)))
    torch.cuda.synchronize()
    # oracle for the window after each push (index -1: before the first async push)
    refs = {}
    ks, vs = ost.regions(0, f(kd), f(vd))
    refs[-1] = OA.partitioned_attention(f(q), ks, vs)
    for i in range(len(frames)):
        ost.push(wl.N + i)
        ks, vs = ost.regions(0, f(kd), f(vd))
        refs[i] = OA.partitioned_attention(f(q), ks, vs)
    for i, o in outs:
        got = host64(o)
        errs = [np.abs(got - refs[j]) for j in (i - 1, i)]
        assert any(e.max() <= ATT_MAX and e.mean() <= ATT_MEAN for e in errs), (
            "call after push %d matches neither window" % i)
    assert cache.check_device_error() == 0
    cache.close()


def test_async_push_needs_a_spare_slot(rx):
    import torch
    wl = W.WORKLOADS["c1"]
    cache = rx.Cache(wl.L, wl.Hq, wl.Hkv, wl.D, wl.P, wl.N, wl.F, wl.S)
    fk, fv = W.frame_kv(wl, 0, 0)
    s = torch.cuda.Stream()
    with pytest.raises(rx.RxError) as e:
        cache.push_frame_async(dev(fk), dev(fv), s, s)
    assert e.value.status == -7
    with pytest.raises(rx.RxError) as e:   # F = 16 is not a multiple of 64
        rx.Cache(wl.L, wl.Hq, wl.Hkv, wl.D, wl.P, wl.N, wl.F, wl.S, spare_slot=1)
    assert e.value.status == -6
    cache.close()
