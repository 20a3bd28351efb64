"""Seeded random shapes for partitioned attention against the fp64 oracle.

"Reflex: Real-Time VLA Control through Streaming Inference", §III Eq. (1):
every suffix query attends with one softmax over [pinned; window; dynamic].
Each case draws a head dimension, a grouping of query heads over K/V heads,
pinned / window / suffix sizes (including empty and ragged regions and a
wrapped window), a number of pushes, and a forced or automatic partition of
the key sequence, then compares every output element with the oracle.
"""
import numpy as np
import pytest

from oracle import attention as OA
from oracle.pipeline import OracleStream
from partitioned_kv_cache_gb300 import workload as W
from tests._util import check_attention, dev, ensure_built, few_keys_scale, host64

pytestmark = pytest.mark.gpu

N_CASES = 48


@pytest.fixture(scope="module")
def rx():
    ensure_built()
    from partitioned_kv_cache_gb300 import rx as m
    return m


def _case(i):
    g = np.random.default_rng(1000 + i)
    D = int(g.choice([64, 128, 256]))
    Hkv = int(g.choice([1, 1, 2, 4]))
    G = int(g.choice([1, 2, 4, 8, 16]))
    P = int(g.choice([0, 1, 37, 64, 150]))
    N = int(g.integers(1, 6))
    F = int(g.choice([1, 17, 64, 100, 128]))
    S = int(g.integers(1, 70))
    if P == 0 and S == 0:
        S = 1
    pushes = int(g.integers(0, N + 4))
    splits = int(g.choice([0, 0, 1, 3, 7, 16, 20]))
    dparts = int(g.choice([0, 0, 1, 2, 4]))
    if dparts and D // dparts < 64:
        dparts = 0
    return dict(D=D, Hkv=Hkv, Hq=G * Hkv, P=P, N=N, F=F, S=S, pushes=pushes, splits=splits, dparts=dparts)


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_shape(rx, i):
    c = _case(i)
    wl = W.Workload("fuzz%d" % i, L=2, Hq=c["Hq"], Hkv=c["Hkv"], D=c["D"], P=c["P"], N=c["N"], F=c["F"],
                    S=c["S"], steps=1, ticks=1, d_model=128, emb_dim=16, state_dim=16, hidden=64)
    seed = 77 + i
    cache = rx.Cache(wl.L, wl.Hq, wl.Hkv, wl.D, wl.P, wl.N, wl.F, wl.S)
    if c["P"] > 0:
        pk, pv = W.pinned_kv(wl, seed)
        cache.pin_prefix(dev(pk), dev(pv))
    cache.set_attn_splits(min(c["splits"], 64))
    cache.set_attn_dparts(c["dparts"])
    ost = OracleStream(wl, seed)
    for t in range(c["pushes"]):
        fk, fv = W.frame_kv(wl, seed, t)
        cache.push_frame(dev(fk), dev(fv))
        ost.push(t)
    f = W.bf16_bits_to_f64
    for layer in range(wl.L):
        q, kd, vd = W.suffix_qkv(wl, seed, max(c["pushes"] - 1, 0), 0, layer)
        got = host64(cache.attend_suffix(layer, dev(q), dev(kd), dev(vd)))
        ks, vs = ost.regions(layer, f(kd), f(vd))
        ref = OA.partitioned_attention(f(q), ks, vs)
        # Unit-scale bounds unless a row sees fewer than 64 keys
        # (few_keys_scale: the path's rounding bound, 2^-8 * max|V|).
        vmax = max(float(np.abs(v).max()) for v in vs if v.size)
        check_attention(got, ref, few_keys_scale(sum(v.shape[0] for v in vs), vmax))
    assert cache.check_device_error() == 0
    cache.close()


N_BATCH_CASES = 16


@pytest.mark.parametrize("i", range(N_BATCH_CASES))
def test_random_batch(rx, i):
    """"OxyGen ...", §"Core method": random language batches (streams, query
    tokens per stream, tail capacities and lengths, with or without the action
    suffix in the same launch) over a shared cache of random shape."""
    import torch
    g = np.random.default_rng(2000 + i)
    D = int(g.choice([64, 128, 256]))
    Hkv = int(g.choice([1, 1, 2]))
    Hq = int(g.choice([1, 2, 4, 8])) * Hkv
    B, T = int(g.integers(1, 21)), int(g.integers(1, 4))
    tail_cap = int(g.integers(1, 41))
    S = int(g.integers(1, 60))
    wl = W.Workload("bfuzz%d" % i, L=1, Hq=Hq, Hkv=Hkv, D=D, P=int(g.choice([0, 20, 64])), N=int(g.integers(1, 4)),
                    F=int(g.choice([17, 64])), S=S, steps=1, ticks=1, d_model=128, emb_dim=16, state_dim=16,
                    hidden=64, n_lang=B, tail_max=tail_cap, tail_cap=tail_cap)
    seed = 300 + i
    cache = rx.Cache(wl.L, wl.Hq, wl.Hkv, wl.D, wl.P, wl.N, wl.F, wl.S, wl.tail_cap, B * T)
    if wl.P > 0:
        pk, pv = W.pinned_kv(wl, seed)
        cache.pin_prefix(dev(pk), dev(pv))
    ost = OracleStream(wl, seed)
    for t in range(int(g.integers(0, wl.N + 2))):
        fk, fv = W.frame_kv(wl, seed, t)
        cache.push_frame(dev(fk), dev(fv))
        ost.push(t)
    f = W.bf16_bits_to_f64
    q = W.to_bf16_bits(g.standard_normal((B, T, Hq, D), dtype=np.float32))
    tk = W.to_bf16_bits(g.standard_normal((B, tail_cap, Hkv, D), dtype=np.float32))
    tv = W.to_bf16_bits(g.standard_normal((B, tail_cap, Hkv, D), dtype=np.float32))
    ln = g.integers(0, tail_cap + 1, size=B).astype(np.int32)
    if wl.P == 0 and len(ost.window.window()) == 0:
        ln = np.maximum(ln, 1)   # every stream needs at least one key
    lang = (dev(q), dev(tk), dev(tv), torch.from_numpy(ln).cuda())
    with_action = bool(g.integers(0, 2))
    action = None
    if with_action:
        aq, akd, avd = W.suffix_qkv(wl, seed, 0, 0, 0)
        action = (dev(aq), dev(akd), dev(avd))
    oa, ol = cache.attend_batch(0, action, lang)
    ks, vs = ost.regions(0, np.zeros((0, Hkv, D)), np.zeros((0, Hkv, D)))
    reqs = [(f(q[b]), f(tk[b, :ln[b]]), f(tv[b, :ln[b]])) for b in range(B)]
    refs = OA.shared_cache_attention(ks[:-1], vs[:-1], reqs)
    got = host64(ol)
    vmax = max([float(np.abs(v).max()) for v in vs[:-1] if v.size] + [float(np.abs(f(tv)).max())])
    shared = sum(v.shape[0] for v in vs[:-1])
    for b, ref in enumerate(refs):
        check_attention(got[b], ref, few_keys_scale(shared + int(ln[b]), vmax))
    if with_action:
        aks, avs = ost.regions(0, f(akd), f(avd))
        amax = max(float(np.abs(v).max()) for v in avs if v.size)
        check_attention(host64(oa), OA.partitioned_attention(f(aq), aks, avs),
                        few_keys_scale(sum(v.shape[0] for v in avs), amax))
    assert cache.check_device_error() == 0
    cache.close()
