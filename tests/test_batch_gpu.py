"""Shared-cache multi-request attention in one launch (config 5).

"OxyGen: Unified KV Cache Management for Vision-Language-Action Models under
Multi-Task Parallelism", §"Core method": the action expert reads the prefill
cache read-only while language streams, stacked along a batch dimension, each
append their own KV; nothing one stream appends enters another's view.
Checked against the oracle's per-request attention over [shared; own tail].
"""
import numpy as np
import pytest

from oracle import attention as OA
from oracle.pipeline import OracleStream
from partitioned_kv_cache_gb300 import workload as W
from tests._util import check_attention, dev, ensure_built, host64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rx():
    ensure_built()
    from partitioned_kv_cache_gb300 import rx as m
    return m


def _setup(rx, wl, seed, pushes):
    cache = rx.Cache(wl.L, wl.Hq, wl.Hkv, wl.D, wl.P, wl.N, wl.F, wl.S, wl.tail_cap,
                     wl.n_lang)
    pk, pv = W.pinned_kv(wl, seed)
    cache.pin_prefix(dev(pk), dev(pv))
    ost = OracleStream(wl, seed)
    for t in range(pushes):
        fk, fv = W.frame_kv(wl, seed, t)
        cache.push_frame(dev(fk), dev(fv))
        ost.push(t)
    return cache, ost


def _lang(wl, seed, tick, step, layer, lens=None):
    import torch
    q, tk, tv, ln = W.lang_requests(wl, seed, tick, step, layer)
    if lens is not None:
        ln = np.asarray(lens, dtype=np.int32)
    return q, tk, tv, ln, (dev(q), dev(tk), dev(tv), torch.from_numpy(ln).cuda())


def _check_lang(ost, layer, q, tk, tv, ln, got):
    f = W.bf16_bits_to_f64
    ks, vs = ost.regions(layer, np.zeros((0,) + tk.shape[2:]), np.zeros((0,) + tk.shape[2:]))
    reqs = [(f(q[b]), f(tk[b, :ln[b]]), f(tv[b, :ln[b]])) for b in range(q.shape[0])]
    for b, ref in enumerate(OA.shared_cache_attention(ks[:-1], vs[:-1], reqs)):
        check_attention(got[b], ref)


def test_action_and_language_streams_in_one_launch(rx):
    wl = W.WORKLOADS["c5"]
    seed, tick, step = 31, 0, 2
    cache, ost = _setup(rx, wl, seed, wl.N + 2)
    for layer in (0, wl.L - 1):
        q, kd, vd = W.suffix_qkv(wl, seed, tick, step, layer)
        lq, ltk, ltv, lln, lang = _lang(wl, seed, tick, step, layer)
        n0 = rx.launch_count()
        oa, ol = cache.attend_batch(layer, (dev(q), dev(kd), dev(vd)), lang)
        assert rx.launch_count() - n0 <= 2          # attention kernel (+ split merge)
        f = W.bf16_bits_to_f64
        ks, vs = ost.regions(layer, f(kd), f(vd))
        check_attention(host64(oa), OA.partitioned_attention(f(q), ks, vs))
        _check_lang(ost, layer, lq, ltk, ltv, lln, host64(ol))
        # The action view is the same as the single-request call.
        single = host64(cache.attend_suffix(layer, dev(q), dev(kd), dev(vd)))
        check_attention(host64(oa), single)
    assert cache.check_device_error() == 0
    cache.close()


@pytest.mark.parametrize("lens", [[0] * 16, [32] * 16, [0, 32, 1, 31] * 4])
def test_tail_length_edges(rx, lens):
    wl = W.WORKLOADS["c5"]
    seed = 32
    cache, ost = _setup(rx, wl, seed, 3)
    lq, ltk, ltv, lln, lang = _lang(wl, seed, 0, 0, 1, lens)
    _, ol = cache.attend_batch(1, None, lang)
    _check_lang(ost, 1, lq, ltk, ltv, lln, host64(ol))
    cache.close()


def test_tails_grow_on_the_device(rx):
    """Tail lengths are read on the device: rewriting them in place changes
    what each stream attends to without any host-side re-encoding."""
    import torch
    wl = W.WORKLOADS["c5"]
    seed = 33
    cache, ost = _setup(rx, wl, seed, 2)
    lq, ltk, ltv, lln, lang = _lang(wl, seed, 0, 0, 0, [3] * 16)
    out = torch.empty((wl.n_lang, 1, wl.Hq, wl.D), dtype=torch.bfloat16, device="cuda")
    cache.attend_batch(0, None, lang, out_lang=out)
    _check_lang(ost, 0, lq, ltk, ltv, lln, host64(out))
    lang[3].copy_(torch.arange(16, dtype=torch.int32, device="cuda"))
    cache.attend_batch(0, None, lang, out_lang=out)
    _check_lang(ost, 0, lq, ltk, ltv, np.arange(16), host64(out))
    cache.close()


def test_streams_with_several_query_tokens(rx):
    """T > 1 tokens per stream (e.g. a draft of several tokens)."""
    import torch
    wl = W.Workload("c5-multi", L=1, Hq=8, Hkv=1, D=256, P=64, N=2, F=256, S=51, steps=1,
                    ticks=1, d_model=1024, emb_dim=16, state_dim=16, hidden=512, n_lang=4,
                    tail_max=30, tail_cap=32)
    seed = 34
    cache = rx.Cache(wl.L, wl.Hq, wl.Hkv, wl.D, wl.P, wl.N, wl.F, wl.S, wl.tail_cap, 12)
    pk, pv = W.pinned_kv(wl, seed)
    cache.pin_prefix(dev(pk), dev(pv))
    ost = OracleStream(wl, seed)
    fk, fv = W.frame_kv(wl, seed, 0)
    cache.push_frame(dev(fk), dev(fv))
    ost.push(0)
    g = np.random.default_rng(5)
    q = W.to_bf16_bits(g.standard_normal((4, 3, wl.Hq, wl.D), dtype=np.float32))
    _, tk, tv, ln = W.lang_requests(wl, seed, 0, 0, 0)
    lang = (dev(q), dev(tk), dev(tv), torch.from_numpy(ln).cuda())
    _, ol = cache.attend_batch(0, None, lang)
    _check_lang(ost, 0, q, tk, tv, ln, host64(ol))
    cache.close()


def test_batch_argument_errors(rx):
    import torch
    wl = W.WORKLOADS["c5"]
    cache, _ = _setup(rx, wl, 35, 1)
    lq, ltk, ltv, lln, lang = _lang(wl, 35, 0, 0, 0)
    big = torch.zeros((17, 1, wl.Hq, wl.D), dtype=torch.bfloat16, device="cuda")
    big_tail = torch.zeros((17, wl.tail_cap, wl.Hkv, wl.D), dtype=torch.bfloat16, device="cuda")
    big_len = torch.zeros(17, dtype=torch.int32, device="cuda")
    with pytest.raises(rx.RxError) as e:      # 17 query tokens > max_req = 16
        cache.attend_batch(0, None, (big, big_tail, big_tail, big_len))
    assert e.value.status == -3
    with pytest.raises(ValueError):           # tails of 16 streams for 17 queries
        cache.attend_batch(0, None, (big, lang[1], lang[2], lang[3]))
    with pytest.raises(rx.RxError) as e:
        cache.attend_batch(wl.L, None, lang)
    assert e.value.status == -2
    cache.close()
