"""A stream tick captured once as a CUDA graph and replayed tick after tick.

"Reflex: Real-Time VLA Control through Streaming Inference", §III "System
architecture" (each tick enqueues the newest frame and evicts the oldest) and
Eq. (1).  The ring state lives on the device and the append kernel advances
it, so replaying one captured {push, attention over every layer and step}
must walk the window exactly as eager calls do.  After every replay each
output is compared with the oracle and layer 0's window with the oracle's
frames, bit for bit.
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


@pytest.mark.parametrize("spare", [0, 1])
def test_replayed_tick_matches_the_oracle(rx, spare):
    import torch
    wl = W.Workload("graph-3L", L=3, Hq=8, Hkv=1, D=256, P=48, N=4, F=256, S=51, steps=2, ticks=1,
                    d_model=128, emb_dim=16, state_dim=16, hidden=64)
    seed = 21
    f = W.bf16_bits_to_f64
    cache = rx.Cache(wl.L, wl.Hq, wl.Hkv, wl.D, wl.P, wl.N, wl.F, wl.S, spare_slot=spare)
    pk, pv = W.pinned_kv(wl, seed)
    cache.pin_prefix(dev(pk), dev(pv))
    ost = OracleStream(wl, seed)

    bf = dict(dtype=torch.bfloat16, device="cuda")
    fk = torch.empty((wl.L, wl.F, wl.Hkv, wl.D), **bf)
    fv = torch.empty_like(fk)
    q = torch.empty((wl.steps, wl.L, wl.S, wl.Hq, wl.D), **bf)
    kd = torch.empty((wl.steps, wl.L, wl.S, wl.Hkv, wl.D), **bf)
    vd = torch.empty_like(kd)
    o = torch.empty_like(q)
    s = torch.cuda.Stream()

    def load(t):   # tick t's inputs into the captured buffers, ordered on s
        a, b = W.frame_kv(wl, seed, t)
        fk.copy_(dev(a))
        fv.copy_(dev(b))
        for k in range(wl.steps):
            for l in range(wl.L):
                qq, kk, vv = W.suffix_qkv(wl, seed, t, k, l)
                q[k, l].copy_(dev(qq))
                kd[k, l].copy_(dev(kk))
                vd[k, l].copy_(dev(vv))

    def tick():
        cache.push_frame(fk, fv)
        for k in range(wl.steps):
            for l in range(wl.L):
                cache.attend_suffix(l, q[k, l], kd[k, l], vd[k, l], out=o[k, l])

    def check(t):
        ost.push(t)
        for k in range(wl.steps):
            for l in range(wl.L):
                qq, kk, vv = (f(a) for a in W.suffix_qkv(wl, seed, t, k, l))
                ks, vs = ost.regions(l, kk, vv)
                check_attention(host64(o[k, l]), OA.partitioned_attention(qq, ks, vs))
        kw, _ = cache.export_window(0)
        want = np.concatenate([fr[1][0] for fr in ost.window.window()])
        np.testing.assert_array_equal(host64(kw), want)

    with torch.cuda.stream(s):   # tick 0 eagerly (first launches set kernel attributes)
        load(0)
        tick()
    torch.cuda.synchronize()
    check(0)
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr, stream=s):
        tick()
    for t in range(1, 2 * wl.N + 2):
        with torch.cuda.stream(s):
            load(t)
            gr.replay()
        torch.cuda.synchronize()
        check(t)
    assert cache.debug_window() is not None
    assert cache.check_device_error() == 0
    cache.close()


def test_replayed_benchmark_tick_matches_the_oracle_stream(rx):
    """The benchmark's tick, captured once and replayed tick after tick: one
    gamma launch for every (layer, site, step), the frame push, then per step
    and layer one launch of the attention with the layer's two AdaRMSNorms
    (rx_attend_suffix_norms).  After every replay each of the three outputs
    of every (step, layer) is compared with the oracle's stream tick ("Reflex
    ...", §III Eq. (1) and Eq. (2)): the norms within the norm tolerance, the
    attention within the attention tolerance."""
    import torch
    from tests._util import check_norm
    wl = W.Workload("tick-2L", L=2, Hq=8, Hkv=1, D=256, P=64, N=3, F=256, S=51, steps=3, ticks=1,
                    d_model=1024, emb_dim=16, state_dim=16, hidden=512)
    seed = 22
    cache = rx.Cache(wl.L, wl.Hq, wl.Hkv, wl.D, wl.P, wl.N, wl.F, wl.S)
    pk, pv = W.pinned_kv(wl, seed)
    cache.pin_prefix(dev(pk), dev(pv))
    ost = OracleStream(wl, seed)
    bf = dict(dtype=torch.bfloat16, device="cuda")
    K, L = wl.steps, wl.L
    fk = torch.empty((L, wl.F, wl.Hkv, wl.D), **bf)
    fv = torch.empty_like(fk)
    q = torch.empty((K, L, wl.S, wl.Hq, wl.D), **bf)
    kd = torch.empty((K, L, wl.S, wl.Hkv, wl.D), **bf)
    vd = torch.empty_like(kd)
    x = torch.empty((K, L, 2, wl.S, wl.d_model), **bf)
    o = torch.empty_like(q)
    y = torch.empty_like(x)
    mlp = [W.mlp_weights(wl, seed, l, site) for l in range(L) for site in (0, 1)]
    W1, b1, W2, b2 = (torch.stack([dev(m[i]) for m in mlp]) for i in range(4))
    tk = torch.tensor(W.timesteps(wl), device="cuda")
    state = torch.empty((K, wl.state_dim), dtype=torch.float32, device="cuda")
    gamma = torch.empty((2 * L, K, wl.d_model), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()

    def load(t):
        a, b = W.frame_kv(wl, seed, t)
        fk.copy_(dev(a))
        fv.copy_(dev(b))
        state.copy_(torch.from_numpy(np.tile(W.robot_state(wl, seed, t), (K, 1))).cuda())
        for k in range(K):
            for l in range(L):
                qq, kk, vv = W.suffix_qkv(wl, seed, t, k, l)
                q[k, l].copy_(dev(qq))
                kd[k, l].copy_(dev(kk))
                vd[k, l].copy_(dev(vv))
                for site in (0, 1):
                    x[k, l, site].copy_(dev(W.norm_input(wl, seed, t, k, l, site)))

    def tick():
        rx.ada_gamma(tk, state, W1, b1, W2, b2, wl.emb_dim, out=gamma)
        cache.push_frame(fk, fv)
        for k in range(K):
            for l in range(L):
                cache.attend_suffix(l, q[k, l], kd[k, l], vd[k, l], out=o[k, l],
                                    norms=[(x[k, l, 0], gamma[2 * l, k], wl.eps, y[k, l, 0]),
                                           (x[k, l, 1], gamma[2 * l + 1, k], wl.eps, y[k, l, 1])])

    def check(t):
        want = ost.tick(t)
        for (k, l), (y0, att, y1) in want.items():
            check_norm(host64(y[k, l, 0]), y0)
            check_attention(host64(o[k, l]), att)
            check_norm(host64(y[k, l, 1]), y1)

    with torch.cuda.stream(s):   # tick 0 eagerly (first launches set kernel attributes)
        load(0)
        tick()
    torch.cuda.synchronize()
    check(0)
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr, stream=s):
        tick()
    for t in range(1, wl.N + 3):
        with torch.cuda.stream(s):
            load(t)
            gr.replay()
        torch.cuda.synchronize()
        check(t)
    assert cache.check_device_error() == 0
    cache.close()


@pytest.mark.parametrize("name", ["c3", "c4"])
def test_full_size_benchmark_tick_matches_the_oracle(rx, name):
    """The benchmark's tick at the workload's full size and in its launch
    configuration: one gamma launch for all 2L sites x K steps, the frame push
    into a full (wrapping) 32-frame window, then K x L launches of the
    attention with the layer's two AdaRMSNorms beside it, on the automatic
    partition (c3: clusters of 12 splits x 2 column shares merged on chip;
    c4: unclustered splits and the combine kernel).  The first
    tick runs eagerly, the next ones from one captured graph.  After each,
    every gamma value is compared with the oracle (Eq. (2)'s MLP, fp64), and
    for sampled (step, layer) pairs every row of both norm outputs and of the
    attention output ("Reflex ...", §III Eq. (1) and (2))."""
    import torch
    from tests._util import check_norm
    wl = W.WORKLOADS[name]
    seed = 23
    K, L = wl.steps, wl.L
    cache = rx.Cache(L, wl.Hq, wl.Hkv, wl.D, wl.P, wl.N, wl.F, wl.S)
    pk, pv = W.pinned_kv(wl, seed)
    cache.pin_prefix(dev(pk), dev(pv))
    ost = OracleStream(wl, seed)
    for t in range(wl.N):             # the window full before the ticks
        fk, fv = W.frame_kv(wl, seed, t)
        cache.push_frame(dev(fk), dev(fv))
        ost.push(t)
    bf = dict(dtype=torch.bfloat16, device="cuda")
    fk = torch.empty((L, wl.F, wl.Hkv, wl.D), **bf)
    fv = torch.empty_like(fk)
    q = torch.empty((K, L, wl.S, wl.Hq, wl.D), **bf)
    kd = torch.empty((K, L, wl.S, wl.Hkv, wl.D), **bf)
    vd = torch.empty_like(kd)
    x = torch.empty((K, L, 2, wl.S, wl.d_model), **bf)
    o = torch.empty_like(q)
    y = torch.empty_like(x)
    mlp = [W.mlp_weights(wl, seed, l, site) for l in range(L) for site in (0, 1)]
    W1, b1, W2, b2 = (torch.stack([dev(m[i]) for m in mlp]) for i in range(4))
    tk = torch.tensor(W.timesteps(wl), device="cuda")
    state = torch.empty((K, wl.state_dim), dtype=torch.float32, device="cuda")
    gamma = torch.empty((2 * L, K, wl.d_model), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()

    def load(t):
        a, b = W.frame_kv(wl, seed, t)
        fk.copy_(dev(a))
        fv.copy_(dev(b))
        state.copy_(torch.from_numpy(np.tile(W.robot_state(wl, seed, t), (K, 1))).cuda())
        for k in range(K):
            for l in range(L):
                qq, kk, vv = W.suffix_qkv(wl, seed, t, k, l)
                q[k, l].copy_(dev(qq))
                kd[k, l].copy_(dev(kk))
                vd[k, l].copy_(dev(vv))
                for site in (0, 1):
                    x[k, l, site].copy_(dev(W.norm_input(wl, seed, t, k, l, site)))

    def tick():
        rx.ada_gamma(tk, state, W1, b1, W2, b2, wl.emb_dim, out=gamma)
        cache.push_frame(fk, fv)
        for k in range(K):
            for l in range(L):
                cache.attend_suffix(l, q[k, l], kd[k, l], vd[k, l], out=o[k, l],
                                    norms=[(x[k, l, 0], gamma[2 * l, k], wl.eps, y[k, l, 0]),
                                           (x[k, l, 1], gamma[2 * l + 1, k], wl.eps, y[k, l, 1])])

    def check(t, pairs):
        ost.push(t)
        g = gamma.cpu().numpy().astype(np.float64)
        for k in range(K):
            for l in range(L):
                for site in (0, 1):
                    np.testing.assert_allclose(g[2 * l + site, k], ost.gamma(t, k, l, site), rtol=0, atol=1e-4)
        for k, l in pairs:
            check_norm(host64(y[k, l, 0]), ost.norm(t, k, l, 0))
            ref = ost.attend(t, k, l)
            # c4's outlier entries (x20): the bounds scale with the output magnitude.
            scale = max(1.0, float(np.abs(ref).max())) if wl.outlier_frac > 0 else 1.0
            check_attention(host64(o[k, l]), ref, scale)
            check_norm(host64(y[k, l, 1]), ost.norm(t, k, l, 1))

    t0 = wl.N
    with torch.cuda.stream(s):   # first tick eagerly (first launches set kernel attributes)
        load(t0)
        tick()
    torch.cuda.synchronize()
    check(t0, [(0, 0), (K - 1, L - 1)])
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr, stream=s):
        tick()
    for t, pairs in ((t0 + 1, [(K // 2, L // 2), (1, L - 2)]), (t0 + 2, [(K - 1, 0)])):
        with torch.cuda.stream(s):
            load(t)
            gr.replay()
        torch.cuda.synchronize()
        check(t, pairs)
    assert cache.check_device_error() == 0
    cache.close()


def test_full_size_batch_tick_matches_the_oracle(rx):
    """c5's benchmark tick at full size: the gamma launch, the push, then per
    step and layer one shared-cache launch (the 51-token action suffix and 16
    one-token language streams with private tails over the same cache,
    "OxyGen ...", §"Core method") with the layer's two AdaRMSNorms beside it.
    The first tick runs eagerly, the next from one captured graph; every
    gamma and, for sampled (step, layer) pairs, every row of the norms, of the
    action output and of each stream's output is compared with the oracle."""
    import torch
    from tests._util import check_norm
    wl = W.WORKLOADS["c5"]
    seed = 24
    K, L, B = wl.steps, wl.L, wl.n_lang
    f = W.bf16_bits_to_f64
    cache = rx.Cache(L, wl.Hq, wl.Hkv, wl.D, wl.P, wl.N, wl.F, wl.S, wl.tail_cap, B)
    pk, pv = W.pinned_kv(wl, seed)
    cache.pin_prefix(dev(pk), dev(pv))
    ost = OracleStream(wl, seed)
    for t in range(wl.N):
        a, b = W.frame_kv(wl, seed, t)
        cache.push_frame(dev(a), dev(b))
        ost.push(t)
    bf = dict(dtype=torch.bfloat16, device="cuda")
    fk = torch.empty((L, wl.F, wl.Hkv, wl.D), **bf)
    fv = torch.empty_like(fk)
    q = torch.empty((K, L, wl.S, wl.Hq, wl.D), **bf)
    kd = torch.empty((K, L, wl.S, wl.Hkv, wl.D), **bf)
    vd = torch.empty_like(kd)
    x = torch.empty((K, L, 2, wl.S, wl.d_model), **bf)
    o = torch.empty_like(q)
    y = torch.empty_like(x)
    ql = torch.empty((K, L, B, 1, wl.Hq, wl.D), **bf)
    ol = torch.empty_like(ql)
    tk_ = torch.empty((L, B, wl.tail_cap, wl.Hkv, wl.D), **bf)
    tv_ = torch.empty_like(tk_)
    tl = torch.empty((L, B), dtype=torch.int32, device="cuda")
    mlp = [W.mlp_weights(wl, seed, l, site) for l in range(L) for site in (0, 1)]
    W1, b1, W2, b2 = (torch.stack([dev(m[i]) for m in mlp]) for i in range(4))
    tk = torch.tensor(W.timesteps(wl), device="cuda")
    state = torch.empty((K, wl.state_dim), dtype=torch.float32, device="cuda")
    gamma = torch.empty((2 * L, K, wl.d_model), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    host = {}

    def load(t):
        a, b = W.frame_kv(wl, seed, t)
        fk.copy_(dev(a))
        fv.copy_(dev(b))
        state.copy_(torch.from_numpy(np.tile(W.robot_state(wl, seed, t), (K, 1))).cuda())
        for l in range(L):
            for k in range(K):
                qq, kk, vv = W.suffix_qkv(wl, seed, t, k, l)
                q[k, l].copy_(dev(qq))
                kd[k, l].copy_(dev(kk))
                vd[k, l].copy_(dev(vv))
                for site in (0, 1):
                    x[k, l, site].copy_(dev(W.norm_input(wl, seed, t, k, l, site)))
                lq, ltk, ltv, lln = W.lang_requests(wl, seed, t, k, l)
                ql[k, l].copy_(dev(lq))
                host[(t, k, l)] = (qq, kk, vv, lq, ltk, ltv, lln)
                if k == 0:   # a stream's tail depends on the tick and layer only
                    tk_[l].copy_(dev(ltk))
                    tv_[l].copy_(dev(ltv))
                    tl[l].copy_(torch.from_numpy(lln).cuda())

    def tick():
        rx.ada_gamma(tk, state, W1, b1, W2, b2, wl.emb_dim, out=gamma)
        cache.push_frame(fk, fv)
        for k in range(K):
            for l in range(L):
                cache.attend_batch(l, (q[k, l], kd[k, l], vd[k, l]), (ql[k, l], tk_[l], tv_[l], tl[l]),
                                   out_act=o[k, l], out_lang=ol[k, l],
                                   norms=[(x[k, l, 0], gamma[2 * l, k], wl.eps, y[k, l, 0]),
                                          (x[k, l, 1], gamma[2 * l + 1, k], wl.eps, y[k, l, 1])])

    def check(t, pairs):
        ost.push(t)
        g = gamma.cpu().numpy().astype(np.float64)
        for k in range(K):
            for l in range(L):
                for site in (0, 1):
                    np.testing.assert_allclose(g[2 * l + site, k], ost.gamma(t, k, l, site), rtol=0, atol=1e-4)
        for k, l in pairs:
            qq, kk, vv, lq, ltk, ltv, lln = host[(t, k, l)]
            check_norm(host64(y[k, l, 0]), ost.norm(t, k, l, 0))
            check_norm(host64(y[k, l, 1]), ost.norm(t, k, l, 1))
            ks, vs = ost.regions(l, f(kk), f(vv))
            check_attention(host64(o[k, l]), OA.partitioned_attention(f(qq), ks, vs))
            reqs = [(f(lq[b]), f(ltk[b, :lln[b]]), f(ltv[b, :lln[b]])) for b in range(B)]
            got = host64(ol[k, l])
            for b, ref in enumerate(OA.shared_cache_attention(ks[:-1], vs[:-1], reqs)):
                check_attention(got[b], ref)

    t0 = wl.N
    with torch.cuda.stream(s):
        load(t0)
        tick()
    torch.cuda.synchronize()
    check(t0, [(0, 0), (K - 1, L - 1)])
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr, stream=s):
        tick()
    with torch.cuda.stream(s):
        load(t0 + 1)
        gr.replay()
    torch.cuda.synchronize()
    check(t0 + 1, [(K // 2, L // 2)])
    assert cache.check_device_error() == 0
    cache.close()
