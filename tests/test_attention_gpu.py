"""Partitioned attention on the GPU against the fp64 oracle.

"Reflex: Real-Time VLA Control through Streaming Inference", §III Eq. (1) and
Proposition A.1 / Table 4 (partitioned output equals full-batch attention).
Tolerance on unit-scale inputs: max-abs 1e-2, mean-abs 1e-3.  Full-size
workloads are checked on sampled suffix tokens that the oracle computes one by
one, in the launch configuration the benchmark uses.
"""
import numpy as np
import pytest

from oracle import attention as OA
from oracle.pipeline import OracleStream
from partitioned_kv_cache_gb300 import workload as W
from tests._util import check_attention, dev, ensure_built, few_keys_scale, host64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rx():
    ensure_built()
    from partitioned_kv_cache_gb300 import rx as m
    return m


def _make(rx, wl, seed, P=None):
    P = wl.P if P is None else P
    cache = rx.Cache(wl.L, wl.Hq, wl.Hkv, wl.D, max(wl.P, P), wl.N, wl.F, wl.S,
                     wl.tail_cap, wl.n_lang)
    pk, pv = W.pinned_kv(wl, seed, P)
    cache.pin_prefix(dev(pk), dev(pv))
    return cache


def _attend(cache, wl, seed, tick, step, layer, S=None):
    q, kd, vd = W.suffix_qkv(wl, seed, tick, step, layer, S)
    return cache.attend_suffix(layer, dev(q), dev(kd), dev(vd))


def _oracle_attend(ost, wl, seed, tick, step, layer, S=None, tokens=None):
    q, kd, vd = (W.bf16_bits_to_f64(a) for a in W.suffix_qkv(wl, seed, tick, step, layer, S))
    if tokens is not None:
        q = q[np.asarray(tokens)]
    ks, vs = ost.regions(layer, kd, vd)
    return OA.partitioned_attention(q, ks, vs)


@pytest.mark.parametrize("name,ticks,steps", [("c1", range(4), (0, 1, 2)),
                                              ("c2", (0, 1, 3, 4, 5), (0, 9))])
def test_stream_parity(rx, name, ticks, steps):
    wl = W.WORKLOADS[name]
    seed = 1
    cache = _make(rx, wl, seed)
    ost = OracleStream(wl, seed)
    done = -1
    for tick in ticks:
        while done < tick:
            done += 1
            fk, fv = W.frame_kv(wl, seed, done)
            cache.push_frame(dev(fk), dev(fv))
            ost.push(done)
        for k in steps:
            for layer in range(wl.L):
                got = host64(_attend(cache, wl, seed, tick, k, layer))
                check_attention(got, _oracle_attend(ost, wl, seed, tick, k, layer))
    assert cache.check_device_error() == 0
    cache.close()


def test_before_any_push_attends_pinned_and_dynamic_only(rx):
    wl = W.WORKLOADS["c2"]
    cache = _make(rx, wl, 2)
    ost = OracleStream(wl, 2)
    got = host64(_attend(cache, wl, 2, 0, 0, 0))
    check_attention(got, _oracle_attend(ost, wl, 2, 0, 0, 0))
    cache.close()


@pytest.mark.parametrize("splits", [1, 2, 3, 7, 16, 18, 0])
def test_split_count_does_not_change_the_result(rx, splits):
    wl = W.WORKLOADS["c2"]
    seed = 3
    cache = _make(rx, wl, seed)
    cache.set_attn_splits(splits)
    ost = OracleStream(wl, seed)
    for t in range(4):
        fk, fv = W.frame_kv(wl, seed, t)
        cache.push_frame(dev(fk), dev(fv))
        ost.push(t)
    got = host64(_attend(cache, wl, seed, 3, 2, 0))
    check_attention(got, _oracle_attend(ost, wl, seed, 3, 2, 0))
    cache.close()


@pytest.mark.parametrize("splits,dparts", [(12, 1), (12, 2), (12, 4), (1, 2), (1, 4), (3, 4),
                                           (20, 2), (20, 4), (0, 0)])
def test_output_column_split_does_not_change_the_result(rx, splits, dparts):
    """Every CTA of a (tile, split) computes the scores in full and the value
    product for its D/dparts columns: fused cluster merge (12, 3 splits),
    single split (1) and the combine kernel (20 splits, clamped to the 18
    key tiles) all agree with the oracle."""
    wl = W.WORKLOADS["c2"]
    seed = 9
    cache = _make(rx, wl, seed)
    cache.set_attn_splits(splits)
    cache.set_attn_dparts(dparts)
    ost = OracleStream(wl, seed)
    for t in range(wl.N + 1):
        fk, fv = W.frame_kv(wl, seed, t)
        cache.push_frame(dev(fk), dev(fv))
        ost.push(t)
    got = host64(_attend(cache, wl, seed, wl.N, 1, 0))
    check_attention(got, _oracle_attend(ost, wl, seed, wl.N, 1, 0))
    assert cache.check_device_error() == 0
    cache.close()


def test_dparts_argument_errors(rx):
    wl = W.WORKLOADS["c1"]   # D = 64: only one 64-column part
    cache = _make(rx, wl, 10)
    for bad in (-1, 3, 2, 4, 8):
        with pytest.raises(rx.RxError):
            cache.set_attn_dparts(bad)
    cache.set_attn_dparts(1)
    cache.set_attn_dparts(0)
    cache.close()


@pytest.mark.parametrize("S", [1, 7, 16, 17, 50, 51])
def test_ragged_suffix_lengths(rx, S):
    wl = W.WORKLOADS["c2"]
    seed = 4
    cache = _make(rx, wl, seed)
    ost = OracleStream(wl, seed)
    for t in range(2):
        fk, fv = W.frame_kv(wl, seed, t)
        cache.push_frame(dev(fk), dev(fv))
        ost.push(t)
    got = host64(_attend(cache, wl, seed, 1, 0, 0, S))
    check_attention(got, _oracle_attend(ost, wl, seed, 1, 0, 0, S))
    cache.close()


@pytest.mark.parametrize("shape", [
    dict(L=2, Hq=8, Hkv=2, D=128, P=40, N=3, F=100, S=20),    # GQA, D = 128, ragged tiles
    dict(L=1, Hq=4, Hkv=4, D=64, P=0, N=2, F=33, S=9),        # MHA, no pinned prefix
    dict(L=1, Hq=16, Hkv=1, D=256, P=1, N=1, F=1, S=3),       # one-token frame
    dict(L=1, Hq=128, Hkv=1, D=64, P=70, N=5, F=64, S=2),     # G = 128: one token per tile
])
def test_other_shapes(rx, shape):
    wl = W.Workload("custom", steps=1, ticks=1, d_model=128, emb_dim=16, state_dim=16,
                    hidden=64, **shape)
    seed = 5
    cache = _make(rx, wl, seed)
    ost = OracleStream(wl, seed)
    for t in range(wl.N + 1):
        fk, fv = W.frame_kv(wl, seed, t)
        cache.push_frame(dev(fk), dev(fv))
        ost.push(t)
        for layer in range(wl.L):
            got = host64(_attend(cache, wl, seed, t, 0, layer))
            ref = _oracle_attend(ost, wl, seed, t, 0, layer)
            # Rows with only a handful of keys get the rounding bound of the
            # path (few_keys_scale); every other row the unit-scale bounds.
            _, vs = ost.regions(layer, *(W.bf16_bits_to_f64(a) for a in W.suffix_qkv(wl, seed, t, 0, layer)[1:]))
            vmax = max(float(np.abs(v).max()) for v in vs if v.size)
            check_attention(got, ref, few_keys_scale(sum(v.shape[0] for v in vs), vmax))
    cache.close()


@pytest.mark.parametrize("name", ["c3", "c4"])
def test_full_size_every_row(rx, name):
    """Full workload (18 layers, wrapped window) in the benchmark's launch
    configuration: every suffix token and head of three layers, so every
    query tile of the launch (including the ragged last one) is compared."""
    wl = W.WORKLOADS[name]
    seed = 6
    cache = _make(rx, wl, seed)
    ost = OracleStream(wl, seed)
    last = wl.N + 2          # the window has wrapped
    for t in range(last + 1):
        fk, fv = W.frame_kv(wl, seed, t)
        cache.push_frame(dev(fk), dev(fv))
        ost.push(t)
    for layer in (0, 9, wl.L - 1):
        got = host64(_attend(cache, wl, seed, last, 3, layer))
        ref = _oracle_attend(ost, wl, seed, last, 3, layer)
        # Outlier entries (x20) make the values non-unit-scale: the bounds
        # scale with the output magnitude (bf16 rounding is relative).
        scale = max(1.0, float(np.abs(ref).max())) if wl.outlier_frac > 0 else 1.0
        check_attention(got, ref, scale)
    assert cache.check_device_error() == 0
    cache.close()


@pytest.mark.parametrize("splits,dparts", [(17, 1), (24, 2), (33, 1), (64, 1)])
def test_more_splits_than_a_cluster_combine_kernel(rx, splits, dparts):
    """More splits than one cluster holds: every split writes its partial to
    the exchange area and a separate kernel combines them, 16 splits per
    chunk with a running maximum (33 leaves a chunk with one live split)."""
    wl = W.WORKLOADS["c4"]
    seed = 12
    cache = _make(rx, wl, seed)
    cache.set_attn_splits(splits)
    cache.set_attn_dparts(dparts)
    ost = OracleStream(wl, seed)
    for t in range(wl.N + 1):
        fk, fv = W.frame_kv(wl, seed, t)
        cache.push_frame(dev(fk), dev(fv))
        ost.push(t)
    for layer in (0, wl.L - 1):
        got = host64(_attend(cache, wl, seed, wl.N, 4, layer))
        ref = _oracle_attend(ost, wl, seed, wl.N, 4, layer)
        check_attention(got, ref, max(1.0, float(np.abs(ref).max())))
    assert cache.check_device_error() == 0
    cache.close()


def test_repeated_calls_are_deterministic(rx):
    wl = W.WORKLOADS["c2"]
    cache = _make(rx, wl, 7)
    for t in range(5):
        fk, fv = W.frame_kv(wl, 7, t)
        cache.push_frame(dev(fk), dev(fv))
    a = _attend(cache, wl, 7, 4, 0, 0)
    b = _attend(cache, wl, 7, 4, 0, 0)
    import torch
    assert torch.equal(a, b)
    cache.close()


def test_argument_errors(rx):
    import torch
    wl = W.WORKLOADS["c1"]
    cache = _make(rx, wl, 8)
    q, kd, vd = (dev(a) for a in W.suffix_qkv(wl, 8, 0, 0, 0))
    with pytest.raises(rx.RxError) as e:
        cache.attend_suffix(1, q, kd, vd)
    assert e.value.status == -2
    big = torch.zeros((wl.S + 1, wl.Hq, wl.D), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(rx.RxError) as e:
        cache.attend_suffix(0, big, big[:, :1].contiguous(), big[:, :1].contiguous())
    assert e.value.status == -3
    with pytest.raises(rx.RxError):
        cache.set_attn_splits(10 ** 6)
    cache.close()


def test_two_caches_on_two_streams_run_concurrently(rx):
    """Each cache owns its exchange workspace: attention on two caches issued
    alternately on two CUDA streams (so their kernels overlap) gives each
    cache's own result."""
    import torch
    wl = W.WORKLOADS["c2"]
    caches, osts, streams = [], [], [torch.cuda.Stream(), torch.cuda.Stream()]
    for seed in (11, 12):
        c = _make(rx, wl, seed)
        o = OracleStream(wl, seed)
        for t in range(wl.N + 1):
            fk, fv = W.frame_kv(wl, seed, t)
            c.push_frame(dev(fk), dev(fv))
            o.push(t)
        caches.append(c)
        osts.append(o)
    torch.cuda.synchronize()
    inputs = [[tuple(dev(a) for a in W.suffix_qkv(wl, 11 + i, wl.N, k, 0)) for k in range(6)] for i in range(2)]
    outs = [[None] * 6 for _ in range(2)]
    for k in range(6):
        for i in range(2):
            with torch.cuda.stream(streams[i]):
                outs[i][k] = caches[i].attend_suffix(0, *inputs[i][k])
    torch.cuda.synchronize()
    for i in range(2):
        for k in range(6):
            check_attention(host64(outs[i][k]), _oracle_attend(osts[i], wl, 11 + i, wl.N, k, 0))
        assert caches[i].check_device_error() == 0
        caches[i].close()


@pytest.mark.parametrize("splits", [0, 16, 40])
def test_long_suffix_many_query_tiles(rx, splits):
    """A 1024-token suffix (8192 query rows, 64 query tiles): more clusters
    than fit at once (several waves), or the global-memory merge with 40
    splits.  Sampled tokens are checked against the oracle."""
    wl = W.Workload("long-suffix", L=1, Hq=8, Hkv=1, D=256, P=48, N=4, F=256, S=1024, steps=1, ticks=1,
                    d_model=128, emb_dim=16, state_dim=16, hidden=64)
    seed = 13
    cache = _make(rx, wl, seed)
    cache.set_attn_splits(splits)
    ost = OracleStream(wl, seed)
    for t in range(wl.N + 1):
        fk, fv = W.frame_kv(wl, seed, t)
        cache.push_frame(dev(fk), dev(fv))
        ost.push(t)
    tokens = [0, 1, 127, 128, 500, 511, 512, 1000, 1022, 1023]
    got = host64(_attend(cache, wl, seed, wl.N, 0, 0))[tokens]
    check_attention(got, _oracle_attend(ost, wl, seed, wl.N, 0, 0, tokens=tokens))
    assert cache.check_device_error() == 0
    cache.close()


@pytest.mark.parametrize("D,dparts", [(64, 1), (128, 1), (128, 2), (256, 1), (256, 2), (256, 4)])
def test_long_key_loop_separate_k_and_v_rings(rx, D, dparts):
    """Key loops longer than four tiles run the deeper build, whose K and V
    tiles go through separate rings: K slots by the score tile, V slots by
    the P V tile, the V ring cut into 2 to 8 slots by the column share.  One
    split walks 14 key tiles (wrapping each ring several times) against the
    oracle."""
    wl = W.Workload("long-loop-d%d" % D, L=1, Hq=4, Hkv=1, D=D, P=64, N=3, F=256, S=40, steps=1, ticks=1,
                    d_model=128, emb_dim=16, state_dim=16, hidden=64)
    seed = 23 + D + dparts
    cache = _make(rx, wl, seed)
    cache.set_attn_splits(1)
    cache.set_attn_dparts(dparts)
    ost = OracleStream(wl, seed)
    for t in range(wl.N + 1):
        fk, fv = W.frame_kv(wl, seed, t)
        cache.push_frame(dev(fk), dev(fv))
        ost.push(t)
    got = host64(_attend(cache, wl, seed, wl.N, 0, 0))
    check_attention(got, _oracle_attend(ost, wl, seed, wl.N, 0, 0))
    assert cache.check_device_error() == 0
    cache.close()


@pytest.mark.parametrize("D,dparts,splits,S", [(64, 1, 2, 250), (128, 2, 2, 250), (256, 1, 2, 250),
                                                (256, 2, 2, 250), (256, 1, 3, 250), (128, 1, 4, 250),
                                                (256, 2, 5, 120), (256, 1, 6, 120), (64, 1, 8, 120)])
def test_small_cluster_builds_long_suffix(rx, D, dparts, splits, S):
    """Long key loops merged by clusters of at most 2, 4 or 8 splits (a long
    suffix over a short window) run builds whose merge takes several rows
    per thread and pass.  250 or 120 tokens x 8 heads leave a ragged last
    query tile."""
    wl = W.Workload("small-cluster-d%d" % D, L=1, Hq=8, Hkv=1, D=D, P=64, N=8, F=256, S=S, steps=1, ticks=1,
                    d_model=128, emb_dim=16, state_dim=16, hidden=64)
    seed = 41 + D + dparts + splits
    cache = _make(rx, wl, seed)
    cache.set_attn_splits(splits)
    cache.set_attn_dparts(dparts)
    ost = OracleStream(wl, seed)
    for t in range(wl.N + 1):
        fk, fv = W.frame_kv(wl, seed, t)
        cache.push_frame(dev(fk), dev(fv))
        ost.push(t)
    got = host64(_attend(cache, wl, seed, wl.N, 0, 0))
    check_attention(got, _oracle_attend(ost, wl, seed, wl.N, 0, 0))
    assert cache.check_device_error() == 0
    cache.close()


def test_2048_token_suffix_one_split_per_tile(rx):
    """A 2048-token suffix over an 8-frame window (16384 query rows, 128 query
    tiles, 4160 keys): the automatic partition gives every query tile one CTA
    that walks all 65 key tiles and writes the output itself (no merge), the
    longest key loop the kernel runs.  Sampled tokens against the oracle."""
    wl = W.Workload("suffix-2048", L=1, Hq=8, Hkv=1, D=256, P=64, N=8, F=256, S=2048, steps=1, ticks=1,
                    d_model=128, emb_dim=16, state_dim=16, hidden=64)
    seed = 17
    cache = _make(rx, wl, seed)
    ost = OracleStream(wl, seed)
    for t in range(wl.N + 2):
        fk, fv = W.frame_kv(wl, seed, t)
        cache.push_frame(dev(fk), dev(fv))
        ost.push(t)
    tokens = [0, 15, 16, 1023, 1024, 2031, 2047]
    assert max(tokens) < wl.S
    got = host64(_attend(cache, wl, seed, wl.N + 1, 0, 0))[tokens]
    check_attention(got, _oracle_attend(ost, wl, seed, wl.N + 1, 0, 0, tokens=tokens))
    assert cache.check_device_error() == 0
    cache.close()


@pytest.mark.parametrize("splits", [1, 2, 0])
def test_running_maximum_rescale(rx, splits):
    """Online softmax with a maximum that jumps by more than 2^8 in the last
    key tile ("Reflex ...", §III Eq. (1): one softmax over all regions).  320
    keys score near 0 and one dynamic key scores ~2^10.6 above them, so the O
    accumulated over the first five tiles must be rescaled in place.  The old
    keys carry ~15% of the weight with values near +1 and the jumping key's
    value is -1, so a wrong rescale factor moves the output visibly.  One split
    walks every tile in order.  The output is of order 1, so the bound is the
    rounding of the path, not the unit-scale tolerance.  bf16 keeps 8
    significant bits (a rounding to nearest is within 2^-8 of the value): the
    output rounding (2^-8 |o|) plus bf16 P in the P V product (2^-8 max|v|).
    With two splits each split's partial is rounded to bf16 too, and the case
    is still held to that two-rounding bound."""
    D, G, S, P, N, F = 64, 8, 51, 64, 4, 64
    rng = np.random.default_rng(77)
    u = np.zeros(D, np.float32)
    u[3] = 1.0
    bits = lambda a: W.to_bf16_bits(np.ascontiguousarray(a, dtype=np.float32))
    near_one = lambda *shape: 1.0 + 0.1 * rng.standard_normal(shape)
    q = bits(np.broadcast_to(4.0 * u, (S, G, D)))
    pin_k = bits(rng.standard_normal((1, P, 1, D)) * 0.1)
    pin_v = bits(near_one(1, P, 1, D))
    frames = [(bits(rng.standard_normal((1, F, 1, D)) * 0.1), bits(near_one(1, F, 1, D))) for _ in range(N)]
    kd = rng.standard_normal((S, 1, D)).astype(np.float32) * 0.1
    kd[7, 0] = 15.0 * u
    vd = (0.1 * rng.standard_normal((S, 1, D))).astype(np.float32)
    vd[7, 0] = -1.0
    kd, vd = bits(kd), bits(vd)
    cache = rx.Cache(1, G, 1, D, P, N, F, S)
    cache.pin_prefix(dev(pin_k), dev(pin_v))
    for fk, fv in frames:
        cache.push_frame(dev(fk), dev(fv))
    cache.set_attn_splits(splits)
    got = host64(cache.attend_suffix(0, dev(q), dev(kd), dev(vd)))
    f = W.bf16_bits_to_f64
    ks = [f(pin_k)[0]] + [f(fk)[0] for fk, _ in frames] + [f(kd)]
    vs = [f(pin_v)[0]] + [f(fv)[0] for _, fv in frames] + [f(vd)]
    ref = OA.partitioned_attention(f(q), ks, vs)
    # the jump really is above the rescale threshold, and the old keys matter
    sc = np.einsum("d,kd->k", f(q)[0, 0], np.concatenate([k[:, 0] for k in ks])) / np.sqrt(D) / np.log(2)
    spike = len(sc) - S + 7
    assert sc[spike] - np.max(np.delete(sc, spike)) > 9.0
    w_old = np.exp2(sc[:len(sc) - S] - sc[spike]).sum() / np.exp2(sc - sc[spike]).sum()
    assert w_old > 0.1
    assert np.all(np.isfinite(got))
    vmax = max(float(np.abs(v).max()) for v in vs)
    bound = 2.0 ** -8 * (np.abs(ref) + vmax)
    err = np.abs(got - ref)
    assert np.all(err <= bound), "worst err / bound %.2f" % float(np.max(err / bound))
    assert cache.check_device_error() == 0
    cache.close()


@pytest.mark.parametrize("splits", [1, 0, 18])
def test_bounded_wait_gives_up_and_reports(rx, splits):
    """A barrier that never completes (the first K tile's barrier of CTA 0
    expects 16 bytes that never arrive): the kernel's waits give up after
    their time limit instead of hanging, the cache's error word reports it
    (bit 1), and the next call on the same cache matches the oracle.  With
    18 splits (more than a cluster) the timed-out CTA's partial is merged by
    the combine kernel with l = 0."""
    import time
    wl = W.WORKLOADS["c2"]
    seed = 31
    cache = _make(rx, wl, seed)
    cache.set_attn_splits(splits)
    ost = OracleStream(wl, seed)
    for t in range(wl.N):
        fk, fv = W.frame_kv(wl, seed, t)
        cache.push_frame(dev(fk), dev(fv))
        ost.push(t)
    with pytest.raises(rx.RxError):
        cache.debug_inject_timeout(15)
    cache.debug_inject_timeout(16)
    t0 = time.time()
    _attend(cache, wl, seed, wl.N - 1, 0, 0)
    assert cache.check_device_error() & 1
    assert time.time() - t0 < 30
    got = host64(_attend(cache, wl, seed, wl.N - 1, 0, 0))
    check_attention(got, _oracle_attend(ost, wl, seed, wl.N - 1, 0, 0))
    assert cache.check_device_error() == 0
    cache.close()
