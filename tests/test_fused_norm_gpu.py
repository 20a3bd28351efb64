"""AdaRMSNorm jobs run inside an attention launch (rx_attend_suffix_norms,
rx_attend_batch_norms).

"Reflex: Real-Time VLA Control through Streaming Inference", §III Eq. (1)
for the attention and Eq. (2) for the norms (AdaRMSNorm before the attention
and before the MLP of every layer, "Model components").  Each case checks
that the norm outputs equal rx_adarmsnorm's bit for bit and the fp64 oracle
within the norm tolerance (elementwise relative 1e-2, finite, inputs of
magnitude 1e-6..1e3).  It also checks that the attention output equals the
separate call's bit for bit and the oracle within the attention tolerance.
"""
import numpy as np
import pytest

from oracle import adarms as OR
from oracle import attention as OA
from oracle.pipeline import OracleStream
from partitioned_kv_cache_gb300 import workload as W
from tests._util import check_attention, check_norm, dev, ensure_built, host64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rx():
    ensure_built()
    from partitioned_kv_cache_gb300 import rx as m
    return m


def _store(rx, wl, seed, pushes):
    cache = rx.Cache(wl.L, wl.Hq, wl.Hkv, wl.D, wl.P, wl.N, wl.F, wl.S, wl.tail_cap, wl.n_lang)
    pk, pv = W.pinned_kv(wl, seed)
    cache.pin_prefix(dev(pk), dev(pv))
    ost = OracleStream(wl, seed)
    for t in range(pushes):
        fk, fv = W.frame_kv(wl, seed, t)
        cache.push_frame(dev(fk), dev(fv))
        ost.push(t)
    return cache, ost


def _jobs(seed, shapes):
    """Norm jobs of the given (rows, d): inputs from the magnitude sweep,
    gamma = 1 + N(0, 0.1)."""
    import torch
    jobs, host = [], []
    for i, (rows, d) in enumerate(shapes):
        x = W.magnitude_sweep(rows, d, seed + i) if rows else np.zeros((0, d), np.uint16)
        g = (1.0 + 0.1 * np.random.default_rng(seed + 100 + i).standard_normal(d)).astype(np.float32)
        y = torch.full((rows, d), float("nan"), dtype=torch.bfloat16, device="cuda")
        jobs.append((dev(x), torch.from_numpy(g).cuda(), 1e-6, y))
        host.append((x, g))
    return jobs, host


def _check_jobs(rx, jobs, host):
    for (x, g, eps, y), (xh, gh) in zip(jobs, host):
        if xh.shape[0] == 0:
            continue
        got = host64(y)
        check_norm(got, OR.ada_rms_norm(W.bf16_bits_to_f64(xh), gh.astype(np.float64), eps))
        import torch
        assert torch.equal(y, rx.adarmsnorm(x, g, eps)), "fused norm differs from rx_adarmsnorm"


@pytest.mark.parametrize("name,shapes,splits", [
    ("c3", [(51, 1024), (51, 1024)], 0),          # the benchmark's two norms per layer
    ("c4", [(51, 1024), (51, 1024)], 0),          # unclustered partition + combine kernel
    ("c2", [(700, 1024), (900, 1024)], 0),        # more rows than the launch has softmax warps
    ("c2", [(51, 128), (0, 1024)], 0),            # a narrow row, an empty job
    ("c2", [(37, 2048)], 0),                      # wide rows: the two-pass form
    ("c2", [(51, 1024), (51, 1024)], 1),          # one split: the CTAs write the output themselves
    ("c2", [(51, 1024), (51, 1024)], 17),         # more splits than a cluster: the combine kernel
])
def test_suffix_with_norm_jobs(rx, name, shapes, splits):
    import dataclasses
    wl = W.WORKLOADS[name]
    if wl.L > 2:
        wl = dataclasses.replace(wl, L=2)
    seed = 51
    cache, ost = _store(rx, wl, seed, wl.N + 1)
    cache.set_attn_splits(splits)
    f = W.bf16_bits_to_f64
    for layer in range(wl.L):
        q, kd, vd = W.suffix_qkv(wl, seed, wl.N, 0, layer)
        jobs, host = _jobs(seed + layer, shapes)
        got = cache.attend_suffix(layer, dev(q), dev(kd), dev(vd), norms=jobs)
        plain = cache.attend_suffix(layer, dev(q), dev(kd), dev(vd))
        import torch
        assert torch.equal(got, plain), "attention output changed by the norm jobs"
        ks, vs = ost.regions(layer, f(kd), f(vd))
        ref = OA.partitioned_attention(f(q), ks, vs)
        scale = max(1.0, float(np.abs(ref).max())) if wl.outlier_frac > 0 else 1.0
        check_attention(host64(got), ref, scale)
        _check_jobs(rx, jobs, host)
    assert cache.check_device_error() == 0
    cache.close()


def test_batch_with_norm_jobs(rx):
    """The shared-cache launch (action suffix + 16 language streams) with the
    layer's two norms."""
    import dataclasses
    import torch
    wl = dataclasses.replace(W.WORKLOADS["c5"], L=2)
    seed = 52
    cache, ost = _store(rx, wl, seed, wl.N + 2)
    f = W.bf16_bits_to_f64
    q, kd, vd = W.suffix_qkv(wl, seed, 0, 1, 1)
    lq, ltk, ltv, lln = W.lang_requests(wl, seed, 0, 1, 1)
    lang = (dev(lq), dev(ltk), dev(ltv), torch.from_numpy(lln).cuda())
    jobs, host = _jobs(seed, [(51, 1024), (51, 1024)])
    oa, ol = cache.attend_batch(1, (dev(q), dev(kd), dev(vd)), lang, norms=jobs)
    pa, pl = cache.attend_batch(1, (dev(q), dev(kd), dev(vd)), lang)
    assert torch.equal(oa, pa) and torch.equal(ol, pl)
    ks, vs = ost.regions(1, f(kd), f(vd))
    check_attention(host64(oa), OA.partitioned_attention(f(q), ks, vs))
    reqs = [(f(lq[b]), f(ltk[b, :lln[b]]), f(ltv[b, :lln[b]])) for b in range(wl.n_lang)]
    for b, ref in enumerate(OA.shared_cache_attention(ks[:-1], vs[:-1], reqs)):
        check_attention(host64(ol[b]), ref)
    _check_jobs(rx, jobs, host)
    # Norm jobs alone (no attention in the call) still run.
    jobs2, host2 = _jobs(seed + 7, [(20, 1024)])
    cache.attend_batch(0, None, None, norms=jobs2)
    _check_jobs(rx, jobs2, host2)
    # The language streams alone (their segment is the launch's only one)
    # with the layer's two norms.
    jobs3, host3 = _jobs(seed + 9, [(51, 1024), (51, 1024)])
    _, ol3 = cache.attend_batch(1, None, lang, norms=jobs3)
    _, pl3 = cache.attend_batch(1, None, lang)
    assert torch.equal(ol3, pl3)
    for b, ref in enumerate(OA.shared_cache_attention(ks[:-1], vs[:-1], reqs)):
        check_attention(host64(ol3[b]), ref)
    _check_jobs(rx, jobs3, host3)
    assert cache.check_device_error() == 0
    cache.close()


def test_norm_job_errors(rx):
    import torch
    wl = W.WORKLOADS["c1"]
    cache, _ = _store(rx, wl, 53, 1)
    q, kd, vd = (dev(a) for a in W.suffix_qkv(wl, 53, 0, 0, 0))
    x = torch.zeros((8, 128), dtype=torch.bfloat16, device="cuda")
    g = torch.ones(128, dtype=torch.float32, device="cuda")
    y = torch.empty_like(x)
    with pytest.raises(ValueError):                  # three jobs
        cache.attend_suffix(0, q, kd, vd, norms=[(x, g, 1e-6, y)] * 3)
    with pytest.raises(rx.RxError) as e:             # y overlaps x
        cache.attend_suffix(0, q, kd, vd, norms=[(x, g, 1e-6, x)])
    assert e.value.status == -1
    with pytest.raises(rx.RxError) as e:             # two jobs write the same rows
        cache.attend_suffix(0, q, kd, vd, norms=[(x, g, 1e-6, y), (x, g, 1e-6, y)])
    assert e.value.status == -1
    with pytest.raises(rx.RxError) as e:             # negative eps
        cache.attend_suffix(0, q, kd, vd, norms=[(x, g, -1.0, y)])
    assert e.value.status == -1
    # The norms run beside the attention of the same launch: a norm output on
    # the attention's q (8 x 2 x 64 = 8 x 128 values), or a norm input under
    # the attention's output, is refused on both entry points.
    with pytest.raises(rx.RxError) as e:
        cache.attend_suffix(0, q, kd, vd, norms=[(x, g, 1e-6, q.view(8, 128))])
    assert e.value.status == -1
    with pytest.raises(rx.RxError) as e:
        cache.attend_suffix(0, q, kd, vd, out=x.view(8, 2, 64), norms=[(x, g, 1e-6, y)])
    assert e.value.status == -1
    with pytest.raises(rx.RxError) as e:
        cache.attend_batch(0, (q, kd, vd), None, norms=[(x, g, 1e-6, q.view(8, 128))])
    assert e.value.status == -1
    assert cache.check_device_error() == 0
    cache.close()
