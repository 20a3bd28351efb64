"""The hot path's follow-on rows on the GPU: the block-causal variant of
Eq. 1, single-token tail append for cross-frame continuous batching, and
ring-state snapshot / restore."""
import numpy as np
import pytest

from oracle import attention as OA
from oracle.pipeline import OracleStream
from oracle.ring import FrameWindow
from partitioned_kv_cache_gb300 import workload as W
from tests._util import check_attention, dev, ensure_built, host64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rx():
    ensure_built()
    from partitioned_kv_cache_gb300 import rx as m
    return m


def _stream_cache(rx, wl, seed, pushes):
    cache = rx.Cache(wl.L, wl.Hq, wl.Hkv, wl.D, wl.P, wl.N, wl.F, wl.S, wl.tail_cap, wl.n_lang)
    pk, pv = W.pinned_kv(wl, seed)
    cache.pin_prefix(dev(pk), dev(pv))
    ost = OracleStream(wl, seed)
    for t in range(pushes):
        fk, fv = W.frame_kv(wl, seed, t)
        cache.push_frame(dev(fk), dev(fv))
        ost.push(t)
    return cache, ost


@pytest.mark.parametrize("name,n_state", [("c2", 1), ("c2", 0), ("c2", 51), ("c2", 17), ("c1", 3)])
def test_block_causal_suffix(rx, name, n_state):
    """State-block tokens see the cache and only the state block's own keys."""
    wl = W.WORKLOADS[name]
    seed = 41
    cache, ost = _stream_cache(rx, wl, seed, wl.N + 1)
    f = W.bf16_bits_to_f64
    for layer in range(wl.L):
        q, kd, vd = W.suffix_qkv(wl, seed, wl.N, 0, layer)
        got = host64(cache.attend_suffix(layer, dev(q), dev(kd), dev(vd), n_state=n_state))
        ks, vs = ost.regions(layer, f(kd), f(vd))
        check_attention(got, OA.block_causal_attention(f(q), ks, vs, n_state))
    cache.close()


@pytest.mark.parametrize("name", ["c3", "c4"])
def test_block_causal_suffix_at_full_size(rx, name):
    """The full-size stores with one state token, as the benchmark times the
    masked call: every row of the first and last layer after a full window
    (c4: 27 key splits merged by the combine kernel, the mask in the last
    split's dynamic tile).  c4's ×20 outlier keys make the output scale
    max|ref|, and both bounds are taken relative to it."""
    wl = W.WORKLOADS[name]
    seed = 43
    cache, ost = _stream_cache(rx, wl, seed, wl.N + 1)
    f = W.bf16_bits_to_f64
    for layer in (0, wl.L - 1):
        q, kd, vd = W.suffix_qkv(wl, seed, wl.N, 3, layer)
        got = host64(cache.attend_suffix(layer, dev(q), dev(kd), dev(vd), n_state=1))
        ks, vs = ost.regions(layer, f(kd), f(vd))
        ref = OA.block_causal_attention(f(q), ks, vs, 1)
        scale = max(1.0, float(np.abs(ref).max())) if wl.outlier_frac > 0 else 1.0
        check_attention(got, ref, scale)
    assert cache.check_device_error() == 0
    cache.close()


def test_tail_append_follows_the_host_model_and_reports_overflow(rx):
    import torch
    B, cap, Hkv, D = 5, 4, 1, 64
    kt = torch.zeros((B, cap, Hkv, D), dtype=torch.bfloat16, device="cuda")
    vt = torch.zeros_like(kt)
    ln = torch.zeros(B, dtype=torch.int32, device="cuda")
    ovf = torch.zeros(1, dtype=torch.int32, device="cuda")
    active = torch.tensor([1, 1, 0, 1, 1], dtype=torch.int32, device="cuda")
    model = [[] for _ in range(B)]
    for step in range(6):
        kn = torch.full((B, Hkv, D), 0.0, device="cuda")
        kn += torch.arange(B, device="cuda").view(B, 1, 1) * 16 + step   # exact small integers
        kn = kn.to(torch.bfloat16)
        rx.tail_append(kt, vt, ln, kn, -kn, active, ovf)
        for b in range(B):
            if active[b] and len(model[b]) < cap:
                model[b].append(b * 16 + step)
    torch.cuda.synchronize()
    assert ln.tolist() == [len(m) for m in model]
    assert int(ovf.item()) == 1          # streams hit their capacity
    for b in range(B):
        got = kt[b, :len(model[b]), 0, 0].float().tolist()
        assert got == [float(x) for x in model[b]]
        assert torch.equal(vt[b, :len(model[b])], -kt[b, :len(model[b])])


def test_continuous_batching_over_frames(rx):
    """OxyGen §"Core method": language streams decode k tokens per frame over a
    shared cache, appending their KV each step; finished streams are retired and
    their slot reused.  Every step's outputs match the oracle."""
    import torch
    wl = W.WORKLOADS["c5"]
    seed, layer, k_per_frame = 42, 3, 3
    cache, ost = _stream_cache(rx, wl, seed, 2)
    B, cap = wl.n_lang, wl.tail_cap
    g = np.random.default_rng(7)
    kt = torch.zeros((B, cap, wl.Hkv, wl.D), dtype=torch.bfloat16, device="cuda")
    vt = torch.zeros_like(kt)
    ln = torch.from_numpy(g.integers(0, 10, size=B).astype(np.int32)).cuda()
    host_tails = [[] for _ in range(B)]
    # pre-fill the tails with their initial lengths
    init = W.to_bf16_bits(g.standard_normal((B, cap, wl.Hkv, wl.D), dtype=np.float32))
    init_v = W.to_bf16_bits(g.standard_normal((B, cap, wl.Hkv, wl.D), dtype=np.float32))
    kt.copy_(dev(init)); vt.copy_(dev(init_v))
    for b in range(B):
        host_tails[b] = [(init[b, j], init_v[b, j]) for j in range(int(ln[b]))]
    f = W.bf16_bits_to_f64
    for frame in range(2):
        fk, fv = W.frame_kv(wl, seed, 100 + frame)
        cache.push_frame(dev(fk), dev(fv))
        ost.push(100 + frame)
        for step in range(k_per_frame):
            q = W.to_bf16_bits(g.standard_normal((B, 1, wl.Hq, wl.D), dtype=np.float32))
            _, out = cache.attend_batch(layer, None, (dev(q), kt, vt, ln))
            got = host64(out)
            ks, vs = ost.regions(layer, f(init[0, :0]), f(init_v[0, :0]))
            for b in range(B):
                tk = np.stack([t[0] for t in host_tails[b]]) if host_tails[b] else init[0, :0]
                tv = np.stack([t[1] for t in host_tails[b]]) if host_tails[b] else init_v[0, :0]
                ref = OA.shared_cache_attention(ks[:-1], vs[:-1], [(f(q[b]), f(tk), f(tv))])[0]
                check_attention(got[b], ref)
            # decode: append this step's new KV; retire streams that are full
            kn = W.to_bf16_bits(g.standard_normal((B, wl.Hkv, wl.D), dtype=np.float32))
            vn = W.to_bf16_bits(g.standard_normal((B, wl.Hkv, wl.D), dtype=np.float32))
            rx.tail_append(kt, vt, ln, dev(kn), dev(vn))
            for b in range(B):
                if len(host_tails[b]) < cap:
                    host_tails[b].append((kn[b], vn[b]))
        # end of frame: stream 0 finished (EOS) and its slot starts a new request
        ln[0] = 0
        host_tails[0] = []
    torch.cuda.synchronize()
    cache.close()


def test_snapshot_restore_reproduces_outputs_bit_exactly(rx):
    import torch
    wl = W.WORKLOADS["c2"]
    seed = 43
    cache, _ = _stream_cache(rx, wl, seed, 3)
    snap = cache.snapshot()
    state = cache.get_state()
    q, kd, vd = (dev(a) for a in W.suffix_qkv(wl, seed, 9, 0, 0))
    outs = []
    for t in (10, 11, 12):
        fk, fv = W.frame_kv(wl, seed, t)
        cache.push_frame(dev(fk), dev(fv))
        outs.append(cache.attend_suffix(0, q, kd, vd).clone())
    cache.restore(snap)
    assert cache.get_state() == state
    for i, t in enumerate((10, 11, 12)):
        fk, fv = W.frame_kv(wl, seed, t)
        ev = cache.push_frame(dev(fk), dev(fv))
        assert ev == (1 if 3 + i + 1 > wl.N else 0)
        assert torch.equal(cache.attend_suffix(0, q, kd, vd), outs[i])
    other = rx.Cache(wl.L, wl.Hq, wl.Hkv, wl.D, wl.P, wl.N + 1, wl.F, wl.S)
    with pytest.raises(rx.RxError):
        other.restore(snap)
    other.close()
    cache.close()
