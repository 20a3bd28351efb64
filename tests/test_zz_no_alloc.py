"""The allocation-free attention entry point (rx_attend_regions_static).

It serves callers that cannot allocate device memory: a real-time control
loop that must never stall on cudaMalloc, an embedded runtime with a fixed
memory budget, or a plugin inside a framework that owns the allocator.  The
same attention kernels run with their scratch in a fixed array inside the
library.  Through the C ABI, every case below checks two calls in a row
against the fp64 oracle ("Reflex: Real-Time VLA Control through Streaming
Inference", §III Eq. (1) over [pinned; window; dynamic]) within the attention
tolerance the other tests use.  It also checks that the calls leave the
device's free memory unchanged.  The file is named so that pytest collects
it last.
"""
import numpy as np
import pytest

from oracle import attention as OA
from partitioned_kv_cache_gb300 import workload as W
from tests._util import check_attention, dev, ensure_built, few_keys_scale, host64

pytestmark = pytest.mark.gpu

# (S, Hq, Hkv, D, P, W, n_dyn): the single-layer benchmark shape (whose
# 408 query rows leave room for 30 of the 64 splits in the scratch), the
# long-history store's 8448 cached keys (27 key splits merged by the combine
# kernel, their partials in the fixed scratch), empty
# regions, a window that is not a multiple of 64 tokens, G of 1 and 2,
# D of 64 and 128, and a 1024-token suffix whose 8192 rows leave room for one
# split only.
CASES = [
    (51, 8, 1, 256, 48, 1024, 51),
    (51, 8, 1, 256, 256, 8192, 51),
    (51, 8, 1, 256, 0, 1024, 51),
    (51, 8, 1, 256, 48, 0, 51),
    (51, 8, 1, 256, 48, 1024, 0),
    (20, 4, 2, 128, 40, 100, 20),
    (33, 2, 2, 64, 17, 300, 33),
    (9, 1, 1, 64, 0, 257, 9),
    (1024, 8, 1, 256, 48, 1024, 64),
]


def _draw(seed, call, S, Hq, Hkv, D, P, Wn, n_dyn):
    g = W.rng(seed, "q", call, S, D)
    bits = lambda *shape: W.to_bf16_bits(g.standard_normal(shape, dtype=np.float32))
    return (bits(S, Hq, D), bits(P, Hkv, D), bits(P, Hkv, D), bits(Wn, Hkv, D), bits(Wn, Hkv, D),
            bits(n_dyn, Hkv, D), bits(n_dyn, Hkv, D))


@pytest.mark.parametrize("case", CASES, ids=["S%d-Hq%d-Hkv%d-D%d-P%d-W%d-dyn%d" % c for c in CASES])
def test_static_entry_matches_the_oracle_on_two_calls(case):
    import torch
    ensure_built()
    from partitioned_kv_cache_gb300 import rx
    S, Hq, Hkv, D, P, Wn, n_dyn = case
    f = W.bf16_bits_to_f64
    calls = []
    for call in range(2):
        host = _draw(40 + call, call, *case)
        tens = [dev(a) if a.shape[0] else None for a in host]
        calls.append((host, tens))
    out = torch.empty((S, Hq, D), dtype=torch.bfloat16, device="cuda")
    # A first call loads the kernels (module loading may allocate); after it,
    # two more calls must leave the free device memory as it was.
    rx.attend_regions_static(*calls[0][1], out)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    results = []
    for host, tens in calls:
        rx.attend_regions_static(*tens, out)
        results.append(out.cpu())     # bf16 straight to the host: no device allocation here
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0, "the static entry point changed free device memory"
    for (host, _), res in zip(calls, results):
        got = host64(res)
        q, kp, vp, kw, vw, kd, vd = (f(a) for a in host)
        ref = OA.partitioned_attention(q, [kp, kw, kd], [vp, vw, vd])
        vmax = max(float(np.abs(v).max()) for v in (vp, vw, vd) if v.size)
        check_attention(got, ref, few_keys_scale(P + Wn + n_dyn, vmax))


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
