"""Small, self-contained cases of the hot-path kernels for profilers.

--op attention builds the store of one named workload with only a few layers
(the K/V of a layer, the suffix and the partition are those of the full
workload), fills the window, and issues a handful of attention calls, so that
one launch of the attention kernel can be captured in isolation:

    python -m partitioned_kv_cache_gb300.attn_case --workload c4 --layers 2 --calls 6

--op gamma issues the gamma-MLP launch of one tick of the workload (all 2L
norm sites x K steps) a few times, each on its own weight set:

    python -m partitioned_kv_cache_gb300.attn_case --workload c3 --op gamma --calls 4

Inputs are seeded random bf16; nothing is checked here (the tests compare with
the oracle).
"""
import argparse

import torch

from . import rx
from . import workload as W


def main(argv=None) -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="c3", choices=sorted(W.WORKLOADS))
    ap.add_argument("--layers", type=int, default=2)
    ap.add_argument("--calls", type=int, default=6)
    ap.add_argument("--op", default="attention", choices=["attention", "gamma"])
    a = ap.parse_args(argv)
    wl = W.WORKLOADS[a.workload]
    L = max(1, min(a.layers, wl.L))
    g = torch.Generator(device="cuda")
    g.manual_seed(0)

    def r(*shape, scale=1.0):
        return (torch.randn(*shape, generator=g, device="cuda") * scale).to(torch.bfloat16)

    if a.op == "gamma":
        n_sets = 2 * wl.L
        t = torch.tensor(W.timesteps(wl), device="cuda")
        state = torch.rand(wl.steps, wl.state_dim, generator=g, device="cuda")
        out = torch.empty((n_sets, wl.steps, wl.d_model), dtype=torch.float32, device="cuda")
        for _ in range(a.calls):
            rx.ada_gamma(t, state, r(n_sets, wl.hidden, wl.cond_dim, scale=0.02), r(n_sets, wl.hidden, scale=0.02),
                         r(n_sets, wl.d_model, wl.hidden, scale=0.02), r(n_sets, wl.d_model, scale=0.02),
                         wl.emb_dim, out=out)
        torch.cuda.synchronize()
        if not bool(torch.isfinite(out).all()):
            raise SystemExit("non-finite gamma")
        print("%s: %d gamma launches of %d sets x %d steps" % (wl.name, a.calls, n_sets, wl.steps))
        return

    cache = rx.Cache(L, wl.Hq, wl.Hkv, wl.D, wl.P, wl.N, wl.F, wl.S)
    cache.pin_prefix(r(L, wl.P, wl.Hkv, wl.D), r(L, wl.P, wl.Hkv, wl.D))
    for _ in range(wl.N):
        cache.push_frame(r(L, wl.F, wl.Hkv, wl.D), r(L, wl.F, wl.Hkv, wl.D))
    q = r(wl.S, wl.Hq, wl.D)
    kd = r(wl.S, wl.Hkv, wl.D)
    vd = r(wl.S, wl.Hkv, wl.D)
    o = torch.empty_like(q)
    for i in range(a.calls):
        cache.attend_suffix(i % L, q, kd, vd, out=o)
    torch.cuda.synchronize()
    if cache.check_device_error() != 0:
        raise SystemExit("a kernel reported a device-side timeout")
    cache.close()
    print("%s: %d attention calls on %d layers" % (wl.name, a.calls, L))


if __name__ == "__main__":
    main()
