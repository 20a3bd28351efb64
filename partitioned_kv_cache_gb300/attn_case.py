"""Small, self-contained cases of the hot-path kernels for profilers.

--op attention builds the store of one named workload with only a few layers
(the K/V of a layer, the suffix and the partition are those of the full
workload), fills the window, and issues a handful of attention calls, so that
one launch of the attention kernel can be captured in isolation:

    python -m partitioned_kv_cache_gb300.attn_case --workload c4 --layers 2 --calls 6

(--suffix replaces the workload's suffix length, e.g. 1024 query tokens;
--splits and --dparts force the partition, 0 = automatic; --norms runs the
layer's two AdaRMSNorms of the suffix in the same launch, as the benchmark's
tick does.)

--op batch runs the shared-cache launch of the workload (the action suffix
plus its language streams, each with a private tail of U{0..tail_max} keys):

    python -m partitioned_kv_cache_gb300.attn_case --workload c5 --op batch --layers 2 --calls 6

--op gamma issues the gamma-MLP launch of one tick of the workload (all 2L
norm sites x K steps) a few times, each on its own weight set:

    python -m partitioned_kv_cache_gb300.attn_case --workload c3 --op gamma --calls 4

--op push pushes distinct frames into a store of the workload's layers
(--frame-mult scales the frame's tokens), and --op norm runs AdaRMSNorm over
--rows rows of the model width (default: the suffix), each call on its own
input:

    python -m partitioned_kv_cache_gb300.attn_case --workload c3 --op push --layers 18 --calls 6
    python -m partitioned_kv_cache_gb300.attn_case --workload c3 --op norm --calls 6

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
    ap.add_argument("--op", default="attention", choices=["attention", "batch", "gamma", "push", "norm"])
    ap.add_argument("--norms", action="store_true")
    ap.add_argument("--frame-mult", type=int, default=1)
    ap.add_argument("--rows", type=int, default=0)
    ap.add_argument("--suffix", type=int, default=0)
    ap.add_argument("--splits", type=int, default=0)
    ap.add_argument("--dparts", type=int, default=0)
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

    if a.op == "push":
        F = wl.F * max(1, a.frame_mult)
        cache = rx.Cache(L, wl.Hq, wl.Hkv, wl.D, wl.P, wl.N, F, wl.S)
        for _ in range(a.calls):
            cache.push_frame(r(L, F, wl.Hkv, wl.D), r(L, F, wl.Hkv, wl.D))
        torch.cuda.synchronize()
        if cache.check_device_error() != 0:
            raise SystemExit("a kernel reported a device-side timeout")
        cache.close()
        print("%s: %d pushes of %d tokens x %d layers" % (wl.name, a.calls, F, L))
        return
    if a.op == "norm":
        rows = a.rows if a.rows > 0 else wl.S
        gamma = (1.0 + 0.1 * torch.randn(wl.d_model, generator=g, device="cuda")).float()
        ys = []
        for _ in range(a.calls):
            ys.append(rx.adarmsnorm(r(rows, wl.d_model), gamma, wl.eps))
        torch.cuda.synchronize()
        if not all(bool(torch.isfinite(y.float()).all()) for y in ys):
            raise SystemExit("non-finite norm output")
        print("%s: %d norms of %d x %d" % (wl.name, a.calls, rows, wl.d_model))
        return

    S = a.suffix if a.suffix > 0 else wl.S
    B = wl.n_lang if a.op == "batch" else 0
    cache = rx.Cache(L, wl.Hq, wl.Hkv, wl.D, wl.P, wl.N, wl.F, S, wl.tail_cap if B else 0, B)
    cache.set_attn_splits(a.splits)
    cache.set_attn_dparts(a.dparts)
    cache.pin_prefix(r(L, wl.P, wl.Hkv, wl.D), r(L, wl.P, wl.Hkv, wl.D))
    for _ in range(wl.N):
        cache.push_frame(r(L, wl.F, wl.Hkv, wl.D), r(L, wl.F, wl.Hkv, wl.D))
    q = r(S, wl.Hq, wl.D)
    kd = r(S, wl.Hkv, wl.D)
    vd = r(S, wl.Hkv, wl.D)
    o = torch.empty_like(q)
    norms = None
    if a.norms:
        gamma = (1.0 + 0.1 * torch.randn(2, wl.d_model, generator=g, device="cuda")).float()
        x = r(2, S, wl.d_model)
        y = torch.empty_like(x)
        norms = [(x[0], gamma[0], wl.eps, y[0]), (x[1], gamma[1], wl.eps, y[1])]
    if B:
        lq = r(B, 1, wl.Hq, wl.D)
        lo = torch.empty_like(lq)
        tails = (r(B, wl.tail_cap, wl.Hkv, wl.D), r(B, wl.tail_cap, wl.Hkv, wl.D))
        lens = torch.randint(0, wl.tail_max + 1, (B,), generator=g, device="cuda", dtype=torch.int32)
    for i in range(a.calls):
        if B:
            cache.attend_batch(i % L, (q, kd, vd), (lq, tails[0], tails[1], lens), out_act=o, out_lang=lo,
                               norms=norms)
        else:
            cache.attend_suffix(i % L, q, kd, vd, out=o, norms=norms)
    torch.cuda.synchronize()
    if cache.check_device_error() != 0:
        raise SystemExit("a kernel reported a device-side timeout")
    cache.close()
    print("%s: %d %s calls on %d layers%s" % (wl.name, a.calls, "shared-cache" if B else "attention", L,
                                             " with two norm jobs each" if norms else ""))


if __name__ == "__main__":
    main()
