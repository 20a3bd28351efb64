#!/usr/bin/env python
"""Benchmark of the partitioned-attention hot path on GB300.

One benchmark step = one stream tick of the whole hot path:
  * gamma of AdaRMSNorm for every (layer, site, denoising step) of the tick
    (one launch: gamma depends only on t_k, the robot state and the weights),
  * ring append of the new frame into all layers' windows,
  * K denoising steps x L layers of {AdaRMSNorm, partitioned attention,
    AdaRMSNorm},
captured once as a CUDA graph and replayed.  value = denoise steps per second
(ticks x K / time).  Inputs are seeded synthetic tensors already resident in
HBM; two input pools larger than L2 alternate between ticks.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload c4]
    python bench.py --impl reference ...   # the CPU fp64 oracle, timed on host cores

Under torchrun (N > 1) every rank runs an independent replica (the method has
no cross-GPU exchange); value = all ranks' denoise steps / max rank time.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from partitioned_kv_cache_gb300 import workload as W  # noqa: E402

METRIC = "partitioned-attn denoise-steps/s; TFLOP/s & HBM GB/s as % of GB300 peak"
UNIT = "denoise-steps/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one attention
# call (its kernels' launches) from an ncu capture of the same workload.  It is
# reported only while the kernel's code (its source file and the headers it
# includes, comments and blank lines removed) still matches the code captured;
# otherwise the line carries null.
ATTN_TRAFFIC = {"sha256_16": "d9b10635b2fe4cd9", "workload": "c4", "bytes": 9.199104e6}
ATTN_SOURCES = ("partitioned_attn.cu", "partition.h", "rx_internal.h", "sm103_ptx.cuh", "norm_row.cuh")


def kernel_code_hash() -> str:
    import hashlib
    import re
    h = hashlib.sha256()
    for name in ATTN_SOURCES:
        text = open(os.path.join(ROOT, "partitioned_kv_cache_gb300", "csrc", name)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        lines = (re.sub(r"//.*$", "", ln).rstrip() for ln in text.splitlines())
        h.update("\n".join(ln for ln in lines if ln).encode())
    return h.hexdigest()[:16]


def attn_traffic(wl_key: str):
    try:
        sha = kernel_code_hash()
    except OSError:
        return None
    if sha == ATTN_TRAFFIC["sha256_16"] and wl_key == ATTN_TRAFFIC["workload"]:
        return ATTN_TRAFFIC["bytes"]
    return None


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def attn_flops(wl: W.Workload) -> float:
    """Algorithmic FLOPs of one attention call (full window): 4*Hq*S*Lk*D for
    the suffix, plus 4*Hq*(cached + mean tail)*D per language stream."""
    f = 4.0 * wl.Hq * wl.S * wl.keys_full * wl.D
    if wl.n_lang:
        f += wl.n_lang * 4.0 * wl.Hq * (wl.cached + wl.tail_max / 2.0) * wl.D
    return f


def describe(wl: W.Workload) -> str:
    d = ("%s: %d layers, %d q / %d kv heads, head_dim %d, pinned %d, window %d x %d, "
         "suffix %d, %d denoising steps per tick, AdaRMSNorm d=%d" %
         (wl.name, wl.L, wl.Hq, wl.Hkv, wl.D, wl.P, wl.N, wl.F, wl.S, wl.steps, wl.d_model))
    if wl.n_lang:
        d += ("; plus %d one-token language streams with private tails U{0..%d} in the same "
              "attention launch" % (wl.n_lang, wl.tail_max))
    return d


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu = gpu_id
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu, "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.close()
        with open(self.path) as f:
            lines = f.readlines()
        os.unlink(self.path)
        return summarise_clock_rows(lines)


def summarise_clock_rows(lines):
    """The clocks entry of the JSON line from nvidia-smi rows in
    ClockSampler.FIELDS order (csv, no header, no units): the median SM clock
    under load, the largest maximum clock seen, and every throttle reason
    that was active in any sample.  Rows that do not parse (an "[N/A]" clock,
    a short line) are skipped; no usable row gives None."""
    rows = []
    for line in lines:
        parts = [p.strip() for p in line.split(",")]
        if len(parts) < 9:
            continue
        try:
            rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
        except ValueError:
            continue
    if not rows:
        return None
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    reasons = sorted({names[i] for r in rows for i, v in enumerate(r[2]) if v.lower().startswith("active")})
    sm = sorted(r[0] for r in rows)
    return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": max(r[1] for r in rows),
            "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------
# CPU fp64 oracle (reference arm and cpu_baseline): timed as it stands
# ---------------------------------------------------------------------------
class OracleTimer:
    """Runs the oracle's functions, as they stand, over the workload and
    accumulates the seconds spent inside them.  The seeded inputs are drawn and
    converted to float64 outside the timed calls (on the GPU the inputs are
    resident before timing starts too).  One push per ``wl.steps`` denoising
    steps, the proportion of the stream tick."""

    def __init__(self, wl: W.Workload, seed: int):
        from oracle.pipeline import OracleStream
        self.wl, self.seed = wl, seed
        self.st = OracleStream(wl, seed)
        for t in range(wl.N):               # a full window before timing
            self.st.push(t)
        for l in range(wl.L):               # site weights drawn once, untimed
            for site in (0, 1):
                self.st.mlp(l, site)
        self.tick = wl.N - 1
        self.done = 0                       # denoising steps run
        self.seconds = 0.0

    def _timed(self, fn, *a):
        t0 = time.perf_counter()
        r = fn(*a)
        self.seconds += time.perf_counter() - t0
        return r

    def denoise_step(self):
        from oracle.adarms import ada_rms_norm, conditioning, gamma_mlp
        from oracle.attention import partitioned_attention, shared_cache_attention
        wl, seed, f = self.wl, self.seed, W.bf16_bits_to_f64
        k = self.done % wl.steps
        if k == 0:                           # the tick's frame enters the ring
            self.tick += 1
            fk, fv = W.frame_kv(wl, seed, self.tick)
            self._timed(self.st.window.push, (self.tick, f(fk), f(fv)))
        t = float(W.timesteps(wl)[k])
        state = W.robot_state(wl, seed, self.tick)
        for l in range(wl.L):
            for site in (0, 1):
                x = f(W.norm_input(wl, seed, self.tick, k, l, site))
                w = self.st.mlp(l, site)
                self._timed(lambda: ada_rms_norm(x, gamma_mlp(conditioning(t, state, wl.emb_dim), *w),
                                                 wl.eps))
                if site == 0:
                    q, kd, vd = (f(a) for a in W.suffix_qkv(wl, seed, self.tick, k, l))
                    ks, vs = self.st.regions(l, kd, vd)
                    self._timed(partitioned_attention, q, ks, vs)
                    if wl.n_lang:   # the language streams of the shared-cache workload
                        lq, tk, tv, ln = W.lang_requests(wl, seed, self.tick, k, l)
                        reqs = [(f(lq[b]), f(tk[b, :ln[b]]), f(tv[b, :ln[b]])) for b in range(wl.n_lang)]
                        self._timed(shared_cache_attention, ks[:-1], vs[:-1], reqs)
        self.done += 1


def oracle_sample(wl: W.Workload, seed: int, target_s: float, max_steps: int):
    """Time the oracle over whole denoising steps until about ``target_s``
    seconds of oracle work (at most ``max_steps``).  Returns (denoise-steps/s,
    oracle seconds, description)."""
    ot = OracleTimer(wl, seed)
    while ot.done < max_steps and (ot.done == 0 or ot.seconds < target_s):
        ot.denoise_step()
    pushes = (ot.done + wl.steps - 1) // wl.steps
    desc = ("%d frame push(es) + %d denoising steps x %d layers of %s {gamma MLP, AdaRMSNorm, attention, "
            "AdaRMSNorm}, oracle time only (seeded inputs drawn untimed)" % (pushes, ot.done, wl.L, wl.name))
    return ot.done / ot.seconds, ot.seconds, desc


def run_reference(args, wl):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    cores = os.cpu_count()
    ot = OracleTimer(wl, args.seed)
    for _ in range(args.warmup):
        ot.denoise_step()
    ot.seconds = 0.0
    for _ in range(args.steps):
        ot.denoise_step()
    dt = ot.seconds
    value = args.steps / dt
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": describe(wl)},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": "per step: one denoising step of all %d layers of %s (gamma MLP, "
                                       "AdaRMSNorm, attention, AdaRMSNorm), plus the frame push every "
                                       "%d steps; oracle time only (seeded inputs drawn untimed)"
                                       % (wl.L, wl.name, wl.steps)},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
def max_over_ranks(ms: float, world: int, device) -> float:
    """The slowest rank's time: barrier, then a MAX all-reduce (replicas run
    the same work, so the job is as fast as its slowest GPU)."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    dist.barrier()
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(units_per_rank: int, world: int, ms: float) -> float:
    """Whole-job units per second: every rank processed units_per_rank."""
    return units_per_rank * world / (ms / 1e3)


def attention_call_us(rx, wl, stream, randn_bf16, reps=3):
    """Per-call time of the workload's attention (every layer, every step of a
    tick, one CUDA graph) on a store with a full window; (us, FLOP per call)."""
    import torch
    L, S, Hq, Hkv, D, K, B = wl.L, wl.S, wl.Hq, wl.Hkv, wl.D, wl.steps, wl.n_lang
    cache = rx.Cache(L, Hq, Hkv, D, wl.P, wl.N, wl.F, S, wl.tail_cap, B)
    cache.pin_prefix(randn_bf16(L, wl.P, Hkv, D), randn_bf16(L, wl.P, Hkv, D))
    q = randn_bf16(K, L, S, Hq, D)
    kd = randn_bf16(K, L, S, Hkv, D)
    vd = randn_bf16(K, L, S, Hkv, D)
    o = torch.empty_like(q)
    if B:
        ql = randn_bf16(K, L, B, 1, Hq, D)
        ol = torch.empty_like(ql)
        tails_k = randn_bf16(L, B, wl.tail_cap, Hkv, D)
        tails_v = randn_bf16(L, B, wl.tail_cap, Hkv, D)
        tail_len = torch.randint(0, wl.tail_max + 1, (L, B), device=q.device, dtype=torch.int32)

    def calls():
        for k in range(K):
            for l in range(L):
                if B:
                    cache.attend_batch(l, (q[k, l], kd[k, l], vd[k, l]),
                                       (ql[k, l], tails_k[l], tails_v[l], tail_len[l]),
                                       out_act=o[k, l], out_lang=ol[k, l])
                else:
                    cache.attend_suffix(l, q[k, l], kd[k, l], vd[k, l], out=o[k, l])

    with torch.cuda.stream(stream):
        for t in range(wl.N):
            cache.push_frame(randn_bf16(L, wl.F, Hkv, D), randn_bf16(L, wl.F, Hkv, D))
        calls()
    torch.cuda.synchronize()
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr, stream=stream):
        calls()
    with torch.cuda.stream(stream):
        gr.replay()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            gr.replay()
        e1.record(stream)
    e1.synchronize()
    assert cache.check_device_error() == 0, "a kernel reported a device-side timeout"
    cache.close()
    return e0.elapsed_time(e1) * 1e3 / (reps * K * L), attn_flops(wl)


def graph_us(fn, stream, calls, reps=3):
    """Per-call time of fn() (`calls` library calls) captured as one CUDA
    graph after one eager run, replayed `reps` times between CUDA events."""
    import torch
    with torch.cuda.stream(stream):
        fn()
    torch.cuda.synchronize()
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr, stream=stream):
        fn()
    with torch.cuda.stream(stream):
        gr.replay()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            gr.replay()
        e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1) * 1e3 / (reps * calls)


def next_rows_kernels(rx, wl, stream, randn_bf16, peaks):
    """The rows beyond the tick, on the workload's shapes: the block-causal
    attention call, the push into a ring with a spare slot (the concurrent
    producer/consumer mode: the frame's tiles are written before the state is
    published), the language streams' one-token tail append, and a snapshot
    of the store."""
    import torch
    L, S, Hq, Hkv, D, K = wl.L, wl.S, wl.Hq, wl.Hkv, wl.D, wl.steps
    hbm = float(peaks["hbm_gbs"])
    out = {}
    cache = rx.Cache(L, Hq, Hkv, D, wl.P, wl.N, wl.F, S)
    cache.pin_prefix(randn_bf16(L, wl.P, Hkv, D), randn_bf16(L, wl.P, Hkv, D))
    with torch.cuda.stream(stream):
        for _ in range(wl.N):
            cache.push_frame(randn_bf16(L, wl.F, Hkv, D), randn_bf16(L, wl.F, Hkv, D))
    q = randn_bf16(K, L, S, Hq, D)
    kd = randn_bf16(K, L, S, Hkv, D)
    vd = randn_bf16(K, L, S, Hkv, D)
    o = torch.empty_like(q)

    def causal():
        for k in range(K):
            for l in range(L):
                cache.attend_suffix(l, q[k, l], kd[k, l], vd[k, l], out=o[k, l], n_state=1)

    us = graph_us(causal, stream, K * L)
    Lk = wl.P + wl.N * wl.F + S
    fl = 4.0 * Hq * D * ((S - 1) * Lk + (Lk - (S - 1)))   # the state token's row skips S-1 keys
    out["attention_block_causal"] = {
        "us_per_call": us, "flops_per_call": fl, "TFLOP/s": fl / us / 1e6,
        "frac_tensor": fl / us / 1e6 / float(peaks["bf16_tflops"]),
        "note": "Eq. 1 with the block-causal mask (the state token sees only its own dynamic key, the "
                "%d action tokens every key); %d calls per graph" % (S - 1, K * L)}
    nb = cache.snapshot_bytes()
    snap = torch.empty(nb, dtype=torch.uint8, device=q.device)
    with torch.cuda.stream(stream):
        cache.snapshot(snap)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(5):
            cache.snapshot(snap)
        e1.record(stream)
    e1.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / 5
    out["snapshot"] = {"us": us, "bytes": 2.0 * nb, "GB/s": 2.0 * nb / us / 1e3,
                       "frac_hbm": 2.0 * nb / us / 1e3 / hbm,
                       "note": "device copy of the store's regions and ring state (%.1f MB read + written)"
                               % (nb / 1e6)}
    assert cache.check_device_error() == 0, "a kernel reported a device-side timeout"
    cache.close()
    del q, kd, vd, o, snap

    sp = rx.Cache(L, Hq, Hkv, D, wl.P, wl.N, wl.F, S, spare_slot=1)
    fb = 2 * L * wl.F * Hkv * D * 2
    nfr = max(2, int(np.ceil(2 * 129e6 / fb)))
    pool = [(randn_bf16(L, wl.F, Hkv, D), randn_bf16(L, wl.F, Hkv, D)) for _ in range(nfr)]

    def pushes():
        for fr in pool:
            sp.push_frame(*fr)

    us = graph_us(pushes, stream, nfr)
    out["ring_append_spare_slot"] = {
        "us": us, "bytes": 2.0 * fb, "GB/s": 2.0 * fb / us / 1e3, "frac_hbm": 2.0 * fb / us / 1e3 / hbm,
        "note": "one push of all %d layers into a ring with a spare slot, graph of %d pushes over distinct "
                "frames (> 2x L2)" % (L, nfr)}
    assert sp.check_device_error() == 0, "a kernel reported a device-side timeout"
    sp.close()
    del pool

    B, cap = max(wl.n_lang, 16), max(wl.tail_cap, 32)
    tk = randn_bf16(L, B, cap, Hkv, D)
    tv = randn_bf16(L, B, cap, Hkv, D)
    tl = torch.zeros((L, B), dtype=torch.int32, device=tk.device)
    nk = randn_bf16(L, B, Hkv, D)
    nv = randn_bf16(L, B, Hkv, D)

    def appends():
        tl.zero_()
        for l in range(L):
            rx.tail_append(tk[l], tv[l], tl[l], nk[l], nv[l])

    us = graph_us(appends, stream, L)
    tb = 2.0 * 2 * B * Hkv * D * 2
    out["tail_append"] = {"us": us, "bytes": tb, "GB/s": tb / us / 1e3,
                          "note": "one token appended to each of %d language streams' tails (one call per "
                                  "layer, %d calls per graph): latency-bound" % (B, L)}
    return out


def run_ours(args, wl):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from partitioned_kv_cache_gb300 import rx

    peaks, peak_kind = load_peaks()
    g = torch.Generator(device=dev)
    g.manual_seed(args.seed * 1000 + rank)

    def randn_bf16(*shape, scale=1.0):
        return (torch.randn(*shape, generator=g, device=dev) * scale).to(torch.bfloat16)

    L, S, Hq, Hkv, D, K = wl.L, wl.S, wl.Hq, wl.Hkv, wl.D, wl.steps
    B = wl.n_lang
    cache = rx.Cache(L, Hq, Hkv, D, wl.P, wl.N, wl.F, S, wl.tail_cap, B)
    if args.splits:
        cache.set_attn_splits(args.splits)
    cache.pin_prefix(randn_bf16(L, wl.P, Hkv, D), randn_bf16(L, wl.P, Hkv, D))

    NSLOT = 2   # alternating input pools, each larger than L2
    frames = [(randn_bf16(L, wl.F, Hkv, D), randn_bf16(L, wl.F, Hkv, D)) for _ in range(NSLOT)]
    q = randn_bf16(NSLOT, K, L, S, Hq, D)
    kd = randn_bf16(NSLOT, K, L, S, Hkv, D)
    vd = randn_bf16(NSLOT, K, L, S, Hkv, D)
    x = randn_bf16(NSLOT, K, L, 2, S, wl.d_model)
    o = torch.empty_like(q)
    y = torch.empty_like(x)
    n_sets = 2 * L
    W1 = randn_bf16(n_sets, wl.hidden, wl.cond_dim, scale=0.02)
    b1 = randn_bf16(n_sets, wl.hidden, scale=0.02)
    W2 = randn_bf16(n_sets, wl.d_model, wl.hidden, scale=0.02)
    b2 = randn_bf16(n_sets, wl.d_model, scale=0.02)
    if B:   # language streams sharing the cache: 1 query token each, private tails
        ql = randn_bf16(NSLOT, K, L, B, 1, Hq, D)
        ol = torch.empty_like(ql)
        tails_k = randn_bf16(L, B, wl.tail_cap, Hkv, D)
        tails_v = randn_bf16(L, B, wl.tail_cap, Hkv, D)
        tail_len = torch.randint(0, wl.tail_max + 1, (L, B), generator=g, device=dev, dtype=torch.int32)
    tk = torch.tensor(W.timesteps(wl), device=dev)
    state = (torch.rand(NSLOT, K, wl.state_dim, generator=g, device=dev) * 2 - 1).contiguous()
    gamma = torch.empty((n_sets, K, wl.d_model), dtype=torch.float32, device=dev)
    for t in range(wl.N):   # fill the window before timing (steady state)
        cache.push_frame(*frames[t % NSLOT])

    def attend(slot, k, l, norms=None):
        if B:
            cache.attend_batch(l, (q[slot, k, l], kd[slot, k, l], vd[slot, k, l]),
                               (ql[slot, k, l], tails_k[l], tails_v[l], tail_len[l]),
                               out_act=o[slot, k, l], out_lang=ol[slot, k, l], norms=norms)
        else:
            cache.attend_suffix(l, q[slot, k, l], kd[slot, k, l], vd[slot, k, l], out=o[slot, k, l],
                                norms=norms)

    def tick(slot, fused=True):
        """One stream tick.  fused: each (step, layer) is one launch that runs
        the layer's two AdaRMSNorms beside its attention; otherwise the norms
        are launches of their own before and after the attention."""
        rx.ada_gamma(tk, state[slot], W1, b1, W2, b2, wl.emb_dim, out=gamma)
        cache.push_frame(*frames[slot])
        for k in range(K):
            for l in range(L):
                jobs = [(x[slot, k, l, 0], gamma[2 * l, k], wl.eps, y[slot, k, l, 0]),
                        (x[slot, k, l, 1], gamma[2 * l + 1, k], wl.eps, y[slot, k, l, 1])]
                if fused:
                    attend(slot, k, l, norms=jobs)
                else:
                    rx.adarmsnorm(*jobs[0][:3], out=jobs[0][3])
                    attend(slot, k, l)
                    rx.adarmsnorm(*jobs[1][:3], out=jobs[1][3])

    def attn_only(slot, fused=True):
        """Every (step, layer) launch of the tick without the gamma and the
        push: the attention with the layer's two norms beside it (fused), or
        the attention alone."""
        for k in range(K):
            for l in range(L):
                if fused:
                    attend(slot, k, l, norms=[(x[slot, k, l, 0], gamma[2 * l, k], wl.eps, y[slot, k, l, 0]),
                                              (x[slot, k, l, 1], gamma[2 * l + 1, k], wl.eps,
                                               y[slot, k, l, 1])])
                else:
                    attend(slot, k, l)

    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        for s in range(NSLOT):   # eager warm-up (first launches set kernel attributes)
            tick(s)
            tick(s, fused=False)
    torch.cuda.synchronize()
    graphs = []
    n0 = rx.launch_count()
    for s in range(NSLOT):
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            tick(s)
        graphs.append(gr)
    launches_per_tick = (rx.launch_count() - n0) // NSLOT
    # The tick's launches without the gamma and the push, one graph per input
    # slot, replayed alternately as the ticks are (the slots' inputs do not
    # stay in L2): with the norm jobs (the tick's launch) and without.
    a_graphs, p_graphs = [], []
    n1 = rx.launch_count()
    for s in range(NSLOT):
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            attn_only(s)
        a_graphs.append(gr)
    attn_kernels_per_call = (rx.launch_count() - n1) / (NSLOT * K * L)
    for s in range(NSLOT):
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            attn_only(s, fused=False)
        p_graphs.append(gr)
    torch.cuda.synchronize()

    for i in range(args.warmup):
        graphs[i % NSLOT].replay()
    torch.cuda.synchronize()
    assert cache.check_device_error() == 0, "a kernel reported a device-side timeout"

    # ---------------- timed region: K ticks ----------------
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        gpu_id = str(local)
    sampler = ClockSampler(gpu_id)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for i in range(args.steps):
            graphs[i % NSLOT].replay()
        e1.record(stream)
    e1.synchronize()
    torch.cuda.synchronize()
    clocks = sampler.stop()
    ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    value = replica_throughput(args.steps * K, world, ms)

    # ---------------- the same tick with the norms as launches of their own ----------------
    sep_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(sep_graph, stream=stream):
        tick(0, fused=False)
    with torch.cuda.stream(stream):
        sep_graph.replay()
        h0 = torch.cuda.Event(enable_timing=True)
        h1 = torch.cuda.Event(enable_timing=True)
        h0.record(stream)
        for _ in range(max(3, args.steps // 4)):
            sep_graph.replay()
        h1.record(stream)
    h1.synchronize()
    sep_ms = h0.elapsed_time(h1) / max(3, args.steps // 4)
    del sep_graph

    # ---------------- attention alone: per-launch time for the roofline ----------------
    reps = 2 * max(2, min(25, args.steps // 20))

    def per_call_us(grs):
        with torch.cuda.stream(stream):
            for gr in grs:
                gr.replay()
            b0 = torch.cuda.Event(enable_timing=True)
            b1 = torch.cuda.Event(enable_timing=True)
            b0.record(stream)
            for i in range(reps):
                grs[i % NSLOT].replay()
            b1.record(stream)
        b1.synchronize()
        return b0.elapsed_time(b1) * 1e3 / (reps * K * L)

    attn_us = per_call_us(a_graphs)
    plain_us = per_call_us(p_graphs)
    del a_graphs, p_graphs
    fl = attn_flops(wl)
    achieved = fl / (attn_us * 1e-6) / 1e12
    peak_tf = float(peaks["bf16_tflops"])

    # ---------------- append and AdaRMSNorm bandwidth (graph replays) ----------------
    kern = {}
    nfr = max(2, int(np.ceil(2 * 129e6 / (2 * L * wl.F * Hkv * D * 2))))
    pool = [(randn_bf16(L, wl.F, Hkv, D), randn_bf16(L, wl.F, Hkv, D)) for _ in range(nfr)]
    with torch.cuda.stream(stream):
        for fr in pool:
            cache.push_frame(*fr)
    torch.cuda.synchronize()
    p_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(p_graph, stream=stream):
        for fr in pool:
            cache.push_frame(*fr)
    with torch.cuda.stream(stream):
        p_graph.replay()
        b0 = torch.cuda.Event(enable_timing=True)
        b1 = torch.cuda.Event(enable_timing=True)
        b0.record(stream)
        for _ in range(3):
            p_graph.replay()
        b1.record(stream)
    b1.synchronize()
    app_us = b0.elapsed_time(b1) * 1e3 / (3 * nfr)
    app_bytes = 2.0 * 2 * L * wl.F * Hkv * D * 2
    kern["ring_append"] = {"us": app_us, "bytes": app_bytes, "GB/s": app_bytes / app_us / 1e3,
                           "frac_hbm": app_bytes / app_us / 1e3 / float(peaks["hbm_gbs"]),
                           "note": "one push of all %d layers (read + write of K and V), graph of %d "
                                   "pushes over distinct frames (> 2x L2)" % (L, nfr)}
    # the same kernel on a push 8x the workload's frame (2048 tokens per layer)
    Fb = 8 * wl.F
    big = rx.Cache(L, Hq, Hkv, D, wl.P, 2, Fb, S)
    fbb = 2 * L * Fb * Hkv * D * 2
    nbig = max(2, int(np.ceil(2 * 129e6 / fbb)))
    bpool = [(randn_bf16(L, Fb, Hkv, D), randn_bf16(L, Fb, Hkv, D)) for _ in range(nbig)]
    with torch.cuda.stream(stream):
        for fr in bpool:
            big.push_frame(*fr)
    torch.cuda.synchronize()
    bp_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(bp_graph, stream=stream):
        for fr in bpool:
            big.push_frame(*fr)
    with torch.cuda.stream(stream):
        bp_graph.replay()
        d0 = torch.cuda.Event(enable_timing=True)
        d1 = torch.cuda.Event(enable_timing=True)
        d0.record(stream)
        for _ in range(3):
            bp_graph.replay()
        d1.record(stream)
    d1.synchronize()
    assert big.check_device_error() == 0, "a kernel reported a device-side timeout"
    bap_us = d0.elapsed_time(d1) * 1e3 / (3 * nbig)
    bap_bytes = 2.0 * fbb
    kern["ring_append_bw_scale"] = {"us": bap_us, "bytes": bap_bytes, "GB/s": bap_bytes / bap_us / 1e3,
                                    "frac_hbm": bap_bytes / bap_us / 1e3 / float(peaks["hbm_gbs"]),
                                    "note": "one push of %d tokens x %d layers, graph of %d pushes over "
                                            "distinct frames (> 2x L2)" % (Fb, L, nbig)}
    del bp_graph, bpool
    big.close()
    rows_bw = S * L * 2 * 64
    xs = [randn_bf16(rows_bw, wl.d_model) for _ in range(2)]
    ys = torch.empty_like(xs[0])
    with torch.cuda.stream(stream):
        rx.adarmsnorm(xs[0], gamma[0, 0], wl.eps, out=ys)
    torch.cuda.synchronize()
    n_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(n_graph, stream=stream):
        for i in range(10):
            rx.adarmsnorm(xs[i % 2], gamma[0, 0], wl.eps, out=ys)
    with torch.cuda.stream(stream):
        n_graph.replay()
        c0 = torch.cuda.Event(enable_timing=True)
        c1 = torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        n_graph.replay()
        c1.record(stream)
    c1.synchronize()
    nrm_us = c0.elapsed_time(c1) * 1e3 / 10
    nrm_bytes = 2.0 * rows_bw * wl.d_model * 2
    kern["adarmsnorm_bw_scale"] = {"us": nrm_us, "rows": rows_bw, "bytes": nrm_bytes,
                                   "GB/s": nrm_bytes / nrm_us / 1e3,
                                   "frac_hbm": nrm_bytes / nrm_us / 1e3 / float(peaks["hbm_gbs"])}
    # The gamma MLP: one launch per tick computes gamma for all 2L sites x K
    # steps.  Timed alone over weight pools whose W2 together exceed 2x L2, so
    # each launch streams its weights from DRAM as the tick's does.  Bytes:
    # the weights (W1, b1, W2, b2, bf16) read once, gamma (fp32) written once.
    w_bytes = 2.0 * n_sets * (wl.hidden * wl.cond_dim + wl.hidden + wl.d_model * wl.hidden + wl.d_model)
    g_bytes = 4.0 * n_sets * K * wl.d_model
    ngp = max(2, int(np.ceil(2 * 129e6 / w_bytes)))
    gpool = [tuple(randn_bf16(*shp, scale=0.02) for shp in
                   ((n_sets, wl.hidden, wl.cond_dim), (n_sets, wl.hidden), (n_sets, wl.d_model, wl.hidden),
                    (n_sets, wl.d_model))) for _ in range(ngp)]
    gam_out = torch.empty_like(gamma)
    with torch.cuda.stream(stream):
        for wp in gpool:
            rx.ada_gamma(tk, state[0], *wp, wl.emb_dim, out=gam_out)
    torch.cuda.synchronize()
    g_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_graph, stream=stream):
        for wp in gpool:
            rx.ada_gamma(tk, state[0], *wp, wl.emb_dim, out=gam_out)
    with torch.cuda.stream(stream):
        g_graph.replay()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(3):
            g_graph.replay()
        e1.record(stream)
    e1.synchronize()
    gam_us = e0.elapsed_time(e1) * 1e3 / (3 * ngp)
    kern["ada_gamma"] = {"us": gam_us, "bytes": w_bytes + g_bytes, "GB/s": (w_bytes + g_bytes) / gam_us / 1e3,
                         "frac_hbm": (w_bytes + g_bytes) / gam_us / 1e3 / float(peaks["hbm_gbs"]),
                         "note": "one launch of %d gamma vectors (%d sites x %d steps), graph of %d launches "
                                 "over distinct weight sets (> 2x L2)" % (n_sets * K, n_sets, K, ngp)}
    del g_graph, gpool, gam_out
    kern.update(next_rows_kernels(rx, wl, stream, randn_bf16, peaks))
    kern["attention"] = {"us_per_call": plain_us, "flops_per_call": fl, "TFLOP/s": fl / plain_us / 1e6,
                         "frac_tensor": fl / plain_us / 1e6 / peak_tf,
                         "note": "the attention call alone, without the norm jobs"}
    kern["attention_with_norms"] = {"us_per_call": attn_us, "kernels_per_call": attn_kernels_per_call,
                                    "flops_per_call": fl, "TFLOP/s": achieved,
                                    "note": "the tick's launch: attention plus the layer's two AdaRMSNorms "
                                            "(the roofline line's figure)"}
    kern["tick_norms_in_own_launches"] = {
        "ms_per_tick": sep_ms, "denoise-steps/s": K / (sep_ms / 1e3),
        "note": "the same tick with each AdaRMSNorm as a launch of its own (3 launches per step "
                "and layer instead of 1)"}
    del pool, xs, ys

    # The same kernel with a 1024-token suffix (64 query tiles) over the
    # workload's cached keys, one call per layer of an 18-layer store (larger
    # than L2 for c4): the per-launch latency amortised over 16x the work.
    S_big = 1024
    big_a = rx.Cache(L, Hq, Hkv, D, wl.P, wl.N, wl.F, S_big)
    big_a.pin_prefix(randn_bf16(L, wl.P, Hkv, D), randn_bf16(L, wl.P, Hkv, D))
    with torch.cuda.stream(stream):
        for t in range(wl.N):
            big_a.push_frame(randn_bf16(L, wl.F, Hkv, D), randn_bf16(L, wl.F, Hkv, D))
    qb = randn_bf16(L, S_big, Hq, D)
    kb = randn_bf16(L, S_big, Hkv, D)
    vb = randn_bf16(L, S_big, Hkv, D)
    ob = torch.empty_like(qb)

    def big_calls():
        for l in range(L):
            big_a.attend_suffix(l, qb[l], kb[l], vb[l], out=ob[l])

    with torch.cuda.stream(stream):
        big_calls()
    torch.cuda.synchronize()
    bg = torch.cuda.CUDAGraph()
    with torch.cuda.graph(bg, stream=stream):
        big_calls()
    with torch.cuda.stream(stream):
        bg.replay()
        g0 = torch.cuda.Event(enable_timing=True)
        g1 = torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for _ in range(3):
            bg.replay()
        g1.record(stream)
    g1.synchronize()
    assert big_a.check_device_error() == 0, "a kernel reported a device-side timeout"
    big_us = g0.elapsed_time(g1) * 1e3 / (3 * L)
    big_fl = 4.0 * Hq * S_big * (wl.cached + S_big) * D
    kern["attention_1024_token_suffix"] = {
        "us_per_call": big_us, "flops_per_call": big_fl, "TFLOP/s": big_fl / big_us / 1e6,
        "frac_tensor": big_fl / big_us / 1e6 / peak_tf,
        "note": "%d-token suffix x %d heads over %d cached + %d dynamic keys, one call per layer of "
                "the %d-layer store" % (S_big, Hq, wl.cached, S_big, L)}
    big_a.close()
    del qb, kb, vb, ob, bg

    # ---------------- end to end through the API with host buffers ----------------
    # Every tick moves all of its inputs from pinned host memory (the frame's
    # K/V, the robot state, and every step's and layer's q, k_dyn, v_dyn and
    # norm inputs) and reads all of its outputs back (every attention output
    # and both norms' outputs).  The next tick's inputs upload on a copy
    # stream into the other input slot while this tick computes, and this
    # tick's outputs download on a second copy stream while the next one
    # computes, as a streaming deployment would overlap them.  A slot's
    # upload waits for the tick that last read it, and a tick waits for the
    # download of the outputs it is about to overwrite.  Every copy is inside
    # the timed region.
    ins = [lambda s_: frames[s_][0], lambda s_: frames[s_][1], lambda s_: state[s_],
           lambda s_: q[s_], lambda s_: kd[s_], lambda s_: vd[s_], lambda s_: x[s_]]
    outs = [lambda s_: o[s_], lambda s_: y[s_]]
    if B:
        ins.append(lambda s_: ql[s_])
        outs.append(lambda s_: ol[s_])
    h_in = [fn(0).cpu().pin_memory() for fn in ins]
    h_out = [torch.empty(fn(0).shape, dtype=fn(0).dtype).pin_memory() for fn in outs]
    h2d = sum(t.numel() * t.element_size() for t in h_in)
    d2h = sum(t.numel() * t.element_size() for t in h_out)
    # As many ticks as the timed region, so that the first upload and the
    # last read-back (which nothing overlaps) weigh as they do in a stream.
    e2e_steps = max(16, args.steps)
    up_stream = torch.cuda.Stream(device=dev)
    down_stream = torch.cuda.Stream(device=dev)
    ready = [torch.cuda.Event() for _ in range(NSLOT)]      # slot's inputs uploaded
    consumed = [torch.cuda.Event() for _ in range(NSLOT)]   # slot's tick finished
    drained = [torch.cuda.Event() for _ in range(NSLOT)]    # slot's outputs downloaded

    def upload(s_):
        with torch.cuda.stream(up_stream):
            up_stream.wait_event(consumed[s_])
            for fn, h in zip(ins, h_in):
                fn(s_).copy_(h, non_blocking=True)
            ready[s_].record(up_stream)

    def download(s_):
        with torch.cuda.stream(down_stream):
            down_stream.wait_event(consumed[s_])
            for fn, h in zip(outs, h_out):
                h.copy_(fn(s_), non_blocking=True)
            drained[s_].record(down_stream)

    with torch.cuda.stream(stream):
        for s_ in range(NSLOT):
            consumed[s_].record(stream)
            drained[s_].record(stream)
        f0 = torch.cuda.Event(enable_timing=True)
        f1 = torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        up_stream.wait_stream(stream)     # every copy is inside the timed region
        down_stream.wait_stream(stream)
        upload(0)
        for i in range(e2e_steps):
            s_ = i % NSLOT
            if i + 1 < e2e_steps:
                upload((i + 1) % NSLOT)
            stream.wait_event(ready[s_])
            stream.wait_event(drained[s_])
            graphs[s_].replay()
            consumed[s_].record(stream)
            download(s_)
        stream.wait_stream(down_stream)
        f1.record(stream)
    f1.synchronize()
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(f0.elapsed_time(f1), world, dev)
    e2e_val = replica_throughput(e2e_steps * K, world, e2e_ms)
    assert cache.check_device_error() == 0, "a kernel reported a device-side timeout"
    del h_in, h_out

    # ---------------- the other multi-layer workloads' attention calls ----------------
    for other in ("c3", "c4", "c5"):
        if other == args.workload:
            continue
        us, flo = attention_call_us(rx, W.WORKLOADS[other], stream, randn_bf16, reps=3)
        kern["attention_" + other] = {
            "us_per_call": us, "flops_per_call": flo, "TFLOP/s": flo / us / 1e6,
            "frac_tensor": flo / us / 1e6 / peak_tf,
            "note": "%s, graph of %d x %d calls over one input set" % (
                describe(W.WORKLOADS[other]), W.WORKLOADS[other].steps, W.WORKLOADS[other].L)}

    if rank != 0:
        return
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        v, dt, desc = oracle_sample(wl, args.seed, args.cpu_seconds, args.cpu_max_steps)
        cpu = {"value": v, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
               "sample": desc + " (%.1f s)" % dt}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": describe(wl), "step": "one stream tick: gamma for all sites and "
                   "steps, 1 ring append, %d denoising steps x %d layers x {AdaRMSNorm, attention, "
                   "AdaRMSNorm} (one launch per step and layer: the two norms run in the attention "
                   "launch), one CUDA graph" % (K, L),
                   "keys_per_query": wl.keys_full, "attn_splits": "auto" if not args.splits else args.splits,
                   "l2": "inputs larger than L2: two alternating input pools of %.0f MB each; the "
                         "%.1f MB per-layer K/V store is reused across the %d steps of a tick by design"
                         % ((q[0].numel() + kd[0].numel() * 2 + x[0].numel()) * 2 / 1e6,
                            wl.cached * Hkv * D * 4 / 1e6, K),
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak_tf, "unit": "TFLOP/s",
                     "frac": achieved / peak_tf, "traffic": attn_traffic(args.workload),
                     "traffic_source": "ncu dram__bytes_read.sum + dram__bytes_write.sum of one call "
                                       "from a capture of this workload, reported only while the kernel "
                                       "code hash matches that capture (else null)",
                     "kernel": "partitioned attention with the layer's two AdaRMSNorms in the same "
                               "launch (split-KV kernel + merge), as the tick runs it: %.2f us per call, "
                               "%.3g algorithmic attention FLOP per call (4*Hq*S*Lk*D; the norms' bytes "
                               "are not counted)" % (attn_us, fl),
                     "peak_kind": "%s bf16 dense burst" % peak_kind},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_val, "unit": UNIT, "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h)},
        "gpu_launches": int(launches_per_tick * args.steps),
        "clocks": clocks,
        "kernels": kern,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="c4", choices=["c2", "c3", "c4", "c5"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--splits", type=int, default=0, help="split-KV partitions (0 = automatic)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="oracle seconds the CPU sample aims for (whole denoising steps)")
    ap.add_argument("--cpu-max-steps", type=int, default=200, help="most denoising steps in the CPU sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    wl = W.WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, wl)
    else:
        run_ours(args, wl)


if __name__ == "__main__":
    main()
