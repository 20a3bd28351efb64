"""Seeded synthetic workloads for the partitioned-attention hot path.

This module only draws random numbers and fixes shapes.  It holds none of the
method's arithmetic (no attention, no normalisation, no embedding): both the
CUDA path and the CPU oracle consume what it produces, so it must stay neutral.

Shapes follow the Reflex streaming setting ("Reflex: Real-Time VLA Control
through Streaming Inference", §III "System architecture" and "Model
components"): a pinned instruction prefix, a FIFO of N observation frames of F
tokens each, and a dynamic suffix of S flow-state tokens that changes at every
denoising step.  The action chunk of 50 tokens plus one state token gives
S = 51 (Table 9, default chunk 50); ten denoising steps per tick (Table 7,
"denoise loop (x10)").  The shared-cache multi-request workload follows
"OxyGen: Unified KV Cache Management for Vision-Language-Action Models under
Multi-Task Parallelism", §"Core method" (one read-only prefill cache, language
streams with private appended KV).

Every tensor is returned as bf16 bit patterns (``np.uint16``) rounded to
nearest-even from float32 draws, so the GPU side and the oracle see the same
numbers exactly.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Tuple

import numpy as np


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    L: int            # layers
    Hq: int           # query heads
    Hkv: int          # key/value heads
    D: int            # head dimension
    P: int            # pinned prefix tokens
    N: int            # frames in the sliding window
    F: int            # tokens per frame
    S: int            # dynamic suffix tokens (1 state + action chunk)
    steps: int        # denoising steps per tick
    ticks: int        # stream ticks (frames pushed)
    d_model: int      # AdaRMSNorm width
    emb_dim: int      # sinusoidal timestep embedding width
    state_dim: int    # proprioceptive state width
    hidden: int       # gamma-MLP hidden width
    eps: float = 1e-6
    outlier_frac: float = 0.0   # fraction of K/V entries scaled up
    outlier_scale: float = 1.0
    n_lang: int = 0             # language streams sharing the cache
    tail_max: int = 0           # largest private tail length (inclusive)
    tail_cap: int = 0           # private tail capacity per stream

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def cond_dim(self) -> int:
        return self.emb_dim + self.state_dim

    @property
    def cached(self) -> int:
        """Keys held in the store per layer once the window is full."""
        return self.P + self.N * self.F

    @property
    def keys_full(self) -> int:
        """Keys one suffix query sees once the window is full."""
        return self.cached + self.S


WORKLOADS: Dict[str, Workload] = {
    # tiny oracle check
    "c1": Workload("c1-tiny", L=1, Hq=2, Hkv=1, D=64, P=16, N=2, F=16, S=8,
                   steps=3, ticks=4, d_model=128, emb_dim=16, state_dim=16,
                   hidden=64),
    # single layer, MQA 8/1, head_dim 256
    "c2": Workload("c2-single-layer", L=1, Hq=8, Hkv=1, D=256, P=48, N=4,
                   F=256, S=51, steps=10, ticks=100, d_model=1024, emb_dim=16,
                   state_dim=16, hidden=512),
    # 18-layer action-expert stack
    "c3": Workload("c3-action-expert-18L", L=18, Hq=8, Hkv=1, D=256, P=64,
                   N=8, F=256, S=51, steps=10, ticks=100, d_model=1024,
                   emb_dim=16, state_dim=16, hidden=512),
    # long history with outliers
    "c4": Workload("c4-long-history-18L", L=18, Hq=8, Hkv=1, D=256, P=256,
                   N=32, F=256, S=51, steps=10, ticks=40, d_model=1024,
                   emb_dim=16, state_dim=16, hidden=512, outlier_frac=0.01,
                   outlier_scale=20.0),
    # shared cache, 1 action suffix + 16 one-token language streams
    "c5": Workload("c5-shared-cache-18L", L=18, Hq=8, Hkv=1, D=256, P=64,
                   N=8, F=256, S=51, steps=10, ticks=20, d_model=1024,
                   emb_dim=16, state_dim=16, hidden=512, n_lang=16,
                   tail_max=30, tail_cap=32),
}


# --------------------------------------------------------------------------
# bf16 bit patterns
# --------------------------------------------------------------------------
def to_bf16_bits(x) -> np.ndarray:
    """float -> bf16 bit pattern, round to nearest even (finite inputs)."""
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = f.view(np.uint32)
    # u + 0x7FFF + lsb stays below 2^32 for every finite float32
    r = (u >> 16) & np.uint32(1)
    r += np.uint32(0x7FFF)
    r += u
    r >>= np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f64(bits) -> np.ndarray:
    """bf16 bit pattern -> float64 (exact)."""
    b = np.ascontiguousarray(np.asarray(bits, dtype=np.uint16))
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_bits_to_f32(bits) -> np.ndarray:
    b = np.ascontiguousarray(np.asarray(bits, dtype=np.uint16))
    return (b.astype(np.uint32) << 16).view(np.float32)


# --------------------------------------------------------------------------
# seeded draws
# --------------------------------------------------------------------------
_TAGS = {"pin": 1, "frame": 2, "q": 3, "kdyn": 4, "vdyn": 5, "x": 6,
         "state": 7, "mlp": 8, "tail": 9, "qlang": 10, "taillen": 11,
         "xmlp": 12, "sweep": 13}


def rng(seed: int, tag: str, *idx: int) -> np.random.Generator:
    """Independent stream per (seed, tag, indices)."""
    return np.random.Generator(np.random.PCG64(
        np.random.SeedSequence([int(seed), _TAGS[tag]] + [int(i) for i in idx])))


def _normal(g: np.random.Generator, shape, wl: Workload | None = None,
            outliers: bool = False) -> np.ndarray:
    a = g.standard_normal(shape, dtype=np.float32)
    if outliers and wl is not None and wl.outlier_frac > 0.0:
        mask = g.random(shape, dtype=np.float32) < wl.outlier_frac
        a = np.where(mask, a * np.float32(wl.outlier_scale), a)
    return to_bf16_bits(a)


def pinned_kv(wl: Workload, seed: int, P: int | None = None) -> Tuple[np.ndarray, np.ndarray]:
    """Instruction-prefix K, V for all layers: [L][P][Hkv][D] bf16 bits."""
    P = wl.P if P is None else P
    g = rng(seed, "pin")
    shape = (wl.L, P, wl.Hkv, wl.D)
    return _normal(g, shape, wl, True), _normal(g, shape, wl, True)


def frame_kv(wl: Workload, seed: int, tick: int) -> Tuple[np.ndarray, np.ndarray]:
    """One observation frame's K, V for all layers: [L][F][Hkv][D] bf16 bits."""
    g = rng(seed, "frame", tick)
    shape = (wl.L, wl.F, wl.Hkv, wl.D)
    return _normal(g, shape, wl, True), _normal(g, shape, wl, True)


def suffix_qkv(wl: Workload, seed: int, tick: int, step: int, layer: int,
               S: int | None = None) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Flow-state suffix q [S][Hq][D], k_dyn, v_dyn [S][Hkv][D] (bf16 bits)."""
    S = wl.S if S is None else S
    g = rng(seed, "q", tick, step, layer)
    q = _normal(g, (S, wl.Hq, wl.D))
    g = rng(seed, "kdyn", tick, step, layer)
    k = _normal(g, (S, wl.Hkv, wl.D), wl, True)
    v = _normal(g, (S, wl.Hkv, wl.D), wl, True)
    return q, k, v


def norm_input(wl: Workload, seed: int, tick: int, step: int, layer: int,
               site: int, rows: int | None = None) -> np.ndarray:
    """Suffix activations entering an AdaRMSNorm: [S][d_model] ~ N(0, I)."""
    rows = wl.S if rows is None else rows
    g = rng(seed, "x", tick, step, layer, site)
    return _normal(g, (rows, wl.d_model))


def magnitude_sweep(rows: int, d: int, seed: int, lo: float = -6.0,
                    hi: float = 3.0) -> np.ndarray:
    """Rows of N(0,1) scaled by 10**u, u ~ U(lo, hi): magnitudes 1e-6..1e3."""
    g = rng(seed, "sweep", rows, d)
    a = g.standard_normal((rows, d), dtype=np.float32)
    u = g.uniform(lo, hi, size=(rows, 1)).astype(np.float32)
    return to_bf16_bits(a * np.power(np.float32(10.0), u))


def robot_state(wl: Workload, seed: int, tick: int) -> np.ndarray:
    """Proprioceptive state for one tick: [state_dim] ~ U(-1, 1), float32."""
    g = rng(seed, "state", tick)
    return g.uniform(-1.0, 1.0, size=(wl.state_dim,)).astype(np.float32)


def timesteps(wl: Workload) -> np.ndarray:
    """Flow-matching time of each denoising step: t_k = 1 - k/K (float32)."""
    K = wl.steps
    return np.array([1.0 - k / K for k in range(K)], dtype=np.float32)


def mlp_weights(wl: Workload, seed: int, layer: int, site: int):
    """Gamma-MLP parameters of one norm site, nn.Linear layout, ~N(0, 0.02).

    Returns W1 [hidden][cond_dim], b1 [hidden], W2 [d_model][hidden],
    b2 [d_model] as bf16 bits.
    """
    g = rng(seed, "mlp", layer, site)
    s = np.float32(0.02)
    W1 = to_bf16_bits(g.standard_normal((wl.hidden, wl.cond_dim), dtype=np.float32) * s)
    b1 = to_bf16_bits(g.standard_normal((wl.hidden,), dtype=np.float32) * s)
    W2 = to_bf16_bits(g.standard_normal((wl.d_model, wl.hidden), dtype=np.float32) * s)
    b2 = to_bf16_bits(g.standard_normal((wl.d_model,), dtype=np.float32) * s)
    return W1, b1, W2, b2


def lang_requests(wl: Workload, seed: int, tick: int, step: int, layer: int):
    """Language streams sharing the cache: one query token each plus a
    private tail of U{0..tail_max} appended tokens.

    Returns q [n_lang][1][Hq][D], tails_k/tails_v [n_lang][tail_cap][Hkv][D]
    and tail lengths [n_lang] (int32).
    """
    g = rng(seed, "taillen", tick, layer)
    lens = g.integers(0, wl.tail_max + 1, size=(wl.n_lang,)).astype(np.int32)
    g = rng(seed, "qlang", tick, step, layer)
    q = _normal(g, (wl.n_lang, 1, wl.Hq, wl.D))
    g = rng(seed, "tail", tick, layer)
    shape = (wl.n_lang, wl.tail_cap, wl.Hkv, wl.D)
    return q, _normal(g, shape, wl, True), _normal(g, shape, wl, True), lens
