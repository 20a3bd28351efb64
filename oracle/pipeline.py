"""One stream tick of the hot path, composed from the oracle's parts
(test infrastructure only).

"Reflex: Real-Time VLA Control through Streaming Inference", §III "System
architecture" and "Core formulas": each stream tick enqueues the newest
observation frame (evicting the oldest once N frames are held); then, for each
of the K denoising steps, every layer normalises the suffix with AdaRMSNorm
(Eq. 2) before attention and before the MLP, and attends the suffix queries
over [pinned; sliding; dynamic] (Eq. 1).  The encoder is timestep-invariant
(Proposition A.1), so one frame's K/V serve all K steps of its tick; only the
suffix q, k_dyn, v_dyn change per step.

There is no model here: every per-step input comes from the seeded generator
``partitioned_kv_cache_gb300.workload`` and every output is returned, not fed
forward.
"""
from __future__ import annotations

from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

from partitioned_kv_cache_gb300 import workload as W

from .adarms import ada_rms_norm, conditioning, gamma_mlp
from .attention import partitioned_attention
from .ring import FrameWindow


class OracleStream:
    """Pinned prefix + per-layer FIFO window, advanced one tick at a time."""

    def __init__(self, wl: W.Workload, seed: int, P: Optional[int] = None):
        self.wl = wl
        self.seed = seed
        pk, pv = W.pinned_kv(wl, seed, P)
        self.pin_k = W.bf16_bits_to_f64(pk)   # [L][P][Hkv][D]
        self.pin_v = W.bf16_bits_to_f64(pv)
        self.window = FrameWindow(wl.N)       # frames hold (tick, K, V)
        self._mlp: Dict[Tuple[int, int], tuple] = {}

    # ---- ring ----------------------------------------------------------
    def push(self, tick: int) -> int:
        fk, fv = W.frame_kv(self.wl, self.seed, tick)
        return self.window.push((tick, W.bf16_bits_to_f64(fk), W.bf16_bits_to_f64(fv)))

    def window_ticks(self) -> List[int]:
        return [f[0] for f in self.window.window()]

    def regions(self, layer: int, k_dyn, v_dyn):
        ks = [self.pin_k[layer]] + [f[1][layer] for f in self.window.window()] + [k_dyn]
        vs = [self.pin_v[layer]] + [f[2][layer] for f in self.window.window()] + [v_dyn]
        return ks, vs

    # ---- Eq. 1 ---------------------------------------------------------
    def attend(self, tick: int, step: int, layer: int,
               tokens: Optional[Sequence[int]] = None) -> np.ndarray:
        """Attention output [S][Hq][D] (or only the listed suffix tokens)."""
        q, kd, vd = W.suffix_qkv(self.wl, self.seed, tick, step, layer)
        q = W.bf16_bits_to_f64(q)
        if tokens is not None:
            q = q[np.asarray(tokens)]
        ks, vs = self.regions(layer, W.bf16_bits_to_f64(kd), W.bf16_bits_to_f64(vd))
        return partitioned_attention(q, ks, vs)

    # ---- Eq. 2 ---------------------------------------------------------
    def mlp(self, layer: int, site: int):
        key = (layer, site)
        if key not in self._mlp:
            self._mlp[key] = tuple(W.bf16_bits_to_f64(a) for a in
                                   W.mlp_weights(self.wl, self.seed, layer, site))
        return self._mlp[key]

    def gamma(self, tick: int, step: int, layer: int, site: int) -> np.ndarray:
        t = float(W.timesteps(self.wl)[step])
        c = conditioning(t, W.robot_state(self.wl, self.seed, tick), self.wl.emb_dim)
        return gamma_mlp(c, *self.mlp(layer, site))

    def norm(self, tick: int, step: int, layer: int, site: int) -> np.ndarray:
        x = W.bf16_bits_to_f64(W.norm_input(self.wl, self.seed, tick, step, layer, site))
        return ada_rms_norm(x, self.gamma(tick, step, layer, site), self.wl.eps)

    # ---- one tick --------------------------------------------------------
    def tick(self, tick: int, steps: Optional[int] = None, layers: Optional[int] = None):
        """Push frame ``tick`` then run the denoising steps.

        Returns {(step, layer): (y_attn_norm, attn_out, y_mlp_norm)}.
        """
        self.push(tick)
        out = {}
        for k in range(self.wl.steps if steps is None else steps):
            for l in range(self.wl.L if layers is None else layers):
                out[(k, l)] = (self.norm(tick, k, l, 0),
                               self.attend(tick, k, l),
                               self.norm(tick, k, l, 1))
        return out
