"""Partitioned attention, plain fp64 (test infrastructure only).

"Reflex: Real-Time VLA Control through Streaming Inference", §III "Core
formulas", Eq. (1):

    Attn(x^(k)) = Softmax( Q^(k) [K_pin; K_slide(t); K_dyn(k)]^T / sqrt(d) )
                  x [V_pin; V_slide(t); V_dyn(k)]

The keys and values of the three regions are concatenated along the token
axis and one ordinary softmax attention is taken over the concatenation.
Proposition A.1 states that evaluating the regions separately gives exactly
the full-batch result because softmax does not care how its logit set is
partitioned or permuted.

Readings where the page is silent:
* ``d`` in Eq. (1) is the head dimension D (the usual scaled dot product).
* No mask: every suffix query sees every key of the three regions.
* Grouped heads: query head h reads key/value head floor(h / G), G = Hq/Hkv.

Layouts: q [S][Hq][D]; every K/V region [T_i][Hkv][D]; output [S][Hq][D].
Inputs are converted to float64 before any arithmetic.
"""
from __future__ import annotations

import math
from typing import List, Sequence, Tuple

import numpy as np


def _check(q: np.ndarray, K: np.ndarray, V: np.ndarray) -> Tuple[int, int, int, int, int]:
    S, Hq, D = q.shape
    T, Hkv, Dk = K.shape
    if V.shape != K.shape or Dk != D:
        raise ValueError("K/V shapes disagree with q")
    if Hkv < 1 or Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    return S, Hq, D, T, Hkv


def attention_weights(q, K) -> np.ndarray:
    """Softmax weights alpha [S][Hq][T] of Eq. (1) over the key set K."""
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    S, Hq, D, T, Hkv = _check(q, K, K)
    G = Hq // Hkv
    alpha = np.empty((S, Hq, T), dtype=np.float64)
    for h in range(Hq):
        g = h // G
        logits = (q[:, h, :] @ K[:, g, :].T) / math.sqrt(D)
        logits -= logits.max(axis=1, keepdims=True)
        e = np.exp(logits)
        alpha[:, h, :] = e / e.sum(axis=1, keepdims=True)
    return alpha


def full_attention(q, K, V) -> np.ndarray:
    """softmax(q K^T / sqrt(D)) V over one explicit key/value set."""
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    S, Hq, D, T, Hkv = _check(q, K, V)
    if T == 0:
        raise ValueError("attention over an empty key set is undefined")
    G = Hq // Hkv
    alpha = attention_weights(q, K)
    out = np.empty((S, Hq, D), dtype=np.float64)
    for h in range(Hq):
        out[:, h, :] = alpha[:, h, :] @ V[:, h // G, :]
    return out


def partitioned_attention(q, k_regions: Sequence, v_regions: Sequence) -> np.ndarray:
    """Eq. (1): concatenate the regions' K/V along tokens, then attend.

    ``k_regions`` / ``v_regions`` list the pinned prefix, the window's frames
    in logical order (oldest first) and the dynamic suffix, each [T_i][Hkv][D].
    Empty regions are allowed (e.g. no frame pushed yet).
    """
    ks = [np.asarray(k, dtype=np.float64) for k in k_regions]
    vs = [np.asarray(v, dtype=np.float64) for v in v_regions]
    K = np.concatenate(ks, axis=0)
    V = np.concatenate(vs, axis=0)
    return full_attention(q, K, V)


def block_causal_attention(q, k_regions: Sequence, v_regions: Sequence, n_state: int) -> np.ndarray:
    """Eq. (1) with a block-causal suffix (the other plain reading of the
    attention-mask figure of "Reflex: ...", §III "System architecture"): the
    last region is the dynamic suffix; its first ``n_state`` tokens (the state
    block) see the cached regions and only the state block's own keys, while
    the remaining (action) tokens see every key.  n_state = 0 is Eq. (1).
    """
    q = np.asarray(q, dtype=np.float64)
    S = q.shape[0]
    ks = [np.asarray(k, dtype=np.float64) for k in k_regions]
    vs = [np.asarray(v, dtype=np.float64) for v in v_regions]
    n_state = max(0, min(int(n_state), S))
    out = np.empty(q.shape, dtype=np.float64)
    if n_state:
        out[:n_state] = partitioned_attention(q[:n_state], ks[:-1] + [ks[-1][:n_state]],
                                              vs[:-1] + [vs[-1][:n_state]])
    if n_state < S:
        out[n_state:] = partitioned_attention(q[n_state:], ks, vs)
    return out


def region_split_attention(q, k_regions: Sequence, v_regions: Sequence) -> np.ndarray:
    """Proposition A.1, evaluated region by region.

    Each region r gives its own logits; keep its row maximum m_r, the sum of
    exp(logit - m_r) and the exp-weighted sum of its values.  The regions are
    then combined with the global maximum.  Mathematically identical to
    ``partitioned_attention``; used to pin the oracle to the proposition.
    """
    q = np.asarray(q, dtype=np.float64)
    S, Hq, D = q.shape
    parts = []
    for k, v in zip(k_regions, v_regions):
        k = np.asarray(k, dtype=np.float64)
        v = np.asarray(v, dtype=np.float64)
        if k.shape[0] == 0:
            continue
        Hkv = k.shape[1]
        G = Hq // Hkv
        m = np.empty((S, Hq))
        l = np.empty((S, Hq))
        o = np.empty((S, Hq, D))
        for h in range(Hq):
            logits = (q[:, h, :] @ k[:, h // G, :].T) / math.sqrt(D)
            m[:, h] = logits.max(axis=1)
            e = np.exp(logits - m[:, h][:, None])
            l[:, h] = e.sum(axis=1)
            o[:, h, :] = e @ v[:, h // G, :]
        parts.append((m, l, o))
    if not parts:
        raise ValueError("attention over an empty key set is undefined")
    M = np.max(np.stack([p[0] for p in parts]), axis=0)
    num = np.zeros((S, Hq, D))
    den = np.zeros((S, Hq))
    for m, l, o in parts:
        w = np.exp(m - M)
        num += w[:, :, None] * o
        den += w * l
    return num / den[:, :, None]


def brute_force_attention(q, K, V) -> List[List[List[float]]]:
    """Eq. (1) with nothing but Python scalars and loops (tiny shapes only)."""
    S, Hq, D = len(q), len(q[0]), len(q[0][0])
    T, Hkv = len(K), len(K[0])
    G = Hq // Hkv
    out = []
    for s in range(S):
        row = []
        for h in range(Hq):
            g = h // G
            logits = []
            for j in range(T):
                acc = 0.0
                for c in range(D):
                    acc += float(q[s][h][c]) * float(K[j][g][c])
                logits.append(acc / math.sqrt(D))
            mx = max(logits)
            w = [math.exp(z - mx) for z in logits]
            tot = sum(w)
            o = []
            for c in range(D):
                acc = 0.0
                for j in range(T):
                    acc += w[j] * float(V[j][g][c])
                o.append(acc / tot)
            row.append(o)
        out.append(row)
    return out


def shared_cache_attention(k_shared: Sequence, v_shared: Sequence, requests) -> List[np.ndarray]:
    """Several requests over one read-only shared cache plus private keys.

    "OxyGen ...", §"Core method": the action expert reads the prefill cache as
    read-only context while language streams append their own KV per decoded
    token; each stream attends over [shared; its own appended KV] and nothing
    a stream appends enters another stream's view.

    ``requests`` is a list of (q [n][Hq][D], k_priv [t][Hkv][D], v_priv) and
    the result lists each request's output [n][Hq][D].
    """
    outs = []
    for q, kp, vp in requests:
        outs.append(partitioned_attention(q, list(k_shared) + [kp], list(v_shared) + [vp]))
    return outs
