"""AdaRMSNorm and its conditioning, plain fp64 (test infrastructure only).

"Reflex: Real-Time VLA Control through Streaming Inference", §III "Core
formulas", Eq. (2):

    AdaRMSNorm(x, c) = x / RMS(x) (.) gamma(c),   gamma(c) = 1 + MLP(c),
    RMS(x) = sqrt( (1/d) sum_i x_i^2 + eps )

with c = [t_k, s_t], the sinusoidal embedding of the denoising time joined to
the proprioceptive robot state.  §III "Model components": the MLP is
Linear(cond_dim -> hidden) -> SiLU -> Linear(hidden -> model_dim).  §V "Key
implementation": the mean of squares is taken in FP32, x is scaled by
rsqrt(mean + eps), and the gate 1 + MLP(cond) multiplies the result.

Readings where the page is silent:
* Embedding: width E, half = E/2 frequencies w_i = 10000^(-i/half),
  emb(t) = [sin(t w_0..w_{half-1}), cos(t w_0..w_{half-1})].
* Weights follow nn.Linear: W1 [hidden][cond_dim], W2 [d][hidden], biases.
* ``d`` in Eq. (2) is the model width over which the mean is taken.

Everything is computed in float64 from the exact bf16 input values.
"""
from __future__ import annotations

import numpy as np


def sinusoidal_embedding(t: float, dim: int) -> np.ndarray:
    """Sinusoidal embedding of a scalar time t: [sin(t w_i)..., cos(t w_i)...]."""
    if dim % 2:
        raise ValueError("embedding width must be even")
    half = dim // 2
    i = np.arange(half, dtype=np.float64)
    w = np.power(10000.0, -i / half)
    return np.concatenate([np.sin(float(t) * w), np.cos(float(t) * w)])


def conditioning(t: float, state, emb_dim: int) -> np.ndarray:
    """c = [emb(t_k); s_t]."""
    return np.concatenate([sinusoidal_embedding(t, emb_dim),
                           np.asarray(state, dtype=np.float64)])


def silu(z: np.ndarray) -> np.ndarray:
    return z / (1.0 + np.exp(-z))


def gamma_mlp(c, W1, b1, W2, b2) -> np.ndarray:
    """gamma(c) = 1 + W2 SiLU(W1 c + b1) + b2."""
    c = np.asarray(c, dtype=np.float64)
    W1 = np.asarray(W1, dtype=np.float64)
    b1 = np.asarray(b1, dtype=np.float64)
    W2 = np.asarray(W2, dtype=np.float64)
    b2 = np.asarray(b2, dtype=np.float64)
    h = W1 @ c + b1
    return 1.0 + W2 @ silu(h) + b2


def ada_rms_norm(x, gamma, eps: float) -> np.ndarray:
    """Eq. (2) applied row-wise: x [rows][d], gamma [d] -> [rows][d]."""
    x = np.asarray(x, dtype=np.float64)
    gamma = np.asarray(gamma, dtype=np.float64)
    rms = np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    return x / rms * gamma
