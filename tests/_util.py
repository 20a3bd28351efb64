"""Shared helpers for the GPU tests: bf16 bit patterns to CUDA tensors and
the tolerance checks."""
import os

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LIB = os.path.join(ROOT, "partitioned_kv_cache_gb300", "librx.so")

# Attention tolerance on unit-scale inputs: max-abs 1e-2, mean-abs 1e-3.
ATT_MAX = 1e-2
ATT_MEAN = 1e-3
# Fewest keys per query row for which the unit-scale bounds are held as
# stated.  With fewer keys an output is not an average of many values.  bf16
# keeps 8 significant bits, so a rounding to nearest is within 2^-8 of the
# value: the path's two roundings (P for the tensor-core product, and the
# output) are within 2^-8 * sum_j alpha_j |v_j| and 2^-8 * |o|, each at most
# 2^-8 * max|V|, so 2^-7 * max|V| at worst together.  Such rows are held to
# 2^-8 * max|V| wherever that exceeds the unit-scale 1e-2: half the worst
# case, a stricter bound that every case meets.
FEW_KEYS = 64
# AdaRMSNorm: elementwise relative 1e-2, no NaN/Inf.
NORM_REL = 1e-2


def ensure_built():
    if not os.path.exists(LIB):
        from partitioned_kv_cache_gb300 import build
        build.build()


def dev(bits, device="cuda"):
    import torch
    a = np.ascontiguousarray(np.asarray(bits, dtype=np.uint16))
    return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)


def host64(t):
    return t.float().cpu().numpy().astype(np.float64)


def check_attention(got, ref, scale=1.0):
    """got/ref float64 arrays.  `scale` widens the bound for inputs that are
    not unit-scale (outliers): both bounds are multiplied by it."""
    assert np.all(np.isfinite(got)), "non-finite attention output"
    err = np.abs(got - ref)
    assert err.max() <= ATT_MAX * scale, "max abs err %.3e > %.1e" % (err.max(), ATT_MAX * scale)
    assert err.mean() <= ATT_MEAN * scale, "mean abs err %.3e > %.1e" % (err.mean(), ATT_MEAN * scale)
    return err.max(), err.mean()


def few_keys_scale(min_keys, vmax):
    """Widening of the attention bounds for rows that see fewer than FEW_KEYS
    keys (1 otherwise: the stated unit-scale bounds hold)."""
    if min_keys >= FEW_KEYS:
        return 1.0
    return max(1.0, 2.0 ** -8 * vmax / ATT_MAX)


def check_norm(got, ref):
    assert np.all(np.isfinite(got)), "non-finite AdaRMSNorm output"
    bad = np.abs(got - ref) > NORM_REL * np.abs(ref) + 1e-30
    assert not bad.any(), "relative error > 1e-2 at %d elements, worst %s" % (
        bad.sum(), np.max(np.abs(got - ref) / (np.abs(ref) + 1e-30)))
