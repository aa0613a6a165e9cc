"""Shared helpers of the GPU parity tests: the oracle side of each comparison
and the normalised error metric |gpu - ref| / sum|w x| of the fp32 paths."""
from __future__ import annotations

import numpy as np

import datagen
import oracle

TOL_FP32 = 2e-5   # fp32-accumulate paths: max |gpu - ref| / sum_k |w_k x_k|
TOL_BF16 = 1e-2   # bf16 tensor-core prefill path
TOL_W = 1e-6      # routing weights, relative


def norm_err(gpu, ref, den) -> float:
    """max |gpu - ref| / den; where den == 0 the reference is exactly 0 and so must gpu be."""
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.asarray(den, np.float64)
    zero = den == 0
    if np.any(zero):
        assert np.all(gpu[zero] == 0) and np.all(ref[zero] == 0)
    d = np.where(zero, 1.0, den)
    return float(np.max(np.abs(gpu - ref) / d)) if gpu.size else 0.0


def moe_oracle(E, H, I, x64, ids, w, want_h=False, weights=None):
    """Oracle FFN over the experts the ids touch (weights regenerated per expert)."""
    touched = np.unique(ids[(ids >= 0) & (ids < E)])
    if weights is None:
        sub = datagen.moe_weights(E, H, I, experts=touched)
    else:
        sub = {k: v[touched] for k, v in weights.items()}
    pos = np.full(E, -1, np.int64)
    pos[touched] = np.arange(len(touched))
    valid = (ids >= 0) & (ids < E)
    mids = np.where(valid, pos[np.clip(ids, 0, E - 1)], 0).astype(np.int32)
    mw = np.where(valid, w, 0).astype(np.float32)
    return oracle.moe_ffn(sub, x64, mids, mw, want_h=want_h)
