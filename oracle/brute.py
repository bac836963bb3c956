"""Brute-force attention on contiguous K/V (test infrastructure).

An independent restatement used to pin the C oracle: no paging, no gather,
one dense score matrix per head, written with NumPy matrix products.  Query
row r sits at absolute position ``positions[r]`` and sees keys 0..positions[r]
of its own sequence; query head h reads KV head h // (Hq // Hkv).
"""

from __future__ import annotations

import numpy as np


def attention_contiguous(q: np.ndarray, K: np.ndarray, V: np.ndarray, positions,
                         scale: float) -> np.ndarray:
    """q [n, Hq, D], K/V [L, Hkv, D] (float64), positions [n] -> out [n, Hq, D]."""
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    positions = np.asarray(positions, dtype=np.int64)
    n, Hq, D = q.shape
    L, Hkv, _ = K.shape
    group = Hq // Hkv
    out = np.zeros((n, Hq, D))
    visible = np.arange(L)[None, :] <= positions[:, None]          # [n, L]
    for h in range(Hq):
        scores = (q[:, h, :] @ K[:, h // group, :].T) * scale      # [n, L]
        scores = np.where(visible, scores, -np.inf)
        rows = visible.any(axis=1)
        top = np.where(rows, scores.max(axis=1, initial=-np.inf), 0.0)
        w = np.where(visible, np.exp(scores - top[:, None]), 0.0)
        denom = w.sum(axis=1)
        safe = np.where(rows, denom, 1.0)
        out[:, h, :] = (w @ V[:, h // group, :]) / safe[:, None]
    return out
