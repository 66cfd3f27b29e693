"""Second, independent attention path: full causal recompute over a logically
contiguous sequence (numpy, fp64).

TEST INFRASTRUCTURE ONLY.  Page "جعل inference رخيصًا: KV cache وbatching
والتكميم", KV-cache section: the cache is not an approximation -- attending the
new token's query over the stored keys and values gives exactly what re-running
the whole sequence through causal attention gives.  Page "CS336, лекции 10 и
12", §"Арифметическая интенсивность инференса": naive inference re-feeds the
whole history.  So the paged oracle's row for query position p must equal row p
of the full causal score matrix softmax(Q K^T * scale + mask) V built here.
With a window the mask is a band, and tokens outside it must not matter.
"""
from __future__ import annotations

import numpy as np


def causal_attention_full(q_all: np.ndarray, k_all: np.ndarray, v_all: np.ndarray,
                          scale: float, window: int = 0) -> np.ndarray:
    """q_all [S,N,H], k_all/v_all [S,K,H] (float64, positions in logical order).
    Query head n reads KV head n // (N/K).  Returns out [S,N,H]: position i
    attends positions 0..i, or with window > 0 the band i-window+1..i (local
    attention: each position sees the last `window` tokens up to itself)."""
    S, N, H = q_all.shape
    K = k_all.shape[1]
    G = N // K
    out = np.empty((S, N, H), np.float64)
    mask = np.triu(np.ones((S, S), dtype=bool), k=1)  # j > i is hidden
    if window > 0:
        mask |= np.tril(np.ones((S, S), dtype=bool), k=-window)  # j <= i - window hidden
    for n in range(N):
        kh = n // G
        a = (q_all[:, n, :] @ k_all[:, kh, :].T) * scale  # [S, S] library matmul
        a[mask] = -np.inf
        a -= a.max(axis=1, keepdims=True)
        w = np.exp(a)
        w /= w.sum(axis=1, keepdims=True)
        out[:, n, :] = w @ v_all[:, kh, :]
    return out
