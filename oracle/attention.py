"""Brute-force dense softmax attention in float64.

Test infrastructure only (see the package docstring).

This is the plain definition the method reduces to when skipping is off
(λ = 0): for each sequence of a packed batch and each query head h,

    S = Q_h K_g^T * scale,   g = h // (Hq / Hkv)      (grouped-query heads)
    S[r, c] = -inf where c > r                        (causal mask)
    P = softmax(S) row by row,   O_h = P V_g,   lse_r = log sum_c exp(S[r, c])

computed on the whole score matrix at once (no tiling, no online update).
The deployment guide's §5 step 4 asks that GQA variants be supported, which
fixes the head mapping; the causal mask is the one of decoder prefill.

``allowed`` restricts the key set per row: ``allowed(s, h)`` returns a
boolean ``[L, L]`` matrix, ``False`` entries are excluded exactly like the
causal mask. With the tile mask of a skip bitmap this is "attention over the
kept tiles only", the closed form of the skipping path once its decisions
are fixed.
"""
from __future__ import annotations

import math

import numpy as np


def dense(q: np.ndarray, k: np.ndarray, v: np.ndarray, cu_seqlens, Hq: int, Hkv: int,
          causal: bool = True, scale: float | None = None, allowed=None, heads=None,
          cu_seqlens_k=None):
    """Return ``(out [T, Hq, d], lse [Hq, T])`` as float64.

    q, k, v are float64 ``[T, H, d]`` values. Rows of heads not listed in
    ``heads`` are left as NaN. ``cu_seqlens_k`` gives separate key boundaries
    (chunked prefill): the Lq queries of a sequence are its last Lq
    positions, so query r may see key c when c <= Lk - Lq + r.
    """
    T, _, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    G = Hq // Hkv
    out = np.full((T, Hq, d), np.nan)
    lse = np.full((Hq, T), np.nan)
    cu = [int(x) for x in cu_seqlens]
    cuk = cu if cu_seqlens_k is None else [int(x) for x in cu_seqlens_k]
    for s in range(len(cu) - 1):
        a, b = cu[s], cu[s + 1]
        ak, bk = cuk[s], cuk[s + 1]
        Lq, Lk = b - a, bk - ak
        if Lq == 0:
            continue
        for h in (range(Hq) if heads is None else heads):
            g = h // G
            S = (q[a:b, h, :] @ k[ak:bk, g, :].T) * scale
            keep = np.ones((Lq, Lk), bool)
            if causal:
                keep &= np.tri(Lq, Lk, Lk - Lq, dtype=bool)
            if allowed is not None:
                keep &= allowed(s, h)
            S = np.where(keep, S, -np.inf)
            mx = S.max(axis=1, keepdims=True)
            E = np.exp(S - mx)
            z = E.sum(axis=1, keepdims=True)
            out[a:b, h, :] = (E / z) @ v[ak:bk, g, :]
            lse[h, a:b] = (mx + np.log(z))[:, 0]
    return out, lse


def direct_logsumexp(x: np.ndarray) -> float:
    """log(sum(exp(x))) of a 1-D array by the textbook max shift."""
    x = np.asarray(x, np.float64)
    x = x[np.isfinite(x)]
    mx = x.max()
    return float(mx + math.log(np.exp(x - mx).sum()))
