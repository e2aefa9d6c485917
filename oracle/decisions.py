"""Skip decisions without the tile walk: the prefix-max closed form.

Test infrastructure only (see the package docstring).

Under the threshold reading of ``tile_walk`` (skip tile j when every valid
row has ``rm_j < m + ln λ``), a skipped tile never raises the running max,
because ``rm_j < m + ln λ < m`` for λ < 1. So the running max before tile j
is the plain prefix maximum of the tile row maxima,

    M_j[r] = max_{j' < j} rm_{j'}[r],

whatever was skipped before, and

    skip_j  <=>  for all valid rows r:  rm_j[r] < M_j[r] + ln λ.

This routine computes every tile's row maxima first, takes the exclusive
prefix maximum with ``np.maximum.accumulate`` and applies the test, with no
online-softmax state. It is a second statement of the decisions against
which the tile walk is checked; it also makes the decisions monotone in λ
(a larger λ raises every threshold).
"""
from __future__ import annotations

import math

import numpy as np

from . import layout

TILE = 128


def tile_row_max(q, k, cu_seqlens, Hq, Hkv, causal, scale, item, cu_seqlens_k=None) -> np.ndarray:
    """``rm[j, r]``: the max score of query row r over key tile j (visited tiles).

    With ``cu_seqlens_k`` the queries are the last positions of their
    sequence (chunked prefill, bottom-right causal alignment)."""
    s, h, i = item
    cu = [int(x) for x in cu_seqlens]
    cuk = cu if cu_seqlens_k is None else [int(x) for x in cu_seqlens_k]
    a, Lq = cu[s], cu[s + 1] - cu[s]
    ak, Lk = cuk[s], cuk[s + 1] - cuk[s]
    off = Lk - Lq
    n = layout.tiles(Lk)
    g = h // (Hq // Hkv)
    r0, r1 = i * TILE, min((i + 1) * TILE, Lq)
    last = min((off + r1 - 1) // TILE, n - 1) if causal else n - 1
    keys = np.arange(0, min((last + 1) * TILE, Lk))
    S = (q[a + r0:a + r1, h, :] @ k[ak + keys, g, :].T) * scale      # [rows, keys]
    if causal:
        S = np.where(keys[None, :] > off + np.arange(r0, r1)[:, None], -np.inf, S)
    pad = (last + 1) * TILE - S.shape[1]
    S = np.pad(S, ((0, 0), (0, pad)), constant_values=-np.inf)
    return S.reshape(S.shape[0], last + 1, TILE).max(axis=2).T        # [tiles, rows]


def skip_bits(q, k, cu_seqlens, Hq, Hkv, causal, lam, scale=None, item=(0, 0, 0),
              cu_seqlens_k=None) -> np.ndarray:
    """Bool array over visited key tiles: True where the tile is skipped."""
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[2])
    rm = tile_row_max(q, k, cu_seqlens, Hq, Hkv, causal, scale, item, cu_seqlens_k)
    if lam == 0:
        return np.zeros(rm.shape[0], bool)
    prefix = np.maximum.accumulate(rm, axis=0)
    before = np.vstack([np.full((1, rm.shape[1]), -np.inf), prefix[:-1]])
    return np.all(rm < before + math.log(lam), axis=1)
