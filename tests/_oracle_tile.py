"""The oracle's reference for one query tile (test infrastructure).

``reference`` recomputes one query tile (sequence s, query head h, tile i)
with the oracle's tile walk twice: with its own decisions (the skip bits and
decision margins the GPU's bits are checked against) and in mask-replay mode
with the GPU's bits (the output and lse the GPU's are checked against).
Only the key tiles the walk visits are read, so a sampled tile of a 128K
layer costs at most its 1024 tile visits (a few tenths of a second).
This module imports no GPU code.
"""
from __future__ import annotations

import math

import numpy as np

from oracle import layout, numerics, tile_walk


def _values(arrays, scales, qrows, krows, h, g):
    """fp64 values of query rows ``qrows`` of head h and key/value rows
    ``krows`` of head g: bf16 bit patterns, or E4M3 codes times their scale."""
    q, k, v = arrays
    if scales is None:
        return (numerics.bf16_to_f64(q[qrows][:, [h]]), numerics.bf16_to_f64(k[krows][:, [g]]),
                numerics.bf16_to_f64(v[krows][:, [g]]))
    sq, sk, sv = (np.asarray(x, np.float64) for x in scales)
    return (numerics.e4m3_to_f64(q[qrows][:, [h]]) * sq[h],
            numerics.e4m3_to_f64(k[krows][:, [g]]) * sk[g],
            numerics.e4m3_to_f64(v[krows][:, [g]]) * sv[g])


def reference(arrays, scales, cu, cuk, Hq, Hkv, causal, lam, item, got):
    """Oracle for one query tile.

    ``got``: the GPU's skip bits of the tile's row (bool per key tile, the
    row's visited prefix). Returns (want bits, margins, out rows, lse rows,
    last visited key tile).
    """
    s, h, i = item
    a, L = int(cu[s]), int(cu[s + 1] - cu[s])
    ak, Lk = int(cuk[s]), int(cuk[s + 1] - cuk[s])
    off = Lk - L
    r1 = min(i * 128 + 128, L)
    last = min((off + r1 - 1) // 128, layout.tiles(Lk) - 1) if causal else layout.tiles(Lk) - 1
    hi = min((last + 1) * 128, Lk)
    # causal: keys past the last visited tile are never read, so the sequence
    # truncated after it (queries keep their positions, so the chunk keeps the
    # rows that end at key hi) walks identically
    q_hi = hi - off if causal else L
    q, k, v = _values(arrays, scales, slice(a, a + q_hi), slice(ak, ak + hi), h, h // (Hq // Hkv))
    scale = 1.0 / math.sqrt(q.shape[2])
    sub_q, sub_k = [0, q_hi], [0, hi]
    _, _, want, mg, _ = tile_walk.walk_one(q, k, v, sub_q, 1, 1, causal, lam, scale, (0, 0, i),
                                           cu_seqlens_k=sub_k)
    o_ref, lse_ref, _, _, _ = tile_walk.walk_one(q, k, v, sub_q, 1, 1, causal, lam, scale,
                                                 (0, 0, i), replay=np.asarray(got, bool),
                                                 cu_seqlens_k=sub_k)
    return want[:last + 1], mg, o_ref, lse_ref, last
