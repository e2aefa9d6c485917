"""The method: causal prefill attention with dynamic block skipping, in fp64.

Test infrastructure only (see the package docstring).

Source: the dynamic sparse attention deployment guide
("长上下文推理加速方案部署实战：基于动态稀疏注意力机制的推理服务优化指南"),
§3.2 "dynamic sparse attention kernel": the kernel sits inside the online
softmax, keeps the running maximum of the scores, computes each block's local
maximum block by block in order, and declares a block negligible by comparing
that local maximum with the running maximum through the threshold λ; a
negligible block skips the softmax exponentials, the load of its V block and
the product with V. §3.3 and §6.1 say a larger λ prunes more blocks (0.001
conservative, 0.1 aggressive, 0.01 the default of §5 step 3, block size 128).

Readings (where the page is silent or self-contradictory):

* threshold form: the block is skipped when its max is below the running max
  by more than ``-ln λ``, i.e. ``rm < m + ln λ`` (the probability ratio
  ``exp(rm - m)`` is below λ). This is the only form under which a larger λ
  prunes more, as §3.3/§6.1 state. λ = 0 disables skipping.
* granularity: the test is per query row and the tile is skipped only if it
  holds for every valid row of the 128-row query tile.
* running max: the maximum over the tiles before j (skipped ones included;
  a skipped tile cannot raise it since ``rm < m + ln λ < m`` for λ < 1).
* order: key tiles ascending from 0 up to the diagonal tile (causal), one
  query tile at a time; the first tile is never skipped (m = -inf).
* strict ``<``; rows past the sequence end take no part in the vote.
* lse is the natural-log log-sum-exp over the kept entries.

Per query tile (sequence s, query head h, tile i) with g = h // (Hq/Hkv):

    m = -inf, l = 0, O = 0
    for j = 0 .. i (causal) or n-1:
        S  = Q_i K_j^T * scale          (-inf where key > query, or key >= L)
        rm = max over keys of S         (per row)
        skip = all over valid rows of (rm < m + ln λ)
        if skip: record bit (i, j); continue
        m' = max(m, rm);  a = exp(m - m')
        P = exp(S - m');  l = a l + rowsum(P);  O = a O + P V_j;  m = m'
    out = O / l,  lse = m + ln l

Mask-replay mode takes ``skip`` from a given bitmap instead of the rule
(used to compare outputs with a GPU run whose decisions are known).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

from . import layout

TILE = 128


@dataclasses.dataclass
class Result:
    out: np.ndarray            # float64 [T, Hq, d]; NaN on rows not computed
    lse: np.ndarray            # float64 [Hq, T]; NaN on rows not computed
    bitmap: np.ndarray         # uint32 words, layout of ``oracle.layout``
    margins: dict              # (s, h, i) -> float64 [n_visited]: min_r (m + ln λ - rm)
    kept: dict                 # (s, h, i) -> list of kept key tiles


def all_items(cu_seqlens, Hq: int):
    cu = [int(x) for x in cu_seqlens]
    items = []
    for s in range(len(cu) - 1):
        n = layout.tiles(cu[s + 1] - cu[s])
        for h in range(Hq):
            for i in range(n):
                items.append((s, h, i))
    return items


def walk_one(q, k, v, cu_seqlens, Hq, Hkv, causal, lam, scale, item, replay=None,
             cu_seqlens_k=None):
    """Run the tile walk for one query tile; return (out rows, lse rows, bits, margins, kept).

    ``replay``: optional bool array over key tiles; when given, the skip
    decisions are read from it instead of computed.

    ``cu_seqlens_k`` (chunked prefill): key/value sequence boundaries when they
    differ from the queries'. Sequence s then has Lk keys and its Lq queries
    are the last Lq positions of the sequence (query row r sits at position
    Lk - Lq + r, bottom-right causal alignment), as when a long prompt is
    prefilled chunk by chunk against the KV of the chunks before it (the
    prefill-acceleration blog's §3.1 chunked prefill; FlowPrefill's chunked
    prefill baseline). Without it, Lk = Lq and positions start at 0.
    """
    s, h, i = item
    cuq = [int(x) for x in cu_seqlens]
    cuk = cuq if cu_seqlens_k is None else [int(x) for x in cu_seqlens_k]
    aq, Lq = cuq[s], cuq[s + 1] - cuq[s]
    ak, Lk = cuk[s], cuk[s + 1] - cuk[s]
    off = Lk - Lq
    if causal and off < 0:
        raise ValueError("causal chunked prefill needs at least as many keys as queries")
    n = layout.tiles(Lk)
    g = h // (Hq // Hkv)
    r0, r1 = i * TILE, min((i + 1) * TILE, Lq)
    Qi = q[aq + r0:aq + r1, h, :]
    qpos = off + np.arange(r0, r1)
    nrow = r1 - r0
    m = np.full(nrow, -np.inf)
    l = np.zeros(nrow)
    O = np.zeros((nrow, q.shape[2]))
    last = min((off + r1 - 1) // TILE, n - 1) if causal else n - 1
    ln_lam = math.log(lam) if lam > 0 else -np.inf
    bits = np.zeros(n, bool)
    margins = np.full(last + 1, -np.inf)
    kept = []
    for j in range(last + 1):
        c0, c1 = j * TILE, min((j + 1) * TILE, Lk)
        Kj = k[ak + c0:ak + c1, g, :]
        Vj = v[ak + c0:ak + c1, g, :]
        S = (Qi @ Kj.T) * scale
        if causal:
            S = np.where(np.arange(c0, c1)[None, :] > qpos[:, None], -np.inf, S)
        rm = S.max(axis=1)
        with np.errstate(invalid="ignore"):
            margins[j] = np.min(m + ln_lam - rm)
        if replay is not None:
            skip = bool(replay[j])
        else:
            skip = bool(np.all(rm < m + ln_lam))
        if skip:
            bits[j] = True
            continue
        kept.append(j)
        m_new = np.maximum(m, rm)
        with np.errstate(invalid="ignore"):
            alpha = np.where(m_new == -np.inf, 0.0, np.exp(m - m_new))
            P = np.where(m_new[:, None] == -np.inf, 0.0, np.exp(S - m_new[:, None]))
        l = alpha * l + P.sum(axis=1)
        O = alpha[:, None] * O + P @ Vj
        m = m_new
    if not kept or np.any(l <= 0):
        raise ValueError(f"item {item}: a row has no kept key (invalid replay bitmap)")
    return O / l[:, None], m + np.log(l), bits, margins, kept


def prefill_fwd(q, k, v, cu_seqlens, Hq: int, Hkv: int, causal: bool = True, lam: float = 0.01,
                scale: float | None = None, items=None, replay_bitmap=None,
                cu_seqlens_k=None) -> Result:
    """Tile walk over ``items`` (all query tiles by default).

    q, k, v: float64 values ``[T, H, d]`` (k, v over the key tokens when
    ``cu_seqlens_k`` is given). ``replay_bitmap``: uint32 words in the
    interface layout; when given, decisions come from it (mask replay).
    """
    if not (lam == 0 or 0 < lam < 1):
        raise ValueError("lambda must be 0 or in (0, 1)")
    T, _, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    cu = np.asarray(cu_seqlens, np.int64)
    cuk = cu if cu_seqlens_k is None else np.asarray(cu_seqlens_k, np.int64)
    out = np.full((T, Hq, d), np.nan)
    lse = np.full((Hq, T), np.nan)
    bitmap = np.zeros(layout.total_words(cu, Hq, cuk), np.uint32)
    margins, kept_all = {}, {}
    for item in (all_items(cu, Hq) if items is None else items):
        s, h, i = item
        replay = None
        if replay_bitmap is not None:
            replay = layout.row_bits(replay_bitmap, cu, Hq, s, h, i, cuk)
        o, ls, bits, mg, kept = walk_one(q, k, v, cu, Hq, Hkv, causal, lam, scale, item, replay,
                                         cu_seqlens_k=cuk)
        a, L = int(cu[s]), int(cu[s + 1] - cu[s])
        r0, r1 = i * TILE, min((i + 1) * TILE, L)
        out[a + r0:a + r1, h, :] = o
        lse[h, a + r0:a + r1] = ls
        base = layout.row_offset(cu, Hq, s, h, i, cuk)
        for j in np.nonzero(bits)[0]:
            bitmap[base + j // 32] |= np.uint32(1 << (int(j) % 32))
        margins[item] = mg
        kept_all[item] = kept
    return Result(out, lse, bitmap, margins, kept_all)
