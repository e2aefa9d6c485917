"""Skip-bitmap word layout of the C interface, restated for the oracle.

Test infrastructure only (see the package docstring).

The deployment guide's §3.5 (observability) asks for the number of skipped
blocks per request to be recorded. The interface records every decision:
one bit per (sequence s, query head h, query tile i, key tile j), set when
tile (i, j) was skipped. For sequence s with n_s = ceil(L_s / 128) tiles a
row (s, h, i) holds W_s = ceil(n_s / 32) uint32 words; bit j % 32 of word
j // 32 is tile j. Rows are ordered h-major then i; sequences follow each
other, so sequence s starts at word sum_{t<s} Hq * n_t * W_t. Bits of tiles
that are not visited (j > i when causal) are zero.
"""
from __future__ import annotations

import numpy as np

TILE = 128


def tiles(L: int) -> int:
    return (int(L) + TILE - 1) // TILE


def row_words(L: int) -> int:
    return (tiles(L) + 31) // 32


def _lens(cu_seqlens, cu_seqlens_k, s):
    cu = np.asarray(cu_seqlens, np.int64)
    cuk = cu if cu_seqlens_k is None else np.asarray(cu_seqlens_k, np.int64)
    return int(cu[s + 1] - cu[s]), int(cuk[s + 1] - cuk[s])


def seq_offsets(cu_seqlens, Hq: int, cu_seqlens_k=None) -> np.ndarray:
    """Word offset of each sequence's block of rows; last entry = total words.

    With separate key boundaries (chunked prefill) a sequence has one row per
    query tile and ceil(key tiles / 32) words per row."""
    off = [0]
    for s in range(len(cu_seqlens) - 1):
        Lq, Lk = _lens(cu_seqlens, cu_seqlens_k, s)
        off.append(off[-1] + Hq * tiles(Lq) * row_words(Lk))
    return np.asarray(off, np.int64)


def total_words(cu_seqlens, Hq: int, cu_seqlens_k=None) -> int:
    return int(seq_offsets(cu_seqlens, Hq, cu_seqlens_k)[-1])


def row_offset(cu_seqlens, Hq: int, s: int, h: int, i: int, cu_seqlens_k=None) -> int:
    Lq, Lk = _lens(cu_seqlens, cu_seqlens_k, s)
    return int(seq_offsets(cu_seqlens, Hq, cu_seqlens_k)[s]) + (h * tiles(Lq) + i) * row_words(Lk)


def get_bit(bitmap: np.ndarray, cu_seqlens, Hq: int, s: int, h: int, i: int, j: int,
            cu_seqlens_k=None) -> bool:
    w = int(bitmap[row_offset(cu_seqlens, Hq, s, h, i, cu_seqlens_k) + j // 32])
    return bool((w >> (j % 32)) & 1)


def row_bits(bitmap: np.ndarray, cu_seqlens, Hq: int, s: int, h: int, i: int,
             cu_seqlens_k=None) -> np.ndarray:
    """The row's bits as a bool array over the sequence's key tiles."""
    Lq, Lk = _lens(cu_seqlens, cu_seqlens_k, s)
    n, W = tiles(Lk), row_words(Lk)
    base = row_offset(cu_seqlens, Hq, s, h, i, cu_seqlens_k)
    words = np.asarray(bitmap[base:base + W], np.uint64)
    return np.array([(int(words[j // 32]) >> (j % 32)) & 1 for j in range(n)], bool)
