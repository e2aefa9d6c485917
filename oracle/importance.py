"""Token-block importance and top-p block selection, in fp64.

Test infrastructure only (see the package docstring).

Source: "UniPrefill：通过分块动态稀疏化实现通用长上下文预填充加速"
(bittide.aicompass.dev article), §3.2 "token importance estimation",
Eq. (3)-(4), and §3.3 "top-p percent token selection".

§3.2: the weight token i carries for the next-token prediction is its
attention weight from the last position; to lower the variance the page
averages the weights of the last n query positions (Eq. 3), and works on
blocks of G consecutive keys: the partial product S = Q[N-n:N] K^T is taken,
the softmax is normalised across the whole key range first, and only then
are the weights summed inside each block and divided by G (Eq. 4).

§3.3: with the block scores sorted in descending order, the kept set is the
shortest prefix of that order whose scores add up to at least p times the
sum of all block scores.

Readings where the page is silent:

* causal: window row j attends the keys i <= j (the weights a causal model
  computes); ``causal=False`` lets every window row see all N keys, which is
  Eq. (2)'s form for the last row.
* heads: the page writes one head. Scores are per query head (GQA: head h
  uses KV head h // (Hq/Hkv)); the selection takes the mean over query heads.
* block size G = 128 (the tile and page size of this library); Eq. (4)
  divides by G for every block, the short last block included.
* window: n_eff = min(n, N) rows; the average is over those rows.
* score scale 1/sqrt(d_k).
* ties in the sort keep ascending block order; p in (0, 1].
* k* = the first prefix length (from 1) whose running sum reaches p times
  the total, the total being the running sum over all blocks.
"""
from __future__ import annotations

import math

import numpy as np

from .numerics import bf16_to_f64

BLOCK = 128


def window_weights(qh: np.ndarray, kh: np.ndarray, n: int, causal: bool) -> np.ndarray:
    """Softmax weights A[j, i] of the last n_eff query rows over all N keys.

    qh: float64 [N, d] queries of one head; kh: float64 [N, d] its keys.
    Row r of the result is query position N - n_eff + r.
    """
    N, d = qh.shape
    ne = min(int(n), N)
    pos = np.arange(N - ne, N)
    S = (qh[N - ne:] @ kh.T) / math.sqrt(d)
    if causal:
        S = np.where(np.arange(N)[None, :] <= pos[:, None], S, -np.inf)
    S = S - S.max(axis=1, keepdims=True)
    E = np.exp(S)
    return E / E.sum(axis=1, keepdims=True)


def sequence_scores(qh: np.ndarray, kh: np.ndarray, n: int, causal: bool,
                    G: int = BLOCK) -> np.ndarray:
    """Eq. (4) for one head: block score s_g = (1/G) sum_{i in B_g} (1/n) sum_j A[j, i]."""
    A = window_weights(qh, kh, n, causal)
    s = A.mean(axis=0)                      # Eq. (3): average over the window rows
    N = s.shape[0]
    nb = (N + G - 1) // G
    out = np.zeros(nb)
    for g in range(nb):
        out[g] = s[g * G:min((g + 1) * G, N)].sum() / G
    return out


def block_offsets(cu_seqlens, G: int = BLOCK) -> np.ndarray:
    """First block of every sequence in the packed block axis (n_seqs + 1 entries)."""
    L = np.diff(np.asarray(cu_seqlens, np.int64))
    return np.concatenate([[0], np.cumsum((L + G - 1) // G)]).astype(np.int64)


def block_importance(q_bits, k_bits, cu_seqlens, Hq: int, Hkv: int, n: int, causal: bool = True,
                     G: int = BLOCK) -> np.ndarray:
    """Per-head block scores [Hq, total_blocks] of a packed batch (bf16 bit inputs)."""
    cu = np.asarray(cu_seqlens, np.int64)
    off = block_offsets(cu, G)
    grp = Hq // Hkv
    out = np.zeros((Hq, int(off[-1])))
    for s in range(len(cu) - 1):
        a, b = int(cu[s]), int(cu[s + 1])
        if b == a:
            continue
        for h in range(Hq):
            qh = bf16_to_f64(q_bits[a:b, h])
            kh = bf16_to_f64(k_bits[a:b, h // grp])
            out[h, off[s]:off[s + 1]] = sequence_scores(qh, kh, n, causal, G)
    return out


def head_mean(scores: np.ndarray) -> np.ndarray:
    """The selection score of a block: the mean of its per-head scores."""
    return np.asarray(scores, np.float64).mean(axis=0)


def top_p(scores, p: float):
    """§3.3 on one sequence's block scores: (order, k*).

    order lists the block indices by descending score (ties: ascending
    index); the kept blocks are order[:k*].
    """
    s = np.asarray(scores, np.float64)
    if s.size == 0:
        return np.zeros(0, np.int64), 0
    order = np.array(sorted(range(s.size), key=lambda i: (-s[i], i)), np.int64)
    run = np.cumsum(s[order])
    k_star = int(np.argmax(run >= p * run[-1])) + 1
    return order, k_star


def select(mean_scores, cu_seqlens, p: float, G: int = BLOCK):
    """§3.3 for every sequence of a packed batch: (order, k*, keep) in the C layout.

    order[off_s + r] is the r-th block of sequence s by score (index within
    the sequence), keep[off_s + g] is 1 for a kept block.
    """
    off = block_offsets(cu_seqlens, G)
    order = np.zeros(int(off[-1]), np.int64)
    keep = np.zeros(int(off[-1]), np.uint8)
    ks = np.zeros(len(off) - 1, np.int64)
    for s in range(len(off) - 1):
        a, b = int(off[s]), int(off[s + 1])
        o, k = top_p(mean_scores[a:b], p)
        order[a:b] = o
        keep[a + o[:k]] = 1
        ks[s] = k
    return order, ks, keep
