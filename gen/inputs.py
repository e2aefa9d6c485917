"""Seeded synthetic inputs for block-skipping causal prefill attention.

This module only draws and packs input data. It holds none of the
attention arithmetic: no scores, no softmax, no skip rule. Both the CPU
oracle and the GPU path consume what it returns, so neither has to trust
the other's inputs.

Recipe (one sequence of length L, Hq query heads, Hkv key/value heads,
head dim d, G = Hq / Hkv):

* one random direction per KV head: ``u_g = sqrt(d) * z / |z|`` with
  ``z ~ N(0, I_d)``;
* ``Q[t, h] = 0.5 * N(0, 1) + u_{h // G}`` (query heads of a group share u);
* ``K[t, g] = 0.5 * N(0, 1) + sink * u_g`` on keys ``t < sink_len``
  (an attention sink) ``+ window * u_g`` on the last ``window_len``
  positions of every ``window_period`` segment (a local-window bias);
* ``V = N(0, 1)``.

Values are drawn in float32 from numpy's PCG64 ``default_rng`` (platform
independent) and rounded to bfloat16 with round-to-nearest-even. bf16 data
is carried as ``uint16`` bit patterns. Sequences of a packed (varlen) batch
each draw from their own generator ``default_rng([seed, s])``.

The named workloads are the synthetic stand-ins for the long-context
prefill inputs the block-sparse prefill pages talk about (Llama-3-8B
attention shape: 32 query heads, 8 KV heads, head dim 128).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

TILE = 128
HEAD_DIM = 128
_CHUNK_TOKENS = 4096


@dataclasses.dataclass
class Problem:
    """One packed prefill-attention input.

    q: uint16 bf16 bits ``[total_tokens, Hq, d]``
    k, v: uint16 bf16 bits ``[total_tokens, Hkv, d]``
    cu_seqlens: int32 ``[n_seqs + 1]`` prefix sums of the sequence lengths
    """

    name: str
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    cu_seqlens: np.ndarray
    Hq: int
    Hkv: int
    d: int
    causal: bool = True
    lam: float = 0.01
    # chunked prefill: key/value boundaries when q holds only each sequence's
    # last positions (k, v are then packed by these instead of cu_seqlens)
    cu_seqlens_k: np.ndarray | None = None

    @property
    def n_seqs(self) -> int:
        return int(self.cu_seqlens.shape[0] - 1)

    @property
    def total_tokens(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def seqlens(self) -> np.ndarray:
        return np.diff(self.cu_seqlens.astype(np.int64))


def bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); return bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounding = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + rounding) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns to float32."""
    b = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32)


def _directions(rng: np.random.Generator, hkv: int, d: int) -> np.ndarray:
    z = rng.standard_normal((hkv, d))
    return (z / np.linalg.norm(z, axis=1, keepdims=True) * math.sqrt(d)).astype(np.float32)


def sequence(rng: np.random.Generator, L: int, Hq: int, Hkv: int, d: int = HEAD_DIM,
             sink: float = 4.0, sink_len: int = 64,
             window: float = 0.0, window_period: int = 4096, window_len: int = 512):
    """Draw Q, K, V (bf16 bits) of one sequence following the module recipe."""
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    G = Hq // Hkv
    u = _directions(rng, Hkv, d)
    uq = np.repeat(u, G, axis=0)  # query head h uses its group's direction
    q = np.empty((L, Hq, d), np.uint16)
    k = np.empty((L, Hkv, d), np.uint16)
    v = np.empty((L, Hkv, d), np.uint16)
    for t0 in range(0, L, _CHUNK_TOKENS):
        t1 = min(L, t0 + _CHUNK_TOKENS)
        q[t0:t1] = bf16_bits_from_f32(
            np.float32(0.5) * rng.standard_normal((t1 - t0, Hq, d), dtype=np.float32) + uq)
    for t0 in range(0, L, _CHUNK_TOKENS):
        t1 = min(L, t0 + _CHUNK_TOKENS)
        kk = np.float32(0.5) * rng.standard_normal((t1 - t0, Hkv, d), dtype=np.float32)
        pos = np.arange(t0, t1)
        bias = np.zeros(t1 - t0, np.float32)
        bias[pos < sink_len] += np.float32(sink)
        if window:
            bias[(pos % window_period) >= window_period - window_len] += np.float32(window)
        kk += bias[:, None, None] * u[None, :, :]
        k[t0:t1] = bf16_bits_from_f32(kk)
    for t0 in range(0, L, _CHUNK_TOKENS):
        t1 = min(L, t0 + _CHUNK_TOKENS)
        v[t0:t1] = bf16_bits_from_f32(rng.standard_normal((t1 - t0, Hkv, d), dtype=np.float32))
    return q, k, v


def packed(name: str, lengths, Hq: int, Hkv: int, seed: int = 0, d: int = HEAD_DIM,
           causal: bool = True, lam: float = 0.01, **recipe) -> Problem:
    """Pack several sequences, each drawn from ``default_rng([seed, s])``."""
    lengths = [int(x) for x in lengths]
    if not lengths or min(lengths) < 1:
        raise ValueError("every sequence needs at least one token")
    cu = np.zeros(len(lengths) + 1, np.int32)
    cu[1:] = np.cumsum(lengths)
    T = int(cu[-1])
    q = np.empty((T, Hq, d), np.uint16)
    k = np.empty((T, Hkv, d), np.uint16)
    v = np.empty((T, Hkv, d), np.uint16)
    for s, L in enumerate(lengths):
        rng = np.random.default_rng([seed, s])
        a, b = int(cu[s]), int(cu[s + 1])
        q[a:b], k[a:b], v[a:b] = sequence(rng, L, Hq, Hkv, d, **recipe)
    return Problem(name, q, k, v, cu, Hq, Hkv, d, causal, lam)


def chunk(p: Problem, lq) -> Problem:
    """Keep only the last ``lq[s]`` queries of every sequence of ``p`` (all keys stay)."""
    qs, cuq = [], [0]
    for s, n in enumerate(lq):
        b = int(p.cu_seqlens[s + 1])
        qs.append(p.q[b - int(n):b])
        cuq.append(cuq[-1] + int(n))
    return Problem(p.name + "_chunk", np.concatenate(qs), p.k, p.v, np.asarray(cuq, np.int32),
                   p.Hq, p.Hkv, p.d, p.causal, p.lam, cu_seqlens_k=p.cu_seqlens.copy())


def varlen_lengths(seed: int = 0, n: int = 16, lo: int = 4096, hi: int = 65536) -> list:
    """Log-uniform lengths in [lo, hi], rounded to a multiple of the tile."""
    rng = np.random.default_rng(seed)
    x = np.exp(rng.uniform(math.log(lo), math.log(hi), n))
    L = np.clip(np.rint(x / TILE).astype(np.int64) * TILE, lo, hi)
    return [int(a) for a in L]


# Named workloads.  C0 is the small single-head case; C1 the Llama-3-8B
# attention shape at 32K; C2 the same heads at 128K (the headline layer);
# C3 a continuous-batching mix; C4 reuses C2's values (the FP8 variant
# quantises them).  ``scale`` of the sink is the recipe's 4.0 unless the
# diagnostic weak-sink run asks for less.
_LLAMA = dict(Hq=32, Hkv=8)
_WINDOW = dict(window=2.0, window_period=4096, window_len=512)


def config(name: str, seed: int = 0, lam: float = 0.01, sink: float = 4.0) -> Problem:
    if name == "C0":
        return packed(name, [2048], 1, 1, seed, lam=lam, sink=sink)
    if name == "C1":
        return packed(name, [32768], seed=seed, lam=lam, sink=sink, **_LLAMA, **_WINDOW)
    if name in ("C2", "C4"):
        return packed(name, [131072], seed=seed, lam=lam, sink=sink, **_LLAMA, **_WINDOW)
    if name == "C3":
        return packed(name, varlen_lengths(seed), seed=seed, lam=lam, sink=sink,
                      **_LLAMA, **_WINDOW)
    raise KeyError(name)


def small(name: str, lengths, Hq: int = 4, Hkv: int = 2, seed: int = 0, lam: float = 0.01,
          causal: bool = True, sink: float = 4.0, window: float = 2.0,
          window_period: int = 1024, window_len: int = 256) -> Problem:
    """A parity-sized problem with the same recipe and a shorter window period."""
    return packed(name, lengths, Hq, Hkv, seed, causal=causal, lam=lam, sink=sink,
                  window=window, window_period=window_period, window_len=window_len)


def head_range(Hkv: int, world: int, rank: int) -> tuple:
    """KV heads [lo, hi) of rank ``rank`` when a layer's heads are split over
    ``world`` processes: contiguous, sizes differing by at most one."""
    if not 0 <= rank < world or world > Hkv:
        raise ValueError("need 0 <= rank < world <= Hkv")
    return rank * Hkv // world, (rank + 1) * Hkv // world


def split_heads(p: Problem, rank: int, world: int) -> Problem:
    """The part of ``p`` one process computes when the KV heads are split over
    ``world`` processes: KV heads ``head_range`` and the query heads of their
    groups, as contiguous arrays (query head h of the piece is query head
    lo * G + h of the layer). Sequences, lengths and values are unchanged."""
    G = p.Hq // p.Hkv
    lo, hi = head_range(p.Hkv, world, rank)
    return Problem(f"{p.name}_heads{lo}-{hi}", np.ascontiguousarray(p.q[:, lo * G:hi * G]),
                   np.ascontiguousarray(p.k[:, lo:hi]), np.ascontiguousarray(p.v[:, lo:hi]),
                   p.cu_seqlens, (hi - lo) * G, hi - lo, p.d, p.causal, p.lam,
                   cu_seqlens_k=p.cu_seqlens_k)
