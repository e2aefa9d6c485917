"""Shared test inputs: planted tiles and small seeded problems.

Only builds inputs (bf16 bit patterns); holds no attention arithmetic.
"""
from __future__ import annotations

import json
import os
import functools

import numpy as np

from gen import inputs as gi

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def planted_golden():
    with open(os.path.join(GOLDEN, "planted_tiles.json")) as f:
        return json.load(f)


def planted_problem(tokens=None, causal=True, lam=0.01, lengths=None) -> gi.Problem:
    """Q rows = e_0; K rows of tile j = b[j] e_0; V rows = c[j] e_0 + e_1.

    ``lengths`` packs several copies (each sequence restarts at tile 0).
    """
    g = planted_golden()["construction"]
    b = np.asarray(g["b"], np.float32)
    c = np.asarray(g["c"], np.float32)
    if lengths is None:
        lengths = [tokens or g["tokens"]]
    d = 128
    qs, ks, vs = [], [], []
    for L in lengths:
        t = np.arange(L)
        q = np.zeros((L, 1, d), np.float32)
        q[:, 0, 0] = 1.0
        k = np.zeros((L, 1, d), np.float32)
        k[:, 0, 0] = b[t // 128]
        v = np.zeros((L, 1, d), np.float32)
        v[:, 0, 0] = c[t // 128]
        v[:, 0, 1] = 1.0
        qs.append(q), ks.append(k), vs.append(v)
    cu = np.zeros(len(lengths) + 1, np.int32)
    cu[1:] = np.cumsum(lengths)
    cat = lambda xs: gi.bf16_bits_from_f32(np.concatenate(xs))  # noqa: E731
    return gi.Problem("planted", cat(qs), cat(ks), cat(vs), cu, 1, 1, d, causal, lam)


@functools.lru_cache(maxsize=None)
def small_problem(key: str) -> gi.Problem:
    """Named parity-sized problems (seeded, same recipe as the workloads)."""
    if key == "C0":
        return gi.config("C0")
    if key == "gqa_ragged":      # several tiles, ragged tails, GQA G = 2
        return gi.small(key, [300, 1000, 129, 640], Hq=4, Hkv=2, seed=1)
    if key == "gqa4":            # the Llama grouping G = 4, two sequences
        return gi.small(key, [1536, 777], Hq=8, Hkv=2, seed=2)
    if key == "weak_sink":       # sink too weak to dominate: mixed keep / skip
        return gi.small(key, [1024, 900], Hq=2, Hkv=1, seed=3, sink=1.0, window=1.0)
    if key == "no_sink":         # running max grows tile by tile
        return gi.small(key, [700], Hq=2, Hkv=2, seed=4, sink=0.0, window=0.0)
    if key == "tiny":            # shorter than one tile
        return gi.small(key, [1, 77, 128], Hq=2, Hkv=1, seed=5)
    raise KeyError(key)


def full_problem(name: str, sink: float = 4.0) -> gi.Problem:
    """A full-size workload (C1, C2, C3; C4 is C2's values, quantised by the
    FP8 tests), generated once per test session and shared by every module."""
    return _full("C2" if name == "C4" else name, sink)


@functools.lru_cache(maxsize=4)
def _full(name: str, sink: float) -> gi.Problem:
    return gi.config(name, sink=sink)


def f64(bits):
    w = np.asarray(bits, np.uint16).astype(np.uint32) << np.uint32(16)
    return w.view(np.float32).astype(np.float64)
