"""GPU parity: the CUDA library (through its C interface) against the oracle.

Skip bits must match bit for bit outside the 1e-3 decision margin; outputs
are compared with the oracle in mask-replay mode (the oracle takes the GPU's
decisions) within max-abs 2e-2 / mean-abs 2e-3 (bf16) and lse within 1e-3.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import _cases
import _gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("lam", [0.01, 0.0])
def test_c0(lam):
    p = _cases.small_problem("C0")
    g = _gpu.run(p, lam=lam)
    out, lse = _gpu.host(g)
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    _gpu.compare(p, g)
    if lam == 0:
        assert not g["bitmap"].any()


@pytest.mark.parametrize("lam", ["0", "0.0001", "0.01", "0.05", "0.5"])
@pytest.mark.parametrize("causal,L", [(True, 1024), (False, 1024), (True, 1000), (False, 1000)])
def test_planted_golden(lam, causal, L):
    """Decisions enumerated by hand (tests/golden/planted_tiles.json)."""
    golden = _cases.planted_golden()
    p = _cases.planted_problem(tokens=L, causal=causal)
    g = _gpu.run(p, lam=float(lam), causal=causal)
    from oracle import layout
    skipped = set(golden["skipped"][lam])
    n = layout.tiles(L)
    for i in range(n):
        visited = range(i + 1) if causal else range(n)
        want = np.array([(j in skipped) and (j in visited) for j in range(n)])
        assert np.array_equal(layout.row_bits(g["bitmap"], p.cu_seqlens, 1, 0, 0, i), want), i
    _gpu.compare(p, g)


@pytest.mark.parametrize("key,lam", [("gqa_ragged", 0.01), ("gqa_ragged", 0.0), ("gqa4", 0.01),
                                     ("weak_sink", 0.05), ("weak_sink", 0.5), ("no_sink", 0.0),
                                     ("no_sink", 0.3), ("tiny", 0.01), ("tiny", 0.0)])
@pytest.mark.parametrize("causal", [True, False])
def test_small_cases(key, lam, causal):
    p = _cases.small_problem(key)
    g = _gpu.run(p, lam=lam, causal=causal)
    out, lse = _gpu.host(g)
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    _gpu.compare(p, g)


def test_deterministic():
    p = _cases.small_problem("weak_sink")
    a = _gpu.run(p, lam=0.05)
    b = _gpu.run(p, lam=0.05)
    assert torch.equal(a["out"], b["out"]) and torch.equal(a["lse"], b["lse"])
    assert np.array_equal(a["bitmap"], b["bitmap"])


def test_packed_equals_separate():
    """A packed batch gives the same rows as each sequence run alone."""
    p = _cases.small_problem("gqa_ragged")
    whole = _gpu.run(p, lam=0.01)
    from gen import inputs as gi
    for s in range(p.n_seqs):
        a, b = int(p.cu_seqlens[s]), int(p.cu_seqlens[s + 1])
        one = gi.Problem("one", p.q[a:b], p.k[a:b], p.v[a:b], np.array([0, b - a], np.int32),
                         p.Hq, p.Hkv, p.d, True, 0.01)
        g = _gpu.run(one, lam=0.01)
        assert torch.equal(g["out"], whole["out"][a:b])
        assert torch.equal(g["lse"], whole["lse"][:, a:b])
