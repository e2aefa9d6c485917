"""Pins of the block-importance and top-p oracle (UniPrefill page, §3.2 Eq. 3-4, §3.3).

Each test checks the oracle against something other than its own formula:
closed forms for keys that make the scores constant per block, the mass
invariant (every window row's weights add up to 1), GQA symmetry, a
hand-worked top-p fixture and brute-force subset search.
"""
from __future__ import annotations

import itertools
import json
import math
import os

import numpy as np
import pytest

from gen import inputs as gi
from oracle import importance as imp

G = 128
HERE = os.path.dirname(__file__)


def bits(x):
    return gi.bf16_bits_from_f32(np.asarray(x, np.float32))


def count_in_block(g, P, N):
    """Keys of block g at positions <= P (a causal row at position P)."""
    lo, hi = g * G, min((g + 1) * G, N)
    return max(0, min(hi, P + 1) - lo)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("N,n", [(300, 5), (128, 128), (1000, 64), (77, 200)])
def test_identical_keys_give_uniform_weights(causal, N, n):
    # all keys equal: every key a row may see gets weight 1 / (number it may see)
    rng = np.random.default_rng(1)
    q = bits(rng.standard_normal((N, 1, 128)))
    k = bits(np.broadcast_to(rng.standard_normal((1, 1, 128)), (N, 1, 128)))
    got = imp.block_importance(q, k, np.array([0, N]), 1, 1, n, causal)[0]
    ne = min(n, N)
    nb = (N + G - 1) // G
    want = np.zeros(nb)
    for P in range(N - ne, N):
        seen = P + 1 if causal else N
        for g in range(nb):
            c = count_in_block(g, P, N) if causal else min((g + 1) * G, N) - g * G
            want[g] += c / seen
    want /= ne * G
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=0)


@pytest.mark.parametrize("causal", [True, False])
def test_block_constant_scores_closed_form(causal):
    # q = e0, keys of block g = a_g e0: every score in block g is a_g / sqrt(d),
    # so a row's weight on block g is c_g exp(S_g) / sum_g' c_g' exp(S_g')
    # with c_g the keys of block g the row may see
    N, n, d = 450, 9, 128
    a = np.array([0.0, 8.0, -8.0, 16.0])
    q = np.zeros((N, 1, d), np.float32)
    q[:, 0, 0] = 1.0
    k = np.zeros((N, 1, d), np.float32)
    for i in range(N):
        k[i, 0, 0] = a[i // G]
    got = imp.block_importance(bits(q), bits(k), np.array([0, N]), 1, 1, n, causal)[0]
    S = a / math.sqrt(d)
    want = np.zeros(4)
    for P in range(N - n, N):
        c = np.array([count_in_block(g, P, N) if causal else min((g + 1) * G, N) - g * G
                      for g in range(4)], np.float64)
        w = c * np.exp(S)
        want += w / w.sum()
    want /= n * G
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=0)


@pytest.mark.parametrize("causal", [True, False])
def test_mass_invariant(causal):
    # sum over blocks of G * s_g = mean over window rows of (sum of the row's weights) = 1
    p = gi.small("imp", [700, 129, 1, 300], Hq=4, Hkv=2, seed=5)
    sc = imp.block_importance(p.q, p.k, p.cu_seqlens, 4, 2, 37, causal)
    off = imp.block_offsets(p.cu_seqlens)
    for s in range(p.n_seqs):
        tot = sc[:, off[s]:off[s + 1]].sum(axis=1) * G
        np.testing.assert_allclose(tot, 1.0, rtol=0, atol=1e-12)
    assert (sc >= 0).all()


def test_gqa_heads_follow_their_kv_head():
    N, d = 512, 128
    rng = np.random.default_rng(2)
    u = rng.standard_normal(d).astype(np.float32)
    q = np.broadcast_to(u, (N, 4, d)).copy()                  # every query row of every head is u
    k = (0.1 * rng.standard_normal((N, 2, d))).astype(np.float32)
    k[256:384, 1] = 3.0 * u                                   # KV head 1: block 2 aligned with u
    sc = imp.block_importance(bits(q), bits(k), np.array([0, N]), 4, 2, 16, True)
    assert np.array_equal(sc[0], sc[1]) and np.array_equal(sc[2], sc[3])
    # heads 2, 3 put almost all their weight on block 2; heads 0, 1 spread it
    assert sc[2, 2] * G > 0.99
    assert sc[0].max() * G < 0.5


def test_window_longer_than_sequence_is_whole_sequence():
    p = gi.small("imp", [200], Hq=1, Hkv=1, seed=3)
    a = imp.block_importance(p.q, p.k, p.cu_seqlens, 1, 1, 200, True)
    b = imp.block_importance(p.q, p.k, p.cu_seqlens, 1, 1, 1000, True)
    assert np.array_equal(a, b)


def test_head_mean():
    s = np.array([[1.0, 2.0], [3.0, 6.0]])
    assert np.array_equal(imp.head_mean(s), [2.0, 4.0])


def test_top_p_golden():
    with open(os.path.join(HERE, "golden", "top_p_cases.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        for sel in c["select"]:
            order, k = imp.top_p(np.array(c["scores"]), sel["p"])
            assert order.tolist() == c["order"]
            assert k == sel["k"], (c["scores"], sel)
            assert sorted(order[:k].tolist()) == sel["kept"]


def test_top_p_is_the_smallest_subset():
    # brute force: the fewest blocks whose scores reach p * total (dyadic scores: exact sums)
    rng = np.random.default_rng(4)
    for _ in range(200):
        nb = int(rng.integers(1, 9))
        s = rng.integers(0, 9, nb) / 64.0
        if s.sum() == 0:
            s[0] = 1 / 64.0
        p = float(rng.choice([0.1, 0.25, 0.5, 0.7, 0.9, 0.95, 1.0]))
        order, k = imp.top_p(s, p)
        best = min(r for r in range(1, nb + 1)
                   for sub in itertools.combinations(range(nb), r)
                   if s[list(sub)].sum() >= p * s.sum())
        assert k == best
        assert s[order[:k]].sum() >= p * s.sum()
        assert all(s[order[i]] >= s[order[i + 1]] for i in range(nb - 1))


def test_select_packed_layout():
    cu = np.array([0, 300, 301, 1000])
    off = imp.block_offsets(cu)
    assert off.tolist() == [0, 3, 4, 10]
    rng = np.random.default_rng(6)
    m = rng.random(10)
    order, ks, keep = imp.select(m, cu, 0.5)
    for s in range(3):
        a, b = off[s], off[s + 1]
        o, k = imp.top_p(m[a:b], 0.5)
        assert np.array_equal(order[a:b], o) and ks[s] == k
        assert set(np.flatnonzero(keep[a:b])) == set(o[:k])
