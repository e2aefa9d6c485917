"""Pins for the chunked-prefill (query offset) form of the oracle.

A chunk of Lq queries is the last Lq positions of a sequence whose keys and
values (earlier chunks included) number Lk; query r sits at position
Lk - Lq + r (bottom-right causal alignment).

* dense attention with the offset vs torch SDPA with an explicit mask;
* tile walk at λ = 0 vs that dense attention;
* tile walk at λ > 0 vs dense attention over exactly the kept tiles;
* decisions vs the prefix-max closed form;
* with a tile-aligned offset the chunk's rows, lse and skip bits equal those
  of the same rows in a walk over the whole sequence (the walk of a query
  tile does not depend on which other query tiles exist).
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import _cases
from oracle import attention, decisions, layout, numerics, tile_walk

TOL = 1e-12


def chunk_of(p, lq_list):
    """Queries = the last lq tokens of every sequence of ``p``; keys = all."""
    qs, cuq = [], [0]
    for s, lq in enumerate(lq_list):
        b = int(p.cu_seqlens[s + 1])
        qs.append(p.q[b - lq:b])
        cuq.append(cuq[-1] + lq)
    q = np.concatenate(qs)
    return (numerics.bf16_to_f64(q), numerics.bf16_to_f64(p.k), numerics.bf16_to_f64(p.v),
            np.asarray(cuq, np.int64), p.cu_seqlens.astype(np.int64))


CASES = [("gqa_ragged", [300, 1000, 129, 640], [100, 777, 1, 200]),   # offsets 200, 223, 128, 440
         ("weak_sink", [1024, 900], [384, 900]),                      # 640 (aligned), 0
         ("gqa4", [1536, 777], [1000, 129])]


@pytest.mark.parametrize("key,lens,lq", CASES)
def test_dense_offset_matches_torch_sdpa_with_mask(key, lens, lq):
    p = _cases.small_problem(key)
    q, k, v, cuq, cuk = chunk_of(p, lq)
    out, lse = attention.dense(q, k, v, cuq, p.Hq, p.Hkv, cu_seqlens_k=cuk)
    G = p.Hq // p.Hkv
    for s in range(len(lq)):
        a, b, ak, bk = int(cuq[s]), int(cuq[s + 1]), int(cuk[s]), int(cuk[s + 1])
        Lq, Lk = b - a, bk - ak
        Q = torch.from_numpy(q[a:b]).permute(1, 0, 2)
        K = torch.from_numpy(np.repeat(k[ak:bk], G, axis=1)).permute(1, 0, 2)
        V = torch.from_numpy(np.repeat(v[ak:bk], G, axis=1)).permute(1, 0, 2)
        qpos = torch.arange(Lq)[:, None] + (Lk - Lq)
        mask = torch.arange(Lk)[None, :] <= qpos
        ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V, attn_mask=mask)
        np.testing.assert_allclose(out[a:b], ref.permute(1, 0, 2).numpy(), rtol=0, atol=TOL)


@pytest.mark.parametrize("key,lens,lq", CASES)
def test_chunked_walk_lambda0_is_dense(key, lens, lq):
    p = _cases.small_problem(key)
    q, k, v, cuq, cuk = chunk_of(p, lq)
    r = tile_walk.prefill_fwd(q, k, v, cuq, p.Hq, p.Hkv, lam=0.0, cu_seqlens_k=cuk)
    out, lse = attention.dense(q, k, v, cuq, p.Hq, p.Hkv, cu_seqlens_k=cuk)
    assert not r.bitmap.any()
    np.testing.assert_allclose(r.out, out, rtol=0, atol=TOL)
    np.testing.assert_allclose(r.lse, lse, rtol=0, atol=TOL)


@pytest.mark.parametrize("key,lens,lq", CASES)
@pytest.mark.parametrize("lam", [0.01, 0.3])
def test_chunked_walk_is_dense_over_kept_tiles(key, lens, lq, lam):
    p = _cases.small_problem(key)
    q, k, v, cuq, cuk = chunk_of(p, lq)
    r = tile_walk.prefill_fwd(q, k, v, cuq, p.Hq, p.Hkv, lam=lam, cu_seqlens_k=cuk)

    def allowed(s, h):
        Lq, Lk = int(cuq[s + 1] - cuq[s]), int(cuk[s + 1] - cuk[s])
        nq, nk = layout.tiles(Lq), layout.tiles(Lk)
        ok = np.ones((nq, nk), bool)
        for i in range(nq):
            ok[i] = ~layout.row_bits(r.bitmap, cuq, p.Hq, s, h, i, cuk)
        return ok[(np.arange(Lq) // 128)[:, None], (np.arange(Lk) // 128)[None, :]]

    out, lse = attention.dense(q, k, v, cuq, p.Hq, p.Hkv, allowed=allowed, cu_seqlens_k=cuk)
    np.testing.assert_allclose(r.out, out, rtol=0, atol=TOL)
    np.testing.assert_allclose(r.lse, lse, rtol=0, atol=TOL)
    for item in r.kept:
        s, h, i = item
        want = decisions.skip_bits(q, k, cuq, p.Hq, p.Hkv, True, lam, item=item, cu_seqlens_k=cuk)
        got = layout.row_bits(r.bitmap, cuq, p.Hq, s, h, i, cuk)
        assert np.array_equal(got[:len(want)], want) and not got[len(want):].any()


def test_aligned_offset_chunk_equals_full_walk_rows():
    p = _cases.small_problem("weak_sink")          # lengths 1024, 900
    lq = [384, 900]                                 # offsets 640 (5 tiles) and 0
    q, k, v, cuq, cuk = chunk_of(p, lq)
    qf, kf, vf = (numerics.bf16_to_f64(x) for x in (p.q, p.k, p.v))
    for lam in (0.0, 0.05, 0.5):
        rc = tile_walk.prefill_fwd(q, k, v, cuq, p.Hq, p.Hkv, lam=lam, cu_seqlens_k=cuk)
        rf = tile_walk.prefill_fwd(qf, kf, vf, p.cu_seqlens, p.Hq, p.Hkv, lam=lam)
        for s, L in enumerate([1024, 900]):
            off_tiles = (L - lq[s]) // 128
            a, b = int(cuq[s]), int(cuq[s + 1])
            af = int(p.cu_seqlens[s]) + L - lq[s]
            assert np.array_equal(rc.out[a:b], rf.out[af:af + lq[s]])
            assert np.array_equal(rc.lse[:, a:b], rf.lse[:, af:af + lq[s]])
            for h in range(p.Hq):
                for i in range(layout.tiles(lq[s])):
                    assert np.array_equal(
                        layout.row_bits(rc.bitmap, cuq, p.Hq, s, h, i, cuk),
                        layout.row_bits(rf.bitmap, p.cu_seqlens, p.Hq, s, h, i + off_tiles))


def test_chunked_layout_by_hand():
    # one sequence: 200 queries against 1000 keys -> 2 query tiles, 8 key tiles, 1 word
    assert layout.total_words([0, 200], 3, [0, 1000]) == 3 * 2 * 1
    # 40 key tiles -> 2 words per row
    assert layout.row_offset([0, 10, 300], 2, 1, 1, 2, [0, 100, 5220]) == 2 * 1 * 1 + (3 + 2) * 2
