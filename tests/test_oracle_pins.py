"""Pins for the CPU oracle: each check ties it to something other than itself.

* brute-force dense attention vs torch's SDPA and scipy's logsumexp
  (library routines) -- pins ``oracle.attention``;
* tile walk at λ = 0 vs dense attention (closed form: skipping off);
* tile walk at λ > 0 vs dense attention over exactly the kept tiles;
* kept normalised weights sum to one / lse is the direct log-sum-exp;
* tile-walk decisions vs the prefix-max closed form (``oracle.decisions``),
  and their monotonicity in λ;
* a planted case whose decisions were enumerated by hand
  (``tests/golden/planted_tiles.json``) and whose outputs have a closed form;
* GQA equals MHA with repeated K/V heads (``np.repeat``);
* E4M3 codes vs the format definition and torch's float8 cast;
* bitmap layout sizes counted by hand.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import scipy.special
import torch

import _cases
from oracle import attention, decisions, layout, numerics, tile_walk

TOL = 1e-12


def vals(p):
    return numerics.bf16_to_f64(p.q), numerics.bf16_to_f64(p.k), numerics.bf16_to_f64(p.v)


# ----------------------------------------------------------------- dense

@pytest.mark.parametrize("causal", [True, False])
def test_dense_matches_torch_sdpa(causal):
    p = _cases.small_problem("gqa_ragged")
    q, k, v = vals(p)
    out, lse = attention.dense(q, k, v, p.cu_seqlens, p.Hq, p.Hkv, causal=causal)
    G = p.Hq // p.Hkv
    for s in range(p.n_seqs):
        a, b = int(p.cu_seqlens[s]), int(p.cu_seqlens[s + 1])
        Q = torch.from_numpy(q[a:b]).permute(1, 0, 2)
        K = torch.from_numpy(np.repeat(k[a:b], G, axis=1)).permute(1, 0, 2)
        V = torch.from_numpy(np.repeat(v[a:b], G, axis=1)).permute(1, 0, 2)
        ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V, is_causal=causal)
        np.testing.assert_allclose(out[a:b], ref.permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)
        S = torch.einsum("hqd,hkd->hqk", Q, K) / math.sqrt(p.d)
        if causal:
            S = S.masked_fill(torch.ones(b - a, b - a, dtype=torch.bool).triu(1), -math.inf)
        ref_lse = scipy.special.logsumexp(S.numpy(), axis=-1)
        np.testing.assert_allclose(lse[:, a:b], ref_lse, rtol=0, atol=1e-12)


def test_direct_logsumexp_textbook():
    x = np.array([0.5, -3.0, 2.25, -np.inf])
    assert abs(attention.direct_logsumexp(x) - math.log(math.exp(0.5) + math.exp(-3) + math.exp(2.25))) < 1e-15


# ----------------------------------------------------------------- λ = 0

@pytest.mark.parametrize("key", ["C0", "gqa_ragged", "no_sink", "tiny"])
@pytest.mark.parametrize("causal", [True, False])
def test_walk_lambda0_is_dense(key, causal):
    p = _cases.small_problem(key)
    q, k, v = vals(p)
    r = tile_walk.prefill_fwd(q, k, v, p.cu_seqlens, p.Hq, p.Hkv, causal=causal, lam=0.0)
    out, lse = attention.dense(q, k, v, p.cu_seqlens, p.Hq, p.Hkv, causal=causal)
    assert not r.bitmap.any()
    np.testing.assert_allclose(r.out, out, rtol=0, atol=TOL)
    np.testing.assert_allclose(r.lse, lse, rtol=0, atol=TOL)


# ----------------------------------------------------------------- λ > 0

def kept_mask(p, bitmap, causal):
    cu = p.cu_seqlens

    def allowed(s, h):
        L = int(cu[s + 1] - cu[s])
        n = layout.tiles(L)
        tile_ok = np.ones((n, n), bool)
        for i in range(n):
            tile_ok[i] = ~layout.row_bits(bitmap, cu, p.Hq, s, h, i)
        t = np.arange(L) // 128
        return tile_ok[t[:, None], t[None, :]]
    return allowed


@pytest.mark.parametrize("key,lam", [("C0", 0.01), ("gqa_ragged", 0.01), ("weak_sink", 0.05),
                                     ("weak_sink", 0.5), ("gqa4", 0.01)])
@pytest.mark.parametrize("causal", [True, False])
def test_walk_is_dense_over_kept_tiles(key, lam, causal):
    p = _cases.small_problem(key)
    q, k, v = vals(p)
    r = tile_walk.prefill_fwd(q, k, v, p.cu_seqlens, p.Hq, p.Hkv, causal=causal, lam=lam)
    assert r.bitmap.any(), "case should skip something"
    out, lse = attention.dense(q, k, v, p.cu_seqlens, p.Hq, p.Hkv, causal=causal,
                               allowed=kept_mask(p, r.bitmap, causal))
    np.testing.assert_allclose(r.out, out, rtol=0, atol=TOL)
    np.testing.assert_allclose(r.lse, lse, rtol=0, atol=TOL)


@pytest.mark.parametrize("key,lam", [("weak_sink", 0.05), ("gqa_ragged", 0.01)])
def test_kept_weights_sum_to_one(key, lam):
    """Normalised weights exp(S - lse) over the kept entries sum to 1 per row,
    and lse equals the direct log-sum-exp of the kept scores."""
    p = _cases.small_problem(key)
    q, k, v = vals(p)
    r = tile_walk.prefill_fwd(q, k, v, p.cu_seqlens, p.Hq, p.Hkv, lam=lam)
    G = p.Hq // p.Hkv
    for (s, h, i), kept in list(r.kept.items())[::3]:
        a, L = int(p.cu_seqlens[s]), int(p.cu_seqlens[s + 1] - p.cu_seqlens[s])
        for rr in range(i * 128, min(i * 128 + 128, L), 17):
            keys = np.concatenate([np.arange(j * 128, min(j * 128 + 128, L)) for j in kept])
            keys = keys[keys <= rr]
            sc = k[a + keys, h // G] @ q[a + rr, h] / math.sqrt(p.d)
            lse = r.lse[h, a + rr]
            assert abs(np.exp(sc - lse).sum() - 1.0) < 1e-12
            assert abs(attention.direct_logsumexp(sc) - lse) < 1e-12


# ----------------------------------------------------------------- decisions

@pytest.mark.parametrize("key", ["C0", "gqa_ragged", "weak_sink", "gqa4"])
@pytest.mark.parametrize("causal", [True, False])
def test_walk_decisions_match_prefix_max_closed_form(key, causal):
    p = _cases.small_problem(key)
    q, k, v = vals(p)
    for lam in (0.0, 1e-3, 0.01, 0.05, 0.3, 0.9):
        r = tile_walk.prefill_fwd(q, k, v, p.cu_seqlens, p.Hq, p.Hkv, causal=causal, lam=lam)
        for item in r.kept:
            s, h, i = item
            want = decisions.skip_bits(q, k, p.cu_seqlens, p.Hq, p.Hkv, causal, lam, item=item)
            got = layout.row_bits(r.bitmap, p.cu_seqlens, p.Hq, s, h, i)[:len(want)]
            assert np.array_equal(got, want), (item, lam)


def test_decisions_monotone_in_lambda():
    p = _cases.small_problem("weak_sink")
    q, k, _ = vals(p)
    lams = [0.0, 1e-4, 1e-3, 0.01, 0.02, 0.05, 0.1, 0.3, 0.6, 0.99]
    for item in tile_walk.all_items(p.cu_seqlens, p.Hq):
        prev = None
        for lam in lams:
            cur = decisions.skip_bits(q, k, p.cu_seqlens, p.Hq, p.Hkv, True, lam, item=item)
            if prev is not None:
                assert np.all(cur >= prev)
            prev = cur


@pytest.mark.parametrize("lam", [1e-6, 0.01, 0.5, 0.99])
def test_first_tile_kept_and_no_nan(lam):
    p = _cases.small_problem("weak_sink")
    q, k, v = vals(p)
    r = tile_walk.prefill_fwd(q, k, v, p.cu_seqlens, p.Hq, p.Hkv, lam=lam)
    assert all(kept[0] == 0 for kept in r.kept.values())
    assert np.isfinite(r.out).all() and np.isfinite(r.lse).all()


def test_replay_of_own_bitmap_is_bitwise_identical():
    p = _cases.small_problem("weak_sink")
    q, k, v = vals(p)
    r = tile_walk.prefill_fwd(q, k, v, p.cu_seqlens, p.Hq, p.Hkv, lam=0.05)
    rr = tile_walk.prefill_fwd(q, k, v, p.cu_seqlens, p.Hq, p.Hkv, lam=0.05, replay_bitmap=r.bitmap)
    assert np.array_equal(r.out, rr.out) and np.array_equal(r.lse, rr.lse)
    assert np.array_equal(r.bitmap, rr.bitmap)


def test_replay_rejects_bitmap_without_first_tile():
    p = _cases.small_problem("tiny")
    q, k, v = vals(p)
    bad = np.zeros(layout.total_words(p.cu_seqlens, p.Hq), np.uint32)
    bad[layout.row_offset(p.cu_seqlens, p.Hq, 1, 0, 0)] = 1
    with pytest.raises(ValueError):
        tile_walk.prefill_fwd(q, k, v, p.cu_seqlens, p.Hq, p.Hkv, lam=0.01, replay_bitmap=bad)


# ----------------------------------------------------------------- planted golden

def planted_expected(g, lam, L, causal):
    b = np.asarray(g["construction"]["b"], float) / math.sqrt(128)
    c = np.asarray(g["construction"]["c"], float)
    skipped = set(g["skipped"][lam])
    n = layout.tiles(L)
    out0 = np.zeros(L)
    lse = np.zeros(L)
    for t in range(L):
        i, r = divmod(t, 128)
        w_sum = wc = 0.0
        for j in range(i + 1 if causal else n):
            if j in skipped:
                continue
            if causal:
                nj = 128 if j < i else r + 1
            else:
                nj = min(128, L - 128 * j)
            w = nj * math.exp(b[j])
            w_sum += w
            wc += w * c[j]
        out0[t] = wc / w_sum
        lse[t] = math.log(w_sum)
    return out0, lse


@pytest.mark.parametrize("lam", ["0", "0.0001", "0.01", "0.05", "0.5"])
@pytest.mark.parametrize("causal,L", [(True, 1024), (False, 1024), (True, 1000), (False, 1000)])
def test_planted_tiles_golden(lam, causal, L):
    g = _cases.planted_golden()
    p = _cases.planted_problem(tokens=L, causal=causal)
    q, k, v = vals(p)
    r = tile_walk.prefill_fwd(q, k, v, p.cu_seqlens, 1, 1, causal=causal, lam=float(lam))
    skipped = set(g["skipped"][lam])
    n = layout.tiles(L)
    for i in range(n):
        visited = range(i + 1) if causal else range(n)
        want = np.array([(j in skipped) and (j in visited) for j in range(n)])
        assert np.array_equal(layout.row_bits(r.bitmap, p.cu_seqlens, 1, 0, 0, i), want), i
    out0, lse = planted_expected(g, lam, L, causal)
    np.testing.assert_allclose(r.out[:, 0, 0], out0, rtol=0, atol=1e-12)
    np.testing.assert_allclose(r.out[:, 0, 1], 1.0, rtol=0, atol=1e-12)
    assert np.all(r.out[:, 0, 2:] == 0)
    np.testing.assert_allclose(r.lse[0], lse, rtol=0, atol=1e-12)


# ----------------------------------------------------------------- GQA

def test_gqa_equals_mha_with_repeated_heads():
    p = _cases.small_problem("gqa4")
    q, k, v = vals(p)
    G = p.Hq // p.Hkv
    r1 = tile_walk.prefill_fwd(q, k, v, p.cu_seqlens, p.Hq, p.Hkv, lam=0.01)
    r2 = tile_walk.prefill_fwd(q, np.repeat(k, G, axis=1), np.repeat(v, G, axis=1),
                               p.cu_seqlens, p.Hq, p.Hq, lam=0.01)
    assert np.array_equal(r1.out, r2.out) and np.array_equal(r1.bitmap, r2.bitmap)


# ----------------------------------------------------------------- E4M3

def test_e4m3_decode_table():
    dec = numerics.e4m3_to_f64(np.arange(256, dtype=np.uint8))
    assert dec[0x7E] == 448.0 and dec[0x01] == 2.0 ** -9 and dec[0x08] == 2.0 ** -6
    assert dec[0x38] == 1.0 and dec[0x39] == 1.125 and dec[0xB8] == -1.0
    assert np.isnan(dec[0x7F]) and np.isnan(dec[0xFF])
    pos = dec[:0x7F]
    assert np.all(np.diff(pos) > 0)                     # strictly increasing codes
    assert np.array_equal(dec[0x80:0xFF], -pos)


def test_e4m3_encode_rules():
    enc = numerics.e4m3_from_f32
    f = lambda *x: np.array(x, np.float32)              # noqa: E731
    assert list(enc(f(1.0625, 1.1875, 1.0, -1.0625))) == [0x38, 0x3A, 0x38, 0xB8]   # ties to even
    assert list(enc(f(500.0, -1e9, 448.0, 464.0))) == [0x7E, 0xFE, 0x7E, 0x7E]      # saturation
    assert list(enc(f(2.0 ** -10, 2.0 ** -10 * 3, 2.0 ** -9 * 7.5))) == [0x00, 0x02, 0x08]
    codes = np.arange(0x7F, dtype=np.uint8)
    assert np.array_equal(enc(numerics.e4m3_to_f64(codes).astype(np.float32)), codes)


def test_e4m3_matches_torch_cast():
    rng = np.random.default_rng(7)
    x = np.concatenate([rng.standard_normal(200000) * 50, rng.uniform(-448, 448, 100000),
                        rng.standard_normal(50000) * 1e-2]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(numerics.e4m3_from_f32(x), ref)


def test_per_head_quantiser():
    p = _cases.small_problem("gqa_ragged")
    codes, scale = numerics.quantize_per_head(p.q)
    x = numerics.bf16_to_f64(p.q)
    absmax = np.abs(x).max(axis=(0, 2))
    assert np.array_equal(scale, (absmax.astype(np.float32) / np.float32(448)).astype(np.float32))
    # the largest magnitude of every head maps to the top code
    assert np.all(np.abs(numerics.e4m3_to_f64(codes)).max(axis=(0, 2)) == 448.0)
    err = np.abs(numerics.e4m3_to_f64(codes) * scale[None, :, None] - x)
    assert np.all(err <= np.abs(x) * 2.0 ** -4 + scale[None, :, None] * 2.0 ** -10)


# ----------------------------------------------------------------- layout

def test_bitmap_layout_by_hand():
    # one sequence of 2048 tokens, one head: 16 tiles -> 1 word per row, 16 rows
    assert layout.total_words([0, 2048], 1) == 16
    # lengths 300 (3 tiles, 1 word) and 4700 (37 tiles, 2 words), Hq = 2
    assert layout.total_words([0, 300, 5000], 2) == 2 * 3 * 1 + 2 * 37 * 2
    assert layout.row_offset([0, 300, 5000], 2, 1, 1, 5) == 6 + (37 + 5) * 2
    # the 128K layer: 1024 tiles, 32 words per row, 32 heads -> 4 MiB
    assert layout.total_words([0, 131072], 32) * 4 == 4 << 20
