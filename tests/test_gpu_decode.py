"""GPU parity for the split-KV decode entry point (bsa_decode_fwd).

Decode-shaped problems (a few queries per sequence, at the last positions,
against all keys) are compared with the oracle's tile walk under the same
tolerances as the prefill path: skip bits exact outside the 1e-3 decision
margin, mask-replay outputs within max-abs 2e-2 / mean-abs 2e-3, lse within
1e-3. The decisions of the split path come from prefix maxima of the tile
maxima; the oracle walks the tiles in order, so the comparison also checks
that restatement of the order rule.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import _cases
import _gpu
from gen import inputs as gi

pytestmark = pytest.mark.gpu


def run_decode(p, lam, causal=True, max_q=None, total_k=None, fill=float("nan")):
    b = _gpu.bsa()
    cuk = p.cu_seqlens_k
    T = p.total_tokens
    q, k, v = _gpu.to_dev_bf16(p.q), _gpu.to_dev_bf16(p.k), _gpu.to_dev_bf16(p.v)
    cq = torch.from_numpy(p.cu_seqlens.astype(np.int32)).cuda()
    ck = torch.from_numpy(cuk.astype(np.int32)).cuda()
    max_q = int(p.seqlens.max()) if max_q is None else max_q
    total_k = int(cuk[-1]) if total_k is None else total_k
    out = torch.full((T, p.Hq, p.d), fill, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((p.Hq, T), float("nan"), dtype=torch.float32, device="cuda")
    nw = b.skip_bitmap_words_chunked(p.cu_seqlens, cuk, p.Hq)
    bm = torch.full((max(nw, 1),), -1, dtype=torch.int32, device="cuda")
    st = b.decode_fwd(q, k, v, cq, ck, p.n_seqs, max_q, total_k, p.Hq, p.Hkv, p.d, int(causal),
                      lam, out, lse, bm)
    b.check(st, "bsa_decode_fwd")
    torch.cuda.synchronize()
    status = b.get_device_status()
    return dict(out=out, lse=lse, bitmap=bm[:nw].cpu().numpy().view(np.uint32), lam=lam,
                causal=causal), status


@pytest.fixture(scope="module")
def g16():
    # sixteen query heads on one KV head: the largest group the path takes
    return gi.small("g16", [3000, 700], Hq=16, Hkv=1, seed=7)


CASES = [("weak_sink", [1, 1]), ("gqa_ragged", [1, 3, 1, 2]), ("gqa4", [4, 1]),
         ("tiny", [1, 2, 5]), ("no_sink", [1]), ("C0", [3])]


@pytest.mark.parametrize("key,lq", CASES)
@pytest.mark.parametrize("lam", [0.005, 0.0, 0.3])
@pytest.mark.parametrize("causal", [True, False])
def test_decode_matches_oracle(key, lq, lam, causal):
    p = gi.chunk(_cases.small_problem(key), lq)
    g, st = run_decode(p, lam, causal)
    assert st == 0
    out, lse = _gpu.host(g)
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    print(key, lq, lam, causal, _gpu.compare(p, g))


@pytest.mark.parametrize("lq", [[1, 1], [2, 1]])
def test_decode_group_of_sixteen(g16, lq):
    p = gi.chunk(g16, lq)
    for lam in (0.005, 0.0):
        g, st = run_decode(p, lam)
        assert st == 0
        _gpu.compare(p, g)


def test_decode_max_seqlen_larger_than_needed():
    # max_seqlen_q only bounds the rows; a loose bound gives the same result
    p = gi.chunk(_cases.small_problem("gqa4"), [2, 1])
    a, _ = run_decode(p, 0.005, max_q=2)
    b, _ = run_decode(p, 0.005, max_q=8)
    assert torch.equal(a["out"], b["out"]) and torch.equal(a["lse"], b["lse"])
    assert np.array_equal(a["bitmap"], b["bitmap"])


def test_decode_full_layer_one_query():
    """One new query at the end of the 128K Llama-shaped layer, all 32 heads."""
    p = gi.chunk(_cases.full_problem("C2"), [1])
    for lam in (0.005, 0.0):
        g, st = run_decode(p, lam)
        assert st == 0
        print(lam, _gpu.compare(p, g))


def test_decode_batch_of_four_32k():
    base = gi.packed("dec4", [32768] * 4, Hq=32, Hkv=8, seed=3, window=2.0, window_period=4096,
                     window_len=512)
    p = gi.chunk(base, [1, 2, 1, 1])
    g, st = run_decode(p, 0.005)
    assert st == 0
    _gpu.compare(p, g)


def test_decode_many_work_items():
    """Several work items per SM: 16 KV heads x 80K keys in two sequences,
    so the CTAs claim items from both sequences in turn."""
    base = gi.packed("dec16", [40000, 40064], Hq=32, Hkv=16, seed=4, window=2.0,
                     window_period=4096, window_len=512)
    p = gi.chunk(base, [1, 2])
    for lam in (0.005, 0.0):
        g, st = run_decode(p, lam)
        assert st == 0
        print(lam, _gpu.compare(p, g))


@pytest.mark.parametrize("Hq,L,lq", [(4, 170000, 1), (8, 70000, 4)])
def test_decode_lookback_over_many_splits(Hq, L, lq):
    """One long sequence on one KV head: the last work items have more than
    128 earlier splits (8-tile splits at 4 query rows, 4-tile splits at 32),
    so the look-back for the running max spans several windows of earlier
    splits and stops at published inclusive prefixes."""
    base = gi.packed("declong", [L], Hq=Hq, Hkv=1, seed=9, window=2.0, window_period=4096,
                     window_len=512)
    p = gi.chunk(base, [lq])
    for lam in (0.005, 0.0):
        g, st = run_decode(p, lam)
        assert st == 0
        print(Hq, L, lq, lam, _gpu.compare(p, g))


def test_decode_batch_with_query_free_sequences():
    """Sequences without new queries in the batch (Lq = 0) take no work and no
    bitmap words; the others are unaffected."""
    base = _cases.small_problem("gqa_ragged")             # lengths 300, 1000, 129, 640
    p = gi.chunk(base, [1, 0, 2, 0])
    for lam in (0.005, 0.0):
        g, st = run_decode(p, lam)
        assert st == 0
        _gpu.compare(p, g)


def test_decode_rejects_bad_lengths():
    b = _gpu.bsa()
    p = gi.chunk(_cases.small_problem("gqa4"), [4, 1])
    # a query count above max_seqlen_q, then a wrong key total: nothing written
    g, st = run_decode(p, 0.005, max_q=3, fill=7.0)
    assert st == 6 and bool((g["out"] == 7.0).all())
    g, st = run_decode(p, 0.005, total_k=int(p.cu_seqlens_k[-1]) - 1, fill=7.0)
    assert st == 6 and bool((g["out"] == 7.0).all())
    assert b.get_device_status() == 0


def test_decode_tables_reused_across_shapes():
    """One stream alternates a small and a larger decode problem: the scratch
    is laid out again (and cleared) when a call needs more room, and reused,
    with per-call state told apart by the call count, otherwise. Every call
    equals, bit for bit, the same call on a fresh stream."""
    b = _gpu.bsa()
    small = gi.chunk(_cases.small_problem("gqa_ragged"), [1, 2, 1, 1])
    big = gi.chunk(gi.packed("decbig", [9000, 5000, 7000], Hq=8, Hkv=2, seed=8, window=2.0,
                             window_period=4096, window_len=512), [4, 1, 2])
    probs = [small, big]
    ins = []
    for p in probs:
        ins.append((_gpu.to_dev_bf16(p.q), _gpu.to_dev_bf16(p.k), _gpu.to_dev_bf16(p.v),
                    torch.from_numpy(p.cu_seqlens.astype(np.int32)).cuda(),
                    torch.from_numpy(p.cu_seqlens_k.astype(np.int32)).cuda()))

    def call(t, stream):
        p = probs[t]
        q, k, v, cq, ck = ins[t]
        out = torch.full((p.total_tokens, p.Hq, p.d), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((p.Hq, p.total_tokens), float("nan"), dtype=torch.float32, device="cuda")
        nw = b.skip_bitmap_words_chunked(p.cu_seqlens, p.cu_seqlens_k, p.Hq)
        bm = torch.full((nw,), -1, dtype=torch.int32, device="cuda")
        b.check(b.decode_fwd(q, k, v, cq, ck, p.n_seqs, int(p.seqlens.max()), int(p.cu_seqlens_k[-1]),
                             p.Hq, p.Hkv, p.d, 1, 0.005, out, lse, bm, stream), "decode")
        return out, lse, bm

    refs = []
    for t in range(2):
        s = torch.cuda.Stream()
        refs.append(call(t, s))
        torch.cuda.synchronize()
        assert b.get_device_status(s) == 0
        assert b.release_stream(s) == 0
    s = torch.cuda.Stream()
    for t in (0, 1, 0, 0, 1, 1, 0):
        out, lse, bm = call(t, s)
        torch.cuda.synchronize()
        assert b.get_device_status(s) == 0
        assert torch.equal(out, refs[t][0]) and torch.equal(lse, refs[t][1])
        assert torch.equal(bm, refs[t][2])
    assert b.release_stream(s) == 0
    g, st = run_decode(big, 0.005)
    assert st == 0
    _gpu.compare(big, g)


def test_decode_batch_above_local_table_size():
    """300 sequences (more than the 256 whose tables every CTA builds for
    itself): one CTA writes the per-sequence tables and the others wait for
    it. Mixed lengths (1 to 1100 keys), one or two new queries each."""
    rng = np.random.default_rng(11)
    lens = [int(x) for x in rng.integers(2, 1100, 300)]
    base = gi.packed("dec300", lens, Hq=8, Hkv=2, seed=12)
    lq = [1 + (i % 2) for i in range(300)]
    p = gi.chunk(base, lq)
    for lam in (0.005, 0.0):
        g, st = run_decode(p, lam)
        assert st == 0
        print(lam, _gpu.compare(p, g))
