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


def test_two_streams_concurrently():
    """Calls on two streams may overlap: each stream has its own scratch area."""
    b = _gpu.bsa()
    pa, pb = _cases.small_problem("gqa_ragged"), _cases.small_problem("weak_sink")
    ref_a, ref_b = _gpu.run(pa, lam=0.01), _gpu.run(pb, lam=0.05)

    def launch(p, lam, stream):
        q, k, v = _gpu.to_dev_bf16(p.q), _gpu.to_dev_bf16(p.k), _gpu.to_dev_bf16(p.v)
        cu = torch.from_numpy(p.cu_seqlens).cuda()
        out = torch.empty((p.total_tokens, p.Hq, p.d), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((p.Hq, p.total_tokens), dtype=torch.float32, device="cuda")
        bm = torch.empty((b.skip_bitmap_words(p.cu_seqlens, p.Hq),), dtype=torch.int32, device="cuda")
        torch.cuda.synchronize()
        for _ in range(3):
            b.check(b.prefill_fwd(q, k, v, cu, p.n_seqs, p.Hq, p.Hkv, p.d, 1, lam, b.BSA_BF16,
                                  out, lse, bm, stream), "launch")
        return out, lse, bm, (q, k, v, cu)

    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    oa = launch(pa, 0.01, sa)
    ob = launch(pb, 0.05, sb)
    torch.cuda.synchronize()
    assert b.get_device_status(sa) == 0 and b.get_device_status(sb) == 0
    assert torch.equal(oa[0], ref_a["out"]) and torch.equal(ob[0], ref_b["out"])
    assert np.array_equal(oa[2].cpu().numpy().view(np.uint32), ref_a["bitmap"])
    assert np.array_equal(ob[2].cpu().numpy().view(np.uint32), ref_b["bitmap"])
