"""GPU parity for chunked prefill (bsa_prefill_fwd_chunked): a chunk of Lq
queries against Lk >= Lq keys, queries at the last Lq positions.

Compared with the oracle's chunked tile walk (skip bits outside the 1e-3
margin exact; mask-replay output and lse within the bf16 tolerances), plus
an exact property: with a tile-aligned offset the chunk's outputs, lse and
skip bits equal the same rows of a whole-sequence call.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import _cases
import _gpu
from gen import inputs as gi
from oracle import layout

pytestmark = pytest.mark.gpu

CASES = [("gqa_ragged", [100, 777, 1, 200]),   # offsets 200, 223, 128, 440
         ("weak_sink", [384, 900]),            # 640 (tile-aligned), 0
         ("gqa4", [1000, 129]),                # 536, 648
         ("tiny", [1, 50, 128])]               # 0, 27, 0


@pytest.mark.parametrize("key,lq", CASES)
@pytest.mark.parametrize("lam", [0.01, 0.0, 0.3])
@pytest.mark.parametrize("causal", [True, False])
def test_chunked_matches_oracle(key, lq, lam, causal):
    p = gi.chunk(_cases.small_problem(key), lq)
    g = _gpu.run(p, lam=lam, causal=causal)
    out, lse = _gpu.host(g)
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    _gpu.compare(p, g)


def test_aligned_chunk_equals_whole_sequence_rows():
    full = _cases.small_problem("weak_sink")       # lengths 1024, 900
    lq = [384, 900]
    p = gi.chunk(full, lq)
    for lam in (0.0, 0.05):
        gc = _gpu.run(p, lam=lam)
        gf = _gpu.run(full, lam=lam)
        for s, L in enumerate([1024, 900]):
            a, b = int(p.cu_seqlens[s]), int(p.cu_seqlens[s + 1])
            af = int(full.cu_seqlens[s]) + L - lq[s]
            assert torch.equal(gc["out"][a:b], gf["out"][af:af + lq[s]])
            assert torch.equal(gc["lse"][:, a:b], gf["lse"][:, af:af + lq[s]])
            off_tiles = (L - lq[s]) // 128
            for h in range(p.Hq):
                for i in range(layout.tiles(lq[s])):
                    assert np.array_equal(
                        layout.row_bits(gc["bitmap"], p.cu_seqlens, p.Hq, s, h, i, p.cu_seqlens_k),
                        layout.row_bits(gf["bitmap"], full.cu_seqlens, p.Hq, s, h, i + off_tiles))


def test_chunked_full_size_sampled():
    """The last 8192 queries of the 32K Llama-shaped layer against all its keys."""
    p = gi.chunk(_cases.full_problem("C1"), [8192])
    g = _gpu.run(p, lam=0.01)
    assert bool(torch.isfinite(g["out"]).all())
    _gpu.compare(p, g, items=_gpu.sample_items(p, 12, seed=3))


def test_chunked_rejects_fewer_keys_than_queries():
    b = _gpu.bsa()
    p = _cases.small_problem("tiny")
    q, k, v = _gpu.to_dev_bf16(p.q), _gpu.to_dev_bf16(p.k), _gpu.to_dev_bf16(p.v)
    cuq = torch.tensor([0, 100], dtype=torch.int32, device="cuda")
    cuk = torch.tensor([0, 50], dtype=torch.int32, device="cuda")
    out = torch.full((100, p.Hq, p.d), 3.0, dtype=torch.bfloat16, device="cuda")
    assert b.prefill_fwd_chunked(q, k, v, cuq, cuk, 1, p.Hq, p.Hkv, p.d, 1, 0.01, b.BSA_BF16,
                                 out, None, None) == 0
    assert b.get_device_status() == 6
    assert bool((out == 3.0).all())


@pytest.mark.parametrize("lq", [[1, 1], [3, 4], [1, 128]])
@pytest.mark.parametrize("lam", [0.005, 0.0])
def test_decode_shaped_queries(lq, lam):
    """A few new queries per sequence against all earlier keys (decode /
    speculative-decode shape, the deployment guide's §6.1 decode threshold)."""
    p = gi.chunk(_cases.small_problem("weak_sink"), lq)
    g = _gpu.run(p, lam=lam)
    out, lse = _gpu.host(g)
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    _gpu.compare(p, g)


@pytest.mark.parametrize("key,lq", [("gqa_ragged", [100, 777, 1, 200]), ("weak_sink", [384, 900])])
def test_chunked_fp8(key, lq):
    import test_gpu_fp8
    p = gi.chunk(_cases.small_problem(key), lq)
    f8q = test_gpu_fp8.gpu_quantize(p.q)
    f8k = test_gpu_fp8.gpu_quantize(p.k)
    f8v = test_gpu_fp8.gpu_quantize(p.v)
    f8 = (f8q[0], f8k[0], f8v[0], f8q[1], f8k[1], f8v[1])
    g = _gpu.run(p, lam=0.05, fp8=f8)
    assert bool(torch.isfinite(g["out"]).all())
    _gpu.compare(p, g, fp8=f8)
