"""Calls from two host threads on two streams at once.

Each (device, stream) has its own scratch area and lock, so the host work of
calls on different streams runs concurrently and their kernels may overlap
on the GPU. Every result must equal, bit for bit, the same call made alone
(the kernels are deterministic: a work item's result does not depend on
which CTA runs it), and those match the oracle. Afterwards each stream's
scratch is released.
"""
from __future__ import annotations

import threading

import numpy as np
import pytest
import torch

import _cases
import _gpu

pytestmark = pytest.mark.gpu


def _inputs(p):
    q, k, v = _gpu.to_dev_bf16(p.q), _gpu.to_dev_bf16(p.k), _gpu.to_dev_bf16(p.v)
    cu = torch.from_numpy(p.cu_seqlens.astype(np.int32)).cuda()
    return q, k, v, cu


def _outputs(b, p, n):
    T = p.total_tokens
    nw = b.skip_bitmap_words(p.cu_seqlens, p.Hq)
    return [(torch.empty((T, p.Hq, p.d), dtype=torch.bfloat16, device="cuda"),
             torch.empty((p.Hq, T), dtype=torch.float32, device="cuda"),
             torch.empty((nw,), dtype=torch.int32, device="cuda")) for _ in range(n)]


def test_two_threads_two_streams_match_single_calls_and_oracle():
    b = _gpu.bsa()
    cases = [(_cases.small_problem("gqa_ragged"), 0.01), (_cases.small_problem("weak_sink"), 0.05)]
    refs = []
    for p, lam in cases:
        g = _gpu.run(p, lam=lam)
        _gpu.compare(p, g)
        refs.append(g)
    n_calls = 8
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    ins = [_inputs(p) for p, _ in cases]
    outs = [_outputs(b, p, n_calls) for p, _ in cases]
    torch.cuda.synchronize()
    errors = []
    start = threading.Barrier(2)

    def worker(t):
        try:
            torch.cuda.set_device(0)
            p, lam = cases[t]
            q, k, v, cu = ins[t]
            start.wait()
            for n in range(n_calls):
                out, lse, bm = outs[t][n]
                st = b.prefill_fwd(q, k, v, cu, p.n_seqs, p.Hq, p.Hkv, p.d, 1, lam, b.BSA_BF16,
                                   out, lse, bm, streams[t])
                if st != 0:
                    errors.append((t, n, st))
        except Exception as e:  # reported below
            errors.append((t, repr(e)))

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(2)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    torch.cuda.synchronize()
    for t in range(2):
        assert b.get_device_status(streams[t]) == 0
        ref = refs[t]
        for out, lse, bm in outs[t]:
            assert torch.equal(out, ref["out"]) and torch.equal(lse, ref["lse"])
            assert np.array_equal(bm.cpu().numpy().view(np.uint32), ref["bitmap"])
    for t in range(2):
        assert b.release_stream(streams[t]) == 0
    torch.cuda.synchronize()
    # a released stream gets a fresh scratch area on its next call
    p, lam = cases[0]
    q, k, v, cu = ins[0]
    out, lse, bm = outs[0][0]
    out.fill_(float("nan"))
    b.check(b.prefill_fwd(q, k, v, cu, p.n_seqs, p.Hq, p.Hkv, p.d, 1, lam, b.BSA_BF16, out, lse, bm,
                          streams[0]), "after release")
    torch.cuda.synchronize()
    assert torch.equal(out, refs[0]["out"])


def test_two_threads_two_streams_decode():
    """Decode calls from two host threads on two streams: two persistent
    decode grids may share the GPU. Each grid's work items wait only for items
    its own running CTAs claimed, so both finish; every result equals, bit for
    bit, the same call made alone (which matches the oracle), and a released
    stream's scratch is rebuilt (zero-filled) on its next call."""
    import test_gpu_decode as td
    from gen import inputs as gi
    b = _gpu.bsa()
    bases = [gi.packed("dec2a", [20000, 9000], Hq=8, Hkv=2, seed=5, window=2.0,
                       window_period=4096, window_len=512),
             gi.packed("dec2b", [30000], Hq=16, Hkv=2, seed=6, window=2.0, window_period=4096,
                       window_len=512)]
    probs = [gi.chunk(bases[0], [1, 2]), gi.chunk(bases[1], [3])]
    refs = []
    for p in probs:
        g, st = td.run_decode(p, 0.005)
        assert st == 0
        _gpu.compare(p, g)
        refs.append(g)
    n_calls = 6
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    ins, outs = [], []
    for p in probs:
        q, k, v = _gpu.to_dev_bf16(p.q), _gpu.to_dev_bf16(p.k), _gpu.to_dev_bf16(p.v)
        cq = torch.from_numpy(p.cu_seqlens.astype(np.int32)).cuda()
        ck = torch.from_numpy(p.cu_seqlens_k.astype(np.int32)).cuda()
        ins.append((q, k, v, cq, ck))
        nw = b.skip_bitmap_words_chunked(p.cu_seqlens, p.cu_seqlens_k, p.Hq)
        outs.append([(torch.empty((p.total_tokens, p.Hq, p.d), dtype=torch.bfloat16, device="cuda"),
                      torch.empty((p.Hq, p.total_tokens), dtype=torch.float32, device="cuda"),
                      torch.full((nw,), -1, dtype=torch.int32, device="cuda")) for _ in range(n_calls)])
    torch.cuda.synchronize()
    errors = []
    start = threading.Barrier(2)

    def call(t, n, stream):
        p = probs[t]
        q, k, v, cq, ck = ins[t]
        out, lse, bm = outs[t][n]
        return b.decode_fwd(q, k, v, cq, ck, p.n_seqs, int(p.seqlens.max()), int(p.cu_seqlens_k[-1]),
                            p.Hq, p.Hkv, p.d, 1, 0.005, out, lse, bm, stream)

    def worker(t):
        try:
            torch.cuda.set_device(0)
            start.wait()
            for n in range(n_calls):
                st = call(t, n, streams[t])
                if st != 0:
                    errors.append((t, n, st))
        except Exception as e:  # reported below
            errors.append((t, repr(e)))

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(2)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    torch.cuda.synchronize()
    for t in range(2):
        assert b.get_device_status(streams[t]) == 0
        for out, lse, bm in outs[t]:
            assert torch.equal(out, refs[t]["out"]) and torch.equal(lse, refs[t]["lse"])
            assert np.array_equal(bm.cpu().numpy().view(np.uint32), refs[t]["bitmap"])
    assert b.release_stream(streams[0]) == 0
    torch.cuda.synchronize()
    out, lse, bm = outs[0][0]
    out.fill_(float("nan"))
    b.check(call(0, 0, streams[0]), "after release")
    torch.cuda.synchronize()
    assert torch.equal(out, refs[0]["out"])
    assert np.array_equal(bm.cpu().numpy().view(np.uint32), refs[0]["bitmap"])
