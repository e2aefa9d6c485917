"""Device-side error paths, exercised without faulting the GPU.

* a malformed cu_seqlens (decreasing) is caught by the prologue: nothing is
  written and bsa_get_device_status reports BSA_ERR_BAD_SEQLENS;
* the fault drill drops one K tile load per CTA and bounds every pipeline
  wait to 100 ms: the MMA warp's wait runs out, the kernel records
  BSA_ERR_TIMEOUT, drains its own copies and MMAs, frees tensor memory and
  returns; the next normal call on the same context is correct. The decode
  and block-importance score kernels take the same drill.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import _cases
import _gpu

pytestmark = pytest.mark.gpu


def test_bad_seqlens_reported_and_nothing_written():
    b = _gpu.bsa()
    p = _cases.small_problem("gqa_ragged")
    q, k, v = _gpu.to_dev_bf16(p.q), _gpu.to_dev_bf16(p.k), _gpu.to_dev_bf16(p.v)
    cu = torch.tensor([0, 500, 300, 400], dtype=torch.int32, device="cuda")
    out = torch.full((p.total_tokens, p.Hq, p.d), 7.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((p.Hq, p.total_tokens), 7.0, dtype=torch.float32, device="cuda")
    st = b.prefill_fwd(q, k, v, cu, 3, p.Hq, p.Hkv, p.d, 1, 0.01, b.BSA_BF16, out, lse, None)
    assert st == 0   # the host cannot see device data; the prologue checks it
    assert b.get_device_status() == 6
    assert bool((out == 7.0).all()) and bool((lse == 7.0).all())
    assert b.get_device_status() == 0   # reading clears it


def test_fault_drill_times_out_cleanly_and_context_survives():
    b = _gpu.bsa()
    p = _cases.small_problem("gqa4")
    try:
        b.check(b.debug_fault_drill(5, 100_000_000), "drill")
        b.check(b.prefill_fwd(*_drill_args(p)), "launch")
        torch.cuda.synchronize()
        assert b.get_device_status() == 4   # BSA_ERR_TIMEOUT
    finally:
        b.check(b.debug_fault_drill(-1, 2_000_000_000), "restore")
    g = _gpu.run(p, lam=0.01)
    _gpu.compare(p, g)


_keep = []


def _drill_args(p):
    b = _gpu.bsa()
    q, k, v = _gpu.to_dev_bf16(p.q), _gpu.to_dev_bf16(p.k), _gpu.to_dev_bf16(p.v)
    cu = torch.from_numpy(p.cu_seqlens.astype(np.int32)).cuda()
    out = torch.empty((p.total_tokens, p.Hq, p.d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((p.Hq, p.total_tokens), dtype=torch.float32, device="cuda")
    bm = torch.empty((b.skip_bitmap_words(p.cu_seqlens, p.Hq),), dtype=torch.int32, device="cuda")
    _keep[:] = [q, k, v, cu, out, lse, bm]
    return (q, k, v, cu, p.n_seqs, p.Hq, p.Hkv, p.d, 1, 0.01, b.BSA_BF16, out, lse, bm)


def test_fault_drill_in_decode_and_importance():
    """The same drill in the split-KV decode kernel and the importance
    score kernel: each CTA's first K load is left out, the call records
    BSA_ERR_TIMEOUT, and the next normal calls are correct."""
    import test_gpu_decode as td
    import test_gpu_importance as ti
    from gen import inputs as gi
    from oracle import importance as imp
    b = _gpu.bsa()
    base = _cases.small_problem("gqa4")
    pd = gi.chunk(base, [2, 1])
    try:
        b.check(b.debug_fault_drill(0, 100_000_000), "drill")
        _, st = td.run_decode(pd, 0.005)
        assert st == 4   # BSA_ERR_TIMEOUT (run_decode reads and clears the status)
        _, _, st = ti.run_importance(base, 64)
        assert st == 4
    finally:
        b.check(b.debug_fault_drill(-1, 2_000_000_000), "restore")
    g, st = td.run_decode(pd, 0.005)
    assert st == 0
    _gpu.compare(pd, g)
    sc, mn, st = ti.run_importance(base, 64)
    assert st == 0
    ti.check_scores(sc.cpu().numpy(),
                    imp.block_importance(base.q, base.k, base.cu_seqlens, base.Hq, base.Hkv, 64, True))
