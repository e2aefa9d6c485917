"""GPU parity for the block importance (bsa_block_importance) and the top-p
block selection (bsa_top_p_select), against the fp64 oracle.

Scores: every per-head block score within 5e-4 relative of the oracle plus
1e-9 absolute (a head's scores add up to 1/128 = 7.8e-3). The GPU sums fp32
products of exact bf16 inputs on the tensor cores (scores of up to ~65 in
log2 units on the sink keys, where a relative accumulation error of a few
2^-24 shifts an exponential by ~1e-5), takes 128-term fp32 sums of ex2.approx
values (relative error below 2^-21) and combines up to a few thousand of them
per row in a fp32 log-sum-exp; 5e-4 leaves a margin of about ten over that.
The absolute term covers weights below fp32's range (flushed to zero).

Selection, on the GPU's own float32 scores: the order is compared exactly
(both sides sort the same values, ties by index); k* must equal the
oracle's unless p x total lies within 1e-12 x total of the running sum at
either candidate (the two sides add in different orders). p is passed to the
oracle as the float32 value the library receives.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import _cases
import _gpu
from gen import inputs as gi
from oracle import importance as imp

pytestmark = pytest.mark.gpu

RTOL, ATOL = 5e-4, 1e-9
G = 128


def run_importance(p, n, causal=True, mean=True, total_blocks=None, fill=float("nan")):
    b = _gpu.bsa()
    tb = b.importance_blocks(p.cu_seqlens) if total_blocks is None else total_blocks
    q, k = _gpu.to_dev_bf16(p.q), _gpu.to_dev_bf16(p.k)
    cu = torch.from_numpy(p.cu_seqlens.astype(np.int32)).cuda()
    sc = torch.full((p.Hq, max(tb, 1)), fill, dtype=torch.float32, device="cuda")
    mn = torch.full((max(tb, 1),), fill, dtype=torch.float32, device="cuda") if mean else None
    st = b.block_importance(q, k, cu, p.n_seqs, p.Hq, p.Hkv, p.d, n, int(causal), tb, sc, mn)
    b.check(st, "bsa_block_importance")
    torch.cuda.synchronize()
    return sc, mn, b.get_device_status()


def run_top_p(scores, cu_seqlens, p_sel, keep=True, fill=-7):
    b = _gpu.bsa()
    cu_np = np.asarray(cu_seqlens, np.int32)
    tb = int(np.asarray(scores).shape[0])
    s = torch.from_numpy(np.ascontiguousarray(scores, np.float32)).cuda()
    cu = torch.from_numpy(cu_np).cuda()
    order = torch.full((max(tb, 1),), fill, dtype=torch.int32, device="cuda")
    nsel = torch.full((len(cu_np) - 1,), fill, dtype=torch.int32, device="cuda")
    kp = torch.full((max(tb, 1),), 9, dtype=torch.uint8, device="cuda") if keep else None
    st = b.top_p_select(s, cu, len(cu_np) - 1, tb, p_sel, order, nsel, kp)
    b.check(st, "bsa_top_p_select")
    torch.cuda.synchronize()
    return (order.cpu().numpy()[:tb], nsel.cpu().numpy(),
            kp.cpu().numpy()[:tb] if keep else None, b.get_device_status())


def check_scores(got, want):
    got = np.asarray(got, np.float64)
    err = np.abs(got - want)
    bound = RTOL * np.abs(want) + ATOL
    i = np.unravel_index(np.argmax(err - bound), err.shape)
    assert (err <= bound).all(), f"worst {i}: gpu {got[i]!r} oracle {want[i]!r}"
    return float((err / np.maximum(np.abs(want), 1e-30)).max())


def check_selection(scores, cu, p_sel, order, nsel, keep):
    p64 = float(np.float32(p_sel))
    off = imp.block_offsets(cu)
    for s in range(len(cu) - 1):
        a, b = int(off[s]), int(off[s + 1])
        if a == b:
            assert nsel[s] == 0
            continue
        x = np.asarray(scores[a:b], np.float64)
        o, k = imp.top_p(x, p64)
        assert np.array_equal(order[a:b], o), f"sequence {s}: order differs"
        if nsel[s] != k:
            run = np.cumsum(x[o])
            thr = p64 * run[-1]
            near = [abs(run[j - 1] - thr) <= 1e-12 * run[-1] for j in (k, int(nsel[s]))
                    if 1 <= j <= b - a]
            assert any(near), f"sequence {s}: k* {nsel[s]} vs oracle {k}"
        if keep is not None:
            kk = int(nsel[s])
            want = np.zeros(b - a, np.uint8)
            want[o[:kk]] = 1
            assert np.array_equal(keep[a:b], want)


CASES = [("gqa_ragged", 64), ("gqa4", 128), ("tiny", 37), ("weak_sink", 1), ("no_sink", 100)]


@pytest.mark.parametrize("key,n", CASES)
@pytest.mark.parametrize("causal", [True, False])
def test_scores_match_oracle(key, n, causal):
    p = _cases.small_problem(key)
    sc, mn, st = run_importance(p, n, causal)
    assert st == 0
    want = imp.block_importance(p.q, p.k, p.cu_seqlens, p.Hq, p.Hkv, n, causal)
    print(key, n, causal, "max rel err", check_scores(sc.cpu().numpy(), want))
    check_scores(mn.cpu().numpy(), imp.head_mean(want))


def test_planted_block_scores():
    # block-constant scores: the GPU against the oracle on the planted tiles
    p = _cases.planted_problem()
    for causal in (True, False):
        sc, _, st = run_importance(p, 50, causal, mean=False)
        assert st == 0
        check_scores(sc.cpu().numpy(),
                     imp.block_importance(p.q, p.k, p.cu_seqlens, 1, 1, 50, causal))


def test_empty_sequence_and_window_longer_than_sequence():
    base = gi.small("imp_edge", [300, 1, 129], Hq=2, Hkv=1, seed=9)
    cu = np.array([0, 300, 301, 301, 430], np.int32)             # third sequence empty
    p = gi.Problem("imp_edge", base.q, base.k, base.v, cu, 2, 1, 128)
    sc, mn, st = run_importance(p, 128)
    assert st == 0
    want = imp.block_importance(p.q, p.k, p.cu_seqlens, 2, 1, 128, True)
    check_scores(sc.cpu().numpy(), want)


def test_block_far_above_the_earlier_blocks_of_its_chunk():
    """A key block whose scores exceed every earlier block of its 16-block
    chunk by far more than 127 in log2 units (its keys scaled by 256): the
    kernel takes a tile's (t, e) against the chunk's running maximum, so this
    tile's sum overflows and is taken again against the tile's own maximum.
    Block scores and head means against the oracle, causal and not."""
    base = gi.small("imp_far", [700], Hq=4, Hkv=1, seed=11)
    k = gi.bf16_bits_to_f32(base.k)
    k[3 * G:4 * G] *= 256.0
    p = gi.Problem("imp_far", base.q, gi.bf16_bits_from_f32(k), base.v, base.cu_seqlens, 4, 1, 128)
    qf, kf = gi.bf16_bits_to_f32(p.q), gi.bf16_bits_to_f32(p.k)
    s3 = np.einsum("hd,kd->hk", qf[-1], kf[3 * G:4 * G, 0]) / np.sqrt(128.0) * np.log2(np.e)
    s0 = np.einsum("hd,kd->hk", qf[-1], kf[:3 * G, 0]) / np.sqrt(128.0) * np.log2(np.e)
    assert (s3.max(axis=1) - s0.max(axis=1)).max() > 200   # the case is what it claims
    for n, causal in ((64, True), (128, False)):
        sc, mn, st = run_importance(p, n, causal)
        assert st == 0
        want = imp.block_importance(p.q, p.k, p.cu_seqlens, 4, 1, n, causal)
        print(n, causal, "max rel err", check_scores(sc.cpu().numpy(), want))
        check_scores(mn.cpu().numpy(), imp.head_mean(want))


def test_full_size_mass_and_sampled_heads():
    """The 128K Llama-shaped layer: every head's scores add up to 1/128, and
    four heads (one per KV group pair) match the oracle."""
    p = _cases.full_problem("C2")
    sc, mn, st = run_importance(p, 64)
    assert st == 0
    s = sc.cpu().numpy().astype(np.float64)
    np.testing.assert_allclose(s.sum(axis=1) * G, 1.0, rtol=0, atol=2e-4)
    assert (s >= 0).all()
    L = int(p.cu_seqlens[1])
    for h in (0, 9, 18, 31):
        qh = _cases.f64(p.q[:, h])
        kh = _cases.f64(p.k[:, h // 4])
        want = imp.sequence_scores(qh, kh, 64, True)
        check_scores(s[h], want)
    assert L == 131072


def test_rejects_wrong_block_count():
    p = _cases.small_problem("gqa_ragged")
    b = _gpu.bsa()
    tb = b.importance_blocks(p.cu_seqlens)
    sc, mn, st = run_importance(p, 64, total_blocks=tb - 1, fill=5.0)
    assert st == 6
    assert bool((sc == 5.0).all()) and bool((mn == 5.0).all())


@pytest.mark.parametrize("p_sel", [0.5, 0.9, 0.95, 1.0])
def test_selection_on_importance_scores(p_sel):
    p = _cases.small_problem("gqa4")
    _, mn, _ = run_importance(p, 64)
    m = mn.cpu().numpy()
    order, nsel, keep, st = run_top_p(m, p.cu_seqlens, p_sel)
    assert st == 0
    check_selection(m, p.cu_seqlens, p_sel, order, nsel, keep)


@pytest.mark.parametrize("nb", [1, 2, 3, 1000, 1024, 4097, 16384])
def test_selection_random_scores_with_ties(nb):
    rng = np.random.default_rng(nb)
    x = rng.integers(0, 50, nb).astype(np.float32) / 64.0      # many ties and zeros
    x[rng.integers(0, nb)] = 3.0
    cu = np.array([0, nb * 128 - 5], np.int32)                 # ragged last block
    for p_sel in (0.3, 0.9, 1.0):
        order, nsel, keep, st = run_top_p(x, cu, p_sel)
        assert st == 0
        check_selection(x, cu, p_sel, order, nsel, keep)


def test_selection_packed_batch_and_edges():
    rng = np.random.default_rng(11)
    L = [5000, 0, 1, 128 * 300, 129]
    cu = np.concatenate([[0], np.cumsum(L)]).astype(np.int32)
    tb = int(imp.block_offsets(cu)[-1])
    x = rng.random(tb).astype(np.float32) ** 4
    x[:3] = 0.0
    order, nsel, keep, st = run_top_p(x, cu, 0.8)
    assert st == 0
    check_selection(x, cu, 0.8, order, nsel, keep)
    order, nsel, keep, st = run_top_p(x, cu, 0.8, keep=False)
    assert st == 0 and keep is None
    check_selection(x, cu, 0.8, order, nsel, None)


def test_selection_tiny_p_keeps_the_top_block():
    x = np.array([0.125, 0.5, 0.25, 0.125], np.float32)
    order, nsel, keep, st = run_top_p(x, np.array([0, 500], np.int32), 1e-6)
    assert st == 0 and nsel[0] == 1 and order.tolist() == [1, 2, 0, 3]
    assert keep.tolist() == [0, 1, 0, 0]


def test_selection_p_one_drops_trailing_zeros():
    x = np.array([0.0, 0.25, 0.0, 0.5, 0.0], np.float32)
    order, nsel, keep, st = run_top_p(x, np.array([0, 600], np.int32), 1.0)
    assert st == 0 and nsel[0] == 2 and order.tolist() == [3, 1, 0, 2, 4]
    assert keep.tolist() == [0, 1, 0, 1, 0]


def test_selection_rejects_oversized_sequence_and_bad_total():
    x = np.ones(16385, np.float32)
    order, nsel, keep, st = run_top_p(x, np.array([0, 16385 * 128], np.int32), 0.5)
    assert st == 6 and (order == -7).all() and (nsel == -7).all()
    b = _gpu.bsa()
    s = torch.ones(10, device="cuda")
    cu = torch.tensor([0, 128 * 9], dtype=torch.int32, device="cuda")   # 9 blocks, not 10
    o = torch.full((10,), -7, dtype=torch.int32, device="cuda")
    n = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    assert b.top_p_select(s, cu, 1, 10, 0.5, o, n, None) == 0
    assert b.get_device_status() == 6
    assert bool((o == -7).all()) and int(n[0]) == -7
