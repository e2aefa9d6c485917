"""GPU-side test helpers: run the CUDA library through its C interface and
compare with the CPU oracle under the parity tolerances.

Tolerances (bf16): skip bits bit-exact except on tiles whose oracle decision
margin is within 1e-3 (natural-log units) of the threshold; output in
mask-replay mode within max-abs 2e-2 and mean-abs 2e-3; lse within 1e-3.
FP8: output within max-abs 6e-2.

Comparisons run per query tile (``oracle.tile_walk.walk_one``), so a sample
of tiles of a full-size layer costs only those tiles.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import _oracle_tile
from oracle import layout, tile_walk

MARGIN_TOL = 1e-3
O_MAX_BF16, O_MEAN_BF16 = 2e-2, 2e-3
O_MAX_FP8 = 6e-2
LSE_TOL = 1e-3


def bsa():
    from dynamic_block_sparse_causal_gb300 import bsa as b
    b.lib()
    return b


def to_dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def run(p, lam=None, causal=None, fp8=None, stream=None, out_fill=float("nan")):
    """Run the library on problem ``p``.

    Returns dict(out=device bf16 tensor, lse=device fp32 tensor, bitmap=numpy
    uint32 words, lam, causal). ``fp8``: None for bf16, else ``(q_codes,
    k_codes, v_codes, q_scale, k_scale, v_scale)`` numpy arrays.
    """
    b = bsa()
    lam = p.lam if lam is None else lam
    causal = p.causal if causal is None else causal
    T = p.total_tokens
    cu = torch.from_numpy(p.cu_seqlens.astype(np.int32)).cuda()
    chunked = p.cu_seqlens_k is not None
    cuk = torch.from_numpy(p.cu_seqlens_k.astype(np.int32)).cuda() if chunked else None
    if fp8 is None:
        q, k, v = to_dev_bf16(p.q), to_dev_bf16(p.k), to_dev_bf16(p.v)
        dtype = b.BSA_BF16
    else:
        q, k, v = (torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in fp8[:3])
        scales = [torch.from_numpy(np.asarray(s, np.float32)).cuda() for s in fp8[3:]]
        b.check(b.set_fp8_scales(*scales), "set_fp8_scales")
        dtype = b.BSA_FP8_E4M3
    out = torch.full((T, p.Hq, p.d), out_fill, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((p.Hq, T), float("nan"), dtype=torch.float32, device="cuda")
    if chunked:
        nw = b.skip_bitmap_words_chunked(p.cu_seqlens, p.cu_seqlens_k, p.Hq)
    else:
        nw = b.skip_bitmap_words(p.cu_seqlens, p.Hq)
    bm = torch.full((max(nw, 1),), -1, dtype=torch.int32, device="cuda")
    if chunked:
        st = b.prefill_fwd_chunked(q, k, v, cu, cuk, p.n_seqs, p.Hq, p.Hkv, p.d, int(causal), lam,
                                   dtype, out, lse, bm, stream)
    else:
        st = b.prefill_fwd(q, k, v, cu, p.n_seqs, p.Hq, p.Hkv, p.d, int(causal), lam, dtype,
                           out, lse, bm, stream)
    b.check(st, "bsa_prefill_fwd")
    torch.cuda.synchronize()
    b.check(b.get_device_status(stream), "device status")
    if fp8 is not None:
        b.check(b.set_fp8_scales(None, None, None), "clear scales")
    return dict(out=out, lse=lse, bitmap=bm[:nw].cpu().numpy().view(np.uint32), lam=lam,
                causal=causal)


def host(g):
    """Outputs of a (small) run as float64 numpy arrays."""
    return g["out"].float().cpu().numpy().astype(np.float64), g["lse"].cpu().numpy().astype(np.float64)


def sample_items(p, max_items=None, seed=0, tail_heads=4):
    """All query tiles, or a deterministic sample of ``max_items``: the
    first and middle tiles of every sequence (random heads), its last tile
    (the sequence tail, the longest walk) for up to ``tail_heads`` heads,
    then random tiles."""
    items = tile_walk.all_items(p.cu_seqlens, p.Hq)
    if max_items is None or len(items) <= max_items:
        return items
    rng = np.random.default_rng(seed)
    tails = max(1, min(tail_heads, max_items // (3 * p.n_seqs)))
    pick = set()
    for s in range(p.n_seqs):
        n = layout.tiles(p.seqlens[s])
        pick.add((s, int(rng.integers(p.Hq)), 0))
        pick.add((s, int(rng.integers(p.Hq)), n // 2))
        for h in rng.choice(p.Hq, size=min(tails, p.Hq), replace=False):
            pick.add((s, int(h), n - 1))
    pick = sorted(pick)
    if len(pick) > max_items:
        pick = [pick[k] for k in sorted(rng.choice(len(pick), max_items, replace=False))]
    while len(pick) < max_items:
        it = items[int(rng.integers(len(items)))]
        if it not in pick:
            pick.append(it)
    return sorted(pick)


def compare(p, g, items=None, fp8=None, check_bits=True):
    """Compare a GPU result with the oracle on ``items`` (all query tiles by
    default); return a dict of metrics, asserting the tolerances. The count
    of bits that differ within the decision margin (allowed) is printed."""
    cu = p.cu_seqlens
    cuk = p.cu_seqlens if p.cu_seqlens_k is None else p.cu_seqlens_k
    lam, causal = g["lam"], g["causal"]
    items = tile_walk.all_items(cu, p.Hq) if items is None else list(items)
    arrays = (p.q, p.k, p.v) if fp8 is None else tuple(fp8[:3])
    scales = None if fp8 is None else tuple(fp8[3:])
    gots, visits = [], 0
    for item in items:
        s, h, i = item
        L, Lk = int(cu[s + 1] - cu[s]), int(cuk[s + 1] - cuk[s])
        r1 = min(i * 128 + 128, L)
        last = min((Lk - L + r1 - 1) // 128, layout.tiles(Lk) - 1) if causal else layout.tiles(Lk) - 1
        row = layout.row_bits(g["bitmap"], cu, p.Hq, s, h, i, cuk)
        assert not row[last + 1:].any(), f"bit set on an unvisited tile of {item}"
        gots.append(row[:last + 1])
        visits += last + 1
    refs = [_oracle_tile.reference(arrays, scales, cu, cuk, p.Hq, p.Hkv, causal, lam, it, got)
            for it, got in zip(items, gots)]
    bad_bits = near = 0
    o_max = o_sum = 0.0
    o_cnt = 0
    lse_max = 0.0
    for item, got, (want, mg, o_ref, lse_ref, last) in zip(items, gots, refs):
        s, h, i = item
        for j in np.nonzero(got != want)[0]:
            if j < len(mg) and abs(mg[j]) < MARGIN_TOL:
                near += 1
            else:
                bad_bits += 1
        a, L = int(cu[s]), int(cu[s + 1] - cu[s])
        r0, r1 = a + i * 128, a + min(i * 128 + 128, L)
        o_gpu = g["out"][r0:r1, h].float().cpu().numpy().astype(np.float64)
        l_gpu = g["lse"][h, r0:r1].cpu().numpy().astype(np.float64)
        d = np.abs(o_gpu - o_ref)
        assert np.isfinite(o_gpu).all(), f"non-finite output in {item}"
        o_max = max(o_max, float(d.max()))
        o_sum += float(d.sum())
        o_cnt += d.size
        lse_max = max(lse_max, float(np.abs(l_gpu - lse_ref).max()))
    res = dict(items=len(items), tile_visits=visits, bad_bits=bad_bits, near_margin=near,
               o_max=o_max, o_mean=o_sum / max(o_cnt, 1), lse_max=lse_max, values=o_cnt)
    print(f"parity {p.name} lambda={lam} causal={causal} fp8={fp8 is not None}: {res}")
    if check_bits:
        assert bad_bits == 0, f"{bad_bits} skip bits differ outside the 1e-3 margin: {res}"
    if fp8 is None:
        assert res["o_max"] <= O_MAX_BF16 and res["o_mean"] <= O_MEAN_BF16, res
    else:
        assert res["o_max"] <= O_MAX_FP8, res
    assert res["lse_max"] <= LSE_TOL, res
    return res
