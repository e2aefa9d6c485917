"""GPU-side test helpers: run the CUDA library through its C interface and
compare with the CPU oracle under the parity tolerances.

Tolerances (bf16): skip bits bit-exact except on tiles whose oracle decision
margin is within 1e-3 (natural-log units) of the threshold; output in
mask-replay mode within max-abs 2e-2 and mean-abs 2e-3; lse within 1e-3.
FP8: output within max-abs 6e-2.
"""
from __future__ import annotations

import math

import numpy as np
import torch

from oracle import layout, numerics, tile_walk

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
    """Run the library on problem ``p``; return dict of numpy outputs.

    ``fp8``: None for bf16, else ``(q_codes, k_codes, v_codes, q_scale, k_scale, v_scale)``
    as numpy arrays (device tensors are made here).
    """
    b = bsa()
    lam = p.lam if lam is None else lam
    causal = p.causal if causal is None else causal
    T = p.total_tokens
    cu = torch.from_numpy(p.cu_seqlens.astype(np.int32)).cuda()
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
    nw = b.skip_bitmap_words(p.cu_seqlens, p.Hq)
    bm = torch.full((max(nw, 1),), -1, dtype=torch.int32, device="cuda")
    st = b.prefill_fwd(q, k, v, cu, p.n_seqs, p.Hq, p.Hkv, p.d, int(causal), lam, dtype,
                       out, lse, bm, stream)
    b.check(st, "bsa_prefill_fwd")
    torch.cuda.synchronize()
    b.check(b.get_device_status(stream), "device status")
    if fp8 is not None:
        b.check(b.set_fp8_scales(None, None, None), "clear scales")
    return dict(out=out.float().cpu().numpy().astype(np.float64), lse=lse.cpu().numpy().astype(np.float64),
                bitmap=bm[:nw].cpu().numpy().view(np.uint32), lam=lam, causal=causal)


def sample_items(p, max_items=None, heads=None, seed=0):
    """All query tiles, or a deterministic sample: first / last tiles and a spread."""
    items = tile_walk.all_items(p.cu_seqlens, p.Hq)
    if max_items is None or len(items) <= max_items:
        return items
    rng = np.random.default_rng(seed)
    pick = set()
    for s in range(p.n_seqs):
        n = layout.tiles(p.seqlens[s])
        for i in {0, n - 1, n // 2}:
            pick.add((s, int(rng.integers(p.Hq)) if heads is None else heads[0], i))
    while len(pick) < max_items:
        pick.add(items[int(rng.integers(len(items)))])
    return sorted(pick)[:max_items] if len(pick) > max_items else sorted(pick)


def compare(p, g, items=None, fp8=None, check_bits=True):
    """Compare a GPU result with the oracle; return a dict of metrics (asserts inside)."""
    if fp8 is None:
        q, k, v = (numerics.bf16_to_f64(x) for x in (p.q, p.k, p.v))
    else:
        q, k, v = (numerics.e4m3_to_f64(c) * np.asarray(s, np.float64)[None, :, None]
                   for c, s in zip(fp8[:3], fp8[3:]))
    cu, lam, causal = p.cu_seqlens, g["lam"], g["causal"]
    ref = tile_walk.prefill_fwd(q, k, v, cu, p.Hq, p.Hkv, causal=causal, lam=lam, items=items)
    bad_bits = 0
    near = 0
    for item, mg in ref.margins.items():
        s, h, i = item
        got = layout.row_bits(g["bitmap"], cu, p.Hq, s, h, i)
        want = layout.row_bits(ref.bitmap, cu, p.Hq, s, h, i)
        diff = np.nonzero(got != want)[0]
        for j in diff:
            if j < len(mg) and abs(mg[j]) < MARGIN_TOL:
                near += 1
            else:
                bad_bits += 1
    if check_bits:
        assert bad_bits == 0, f"{bad_bits} skip bits differ outside the 1e-3 margin"
    # mask replay: the oracle takes the GPU's decisions
    rep = tile_walk.prefill_fwd(q, k, v, cu, p.Hq, p.Hkv, causal=causal, lam=lam, items=items,
                                replay_bitmap=g["bitmap"])
    rows = ~np.isnan(rep.out[:, :, 0])
    do = np.abs(g["out"] - rep.out)[rows]
    dl = np.abs(g["lse"] - rep.lse)[~np.isnan(rep.lse)]
    res = dict(bad_bits=bad_bits, near_margin=near, o_max=float(do.max()), o_mean=float(do.mean()),
               lse_max=float(dl.max()), rows=int(rows.sum()))
    if fp8 is None:
        assert res["o_max"] <= O_MAX_BF16 and res["o_mean"] <= O_MEAN_BF16, res
    else:
        assert res["o_max"] <= O_MAX_FP8, res
    assert res["lse_max"] <= LSE_TOL, res
    assert np.isfinite(g["out"][rows]).all()
    return res
