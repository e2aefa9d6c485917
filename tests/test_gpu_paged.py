"""GPU parity for the paged KV cache (bsa_prefill_fwd_paged).

Keys and values are scattered over a pool of 128-token pages in a shuffled
order (unused pages and the unused tail of each sequence's last page hold
finite junk); the page table maps each sequence's key tiles to pages. The
paged call must give exactly the results of the packed chunked call on the
same data, and match the oracle; a page index outside the pool is rejected
on the device.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import _cases
import _gpu
from gen import inputs as gi

pytestmark = pytest.mark.gpu


def page_pool(p, extra_pages=5, seed=0):
    """Scatter p's packed K/V (by cu_seqlens_k) into shuffled 128-token pages."""
    rng = np.random.default_rng(seed)
    cuk = p.cu_seqlens_k if p.cu_seqlens_k is not None else p.cu_seqlens
    lens = np.diff(cuk.astype(np.int64))
    nk = (lens + 127) // 128
    num_pages = int(nk.sum()) + extra_pages
    max_pages = int(nk.max()) + 2
    order = rng.permutation(num_pages)
    junk = gi.bf16_bits_from_f32(rng.standard_normal((num_pages, 128, p.Hkv, p.d), dtype=np.float32))
    kc, vc = junk.copy(), junk[::-1].copy()
    table = np.full((len(lens), max_pages), -1, np.int32)
    nxt = 0
    for s, L in enumerate(lens):
        a = int(cuk[s])
        for j in range(int(nk[s])):
            pg = int(order[nxt])
            nxt += 1
            table[s, j] = pg
            t0, t1 = j * 128, min(j * 128 + 128, int(L))
            kc[pg, :t1 - t0] = p.k[a + t0:a + t1]
            vc[pg, :t1 - t0] = p.v[a + t0:a + t1]
    return kc, vc, table, num_pages, max_pages


def run_paged(p, pool, lam, causal=True):
    b = _gpu.bsa()
    kc, vc, table, num_pages, max_pages = pool
    cuk = p.cu_seqlens_k if p.cu_seqlens_k is not None else p.cu_seqlens
    T = p.total_tokens
    q = _gpu.to_dev_bf16(p.q)
    kd, vd = _gpu.to_dev_bf16(kc), _gpu.to_dev_bf16(vc)
    pt = torch.from_numpy(table).cuda()
    cq = torch.from_numpy(p.cu_seqlens.astype(np.int32)).cuda()
    ck = torch.from_numpy(cuk.astype(np.int32)).cuda()
    out = torch.full((T, p.Hq, p.d), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((p.Hq, T), float("nan"), dtype=torch.float32, device="cuda")
    nw = b.skip_bitmap_words_chunked(p.cu_seqlens, cuk, p.Hq)
    bm = torch.full((max(nw, 1),), -1, dtype=torch.int32, device="cuda")
    st = b.prefill_fwd_paged(q, kd, vd, pt, max_pages, num_pages, cq, ck, p.n_seqs, p.Hq, p.Hkv,
                             p.d, int(causal), lam, b.BSA_BF16, out, lse, bm)
    b.check(st, "bsa_prefill_fwd_paged")
    torch.cuda.synchronize()
    b.check(b.get_device_status(), "device status")
    return dict(out=out, lse=lse, bitmap=bm[:nw].cpu().numpy().view(np.uint32), lam=lam,
                causal=causal)


CASES = [("gqa_ragged", [100, 777, 1, 200]), ("weak_sink", [384, 900]), ("gqa4", [1536, 777])]


@pytest.mark.parametrize("key,lq", CASES)
@pytest.mark.parametrize("lam", [0.01, 0.0, 0.3])
@pytest.mark.parametrize("causal", [True, False])
def test_paged_equals_packed_and_matches_oracle(key, lq, lam, causal):
    base = _cases.small_problem(key)
    p = gi.chunk(base, lq)
    g = run_paged(p, page_pool(p, seed=len(lq)), lam, causal)
    ref = _gpu.run(p, lam=lam, causal=causal)
    assert torch.equal(g["out"], ref["out"]) and torch.equal(g["lse"], ref["lse"])
    assert np.array_equal(g["bitmap"], ref["bitmap"])
    _gpu.compare(p, g)


def test_paged_rejects_page_outside_pool():
    b = _gpu.bsa()
    p = gi.chunk(_cases.small_problem("weak_sink"), [384, 900])
    kc, vc, table, num_pages, max_pages = page_pool(p)
    table[1, 3] = num_pages           # one past the pool
    g_out = torch.full((p.total_tokens, p.Hq, p.d), 5.0, dtype=torch.bfloat16, device="cuda")
    st = b.prefill_fwd_paged(_gpu.to_dev_bf16(p.q), _gpu.to_dev_bf16(kc), _gpu.to_dev_bf16(vc),
                             torch.from_numpy(table).cuda(), max_pages, num_pages,
                             torch.from_numpy(p.cu_seqlens).cuda(),
                             torch.from_numpy(p.cu_seqlens_k).cuda(), p.n_seqs, p.Hq, p.Hkv, p.d,
                             1, 0.01, b.BSA_BF16, g_out, None, None)
    assert st == 0
    assert b.get_device_status() == 6
    assert bool((g_out == 5.0).all())


def test_paged_fp8_equals_packed():
    """FP8 E4M3 codes in the page pool (finite junk in unused slots): the paged
    call equals the packed chunked FP8 call bit for bit and matches the oracle."""
    import test_gpu_fp8
    p = gi.chunk(_cases.small_problem("gqa_ragged"), [100, 777, 1, 200])
    f8q, f8k, f8v = (test_gpu_fp8.gpu_quantize(x) for x in (p.q, p.k, p.v))
    f8 = (f8q[0], f8k[0], f8v[0], f8q[1], f8k[1], f8v[1])
    ref = _gpu.run(p, lam=0.05, fp8=f8)
    rng = np.random.default_rng(3)
    cuk = p.cu_seqlens_k
    lens = np.diff(cuk.astype(np.int64))
    nk = (lens + 127) // 128
    num_pages = int(nk.sum()) + 3
    max_pages = int(nk.max()) + 1
    order = rng.permutation(num_pages)
    junk = rng.integers(0, 0x7F, (num_pages, 128, p.Hkv, p.d)).astype(np.uint8)   # finite codes
    junk |= (rng.integers(0, 2, junk.shape) << 7).astype(np.uint8)                  # either sign
    kc, vc = junk.copy(), junk[::-1].copy()
    table = np.full((p.n_seqs, max_pages), -1, np.int32)
    nxt = 0
    for s, L in enumerate(lens):
        a = int(cuk[s])
        for j in range(int(nk[s])):
            pg = int(order[nxt])
            nxt += 1
            table[s, j] = pg
            t0, t1 = j * 128, min(j * 128 + 128, int(L))
            kc[pg, :t1 - t0] = f8k[0][a + t0:a + t1]
            vc[pg, :t1 - t0] = f8v[0][a + t0:a + t1]
    b = _gpu.bsa()
    scales = [torch.from_numpy(np.asarray(x[1], np.float32)).cuda() for x in (f8q, f8k, f8v)]
    b.check(b.set_fp8_scales(*scales), "scales")
    try:
        T = p.total_tokens
        out = torch.full((T, p.Hq, p.d), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((p.Hq, T), float("nan"), dtype=torch.float32, device="cuda")
        nw = b.skip_bitmap_words_chunked(p.cu_seqlens, cuk, p.Hq)
        bm = torch.full((max(nw, 1),), -1, dtype=torch.int32, device="cuda")
        st = b.prefill_fwd_paged(torch.from_numpy(f8q[0]).cuda(), torch.from_numpy(kc).cuda(),
                                 torch.from_numpy(vc).cuda(), torch.from_numpy(table).cuda(),
                                 max_pages, num_pages, torch.from_numpy(p.cu_seqlens).cuda(),
                                 torch.from_numpy(cuk).cuda(), p.n_seqs, p.Hq, p.Hkv, p.d, 1, 0.05,
                                 b.BSA_FP8_E4M3, out, lse, bm)
        b.check(st, "paged fp8")
        torch.cuda.synchronize()
        b.check(b.get_device_status(), "device status")
    finally:
        b.check(b.set_fp8_scales(None, None, None), "clear scales")
    assert torch.equal(out, ref["out"]) and torch.equal(lse, ref["lse"])
    g = dict(out=out, lse=lse, bitmap=bm[:nw].cpu().numpy().view(np.uint32), lam=0.05, causal=True)
    assert np.array_equal(g["bitmap"], ref["bitmap"])
    _gpu.compare(p, g, fp8=f8)


def test_paged_128k_chunk_as_benched():
    """The bench's paged leg: the last 8192 queries of the 128K layer against
    all 131072 keys, K/V scattered over a shuffled pool of 1024 pages (page j
    of the sequence is pool page perm[j]). Equal bit for bit to the packed
    chunked call, and matching the oracle on sampled query tiles (the last
    tiles of several heads included)."""
    b = _gpu.bsa()
    base = _cases.full_problem("C2")
    p = gi.chunk(base, [8192])
    T, Hq, Hkv, d = base.total_tokens, base.Hq, base.Hkv, base.d
    n_pages = T // 128
    perm = np.random.default_rng(0).permutation(n_pages).astype(np.int32)
    k, v = _gpu.to_dev_bf16(base.k), _gpu.to_dev_bf16(base.v)
    kpool = torch.empty_like(k)
    vpool = torch.empty_like(v)
    pd = torch.from_numpy(perm).cuda()
    kpool.view(n_pages, 128, Hkv, d)[pd.long()] = k.view(n_pages, 128, Hkv, d)
    vpool.view(n_pages, 128, Hkv, d)[pd.long()] = v.view(n_pages, 128, Hkv, d)
    q = _gpu.to_dev_bf16(p.q)
    cq = torch.tensor([0, 8192], dtype=torch.int32, device="cuda")
    ck = torch.from_numpy(base.cu_seqlens).cuda()
    nw = b.skip_bitmap_words_chunked(p.cu_seqlens, base.cu_seqlens, Hq)
    res = []
    for paged in (True, False):
        out = torch.full((8192, Hq, d), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((Hq, 8192), float("nan"), dtype=torch.float32, device="cuda")
        bm = torch.full((nw,), -1, dtype=torch.int32, device="cuda")
        if paged:
            st = b.prefill_fwd_paged(q, kpool, vpool, pd.view(1, n_pages), n_pages, n_pages, cq, ck,
                                     1, Hq, Hkv, d, 1, 0.01, b.BSA_BF16, out, lse, bm)
        else:
            st = b.prefill_fwd_chunked(q, k, v, cq, ck, 1, Hq, Hkv, d, 1, 0.01, b.BSA_BF16, out,
                                       lse, bm)
        b.check(st, "paged" if paged else "chunked")
        torch.cuda.synchronize()
        b.check(b.get_device_status(), "device status")
        res.append(dict(out=out, lse=lse, bitmap=bm.cpu().numpy().view(np.uint32), lam=0.01,
                        causal=True))
    g, ref = res
    assert torch.equal(g["out"], ref["out"]) and torch.equal(g["lse"], ref["lse"])
    assert np.array_equal(g["bitmap"], ref["bitmap"])
    _gpu.compare(p, g, items=_gpu.sample_items(p, 32, seed=5))
