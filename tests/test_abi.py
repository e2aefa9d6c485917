"""The C interface without a GPU: the library loads, exports every entry
point include/bsa.h declares, and rejects invalid arguments before touching
CUDA. Also the host-side bitmap-size helper against the layout restated in
the oracle, and the multi-process max-over-ranks reduction of bench.py on
two gloo ranks.
"""
from __future__ import annotations

import ctypes
import math
import os
import re

import numpy as np
import pytest

from oracle import layout

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from dynamic_block_sparse_causal_gb300 import build, bsa
    if not os.path.exists(build.LIB_PATH):
        build.build()
    return bsa


def declared_functions():
    src = open(os.path.join(ROOT, "include", "bsa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(bsa_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_symbol(L):
    lib = L.lib()
    names = declared_functions()
    assert "bsa_prefill_fwd" in names and len(names) >= 9
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings_and_version(L):
    assert L.status_string(0) == "ok"
    assert "timed out" in L.status_string(4)
    assert L.version() >= 100


def call(L, **over):
    a = dict(q=16, k=32, v=48, cu=64, n_seqs=1, Hq=4, Hkv=2, d=128, causal=1, lam=0.01, dtype=0,
             out=80, lse=None, bm=None)
    a.update(over)
    return L.prefill_fwd(a["q"], a["k"], a["v"], a["cu"], a["n_seqs"], a["Hq"], a["Hkv"], a["d"],
                         a["causal"], a["lam"], a["dtype"], a["out"], a["lse"], a["bm"])


@pytest.mark.parametrize("over,want", [
    (dict(q=None), 1), (dict(k=None), 1), (dict(v=None), 1), (dict(cu=None), 1), (dict(out=None), 1),
    (dict(q=18), 1), (dict(out=8), 1), (dict(cu=66), 1), (dict(lse=2), 1), (dict(bm=6), 1),
    (dict(n_seqs=0), 1), (dict(Hq=0), 1), (dict(Hkv=0), 1), (dict(Hq=6, Hkv=4), 1),
    (dict(causal=2), 1), (dict(lam=-0.1), 1), (dict(lam=1.0), 1), (dict(lam=math.nan), 1),
    (dict(lam=math.inf), 1), (dict(dtype=7), 1), (dict(dtype=1), 1),   # fp8 without scales
    (dict(d=64), 2), (dict(d=256), 2),
])
def test_invalid_arguments_rejected_before_cuda(L, over, want):
    assert call(L, **over) == want


def test_fp8_scales_all_or_nothing(L):
    assert L.set_fp8_scales(16, None, None) == 1
    assert L.set_fp8_scales(None, None, None) == 0


def test_quantize_argument_checks(L):
    assert L.quantize_fp8(None, 10, 2, 128, 16, 16) == 1
    assert L.quantize_fp8(16, -1, 2, 128, 16, 16) == 1
    assert L.quantize_fp8(16, 10, 2, 12, 16, 16) == 1
    assert L.quantize_fp8(18, 10, 2, 128, 16, 16) == 1


def test_fault_drill_argument_checks(L):
    assert L.debug_fault_drill(-2, 10) == 1
    assert L.debug_fault_drill(-1, 0) == 1
    assert L.debug_fault_drill(-1, 2000000000) == 0


@pytest.mark.parametrize("cu,Hq", [([0, 2048], 1), ([0, 300, 5000], 2), ([0, 131072], 32),
                                   ([0, 1, 78, 206], 2), ([0, 0, 129, 129], 3)])
def test_bitmap_words_match_layout(L, cu, Hq):
    assert L.skip_bitmap_words(np.array(cu, np.int32), Hq) == layout.total_words(cu, Hq)


@pytest.mark.parametrize("cuq,cuk,Hq", [([0, 200], [0, 1000], 3), ([0, 10, 300], [0, 100, 5220], 2),
                                        ([0, 2048], [0, 2048], 4), ([0, 0, 77], [0, 64, 77], 1)])
def test_chunked_bitmap_words_match_layout(L, cuq, cuk, Hq):
    assert L.skip_bitmap_words_chunked(np.array(cuq, np.int32), np.array(cuk, np.int32), Hq) == \
        layout.total_words(cuq, Hq, cuk)


def test_chunked_argument_checks(L):
    args = (16, 32, 48, 64, 96, 1, 4, 2, 128, 1, 0.01, 0, 80, None, None)
    assert L.prefill_fwd_chunked(*(args[:4] + (None,) + args[5:])) == 1    # no cu_seqlens_k
    assert L.prefill_fwd_chunked(*(args[:4] + (98,) + args[5:])) == 1      # misaligned
    assert L.prefill_fwd_chunked(*(args[:8] + (64,) + args[9:])) == 2      # d != 128


def test_paged_argument_checks(L):
    a = dict(q=16, k=32, v=48, pt=64, mp=4, npg=10, cuq=80, cuk=96, n=1, Hq=4, Hkv=2, d=128, c=1,
             lam=0.01, dt=0, out=112, lse=None, bm=None)

    def call(**o):
        b = dict(a, **o)
        return L.prefill_fwd_paged(b["q"], b["k"], b["v"], b["pt"], b["mp"], b["npg"], b["cuq"],
                                   b["cuk"], b["n"], b["Hq"], b["Hkv"], b["d"], b["c"], b["lam"],
                                   b["dt"], b["out"], b["lse"], b["bm"])
    assert call(pt=None) == 1 and call(pt=66) == 1 and call(mp=0) == 1 and call(npg=0) == 1
    assert call(npg=1 << 24) == 1           # pool larger than a 32-bit token index
    assert call(cuk=None) == 1 and call(lam=2.0) == 1 and call(d=96) == 2


def test_importance_argument_checks(L):
    a = dict(q=16, k=32, cu=64, n=1, Hq=4, Hkv=2, d=128, nw=64, c=1, tb=10, sc=80, mean=None)

    def call(**o):
        b = dict(a, **o)
        return L.block_importance(b["q"], b["k"], b["cu"], b["n"], b["Hq"], b["Hkv"], b["d"],
                                  b["nw"], b["c"], b["tb"], b["sc"], b["mean"])
    assert call(q=None) == 1 and call(k=None) == 1 and call(cu=None) == 1 and call(sc=None) == 1
    assert call(q=24) == 1 and call(cu=66) == 1 and call(sc=82) == 1 and call(mean=83) == 1
    assert call(n=0) == 1 and call(Hq=6, Hkv=4) == 1 and call(c=2) == 1
    assert call(nw=0) == 1 and call(nw=129) == 1 and call(tb=-1) == 1
    assert call(d=64) == 2


def test_decode_argument_checks(L):
    a = dict(q=16, k=32, v=48, cq=64, ck=80, n=2, mq=1, tk=1000, Hq=32, Hkv=8, d=128, c=1,
             lam=0.005, out=96, lse=None, bm=None)

    def call(**o):
        b = dict(a, **o)
        return L.decode_fwd(b["q"], b["k"], b["v"], b["cq"], b["ck"], b["n"], b["mq"], b["tk"],
                            b["Hq"], b["Hkv"], b["d"], b["c"], b["lam"], b["out"], b["lse"], b["bm"])
    assert call(q=None) == 1 and call(v=None) == 1 and call(ck=None) == 1 and call(out=None) == 1
    assert call(k=40) == 1 and call(cq=66) == 1 and call(lse=2) == 1
    assert call(mq=0) == 1 and call(mq=9) == 1                # 4 x 9 rows > 32
    assert call(Hq=32, Hkv=1) == 1                             # group above 16
    assert call(tk=-1) == 1 and call(tk=1 << 31) == 1 and call(lam=1.0) == 1 and call(c=3) == 1
    assert call(n=0) == 1 and call(Hq=30, Hkv=8) == 1
    assert call(d=64) == 2


def test_top_p_argument_checks(L):
    a = dict(sc=16, cu=32, n=1, tb=10, p=0.9, order=48, nsel=64, keep=None)

    def call(**o):
        b = dict(a, **o)
        return L.top_p_select(b["sc"], b["cu"], b["n"], b["tb"], b["p"], b["order"], b["nsel"],
                              b["keep"])
    assert call(sc=None) == 1 and call(cu=None) == 1 and call(order=None) == 1
    assert call(nsel=None) == 1 and call(order=50) == 1 and call(n=0) == 1 and call(tb=-1) == 1
    for bad_p in (0.0, -0.5, 1.0000001, 2.0, math.nan, math.inf):
        assert call(p=bad_p) == 1


@pytest.mark.parametrize("cu", [[0, 2048], [0, 300, 5000], [0, 1, 78, 206], [0, 0, 129, 129]])
def test_importance_blocks_match_oracle(L, cu):
    from oracle import importance
    assert L.importance_blocks(np.array(cu, np.int32)) == int(importance.block_offsets(cu)[-1])
    assert L.importance_blocks(np.array([0, 5, 3], np.int32)) == -1


def test_bitmap_words_rejects_bad_seqlens(L):
    assert L.skip_bitmap_words(np.array([1, 5], np.int32), 1) == -1
    assert L.skip_bitmap_words(np.array([0, 5, 3], np.int32), 1) == -1


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import sys
    sys.path.insert(0, ROOT)
    import bench
    t = bench.max_over_ranks(10.0 + rank, world)
    bench.barrier(world)
    q.put((rank, t))
    dist.destroy_process_group()


def test_bench_max_over_ranks_gloo():
    import multiprocessing as mp
    import socket
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
    got = sorted(q.get(timeout=5) for _ in range(2))
    assert got == [(0, 11.0), (1, 11.0)]
