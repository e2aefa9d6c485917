"""The multi-GPU split of one layer by KV heads, on two gloo ranks (CPU).

Every KV head (and its query heads) must belong to exactly one rank, and the
per-rank pieces must reassemble the layer's outputs: each rank runs the
oracle on its piece (no GPU), the pieces are gathered on rank 0 and put back
in head order, and the result equals the oracle on the whole layer (out,
lse, skip bits). The GPU path runs the same pieces through the C interface
(bench.py --gpus N); no data crosses ranks, only the timing reduction.
"""
from __future__ import annotations

import multiprocessing as mp
import os
import socket

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("Hkv,world", [(8, 2), (8, 8), (5, 2), (3, 3)])
def test_head_ranges_partition_the_heads(Hkv, world):
    from gen import inputs as gi
    covered = []
    for r in range(world):
        lo, hi = gi.head_range(Hkv, world, r)
        assert hi > lo
        covered += list(range(lo, hi))
    assert covered == list(range(Hkv))


def _problem():
    from gen import inputs as gi
    return gi.small("split", [300, 700], Hq=8, Hkv=4, seed=21, lam=0.01)


def _oracle(p):
    from oracle import numerics, tile_walk
    q, k, v = (numerics.bf16_to_f64(x) for x in (p.q, p.k, p.v))
    return tile_walk.prefill_fwd(q, k, v, p.cu_seqlens, p.Hq, p.Hkv, lam=p.lam)


def _rank_main(rank, world, port, queue):
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from gen import inputs as gi
    piece = gi.split_heads(_problem(), rank, world)
    r = _oracle(piece)
    got = [None] * world
    dist.all_gather_object(got, (rank, gi.head_range(4, world, rank), r.out, r.lse, r.bitmap))
    if rank == 0:
        queue.put(got)
    dist.destroy_process_group()


def test_pieces_reassemble_the_layer_on_two_gloo_ranks():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, queue)) for r in range(2)]
    for p in procs:
        p.start()
    got = queue.get(timeout=300)
    for p in procs:
        p.join(60)
        assert p.exitcode == 0
    from oracle import layout
    full = _problem()
    ref = _oracle(full)
    got.sort(key=lambda g: g[0])
    G = full.Hq // full.Hkv
    # every KV head exactly once, in order
    assert [h for g in got for h in range(*g[1])] == list(range(full.Hkv))
    out = np.concatenate([g[2] for g in got], axis=1)
    lse = np.concatenate([g[3] for g in got], axis=0)
    assert out.shape == ref.out.shape and np.array_equal(out, ref.out)
    assert np.array_equal(lse, ref.lse)
    # skip bits: per sequence the rows of the pieces' heads follow each other
    for s in range(full.n_seqs):
        for g in got:
            lo, hi = g[1]
            piece_Hq = (hi - lo) * G
            for hh in range(piece_Hq):
                for i in range(layout.tiles(full.seqlens[s])):
                    a = layout.row_bits(g[4], full.cu_seqlens, piece_Hq, s, hh, i)
                    b = layout.row_bits(ref.bitmap, full.cu_seqlens, full.Hq, s, lo * G + hh, i)
                    assert np.array_equal(a, b)
