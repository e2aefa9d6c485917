"""Benchmark: block-skipping causal prefill attention on one 128K-token
Llama-3-8B-shaped attention layer (Hq=32, Hkv=8, d=128, causal, bf16,
lambda=0.01), through the library's C interface.

Prints ONE JSON line. ``value`` is dense-equivalent TFLOP/s (the FLOPs of
dense causal attention on the layer divided by the measured time), inputs
resident in HBM; ``e2e`` is the same metric with host buffers copied in and
the result copied out inside the timed region; ``roofline`` compares the
forward kernel's executed tensor FLOPs (QK^T on every causal tile, P.V on
kept tiles) with the measured dense bf16 peak; ``cpu_baseline`` times the
fp64 CPU oracle on a bounded sample of the same layer.

``--impl reference`` times the CPU oracle alone (the reference arm).
Multi-GPU: one process per GPU (torchrun). By default the layer's KV heads
are split over the ranks (rank r computes KV heads [r Hkv / N, (r + 1) Hkv / N)
and their query heads from contiguous copies made before timing; strong
scaling, ``value`` = the whole layer's FLOPs over the slowest rank's time);
``--split replicas`` runs the whole layer on every rank (weak scaling). No
collective is on the data path: the ranks meet only for the barriers and the
max-over-ranks of the times.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "dense-equiv TFLOP/s and ms per 128K prefill attn layer (Llama-3-8B shape)"
TILE = 128
WORKLOADS = {
    "C2": "llama3-8b attention layer, 131072 tokens, Hq=32 Hkv=8 d=128, causal, bf16, lambda=0.01",
    "C1": "llama3-8b attention layer, 32768 tokens, Hq=32 Hkv=8 d=128, causal, bf16, lambda=0.01",
    "C3": "continuous batching, 16 sequences 4K-64K log-uniform, Hq=32 Hkv=8 d=128, causal, bf16",
    "C0": "single head, 2048 tokens, d=128, causal, bf16",
}


# ------------------------------------------------------------------ work model

def dense_flops(seqlens, Hq, d=128):
    """FLOPs of dense causal attention: 2 matmuls x 2 flop x d x L(L+1)/2 per head."""
    return sum(Hq * 4.0 * d * L * (L + 1) / 2.0 for L in seqlens)


def causal_tiles(seqlens, Hq):
    return sum(Hq * n * (n + 1) // 2 for n in ((L + TILE - 1) // TILE for L in seqlens))


def executed_flops(seqlens, Hq, skipped_tiles, d=128):
    """Tensor FLOPs the kernel issues: QK^T on every causal tile, P.V on kept ones."""
    per_tile = 2.0 * TILE * TILE * d
    ct = causal_tiles(seqlens, Hq)
    return per_tile * (ct + (ct - skipped_tiles))


def popcount(words: np.ndarray) -> int:
    return int(np.unpackbits(np.ascontiguousarray(words).view(np.uint8)).sum())


# ------------------------------------------------------------------ measured DRAM traffic

KERNEL_SOURCES = ("dynamic_block_sparse_causal_gb300/csrc/bsa_skip.cu",
                  "dynamic_block_sparse_causal_gb300/csrc/bsa_tile.cuh",
                  "dynamic_block_sparse_causal_gb300/csrc/ptx.cuh",
                  "dynamic_block_sparse_causal_gb300/csrc/bsa_internal.h")
DRAM_PROFILE = os.path.join(ROOT, "profiles", "skip_kernel_c2_dram.md")


def kernel_sources_sha256() -> str:
    import hashlib
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def measured_traffic():
    """DRAM bytes per forward launch on the 128K layer, from the committed
    single-pass ncu capture -- only if it was taken on the current kernel
    sources (otherwise None: the counters no longer describe this kernel)."""
    try:
        text = open(DRAM_PROFILE).read()
    except OSError:
        return None
    fields = {}
    for line in text.splitlines():
        if ":" in line and line.strip().startswith(("kernel_sources_sha256", "traffic_bytes_per_launch")):
            k, v = line.split(":", 1)
            fields[k.strip()] = v.strip().strip("`")
    if fields.get("kernel_sources_sha256") != kernel_sources_sha256():
        return None
    try:
        return int(fields["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# ------------------------------------------------------------------ distributed

def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), \
        int(os.environ.get("LOCAL_RANK", 0))


def max_over_ranks(x: float, world: int, device=None) -> float:
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not self.path:
            return None
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------ CPU oracle timing

def _oracle_item(args):
    """Worker: run the oracle's tile walk on one query tile of the saved layer."""
    path, Hq, Hkv, item = args
    import numpy as np  # noqa: F811
    from oracle import numerics, tile_walk
    q = np.load(os.path.join(path, "q.npy"), mmap_mode="r")
    k = np.load(os.path.join(path, "k.npy"), mmap_mode="r")
    v = np.load(os.path.join(path, "v.npy"), mmap_mode="r")
    s, h, i = item
    g = h // (Hq // Hkv)
    hi = (i + 1) * TILE                       # keys past the diagonal tile are never visited
    qs = numerics.bf16_to_f64(q[:hi, h:h + 1])
    ks = numerics.bf16_to_f64(k[:hi, g:g + 1])
    vs = numerics.bf16_to_f64(v[:hi, g:g + 1])
    t0 = time.perf_counter()
    tile_walk.walk_one(qs, ks, vs, [0, hi], 1, 1, True, 0.01, 1.0 / math.sqrt(128), (0, 0, i))
    return time.perf_counter() - t0


def _c0_walk():
    """The oracle on the whole small single-head layer (2048 tokens, every
    query tile), pinned to one core (run in a child with one BLAS thread)."""
    os.sched_setaffinity(0, {min(os.sched_getaffinity(0))})
    from gen import inputs as gi
    from oracle import numerics, tile_walk
    p = gi.config("C0")
    q, k, v = (numerics.bf16_to_f64(x) for x in (p.q, p.k, p.v))
    t0 = time.perf_counter()
    tile_walk.prefill_fwd(q, k, v, p.cu_seqlens, p.Hq, p.Hkv, lam=0.01)
    ms = (time.perf_counter() - t0) * 1e3
    return {"workload": "single head, 2048 tokens, d=128, causal, lambda=0.01 (all 16 query tiles)",
            "ms": round(ms, 2), "dense_equiv_tflops": round(dense_flops([2048], 1) / (ms * 1e-3) / 1e12, 6),
            "cores": 1}


def oracle_c0_one_core():
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    try:
        r = subprocess.run([sys.executable, "-c", "import bench, json; print(json.dumps(bench._c0_walk()))"],
                           cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
        return json.loads(r.stdout.strip().splitlines()[-1])
    except Exception as e:  # reported, not fatal
        return {"error": str(e)[:200]}


def chunk_dense_flops(lq, lk, Hq, d=128):
    """Dense causal FLOPs of lq queries at the last positions of lk keys."""
    off = lk - lq
    return Hq * 4.0 * d * (lq * (off + 1) + lq * (lq - 1) / 2.0)


def item_dense_flops(i, d=128):
    rows = np.arange(i * TILE, (i + 1) * TILE) + 1
    return 4.0 * d * float(rows.sum())


class SavedLayer:
    """The layer's bf16 arrays saved once under a temporary directory, so
    oracle worker processes can memory-map them."""

    def __init__(self, problem):
        self.problem = problem
        self.dir = tempfile.mkdtemp(prefix="bsa_oracle_")
        for name in ("q", "k", "v"):
            np.save(os.path.join(self.dir, f"{name}.npy"), getattr(problem, name))

    def close(self):
        for name in ("q", "k", "v"):
            os.unlink(os.path.join(self.dir, f"{name}.npy"))
        os.rmdir(self.dir)


def oracle_baseline(problem, budget_s: float = 12.0, cores=None, seed: int = 0, saved=None):
    """Time the oracle on a bounded, random sample of query tiles.

    Returns (dense-equivalent TFLOP/s over the sample, cores, description,
    wall seconds, number of tiles).
    """
    import multiprocessing as mp
    cores = cores or len(os.sched_getaffinity(0))
    own = saved is None
    saved = saved or SavedLayer(problem)
    tmp = saved.dir
    n = (int(problem.seqlens[0]) + TILE - 1) // TILE
    rng = np.random.default_rng(seed)
    env_keep = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
    for k in env_keep:
        os.environ[k] = "1"
    ctx = mp.get_context("spawn")
    try:
        with ctx.Pool(cores) as pool:
            # calibrate on one mid-length tile per worker
            cal = [(tmp, problem.Hq, problem.Hkv, (0, int(rng.integers(problem.Hq)), n // 2))
                   for _ in range(cores)]
            t_cal = statistics.median(pool.map(_oracle_item, cal))
            per_visit = t_cal / (n // 2 + 1)
            visits = max(cores, int(budget_s * cores / per_visit))
            items, total = [], 0
            while total < visits:
                i = int(rng.integers(n))
                items.append((tmp, problem.Hq, problem.Hkv, (0, int(rng.integers(problem.Hq)), i)))
                total += i + 1
            t0 = time.perf_counter()
            pool.map(_oracle_item, items, chunksize=1)
            wall = time.perf_counter() - t0
    finally:
        for k, val in env_keep.items():
            if val is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = val
        if own:
            saved.close()
    flops = sum(item_dense_flops(it[3][2]) for it in items)
    desc = (f"{len(items)} random query tiles (all key tiles up to the diagonal) of the layer, "
            f"{total} tile visits, {cores} worker processes x 1 thread, fp64")
    return flops / wall / 1e12, cores, desc, wall, len(items)


# ------------------------------------------------------------------ GPU helpers

def kv_bytes(bits, seqlens, Hq, Hkv, d, elem=2):
    """Algorithmic HBM bytes of the K/V stream for one launch: every K tile
    once per KV head, and every V tile that at least one query tile of the
    KV head's group keeps, once."""
    G = Hq // Hkv
    total, off = 0, 0
    for L in seqlens:
        n = (L + TILE - 1) // TILE
        W = (n + 31) // 32
        rows = np.ascontiguousarray(bits[off:off + Hq * n * W]).view(np.uint32).reshape(Hq, n, W)
        off += Hq * n * W
        skip = np.unpackbits(rows.view(np.uint8), axis=2, bitorder="little")[:, :, :n].astype(bool)
        visited = np.tril(np.ones((n, n), bool))
        kept = (~skip) & visited[None]
        v_tiles = int(kept.reshape(Hkv, G * n, n).any(axis=1).sum())
        tok_bytes = TILE * d * elem
        total += Hkv * n * tok_bytes + v_tiles * tok_bytes
    return int(total)


def fp8_peak(dev, n=8192, reps=10):
    """Dense E4M3 GEMM rate of the box's library (torch._scaled_mm, n^3,
    bf16 output, best of ``reps``), with and without fast accumulation."""
    import torch
    out = {"how": f"torch._scaled_mm e4m3 {n}^3 -> bf16, best of {reps} (CUDA events)"}
    try:
        a = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn)
        b = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn)
        one = torch.tensor(1.0, device=dev)
        for fast in (False, True):
            def mm():
                return torch._scaled_mm(a, b.t(), scale_a=one, scale_b=one, out_dtype=torch.bfloat16,
                                        use_fast_accum=fast)
            for _ in range(3):
                mm()
            best = float("inf")
            for _ in range(reps):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                mm()
                e1.record()
                torch.cuda.synchronize()
                best = min(best, e0.elapsed_time(e1))
            out["fast_accum" if fast else "tflops"] = round(2.0 * n ** 3 / (best * 1e-3) / 1e12, 1)
        out["peak"] = max(out["tflops"], out["fast_accum"])
        del a, b
    except Exception as e:  # a missing FP8 GEMM is reported, not fatal
        out["error"] = str(e)[:200]
    return out


def sdpa_backends(q, k, v, T, Hq, Hkv, d, dflops, peak, steps, stream):
    """torch SDPA (dense causal) on the same shape with each backend forced;
    K/V heads expanded to Hq outside the timed region. Returns the fastest
    backend's line and every backend's time or error."""
    import torch
    import torch.nn.functional as F
    from torch.nn.attention import SDPBackend, sdpa_kernel
    Q = q.view(1, T, Hq, d).transpose(1, 2)
    K = k.view(1, T, Hkv, d).transpose(1, 2).repeat_interleave(Hq // Hkv, dim=1)
    V = v.view(1, T, Hkv, d).transpose(1, 2).repeat_interleave(Hq // Hkv, dim=1)
    results = {}
    for name, be in (("cudnn", SDPBackend.CUDNN_ATTENTION), ("flash", SDPBackend.FLASH_ATTENTION),
                     ("efficient", SDPBackend.EFFICIENT_ATTENTION)):
        try:
            with sdpa_kernel([be]):
                o = F.scaled_dot_product_attention(Q, K, V, is_causal=True)
                torch.cuda.synchronize()
                n = max(2, steps // 4)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for _ in range(n):
                    o = F.scaled_dot_product_attention(Q, K, V, is_causal=True)
                e1.record(stream)
                torch.cuda.synchronize()
                results[name] = round(e0.elapsed_time(e1) / n, 3)
                del o
        except Exception as e:
            results[name] = "unavailable: " + str(e).splitlines()[0][:160]
    del K, V
    timed_ok = {k_: v_ for k_, v_ in results.items() if isinstance(v_, float)}
    if not timed_ok:
        return {"impl": "torch SDPA", "error": "no backend ran", "backends_ms": results}
    best = min(timed_ok, key=timed_ok.get)
    m = timed_ok[best]
    return {"impl": f"torch.nn.functional.scaled_dot_product_attention, {best} backend (is_causal, "
                    f"K/V heads expanded)", "backend": best, "ms": m,
            "dense_tflops": round(dflops / m / 1e9, 1), "frac_of_peak": round(dflops / m / 1e9 / peak, 4),
            "backends_ms": results}


# ------------------------------------------------------------------ GPU arm

def gpu_arm(args, rank, world, local_rank):
    import torch

    from dynamic_block_sparse_causal_gb300 import bsa
    from gen import inputs as gi

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    bsa.lib()
    p = gi.config(args.config, seed=args.seed, lam=args.lam, sink=args.sink)
    split = world > 1 and args.split == "heads"
    layer_Hq = p.Hq
    if split:   # this rank's KV heads and their query heads (contiguous copies)
        p = gi.split_heads(p, rank, world)
    seqlens = [int(x) for x in p.seqlens]
    T, Hq, Hkv, d = p.total_tokens, p.Hq, p.Hkv, p.d
    dflops = dense_flops(seqlens, Hq, d)
    # FLOPs of the whole job: the layer once (split), or once per rank (replicas)
    job_flops = dense_flops(seqlens, layer_Hq, d) if split else dflops * world
    stream = torch.cuda.current_stream()

    def upload(bits):
        return torch.from_numpy(bits.view(np.int16)).to(dev).view(torch.bfloat16)

    q, k, v = upload(p.q), upload(p.k), upload(p.v)
    cu = torch.from_numpy(p.cu_seqlens).to(dev)
    out = torch.empty((T, Hq, d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((Hq, T), dtype=torch.float32, device=dev)
    nw = bsa.skip_bitmap_words(p.cu_seqlens, Hq)
    bm = torch.empty((nw,), dtype=torch.int32, device=dev)

    def step(lam=args.lam):
        st = bsa.prefill_fwd(q, k, v, cu, p.n_seqs, Hq, Hkv, d, 1, lam, bsa.BSA_BF16, out, lse, bm, stream)
        if st != 0:
            raise bsa.BsaError(st, "bsa_prefill_fwd")

    def timed(nsteps, lam=args.lam):
        """(median, mean) ms per step over nsteps steps: an event before every
        step and one after the last, all on the launching stream."""
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(nsteps + 1)]
        barrier(world)
        torch.cuda.synchronize()
        for i in range(nsteps):
            evs[i].record(stream)
            step(lam)
        evs[nsteps].record(stream)
        torch.cuda.synchronize()
        barrier(world)
        per = [evs[i].elapsed_time(evs[i + 1]) for i in range(nsteps)]
        return statistics.median(per), evs[0].elapsed_time(evs[nsteps]) / nsteps

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    bsa.check(bsa.get_device_status(stream), "device status")
    with ClockSampler(local_rank) as clk:
        ms, ms_mean = timed(args.steps)
    clocks = clk.summary()
    ms = max_over_ranks(ms, world, dev)
    ms_mean = max_over_ranks(ms_mean, world, dev)
    bsa.check(bsa.get_device_status(stream), "device status")
    skipped = popcount(bm.cpu().numpy())
    ctiles = causal_tiles(seqlens, Hq)
    xflops = executed_flops(seqlens, Hq, skipped, d)
    value = job_flops / (ms * 1e-3) / 1e12

    peaks = {}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peaks = json.load(f)
    except OSError:
        pass
    peak = peaks.get("bf16_tflops", 1900.0)
    achieved = xflops / (ms * 1e-3) / 1e12
    traffic = measured_traffic() if args.config == "C2" else None
    kv = kv_bytes(bm.cpu().numpy(), seqlens, Hq, Hkv, d)
    roofline = {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                "frac": round(achieved / peak, 4), "traffic": traffic,
                "algorithmic_bytes": int(2 * (p.q.size + p.k.size + p.v.size + p.q.size) + 4 * Hq * T),
                "peak_source": "MEASURED_PEAKS.json bf16_tflops (burst), of measured"
                if "bf16_tflops" in peaks else "fallback 1900 TFLOP/s, of fallback",
                "flops_per_launch": xflops,
                "kv_hbm": {"bytes": kv, "gbs": round(kv / (ms * 1e-3) / 1e9, 2),
                           "what": "K once per KV head + V of every key tile some query tile keeps, "
                                   "once (the K/V stream's algorithmic HBM bytes)"}}
    if "bf16_tflops_sustained" in peaks and clocks and clocks.get("sm_mhz"):
        # secondary: the seconds-long cuBLAS rate, both normalised by their median SM clock
        pk = peaks.get("clocks_under_load", {}).get("sm_mhz_median")
        if pk:
            roofline["secondary_sustained"] = {
                "peak": peaks["bf16_tflops_sustained"], "peak_sm_mhz": pk, "run_sm_mhz": clocks["sm_mhz"],
                "frac_per_clock": round((achieved / clocks["sm_mhz"]) /
                                        (peaks["bf16_tflops_sustained"] / pk), 4)}

    # end to end through the C interface with host buffers: every step copies
    # its inputs in from pinned host memory and its results (out, lse, skip
    # bitmap) back out. Two device buffer sets and two host result sets let
    # step i + 1's upload and step i - 1's download run on copy streams while
    # step i computes; the timed region includes the first upload and the
    # last download. The same steps run back to back on one stream are
    # reported beside it. Measured right after the resident steps, so that
    # both run in the same state of the GPU (the other legs heat it).
    e2e = None
    if not args.no_e2e:
        hq = torch.from_numpy(p.q.view(np.int16)).pin_memory()
        hk = torch.from_numpy(p.k.view(np.int16)).pin_memory()
        hv = torch.from_numpy(p.v.view(np.int16)).pin_memory()
        hcu = torch.from_numpy(p.cu_seqlens).pin_memory()
        hres = [(torch.empty((T, Hq, d), dtype=torch.int16).pin_memory(),
                 torch.empty((Hq, T), dtype=torch.float32).pin_memory(),
                 torch.empty((nw,), dtype=torch.int32).pin_memory()) for _ in range(2)]
        dbuf = [(q, k, v, cu, out, lse, bm),
                (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v), torch.empty_like(cu),
                 torch.empty_like(out), torch.empty_like(lse), torch.empty_like(bm))]
        s_up, s_down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev = {n: [torch.cuda.Event(), torch.cuda.Event()] for n in ("up", "comp", "down")}
        used = [False, False]

        def e2e_step(i, overlap=True):
            bi = i % 2 if overlap else 0
            dq, dk, dv, dcu, dout, dlse, dbm = dbuf[bi]
            ho, hl, hb = hres[bi]
            s_in = s_up if overlap else stream
            s_out = s_down if overlap else stream
            with torch.cuda.stream(s_in):
                if used[bi]:
                    s_in.wait_event(ev["comp"][bi])       # the forward that last read this set
                dq.view(torch.int16).copy_(hq, non_blocking=True)
                dk.view(torch.int16).copy_(hk, non_blocking=True)
                dv.view(torch.int16).copy_(hv, non_blocking=True)
                dcu.copy_(hcu, non_blocking=True)
                ev["up"][bi].record(s_in)
            stream.wait_event(ev["up"][bi])
            if used[bi]:
                stream.wait_event(ev["down"][bi])         # the download that last read out / lse / bitmap
            st = bsa.prefill_fwd(dq, dk, dv, dcu, p.n_seqs, Hq, Hkv, d, 1, args.lam, bsa.BSA_BF16,
                                 dout, dlse, dbm, stream)
            if st != 0:
                raise bsa.BsaError(st, "bsa_prefill_fwd")
            ev["comp"][bi].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev["comp"][bi])
                ho.copy_(dout.view(torch.int16), non_blocking=True)
                hl.copy_(dlse, non_blocking=True)
                hb.copy_(dbm, non_blocking=True)
                ev["down"][bi].record(s_out)
            used[bi] = True

        def run_e2e(n, overlap):
            for i in range(2):
                e2e_step(i, overlap)
            torch.cuda.synchronize()
            barrier(world)
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            for i in range(n):
                e2e_step(i, overlap)
            torch.cuda.synchronize()
            barrier(world)
            return max_over_ranks((time.perf_counter() - t0) * 1e3 / n, world, dev)

        n_e2e = max(4, args.steps)   # the first upload and last download amortise over these
        ms_e2e = run_e2e(n_e2e, True)
        ms_serial = run_e2e(max(2, args.steps // 2), False)
        h2d = hq.numel() * 2 + hk.numel() * 2 + hv.numel() * 2 + hcu.numel() * 4
        d2h = hres[0][0].numel() * 2 + hres[0][1].numel() * 4 + hres[0][2].numel() * 4
        e2e = {"value": round(job_flops / (ms_e2e * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
               "ms_per_step": round(ms_e2e, 3), "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "steps": n_e2e,
               "overlap": "upload of step i+1 and download of step i-1 on copy streams during the "
                          "forward of step i (two buffer sets); first upload and last download timed",
               "serial_ms_per_step": round(ms_serial, 3),
               "serial_value": round(job_flops / (ms_serial * 1e-3) / 1e12, 2)}
        bsa.check(bsa.get_device_status(stream), "device status")
        del dbuf, hres

    # lambda sweep on the same layer (skip fraction and TFLOP/s for each lambda)
    sweep = []
    if not args.no_sweep:
        for lam in (0.0, 1e-3, 1e-2, 5e-2):
            step(lam)
            torch.cuda.synchronize()
            m, _ = timed(max(2, args.steps // 2), lam)
            sk = popcount(bm.cpu().numpy())
            sweep.append({"lambda": lam, "ms": round(m, 3), "dense_equiv_tflops": round(dflops / m / 1e9, 1),
                          "executed_tflops": round(executed_flops(seqlens, Hq, sk, d) / m / 1e9, 1),
                          "skip_fraction": round(sk / ctiles, 5)})

    # FP8 E4M3 variant of the same layer (C4): per-head quantisation by the
    # library, then the FP8 forward, against the box's measured E4M3 GEMM rate
    fp8 = None
    if not args.no_fp8:
        f8peak = fp8_peak(dev)
        codes = [torch.empty(x.shape, dtype=torch.uint8, device=dev) for x in (q, k, v)]
        scales = [torch.empty((x.shape[1],), dtype=torch.float32, device=dev) for x in (q, k, v)]
        for x, c8, sc in zip((q, k, v), codes, scales):
            bsa.check(bsa.quantize_fp8(x, T, x.shape[1], d, c8, sc, stream), "quantize_fp8")
        bsa.check(bsa.set_fp8_scales(*scales), "set_fp8_scales")

        def step8(lam=args.lam):
            st = bsa.prefill_fwd(codes[0], codes[1], codes[2], cu, p.n_seqs, Hq, Hkv, d, 1, lam,
                                 bsa.BSA_FP8_E4M3, out, lse, bm, stream)
            if st != 0:
                raise bsa.BsaError(st, "bsa_prefill_fwd fp8")
        for _ in range(3):
            step8()
        torch.cuda.synchronize()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n8 = max(2, args.steps // 2)
        ev0.record(stream)
        for _ in range(n8):
            step8()
        ev1.record(stream)
        torch.cuda.synchronize()
        m8 = ev0.elapsed_time(ev1) / n8
        sk8 = popcount(bm.cpu().numpy())
        x8 = executed_flops(seqlens, Hq, sk8, d)
        if "peak" in f8peak:
            p8, p8src = f8peak["peak"], "measured in this run: " + f8peak["how"]
        else:
            p8, p8src = 2 * peak, "measured bf16 burst x nominal FP8/bf16 ratio 2 (FP8 GEMM unavailable)"
        fp8 = {"workload": "the same layer in FP8 E4M3 (per-head absmax scales), bf16 output",
               "lambda": args.lam, "ms": round(m8, 3), "dense_equiv_tflops": round(dflops / m8 / 1e9, 1),
               "executed_tflops": round(x8 / m8 / 1e9, 1), "skip_fraction": round(sk8 / ctiles, 5),
               "roofline_frac": round(x8 / m8 / 1e9 / p8, 4), "peak": p8, "peak_source": p8src,
               "fp8_gemm": f8peak,
               "kv_hbm_gbs": round(kv_bytes(bm.cpu().numpy(), seqlens, Hq, Hkv, d, 1) / (m8 * 1e-3) / 1e9, 2)}
        bsa.check(bsa.set_fp8_scales(None, None, None), "clear scales")
        bsa.check(bsa.get_device_status(stream), "device status")
        del codes, scales

    def time_fn(fn, n):
        """Mean ms of n calls on the stream after 3 untimed ones (CUDA events)."""
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n

    # next rows: chunked prefill (the last 8192 queries against all keys) and
    # the same chunk with K/V in a shuffled pool of 128-token pages
    rows = None
    if not args.no_rows and p.n_seqs == 1:
        lq = 8192
        qc = q[T - lq:]
        cuq = torch.tensor([0, lq], dtype=torch.int32, device=dev)
        outc = torch.empty((lq, Hq, d), dtype=torch.bfloat16, device=dev)
        lsec = torch.empty((Hq, lq), dtype=torch.float32, device=dev)
        nwc = bsa.skip_bitmap_words_chunked(np.array([0, lq]), p.cu_seqlens, Hq)
        bmc = torch.empty((nwc,), dtype=torch.int32, device=dev)
        n_pages = (T + TILE - 1) // TILE
        perm = torch.from_numpy(np.random.default_rng(0).permutation(n_pages).astype(np.int32)).to(dev)
        kpool = torch.empty((n_pages * TILE, Hkv, d), dtype=torch.bfloat16, device=dev)
        vpool = torch.empty_like(kpool)
        kpool.view(n_pages, TILE, Hkv, d)[perm.long()] = k.view(n_pages, TILE, Hkv, d)
        vpool.view(n_pages, TILE, Hkv, d)[perm.long()] = v.view(n_pages, TILE, Hkv, d)
        table = perm.view(1, n_pages)
        cf = chunk_dense_flops(lq, T, Hq, d)

        def chunked():
            bsa.check(bsa.prefill_fwd_chunked(qc, k, v, cuq, cu, 1, Hq, Hkv, d, 1, args.lam,
                                              bsa.BSA_BF16, outc, lsec, bmc, stream), "chunked")

        def paged():
            bsa.check(bsa.prefill_fwd_paged(qc, kpool, vpool, table, n_pages, n_pages, cuq, cu, 1,
                                            Hq, Hkv, d, 1, args.lam, bsa.BSA_BF16, outc, lsec, bmc,
                                            stream), "paged")
        rows = {}
        for name, fn in (("chunked_prefill", chunked), ("paged_kv", paged)):
            for _ in range(3):
                fn()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(args.steps):
                fn()
            e1.record(stream)
            torch.cuda.synchronize()
            m = e0.elapsed_time(e1) / args.steps
            rows[name] = {"workload": f"last {lq} queries of the layer against all {T} keys" +
                          (", K/V in a shuffled pool of 128-token pages" if name == "paged_kv" else ""),
                          "ms": round(m, 3), "dense_equiv_tflops": round(cf / m / 1e9, 1)}
        bsa.check(bsa.get_device_status(stream), "device status")
        del kpool, vpool

        # decode (one new query per sequence, the deployment guide's decode
        # threshold 0.005) through bsa_decode_fwd, the split-KV path, on the
        # whole 128K context and on the layer cut into four 32K contexts; the
        # same call through the chunked prefill entry point for comparison
        hbm_peak = peaks.get("hbm_gbs", 6800.0)
        for name, nseq in (("decode_1_seq", 1), ("decode_4_seqs", 4)):
            cuts = [T * i // nseq for i in range(nseq + 1)]
            cuk_d = torch.tensor(cuts, dtype=torch.int32, device=dev)
            cuq_d = torch.arange(nseq + 1, dtype=torch.int32, device=dev)
            qd = torch.stack([q[c - 1] for c in cuts[1:]]).contiguous()
            outd = torch.empty((nseq, Hq, d), dtype=torch.bfloat16, device=dev)
            lsed = torch.empty((Hq, nseq), dtype=torch.float32, device=dev)
            nwd = bsa.skip_bitmap_words_chunked(np.arange(nseq + 1), np.array(cuts), Hq)
            bmd = torch.empty((nwd,), dtype=torch.int32, device=dev)

            def dec():
                bsa.check(bsa.decode_fwd(qd, k, v, cuq_d, cuk_d, nseq, 1, T, Hq, Hkv, d, 1, 0.005,
                                         outd, lsed, bmd, stream), "decode")

            def dec_prefill_kernel():
                bsa.check(bsa.prefill_fwd_chunked(qd, k, v, cuq_d, cuk_d, nseq, Hq, Hkv, d, 1, 0.005,
                                                  bsa.BSA_BF16, outd, lsed, bmd, stream), "decode")
            m_pf = time_fn(dec_prefill_kernel, args.steps)
            m = time_fn(dec, args.steps)
            bits = bmd.cpu().numpy().view(np.uint32)
            # bytes: every K tile once per KV head, V tiles that some query head kept
            ntiles = [(b - a + TILE - 1) // TILE for a, b in zip(cuts[:-1], cuts[1:])]
            v_kept = 0
            off = 0
            for sq in range(nseq):
                W, nt = (ntiles[sq] + 31) // 32, ntiles[sq]
                rowsb = bits[off:off + Hq * W].reshape(Hq, W)
                off += Hq * W
                sk = np.unpackbits(rowsb.view(np.uint8), bitorder="little").reshape(Hq, -1)[:, :nt]
                v_kept += int((sk == 0).reshape(Hkv, Hq // Hkv, nt).any(axis=1).sum())
            tile_bytes = TILE * d * 2
            nbytes = sum(ntiles) * Hkv * tile_bytes + v_kept * tile_bytes
            gbs = nbytes / (m * 1e-3) / 1e9
            rows[name] = {"workload": f"{nseq} sequence(s) x {T // nseq} keys, one new query each, "
                          f"lambda 0.005, Llama-3-8B heads", "entry": "bsa_decode_fwd",
                          "ms": round(m, 4), "ms_via_prefill_kernel": round(m_pf, 4),
                          "kv_bytes": int(nbytes), "achieved_gbs": round(gbs, 1),
                          "hbm_peak_gbs": hbm_peak, "hbm_frac": round(gbs / hbm_peak, 4),
                          "v_tiles_kept": v_kept, "k_tiles": sum(ntiles) * Hkv}
        bsa.check(bsa.get_device_status(stream), "device status")

        # UniPrefill block importance of the layer (last 64 queries, G = 128)
        # and the top-p (p = 0.9) selection over its head-mean scores
        n_win = 64
        nb = bsa.importance_blocks(p.cu_seqlens)
        sc = torch.empty((Hq, nb), dtype=torch.float32, device=dev)
        mn = torch.empty((nb,), dtype=torch.float32, device=dev)
        order = torch.empty((nb,), dtype=torch.int32, device=dev)
        nsel = torch.empty((1,), dtype=torch.int32, device=dev)
        keep = torch.empty((nb,), dtype=torch.uint8, device=dev)

        def importance():
            bsa.check(bsa.block_importance(q, k, cu, 1, Hq, Hkv, d, n_win, 1, nb, sc, mn, stream), "importance")

        def select():
            bsa.check(bsa.top_p_select(mn, cu, 1, nb, 0.9, order, nsel, keep, stream), "top_p")
        mi = time_fn(importance, args.steps)
        ms_sel = time_fn(select, args.steps)
        bsa.check(bsa.get_device_status(stream), "device status")
        # 128-row tiles issued: with a window of <= 64 rows and an even group
        # one tile carries two query heads
        pair = 2 if (n_win <= 64 and (Hq // Hkv) % 2 == 0) else 1
        mma_flops = Hq // pair * nb * 2 * TILE * TILE * d
        rows["block_importance"] = {
            "workload": f"UniPrefill Eq. 3-4 on the layer: last 64 queries, {nb} blocks of 128 keys, {Hq} heads",
            "ms": round(mi, 4), "top_p_ms": round(ms_sel, 4), "p": 0.9, "kept_blocks": int(nsel[0]),
            "mma_tflops": round(mma_flops / mi / 1e9, 1), "mma_frac": round(mma_flops / mi / 1e9 / peak, 4),
            "query_heads_per_tile": pair,
            "launches": 5}

    # diagnostic, not the headline: the 32K layer with a weak sink (0.25 u),
    # where about two thirds of the causal tiles are skipped and the kept-tile
    # path (exponentials, V loads, P.V) carries a third of the work
    diag = None
    if not args.no_rows and args.config == "C2" and args.sink == 4.0:
        pd = gi.config("C1", seed=args.seed, lam=args.lam, sink=0.25)
        sl = [int(x) for x in pd.seqlens]
        Td = pd.total_tokens
        qd, kd, vd = upload(pd.q), upload(pd.k), upload(pd.v)
        cud = torch.from_numpy(pd.cu_seqlens).to(dev)
        outd = torch.empty((Td, Hq, d), dtype=torch.bfloat16, device=dev)
        lsed = torch.empty((Hq, Td), dtype=torch.float32, device=dev)
        bmd = torch.empty((bsa.skip_bitmap_words(pd.cu_seqlens, Hq),), dtype=torch.int32, device=dev)

        def diag_step():
            bsa.check(bsa.prefill_fwd(qd, kd, vd, cud, pd.n_seqs, Hq, Hkv, d, 1, args.lam, bsa.BSA_BF16,
                                      outd, lsed, bmd, stream), "bsa_prefill_fwd (diagnostic)")
        md = time_fn(diag_step, max(args.steps, 10))
        bsa.check(bsa.get_device_status(stream), "device status")
        skd = popcount(bmd.cpu().numpy())
        xd = executed_flops(sl, Hq, skd, d)
        diag = {"workload": "32K layer (Llama-3-8B heads), sink 0.25 u instead of 4 u", "lambda": args.lam,
                "ms": round(md, 3), "skip_fraction": round(skd / causal_tiles(sl, Hq), 5),
                "dense_equiv_tflops": round(dense_flops(sl, Hq, d) / md / 1e9, 1),
                "executed_tflops": round(xd / md / 1e9, 1), "roofline_frac": round(xd / md / 1e9 / peak, 4)}
        del qd, kd, vd, outd, lsed, bmd

    # dense causal attention from the box's library (torch SDPA, every
    # backend forced in turn) on the same shape: the comparison for the
    # lambda = 0 path
    dense_ref = None
    if not args.no_sweep and p.n_seqs == 1:
        dense_ref = sdpa_backends(q, k, v, T, Hq, Hkv, d, dflops, peak, args.steps, stream)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tf, cores, desc, wall, nitems = oracle_baseline(p, budget_s=args.cpu_budget)
        cpu = {"value": round(tf, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": desc,
               "wall_s": round(wall, 2), "extrapolated": True,
               "extrapolation": "throughput of the sampled query tiles stands for the whole layer",
               "c0_1core": oracle_c0_one_core()}

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
        "ms_per_step_mean": round(ms_mean, 3), "timing": "median of per-step CUDA-event times",
        "higher_is_better": True, "scaling": "strong" if split else "weak", "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded generator: sink + local-window bias, Llama-3-8B attention shape)",
        "config": {"workload": WORKLOADS.get(args.config, args.config), "name": args.config,
                   "tokens": T, "Hq": Hq, "Hkv": Hkv, "d": d, "lambda": args.lam, "causal": True,
                   "sink": args.sink,
                   "parallelism": (f"kv-head split x{world} (this rank: {Hkv} KV heads, {Hq} query heads)"
                                   if split else f"replicas x{world}"),
                   "l2": "inputs larger than L2 (q/out 1.07 GB each, k/v 0.27 GB each); no flush"},
        "skip_fraction": round(skipped / ctiles, 5), "executed_tflop_per_step": round(xflops / 1e12, 3),
        "dense_equiv_tflop_per_step": round(dflops / 1e12, 3),
        "roofline": roofline, "e2e": e2e, "cpu_baseline": cpu, "clocks": clocks,
        "gpu_launches": 2 * args.steps, "lambda_sweep": sweep, "dense_reference": dense_ref,
        "fp8": fp8, "next_rows": rows, "diagnostic_weak_sink": diag,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def reference_arm(args, rank, world):
    """The CPU oracle, as it stands, on a bounded sample of the same layer."""
    if rank != 0:
        return
    from gen import inputs as gi
    p = gi.config(args.config, seed=args.seed, lam=args.lam, sink=args.sink)
    vals = []
    saved = SavedLayer(p)
    try:
        for w in range(args.warmup):
            oracle_baseline(p, budget_s=2.0, saved=saved, seed=1000 + w)
        for k in range(args.steps):
            tf, cores, desc, wall, nitems = oracle_baseline(p, budget_s=args.ref_budget, saved=saved,
                                                            seed=k)
            vals.append((tf, wall))
    finally:
        saved.close()
    tf = statistics.median(v[0] for v in vals)
    dflops = dense_flops([int(x) for x in p.seqlens], p.Hq, p.d)
    ms = dflops / (tf * 1e12) * 1e3
    line = {
        "impl": "reference", "metric": METRIC, "value": round(tf, 6), "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded generator)",
        "config": {"workload": WORKLOADS.get(args.config, args.config), "name": args.config,
                   "lambda": args.lam, "causal": True},
        "cpu_baseline": {"value": round(tf, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": desc + "; ms_per_step extrapolated to the whole layer"},
        "e2e": {"value": round(tf, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gpu", choices=["gpu", "reference"])
    ap.add_argument("--config", default="C2", choices=sorted(WORKLOADS))
    ap.add_argument("--lam", type=float, default=0.01)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--sink", type=float, default=4.0,
                    help="sink strength of the input recipe (4.0; smaller keeps more tiles)")
    ap.add_argument("--split", default="heads", choices=["heads", "replicas"],
                    help="with several GPUs: split the layer's KV heads over the ranks (default) "
                         "or run the whole layer on every rank")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-fp8", action="store_true")
    ap.add_argument("--no-rows", action="store_true", help="skip the chunked / paged legs")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work")
    ap.add_argument("--ref-budget", type=float, default=8.0, help="seconds per reference step")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "gpu":
        ap.error("--warmup must be >= 3")
    rank, world, local_rank = dist_env()
    if args.impl == "reference":
        reference_arm(args, rank, world)
    else:
        gpu_arm(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
