// Split-KV decode with the block-skipping rule, on sm_103a.
//
// Operation: dynamic sparse attention deployment guide
// ("长上下文推理加速方案部署实战：基于动态稀疏注意力机制的推理服务优化指南"),
// §3.2 and §6.1: the same per-block rule as the prefill (a key tile is skipped
// when tile_max < running_max + ln(lambda) for every query row), which the
// guide also applies in decoding (a few new queries per sequence against a
// long key range; §6.1 suggests lambda = 0.005 there).
//
// Splitting the key range needs the order rule restated. A skipped tile never
// raises the running max (tile_max < m + ln(lambda) < m for lambda < 1), so the
// running max before tile j is the prefix max of the tile maxima before j, and
// every decision depends on the tile maxima alone. The path therefore:
//  1. dec_scores_kernel: for every (sequence, KV head, 16-tile split), the
//     scaled scores S (log2 units) of the group's query rows against each key
//     tile (TMA-staged, 3-stage ring) and their per-tile row maxima;
//  2. dec_decide_kernel: per (sequence, KV head), a block-wide prefix-max scan
//     over the tiles gives each tile's decision per query head (the AND over
//     that head's rows) and the skip-bitmap words;
//  3. dec_pv_kernel: per split, the kept tiles' V (TMA, only kept tiles) and
//     an online softmax with the split's own reference max;
//  4. dec_combine_kernel: merges the splits' (max, sum, output) per row.
// The decisions are exactly those of the sequential walk; outputs equal the
// online softmax over the kept tiles up to rounding order. The work is
// bandwidth-bound (K once, kept V once), so the dot products run on the
// CUDA cores: one query row group of at most 32 rows per KV head.
#include <cuda_bf16.h>

#include <climits>
#include <cmath>

#include "bsa_decode.h"
#include "ptx.cuh"

namespace bsa {

namespace {

constexpr uint32_t kTileBytes = 32768;   // 128 keys x 128 bf16
constexpr uint32_t kBoxBytes = 16384;    // one 128-row x 128-byte TMA box
constexpr int kStages = 3;
constexpr float kLn2 = 0.6931471805599453f;

struct DecItem {
  int s, kvh, j0, j1, aq, Lq, ak, Lk;
};

__device__ __forceinline__ void decode_item(const DecParams &p, int item, DecItem &it) {
  int lo = 0, hi = p.n_seqs;   // largest s with item_off[s] <= item
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (p.item_off[mid] <= item) lo = mid; else hi = mid;
  }
  it.s = lo;
  it.aq = p.cu_q[lo];
  it.Lq = p.cu_q[lo + 1] - it.aq;
  it.ak = p.cu_k[lo];
  it.Lk = p.cu_k[lo + 1] - it.ak;
  const int nk = (it.Lk + kTile - 1) / kTile;
  const int ns = (nk + kDecSplit - 1) / kDecSplit;
  // the KV heads of one split are neighbours: CTAs running together read
  // whole token rows of K and V (all heads) from DRAM
  const int local = item - p.item_off[lo];
  const int split = local / p.Hkv;
  it.kvh = local - split * p.Hkv;
  it.j0 = split * kDecSplit;
  it.j1 = min(nk, it.j0 + kDecSplit);
  (void)ns;
}

// Byte offset of 16-byte chunk c (0..15) of row r in a 128-byte-swizzled tile.
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return (uint32_t)((c >> 3) * kBoxBytes + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

__device__ __forceinline__ void load_tile(uint8_t *dst, const CUtensorMap *map, uint64_t *bar,
                                          int head, int row) {
  mbar_expect_tx(bar, kTileBytes);
  tma_load_3d(dst, map, bar, 0, head, row);
  tma_load_3d(dst + kBoxBytes, map, bar, 64, head, row);
}

__device__ __forceinline__ float2 bf2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

}  // namespace

// ============================================================ prologue

__global__ void __launch_bounds__(1024) dec_prologue_kernel(const __grid_constant__ DecParams p) {
  __shared__ int s_bad;
  const int tid = threadIdx.x;
  if (tid == 0)
    s_bad = p.cu_q[0] != 0 || p.cu_k[0] != 0 || (int64_t)p.cu_k[p.n_seqs] != p.total_k;
  __syncthreads();
  for (int s = tid; s < p.n_seqs; s += blockDim.x) {
    const int Lq = p.cu_q[s + 1] - p.cu_q[s], Lk = p.cu_k[s + 1] - p.cu_k[s];
    if (Lq < 0 || Lk < 0 || Lq > p.max_q || (p.causal && Lk < Lq) || (Lq > 0 && Lk == 0))
      atomicOr(&s_bad, 1);
  }
  __syncthreads();
  if (tid == 0) {
    bool bad = s_bad != 0;
    long long tiles = 0, items = 0, words = 0;
    int64_t *tile_off = const_cast<int64_t *>(p.tile_off);
    int64_t *bm_off = const_cast<int64_t *>(p.bm_off);
    int32_t *item_off = const_cast<int32_t *>(p.item_off);
    for (int s = 0; s < p.n_seqs && !bad; ++s) {
      const int Lq = p.cu_q[s + 1] - p.cu_q[s], Lk = p.cu_k[s + 1] - p.cu_k[s];
      const long long nk = (Lk + kTile - 1) / kTile, nq = (Lq + kTile - 1) / kTile;
      tile_off[s] = tiles;
      item_off[s] = (int32_t)min(items, (long long)INT_MAX);
      bm_off[s] = words;
      tiles += nk;
      if (Lq > 0) items += (long long)p.Hkv * ((nk + kDecSplit - 1) / kDecSplit);
      words += (long long)p.Hq * nq * ((nk + 31) / 32);
    }
    tile_off[p.n_seqs] = tiles;
    item_off[p.n_seqs] = (int32_t)min(items, (long long)INT_MAX);
    bm_off[p.n_seqs] = words;
    if (items > INT_MAX) bad = true;
    p.dw->total_items = bad ? 0 : (int32_t)items;
    if (bad) atomicOr(&p.ws->status, kStatusBadSeqlens);
  }
}

// ============================================================ 1: scores

// 32 lanes x 16 consecutive 32-bit TMEM columns; the wait is tied to the
// destination registers.
#define BSA_R8(i) "=r"(v[i]), "=r"(v[i + 1]), "=r"(v[i + 2]), "=r"(v[i + 3]), \
                  "=r"(v[i + 4]), "=r"(v[i + 5]), "=r"(v[i + 6]), "=r"(v[i + 7])
#define BSA_W8(i) "+r"(v[i]), "+r"(v[i + 1]), "+r"(v[i + 2]), "+r"(v[i + 3]), \
                  "+r"(v[i + 4]), "+r"(v[i + 5]), "+r"(v[i + 6]), "+r"(v[i + 7])
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : BSA_R8(0), BSA_R8(8)
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld16(uint32_t (&v)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" : BSA_W8(0), BSA_W8(8) : : "memory");
}
#undef BSA_R8
#undef BSA_W8

// S^T = K Q^T on the tensor cores: M = 128 keys, N = the group's query rows
// padded to 16 or 32, K = head dim. The contraction is tiny (the pass is
// bound by reading K from DRAM) but it takes the dot products off the CUDA
// cores and out of shared memory, whose bandwidth bounded the FMA version.
//   warps 0-3  epilogue: TMEM lane = key; scales, masks and stores S, row maxima
//   warp 4     lane 0: TMA producer of the K ring (all items of this CTA)
//   warp 5     TMEM allocation; lane 0 issues the MMAs
// The query rows of an item are written by the epilogue warps into one of two
// 128-byte-swizzled K-major buffers (the MMA's B operand).
template <int N>
__global__ void __launch_bounds__(kDecScoreThreads + 64, 2)
dec_scores_kernel(const __grid_constant__ DecParams p, const __grid_constant__ CUtensorMap tk) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ float red[2][kDecScoreThreads / 32][kDecMaxRows];
  __shared__ uint64_t kfull[kStages], kempty[kStages], sfull[2], sempty[2], qready[2], qfree[2],
      drain;
  __shared__ uint32_t tmem_sh;
  __shared__ volatile int abort_sh;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t *ring = smem_raw + (sbase - raw);
  uint8_t *qbuf = ring + kStages * kTileBytes;   // two N x 256-byte buffers
  constexpr uint32_t kQBytes = N * 256;
  constexpr uint32_t kIdesc = IDesc<1, false, 128, N>::value;
  constexpr int kEpi = kDecScoreThreads;
  if (t == 0) {
    for (int b = 0; b < kStages; ++b) {
      mbar_init(&kfull[b], 1);
      mbar_init(&kempty[b], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sfull[b], 1);
      mbar_init(&sempty[b], kEpi / 32);
      mbar_init(&qready[b], 1);
      mbar_init(&qfree[b], 1);
    }
    mbar_init(&drain, 1);
    fence_mbar_init();
    abort_sh = 0;
  }
  if (warp == 5) {
    tmem_alloc(&tmem_sh, 2 * N < 32 ? 32 : 2 * N);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_sh;
  const int total = p.dw->total_items;
  const uint64_t limit = p.wait_limit_ns;

  if (warp == 4) {
    // ---------------------------------------------------- TMA producer
    if (lane == 0) {
      uint32_t kc = 0;
      int last_issue[kStages] = {-1, -1, -1};
      bool ok = true;
      for (int item = blockIdx.x; item < total && ok && !abort_sh; item += gridDim.x) {
        DecItem it;
        decode_item(p, item, it);
        for (int j = it.j0; j < it.j1; ++j, ++kc) {
          const uint32_t b = kc % kStages;
          if (!(ok = mbar_wait(&kempty[b], ((kc / kStages) & 1) ^ 1, limit))) break;
          load_tile(ring + b * kTileBytes, &tk, &kfull[b], it.kvh, it.ak + j * kTile);
          last_issue[b] = (int)kc;
        }
      }
      if (!ok) abort_sh = 1;
      if (abort_sh)   // bounded wait for the copies still in flight
        for (int b = 0; b < kStages; ++b)
          if (last_issue[b] >= 0) mbar_wait(&kfull[b], (last_issue[b] / kStages) & 1, limit);
    }
  } else if (warp == 5) {
    // ---------------------------------------------------- MMA issuer
    if (lane == 0) {
      uint32_t kc = 0, sc = 0, i = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < total && ok && !abort_sh; item += gridDim.x, ++i) {
        DecItem it;
        decode_item(p, item, it);
        const uint32_t par = i & 1;
        if (!(ok = mbar_wait(&qready[par], (i >> 1) & 1, limit))) break;
        const uint32_t qs = sbase + kStages * kTileBytes + par * kQBytes;
        for (int j = it.j0; j < it.j1; ++j, ++kc, ++sc) {
          const uint32_t b = kc % kStages, buf = sc & 1;
          if (!(ok = mbar_wait(&kfull[b], (kc / kStages) & 1, limit))) break;
          if (!(ok = mbar_wait(&sempty[buf], ((sc >> 1) & 1) ^ 1, limit))) break;
          tc_fence_after();
          const uint32_t ks = sbase + b * kTileBytes;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t ka = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
            const uint32_t kb = (kk >> 2) * (N * 128) + (kk & 3) * 32;
            mma_f16_ss(tmem + buf * N, sdesc_sw128(ks + ka, 16, 1024), sdesc_sw128(qs + kb, 16, 1024),
                       kIdesc, kk > 0);
          }
          mma_commit(&sfull[buf]);
          mma_commit(&kempty[b]);
        }
        if (!ok) break;
        mma_commit(&qfree[par]);
      }
      if (!ok) abort_sh = 1;
      if (abort_sh) {   // this thread's MMAs finish before TMEM is freed
        mma_commit(&drain);
        mbar_wait(&drain, 0, limit);
      }
    }
  } else {
    // ---------------------------------------------------- epilogue
    const __nv_bfloat16 *q = static_cast<const __nv_bfloat16 *>(p.q);
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    uint32_t sc = 0, i = 0;
    for (int item = blockIdx.x; item < total; item += gridDim.x, ++i) {
      DecItem it;
      decode_item(p, item, it);
      const int R = p.group * it.Lq;
      const uint32_t par = i & 1;
      // B operand: query row r at 128-byte-swizzled K-major position
      // control flow below follows barrier reductions only, so the four
      // warps always agree (abort_sh is also written by the other roles)
      bool ok = i < 2 || mbar_wait(&qfree[par], ((i >> 1) - 1) & 1, limit);
      if (bar_red_or(!ok, 1, kEpi)) {
        abort_sh = 1;
        break;
      }
      bool stop = false;
      uint8_t *qb = qbuf + par * kQBytes;
      for (int c = t; c < N * 16; c += kEpi) {
        const int r = c >> 4, ch = c & 15;
        uint4 w = make_uint4(0u, 0u, 0u, 0u);
        if (r < R) {
          const int h = it.kvh * p.group + r / it.Lq, qi = r % it.Lq;
          w = *reinterpret_cast<const uint4 *>(q + ((size_t)(it.aq + qi) * p.Hq + h) * kTile + ch * 8);
        }
        *reinterpret_cast<uint4 *>(qb + (ch >> 3) * (N * 128) + r * 128 + (((ch & 7) ^ (r & 7)) << 4)) = w;
      }
      fence_proxy_async_smem();
      named_bar_sync(1, kEpi);
      if (t == 0) mbar_arrive(&qready[par]);
      const int64_t toff = p.tile_off[it.s];
      for (int j = it.j0; j < it.j1; ++j, ++sc) {
        const uint32_t buf = sc & 1;
        ok = mbar_wait(&sfull[buf], (sc >> 1) & 1, limit);
        if (bar_red_or(!ok, 1, kEpi)) {
          abort_sh = 1;
          stop = true;
          break;
        }
        tc_fence_after();
        uint32_t v[N];
        tmem_ld16(tmem + lane_off + buf * N, *reinterpret_cast<uint32_t(*)[16]>(&v[0]));
        if (N > 16) tmem_ld16(tmem + lane_off + buf * N + 16, *reinterpret_cast<uint32_t(*)[16]>(&v[N > 16 ? 16 : 0]));
        tmem_wait_ld16(*reinterpret_cast<uint32_t(*)[16]>(&v[0]));
        if (N > 16) tmem_wait_ld16(*reinterpret_cast<uint32_t(*)[16]>(&v[N > 16 ? 16 : 0]));
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sempty[buf]);
        const int kpos = j * kTile + t;
        const int64_t srow = ((toff + j) * p.Hkv + it.kvh) * p.rows;
        const int u = j - it.j0;
#pragma unroll
        for (int r = 0; r < N; ++r) {
          if (r < R) {
            const int pos = it.Lk - it.Lq + r % it.Lq;   // this query's key position
            const bool masked = kpos >= it.Lk || (p.causal && kpos > pos);
            const float s2 = masked ? -INFINITY : __uint_as_float(v[r]) * p.c;
            p.S[(srow + r) * kTile + t] = s2;
            float m = s2;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
            if (lane == 0) red[u & 1][warp][r] = m;
          }
        }
        named_bar_sync(1, kEpi);   // red[u & 1] complete
        if (t < R) {
          const float m = fmaxf(fmaxf(red[u & 1][0][t], red[u & 1][1][t]),
                                fmaxf(red[u & 1][2][t], red[u & 1][3][t]));
          p.rm[(it.kvh * p.max_tiles + toff + j) * p.rows + t] = m;
        }
      }
      if (stop) break;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (abort_sh && t == 0) atomicOr(&p.ws->status, kStatusTimeout);
  if (warp == 5) tmem_dealloc(tmem, 2 * N < 32 ? 32 : 2 * N);
}

// ============================================================ 2: decisions

// One CTA per (sequence, KV head); thread = key tile within a chunk of 1024.
__global__ void __launch_bounds__(1024) dec_decide_kernel(const __grid_constant__ DecParams p) {
  __shared__ float carry[kDecMaxRows];
  __shared__ float wtot[32], wscan[32];
  if (p.dw->total_items == 0) return;
  const int s = blockIdx.x / p.Hkv, kvh = blockIdx.x - s * p.Hkv;
  const int Lq = p.cu_q[s + 1] - p.cu_q[s], Lk = p.cu_k[s + 1] - p.cu_k[s];
  if (Lq == 0) return;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int R = p.group * Lq, nk = (Lk + kTile - 1) / kTile, W = (nk + 31) / 32;
  const int64_t toff = p.tile_off[s];
  if (tid < R) carry[tid] = -INFINITY;
  __syncthreads();
  for (int base = 0; base < nk; base += 1024) {
    const int j = base + tid;
    const bool in = j < nk;
    uint32_t skipb = (1u << p.group) - 1u;   // bit g: query head g of the group skips tile j
    float xs[kDecMaxRows];
    const float *rmj = p.rm + ((int64_t)kvh * p.max_tiles + toff + j) * p.rows;
#pragma unroll
    for (int r = 0; r < kDecMaxRows; ++r) xs[r] = (in && r < R) ? rmj[r] : -INFINITY;
#pragma unroll
    for (int r = 0; r < kDecMaxRows; ++r) {
      if (r >= R) break;
      const float x = xs[r];
      float v = x;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v = fmaxf(v, y);
      }
      if (lane == 31) wtot[warp] = v;
      __syncthreads();
      if (warp == 0) {
        float w = wtot[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float y = __shfl_up_sync(0xffffffffu, w, o);
          if (lane >= o) w = fmaxf(w, y);
        }
        wscan[lane] = w;
      }
      __syncthreads();
      float prev = __shfl_up_sync(0xffffffffu, v, 1);
      if (lane == 0) prev = -INFINITY;
      const float before = fmaxf(carry[r], fmaxf(warp > 0 ? wscan[warp - 1] : -INFINITY, prev));
      // running max before tile j is the prefix max of the earlier tile maxima
      if (!(x < before + p.log2_lambda)) skipb &= ~(1u << (r / Lq));
      const float total = wscan[31];
      __syncthreads();
      if (tid == 0) carry[r] = fmaxf(carry[r], total);
    }
    if (in)
      for (int g = 0; g < p.group; ++g)
        p.skip[(toff + j) * p.Hq + kvh * p.group + g] = (uint8_t)((skipb >> g) & 1u);
    if (p.bitmap) {
      for (int g = 0; g < p.group; ++g) {
        const uint32_t word = __ballot_sync(0xffffffffu, in && ((skipb >> g) & 1u));
        const int w = (base >> 5) + warp;
        if (lane == 0 && w < W)
          p.bitmap[p.bm_off[s] + (int64_t)(kvh * p.group + g) * W + w] = word;
      }
    }
    __syncthreads();
  }
}

// ============================================================ 3: P V per split

// Warps 0-7 (consumers). P: thread t computes key t%128 of the rows r with
// r%2 == t/128. O: thread t accumulates columns 2(t%64), 2(t%64)+1 over keys
// 32(t/64) .. +31, from its slice of the V tile copied to registers (which
// frees the stage at once); the four key quarters are added at the end of
// the split. Warp 8: the producer, which finds the kept tiles of each split
// with one ballot and keeps the V ring full across work items.
// RB >= group x Lq rows.
template <int RB>
__global__ void __launch_bounds__(kDecThreads + 32, RB <= 8 ? 2 : 1)
dec_pv_kernel(const __grid_constant__ DecParams p, const __grid_constant__ CUtensorMap tv) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ float lred[kDecThreads / 32][RB];
  __shared__ uint64_t full[kStages], empty[kStages];
  __shared__ int klist[kDecSplit];
  __shared__ uint32_t kact[kDecSplit], kact_raw[kDecSplit];
  __shared__ int nkept_sh;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t *ring = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  float(*ps)[kTile] = reinterpret_cast<float(*)[kTile]>(ring + kStages * kTileBytes);
  if (t == 0) {
    for (int b = 0; b < kStages; ++b) {
      mbar_init(&full[b], 1);
      mbar_init(&empty[b], kDecThreads / 32);
    }
    fence_mbar_init();
  }
  __syncthreads();
  const int total = p.dw->total_items;
  const uint64_t limit = p.wait_limit_ns;
  bool abort = false;

  if (warp == kDecThreads / 32) {
    // ---------------------------------------------------- V producer
    uint32_t vc = 0;
    int last_issue[kStages] = {-1, -1, -1};
    for (int item = blockIdx.x; item < total && !abort; item += gridDim.x) {
      DecItem it;
      decode_item(p, item, it);
      const int64_t toff = p.tile_off[it.s];
      bool kept_l = false;   // lane l: tile j0 + l kept by some head of the group
      if (lane < it.j1 - it.j0)
        for (int g = 0; g < p.group; ++g)
          kept_l |= !p.skip[(toff + it.j0 + lane) * p.Hq + it.kvh * p.group + g];
      uint32_t kept = __ballot_sync(0xffffffffu, kept_l);
      if (lane == 0) {
        while (kept) {
          const int l = __ffs(kept) - 1;
          kept &= kept - 1;
          const uint32_t b = vc % kStages;
          if (!mbar_wait(&empty[b], ((vc / kStages) & 1) ^ 1, limit)) {
            abort = true;
            break;
          }
          load_tile(ring + b * kTileBytes, &tv, &full[b], it.kvh, it.ak + (it.j0 + l) * kTile);
          last_issue[b] = (int)vc++;
        }
      }
      abort = __shfl_sync(0xffffffffu, abort, 0);
    }
    if (abort && lane == 0)
      for (int b = 0; b < kStages; ++b)
        if (last_issue[b] >= 0) mbar_wait(&full[b], (last_issue[b] / kStages) & 1, limit);
  } else {
    // ---------------------------------------------------- consumers
    const int cp = t & 63, kq = t >> 6, pk = t & (kTile - 1), prow = t >> 7;
    const int col = 2 * cp;
    uint32_t vc = 0;
    for (int item = blockIdx.x; item < total && !abort; item += gridDim.x) {
      DecItem it;
      decode_item(p, item, it);
      const int R = p.group * it.Lq;
      const int64_t toff = p.tile_off[it.s];
      named_bar_sync(1, kDecThreads);   // the previous item is done with klist and ps
      if (t < kDecSplit) kact_raw[t] = 0;
      named_bar_sync(1, kDecThreads);
      {
        const int u = t / p.group, g = t - u * p.group;
        if (u < it.j1 - it.j0 && !p.skip[(toff + it.j0 + u) * p.Hq + it.kvh * p.group + g])
          atomicOr(&kact_raw[u], 1u << g);
      }
      named_bar_sync(1, kDecThreads);
      if (t == 0) {
        int n = 0;
        for (int u = 0; u < it.j1 - it.j0; ++u)
          if (kact_raw[u]) {
            klist[n] = it.j0 + u;
            kact[n] = kact_raw[u];
            ++n;
          }
        nkept_sh = n;
      }
      named_bar_sync(1, kDecThreads);
      const int n = nkept_sh;
      float O[RB][2], mref[RB], lsum[RB];
#pragma unroll
      for (int r = 0; r < RB; ++r) {
        O[r][0] = O[r][1] = 0.f;
        mref[r] = -INFINITY;
        lsum[r] = 0.f;
      }
      for (int u = 0; u < n; ++u, ++vc) {
        const int j = klist[u];
        const uint32_t act = kact[u];
        const int64_t srow = ((toff + j) * p.Hkv + it.kvh) * p.rows;
        const float *rmj = p.rm + ((int64_t)it.kvh * p.max_tiles + toff + j) * p.rows;
        float alpha[RB];
#pragma unroll
        for (int r = 0; r < RB; ++r) {
          alpha[r] = 1.f;
          if (r < R) {
            const bool on = (act >> (r / it.Lq)) & 1u;
            const float mnew = on ? fmaxf(mref[r], rmj[r]) : mref[r];
            alpha[r] = mnew == -INFINITY ? 1.f : ex2_approx(mref[r] - mnew);
            mref[r] = mnew;
            if ((r & 1) == prow) {
              const float pv =
                  (on && mnew != -INFINITY) ? ex2_approx(p.S[(srow + r) * kTile + pk] - mnew) : 0.f;
              ps[r][pk] = pv;
              lsum[r] = lsum[r] * alpha[r] + pv;
            }
          }
        }
        const uint32_t b = vc % kStages;
        const bool ok = mbar_wait(&full[b], (vc / kStages) & 1, limit);
        if (bar_red_or(!ok, 1, kDecThreads)) {   // also publishes ps
          abort = true;
          break;
        }
        const uint8_t *vt = ring + b * kTileBytes;
        uint32_t vr[32];
#pragma unroll
        for (int e = 0; e < 32; ++e)
          vr[e] = *reinterpret_cast<const uint32_t *>(vt + swz(kq * 32 + e, col >> 3) + (col & 7) * 2);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[b]);
#pragma unroll
        for (int r = 0; r < RB; ++r) {
          O[r][0] *= alpha[r];
          O[r][1] *= alpha[r];
        }
#pragma unroll
        for (int k4 = 0; k4 < 8; ++k4) {
          const float2 v0 = bf2(vr[4 * k4]), v1 = bf2(vr[4 * k4 + 1]);
          const float2 v2 = bf2(vr[4 * k4 + 2]), v3 = bf2(vr[4 * k4 + 3]);
#pragma unroll
          for (int r = 0; r < RB; ++r) {
            if (r < R) {
              const float4 pr = *reinterpret_cast<const float4 *>(&ps[r][kq * 32 + 4 * k4]);
              O[r][0] = fmaf(pr.x, v0.x, fmaf(pr.y, v1.x, fmaf(pr.z, v2.x, fmaf(pr.w, v3.x, O[r][0]))));
              O[r][1] = fmaf(pr.x, v0.y, fmaf(pr.y, v1.y, fmaf(pr.z, v2.y, fmaf(pr.w, v3.y, O[r][1]))));
            }
          }
        }
        named_bar_sync(1, kDecThreads);   // ps is free again
      }
      if (abort) break;
      // the four key quarters of O meet in ps; the row sums in lred
      for (int qq = 3; qq >= 0; --qq) {
        if (kq == qq)
#pragma unroll
          for (int r = 0; r < RB; ++r)
            if (r < R) {
              const float a0 = qq == 3 ? 0.f : ps[r][col], a1 = qq == 3 ? 0.f : ps[r][col + 1];
              ps[r][col] = a0 + O[r][0];
              ps[r][col + 1] = a1 + O[r][1];
            }
        named_bar_sync(1, kDecThreads);
      }
#pragma unroll
      for (int r = 0; r < RB; ++r) {
        float x = lsum[r];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
        if (lane == 0) lred[warp][r] = x;
      }
      named_bar_sync(1, kDecThreads);
      const int64_t prow_off = (int64_t)item * p.rows;
      for (int i = t; i < R * kTile; i += kDecThreads)
        p.pO[prow_off * kTile + i] = ps[i >> 7][i & (kTile - 1)];
      if (t < R) {
        float l = 0.f;
#pragma unroll
        for (int w = 0; w < kDecThreads / 32; ++w) l += lred[w][t];
        p.pl[prow_off + t] = l;
#pragma unroll
        for (int r = 0; r < RB; ++r)
          if (r == t) p.pm[prow_off + t] = mref[r];
      }
    }
  }
  __syncthreads();
  if (abort && (t == 0 || t == kDecThreads)) atomicOr(&p.ws->status, kStatusTimeout);
}

// ============================================================ 4: merge

// One CTA per (sequence, query slot, query head); thread t = column t%128 of
// the splits i with i%4 == t/128, the four groups added at the end.
__global__ void __launch_bounds__(4 * kTile) dec_combine_kernel(const __grid_constant__ DecParams p) {
  __shared__ float red[4 * kTile / 32];
  __shared__ float part[3][kTile], lpart[4];
  if (p.dw->total_items == 0) return;
  const int per_seq = p.max_q * p.Hq;
  const int s = blockIdx.x / per_seq, rem = blockIdx.x - s * per_seq;
  const int qi = rem / p.Hq, h = rem - qi * p.Hq;
  const int aq = p.cu_q[s], Lq = p.cu_q[s + 1] - aq;
  if (qi >= Lq) return;
  const int t = threadIdx.x, c = t & (kTile - 1), grp = t >> 7, lane = t & 31, warp = t >> 5;
  const int Lk = p.cu_k[s + 1] - p.cu_k[s];
  const int nk = (Lk + kTile - 1) / kTile, ns = (nk + kDecSplit - 1) / kDecSplit;
  const int kvh = h / p.group, r = (h - kvh * p.group) * Lq + qi;
  const int64_t it0 = (int64_t)p.item_off[s] + kvh;   // split i is item it0 + i * Hkv
  const int64_t H = p.Hkv;
  float m = -INFINITY;
  for (int i = t; i < ns; i += 4 * kTile) m = fmaxf(m, p.pm[(it0 + i * H) * p.rows + r]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) red[warp] = m;
  __syncthreads();
  m = red[0];
#pragma unroll
  for (int w = 1; w < 4 * kTile / 32; ++w) m = fmaxf(m, red[w]);
  float acc = 0.f, l = 0.f;
#pragma unroll 4
  for (int i = grp; i < ns; i += 4) {
    const int64_t ii = it0 + i * H;
    const float mi = p.pm[ii * p.rows + r];
    if (mi == -INFINITY) continue;   // no kept tile of this split for the row
    const float w = ex2_approx(mi - m);
    l = fmaf(p.pl[ii * p.rows + r], w, l);
    acc = fmaf(p.pO[(ii * p.rows + r) * kTile + c], w, acc);
  }
  if (grp > 0) part[grp - 1][c] = acc;
  if (c == 0) lpart[grp] = l;
  __syncthreads();
  if (grp == 0) {
    acc += (part[0][c] + part[1][c]) + part[2][c];
    l = (lpart[0] + lpart[1]) + (lpart[2] + lpart[3]);
    const float inv = l > 0.f ? 1.f / l : 0.f;
    __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(p.out);
    out[((size_t)(aq + qi) * p.Hq + h) * kTile + c] = __float2bfloat16_rn(acc * inv);
    if (p.lse && t == 0) p.lse[(size_t)h * p.cu_q[p.n_seqs] + aq + qi] = (m + log2f(l)) * kLn2;
  }
}

// ============================================================ launchers

namespace {
// K / V ring, then the query rows (scores) or P (P V), fp32, 4..32 rows
size_t dec_smem_bytes(int rows) {
  return (size_t)kStages * kTileBytes + 1024 + (size_t)((rows + 3) & ~3) * kTile * 4;
}
}  // namespace

cudaError_t launch_decode(const DecParams &p, const CUtensorMap &tk, const CUtensorMap &tv,
                          int sm_count, cudaStream_t stream) {
  const int64_t max_tiles = p.total_k / kTile + p.n_seqs;
  const int64_t max_items = (int64_t)p.Hkv * (max_tiles / kDecSplit + p.n_seqs);
  const int grid = (int)(max_items < 8LL * sm_count ? max_items : 8LL * sm_count);
  dec_prologue_kernel<<<1, 1024, 0, stream>>>(p);
  if (p.rows <= 16)
    dec_scores_kernel<16><<<grid, kDecScoreThreads + 64, dec_smem_bytes(16), stream>>>(p, tk);
  else
    dec_scores_kernel<32><<<grid, kDecScoreThreads + 64, dec_smem_bytes(32), stream>>>(p, tk);
  dec_decide_kernel<<<p.n_seqs * p.Hkv, 1024, 0, stream>>>(p);
  if (p.rows <= 4)
    dec_pv_kernel<4><<<grid, kDecThreads + 32, dec_smem_bytes(4), stream>>>(p, tv);
  else if (p.rows <= 8)
    dec_pv_kernel<8><<<grid, kDecThreads + 32, dec_smem_bytes(8), stream>>>(p, tv);
  else if (p.rows <= 16)
    dec_pv_kernel<16><<<grid, kDecThreads + 32, dec_smem_bytes(16), stream>>>(p, tv);
  else
    dec_pv_kernel<32><<<grid, kDecThreads + 32, dec_smem_bytes(32), stream>>>(p, tv);
  dec_combine_kernel<<<p.n_seqs * p.max_q * p.Hq, 4 * kTile, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t prepare_decode() {
  const int smem = (int)dec_smem_bytes(kDecMaxRows);
  cudaError_t e =
      cudaFuncSetAttribute(dec_scores_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(dec_scores_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(dec_pv_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(dec_pv_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(dec_pv_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(dec_pv_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  return e;
}

}  // namespace bsa
