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
//  2. dec_pv_kernel: per split, the decisions (the prefix max of the earlier
//     tiles' maxima, then the split's tiles in order; the AND over each query
//     head's rows), the kept tiles' V (TMA, only kept tiles) and an online
//     softmax with the split's own reference max;
//  3. dec_combine_kernel: merges the splits' (max, sum, output) per row.
// The decisions are exactly those of the sequential walk; outputs equal the
// online softmax over the kept tiles up to rounding order. The work is
// bound by reading K once and the kept V once from DRAM; the two narrow
// contractions (scores, P V) run on the tensor cores because the CUDA-core
// versions were bound by shared-memory traffic, not by DRAM. One query row
// group of at most 32 rows per KV head.
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
  // the KV heads of one split are neighbours: CTAs running together read
  // whole token rows of K and V (all heads) from DRAM
  const int local = item - p.item_off[lo];
  const int split = local / p.Hkv;
  it.kvh = local - split * p.Hkv;
  it.j0 = split * p.split;
  it.j1 = min(nk, it.j0 + p.split);
}

__device__ __forceinline__ void load_tile(uint8_t *dst, const CUtensorMap *map, uint64_t *bar,
                                          int head, int row) {
  mbar_expect_tx(bar, kTileBytes);
  tma_load_3d(dst, map, bar, 0, head, row);
  tma_load_3d(dst + kBoxBytes, map, bar, 64, head, row);
}

// Plain bulk copy global -> shared, completing on an mbarrier (16-byte
// aligned addresses, size a multiple of 16).
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

}  // namespace

// ============================================================ prologue

__global__ void __launch_bounds__(1024) dec_prologue_kernel(const __grid_constant__ DecParams p) {
  __shared__ int s_bad;
  const int tid = threadIdx.x;
  grid_dep_launch();   // the score kernel may set up meanwhile; it waits for this grid
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
      if (Lq > 0) items += (long long)p.Hkv * ((nk + p.split - 1) / p.split);
      words += (long long)p.Hq * nq * ((nk + 31) / 32);
    }
    tile_off[p.n_seqs] = tiles;
    item_off[p.n_seqs] = (int32_t)min(items, (long long)INT_MAX);
    bm_off[p.n_seqs] = words;
    if (items > INT_MAX) bad = true;
    p.dw->total_items = bad ? 0 : (int32_t)items;
    if (bad) atomicOr(&p.ws->status, kStatusBadSeqlens);
    s_bad = bad;
  }
  __syncthreads();
  if (s_bad) return;
  // the split passes OR their skip bits into the bitmap
  if (p.bitmap)
    for (int64_t w = tid; w < p.bm_off[p.n_seqs]; w += blockDim.x) p.bitmap[w] = 0u;
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
  grid_dep_wait();     // tables of the previous kernel
  grid_dep_launch();
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
          if ((int)kc != p.debug_drop_k_load) {
            load_tile(ring + b * kTileBytes, &tk, &kfull[b], it.kvh, it.ak + j * kTile);
            last_issue[b] = (int)kc;
          }
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
      float split_max = -INFINITY;   // thread t < R: row t's max over this split
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
          split_max = fmaxf(split_max, m);
        }
      }
      if (stop) break;
      // the split's row maxima, for the prefix max of the later splits
      if (t < R)
        p.smax[((int64_t)it.kvh * p.max_splits + p.item_off[it.s] / p.Hkv + it.j0 / p.split) *
                   p.rows + t] = split_max;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (abort_sh && t == 0) atomicOr(&p.ws->status, kStatusTimeout);
  if (warp == 5) tmem_dealloc(tmem, 2 * N < 32 ? 32 : 2 * N);
}

// ============================================================ 2: decide, P V

// One work item = (sequence, KV head, 16-tile split), as in the score pass.
//   warps 0-3  decisions of the split: the row maxima of all earlier tiles
//              (prefix max), then a walk over the split's tiles; skip bits go
//              to the bitmap (OR into words the prologue zeroed). Then per
//              kept tile: P (thread t = key t, fp32 exponentials and row sums)
//              into a 128-byte-swizzled bf16 buffer, and O = alpha O + D
//              (thread t = head-dim column t, D read from TMEM).
//   warp 4     V producer for the kept tiles
//   warp 5     TMEM allocation; lane 0 issues O^T = V^T P^T per kept tile:
//              A = the V tile read MN-major (M = head dim), B = P (the
//              group's rows padded to N, keys contiguous), D in one of two
//              TMEM buffers.
// RB >= group x Lq rows; N = RB rounded up to 16.
template <int RB>
__global__ void __launch_bounds__(kDecScoreThreads + 64, RB <= 16 ? 2 : 1)
dec_pv_kernel(const __grid_constant__ DecParams p, const __grid_constant__ CUtensorMap tv) {
  constexpr int N = RB < 16 ? 16 : RB;
  constexpr int kEpi = kDecScoreThreads;
  constexpr uint32_t kPBytes = N * 256;
  // ring stage: the V tile, then the kept tile's scores S (rows x 128 fp32)
  constexpr uint32_t kStage = kTileBytes + RB * kTile * 4;
  // bf16 x bf16 -> f32, A MN-major (bit 15), B K-major, M = 128, N
  constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 15) |
                              ((uint32_t)(N >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
  extern __shared__ uint8_t smem_raw[];
  __shared__ float lred[kEpi / 32][RB];
  __shared__ float mred[kEpi / 32][RB];
  __shared__ float srm[kDecSplit * RB];
  __shared__ uint32_t predmask[RB];
  __shared__ uint64_t vfull[kStages], vempty[kStages], pready[2], pfree[2], dfull[2], dempty[2],
      lready[2], lfree[2], drain;
  __shared__ int klist[2][kDecSplit];
  __shared__ uint32_t kact[2][kDecSplit];
  __shared__ uint32_t act_sh[kDecSplit];
  __shared__ int nkept_sh[2];
  __shared__ uint32_t tmem_sh;
  __shared__ volatile int abort_sh;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t *ring = smem_raw + (sbase - raw);
  uint8_t *pbuf = ring + kStages * kStage;
  if (t == 0) {
    for (int b = 0; b < kStages; ++b) {
      mbar_init(&vfull[b], 1);
      mbar_init(&vempty[b], 2);   // the MMA has read V, the epilogue has read S
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&pready[b], 1);
      mbar_init(&pfree[b], 1);
      mbar_init(&dfull[b], 1);
      mbar_init(&dempty[b], kEpi / 32);
      mbar_init(&lready[b], 1);
      mbar_init(&lfree[b], 2);
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
  grid_dep_wait();     // tables of the previous kernel
  grid_dep_launch();
  const int total = p.dw->total_items;
  const uint64_t limit = p.wait_limit_ns;

  if (warp == 4) {
    // ---------------------------------------------------- V producer
    if (lane == 0) {
      uint32_t kc = 0, i = 0;
      int last_issue[kStages] = {-1, -1, -1};
      bool ok = true;
      for (int item = blockIdx.x; item < total && ok; item += gridDim.x, ++i) {
        DecItem it;
        decode_item(p, item, it);
        const uint32_t par = i & 1;
        if (!(ok = mbar_wait(&lready[par], (i >> 1) & 1, limit))) break;
        const int n = nkept_sh[par];
        const int R = p.group * it.Lq;
        const int64_t toff = p.tile_off[it.s];
        for (int u = 0; u < n; ++u) {
          const uint32_t b = kc % kStages;
          if (!(ok = mbar_wait(&vempty[b], ((kc / kStages) & 1) ^ 1, limit)) || abort_sh) {
            ok = false;
            break;
          }
          const int j = klist[par][u];
          uint8_t *st = ring + b * kStage;
          mbar_expect_tx(&vfull[b], kTileBytes + R * kTile * 4);
          tma_load_3d(st, &tv, &vfull[b], 0, it.kvh, it.ak + j * kTile);
          tma_load_3d(st + kBoxBytes, &tv, &vfull[b], 64, it.kvh, it.ak + j * kTile);
          bulk_load(st + kTileBytes, p.S + ((toff + j) * p.Hkv + it.kvh) * p.rows * kTile,
                    R * kTile * 4, &vfull[b]);
          last_issue[b] = (int)kc++;
        }
        mbar_arrive(&lfree[par]);
      }
      if (!ok) {
        abort_sh = 1;
        for (int b = 0; b < kStages; ++b)
          if (last_issue[b] >= 0) mbar_wait(&vfull[b], (last_issue[b] / kStages) & 1, limit);
      }
    }
  } else if (warp == 5) {
    // ---------------------------------------------------- MMA issuer
    if (lane == 0) {
      uint32_t kc = 0, i = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < total && ok; item += gridDim.x, ++i) {
        const uint32_t par = i & 1;
        if (!(ok = mbar_wait(&lready[par], (i >> 1) & 1, limit))) break;
        const int n = nkept_sh[par];
        mbar_arrive(&lfree[par]);
        for (int u = 0; u < n; ++u, ++kc) {
          const uint32_t b = kc % kStages, slot = kc & 1;
          if (!(ok = mbar_wait(&vfull[b], (kc / kStages) & 1, limit))) break;
          if (!(ok = mbar_wait(&pready[slot], (kc >> 1) & 1, limit))) break;
          if (!(ok = mbar_wait(&dempty[slot], ((kc >> 1) & 1) ^ 1, limit))) break;
          if (abort_sh) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t vs = sbase + b * kStage;
          const uint32_t ps = sbase + kStages * kStage + slot * kPBytes;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            // A: 16 keys = two 8-key swizzle atoms (2048 bytes); the two 64-wide
            // halves of the head dim are one box apart. B: 32 bytes per K step.
            const uint64_t ad = sdesc_sw128(vs + kk * 2048, kBoxBytes, 1024);
            const uint64_t bd = sdesc_sw128(ps + (kk >> 2) * (N * 128) + (kk & 3) * 32, 16, 1024);
            mma_f16_ss(tmem + slot * N, ad, bd, kIdesc, kk > 0);
          }
          mma_commit(&dfull[slot]);
          mma_commit(&vempty[b]);
          mma_commit(&pfree[slot]);
        }
      }
      if (!ok) {
        abort_sh = 1;
        mma_commit(&drain);
        mbar_wait(&drain, 0, limit);
      }
    }
  } else {
    // ---------------------------------------------------- epilogue
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    uint32_t kc = 0, i = 0;
    bool stop = false;
    for (int item = blockIdx.x; item < total && !stop; item += gridDim.x, ++i) {
      DecItem it;
      decode_item(p, item, it);
      const int R = p.group * it.Lq, nt = it.j1 - it.j0;
      const int64_t toff = p.tile_off[it.s];
      const uint32_t par = i & 1;
      const float *rmh = p.rm + ((int64_t)it.kvh * p.max_tiles + toff) * p.rows;
      // ---- decisions. Running max before the split: the max of the earlier
      // splits' row maxima (written by the score pass). Rp (R rounded up to a
      // power of two) divides the thread stride, so thread t always meets row
      // t % Rp; the split's own tile maxima go to shared memory for the walk
      // in order.
      const int Rp = R <= 1 ? 1 : 1 << (32 - __clz(R - 1));
      const int rt = t & (Rp - 1);
      float mp = -INFINITY;
      if (rt < R) {
        const float *sm = p.smax + ((int64_t)it.kvh * p.max_splits + p.item_off[it.s] / p.Hkv) * p.rows;
        const int q = it.j0 / p.split;   // splits before this one
#pragma unroll 4
        for (int idx = t; idx < q * Rp; idx += kEpi)
          mp = fmaxf(mp, sm[(int64_t)(idx / Rp) * p.rows + rt]);
      }
      for (int idx = t; idx < nt * R; idx += kEpi)
        srm[idx] = rmh[(int64_t)(it.j0 + idx / R) * p.rows + idx % R];
      for (int o = 16; o >= Rp; o >>= 1) mp = fmaxf(mp, __shfl_xor_sync(0xffffffffu, mp, o));
      if (lane < Rp) mred[warp][lane] = mp;
      // the lists of item i - 2 are no longer read by the producer and MMA
      const bool okl = i < 2 || mbar_wait(&lfree[par], ((i >> 1) - 1) & 1, limit);
      if (bar_red_or(!okl, 1, kEpi)) {
        stop = true;
        break;
      }
      if (t < R) {   // walk the split's tiles in order, per row
        float mr = fmaxf(fmaxf(mred[0][t], mred[1][t]), fmaxf(mred[2][t], mred[3][t]));
        uint32_t bits = 0;   // bit u: row t would skip tile j0 + u
        for (int u = 0; u < nt; ++u) {
          const float x = srm[u * R + t];
          if (x < mr + p.log2_lambda) bits |= 1u << u;
          mr = fmaxf(mr, x);
        }
        predmask[t] = bits;
      }
      named_bar_sync(1, kEpi);
      if (t < nt) {   // heads of the group that keep tile j0 + t
        uint32_t act = 0;
        for (int g = 0; g < p.group; ++g) {
          bool keep = false;
          for (int qi = 0; qi < it.Lq; ++qi) keep |= !((predmask[g * it.Lq + qi] >> t) & 1u);
          if (keep) act |= 1u << g;
        }
        act_sh[t] = act;
      }
      named_bar_sync(1, kEpi);
      if (t == 0) {
        int n = 0;
        for (int u = 0; u < nt; ++u)
          if (act_sh[u]) {
            klist[par][n] = it.j0 + u;
            kact[par][n] = act_sh[u];
            ++n;
          }
        nkept_sh[par] = n;
        mbar_arrive(&lready[par]);
      }
      if (p.bitmap && t < p.group) {   // this split's 16 bits of each head's row
        uint32_t bits = 0xFFFFu;
        for (int qi = 0; qi < it.Lq; ++qi) bits &= predmask[t * it.Lq + qi];
        bits &= (nt >= 32 ? 0xFFFFFFFFu : ((1u << nt) - 1u));
        const int nk = (it.Lk + kTile - 1) / kTile, W = (nk + 31) / 32;
        if (bits)
          atomicOr(p.bitmap + p.bm_off[it.s] + (int64_t)(it.kvh * p.group + t) * W + (it.j0 >> 5),
                   bits << (it.j0 & 31));
      }
      named_bar_sync(1, kEpi);
      const int n = nkept_sh[par];
      // ---- kept tiles
      float O[RB], mref[RB], lsum[RB], alpha[RB], alpha_prev[RB];
#pragma unroll
      for (int r = 0; r < RB; ++r) {
        O[r] = 0.f;
        mref[r] = -INFINITY;
        lsum[r] = 0.f;
        alpha[r] = alpha_prev[r] = 1.f;
      }
      // O += D of kept tile number kd (its P used the reference alpha_prev)
      auto take_d = [&](uint32_t kd) -> bool {
        const uint32_t slot = kd & 1;
        const bool okd = mbar_wait(&dfull[slot], (kd >> 1) & 1, limit);
        if (bar_red_or(!okd, 1, kEpi)) return false;
        tc_fence_after();
        uint32_t v[N];
#pragma unroll
        for (int h = 0; h < N / 16; ++h)
          tmem_ld16(tmem + lane_off + slot * N + h * 16, *reinterpret_cast<uint32_t(*)[16]>(&v[h * 16]));
#pragma unroll
        for (int h = 0; h < N / 16; ++h) tmem_wait_ld16(*reinterpret_cast<uint32_t(*)[16]>(&v[h * 16]));
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&dempty[slot]);
#pragma unroll
        for (int r = 0; r < RB; ++r) O[r] = fmaf(O[r], alpha_prev[r], __uint_as_float(v[r]));
        return true;
      };
      for (int u = 0; u < n && !stop; ++u, ++kc) {
        const int j = klist[par][u];
        const uint32_t act = kact[par][u], slot = kc & 1, b = kc % kStages;
        const float *rmj = rmh + (int64_t)j * p.rows;
        // P buffer slot free (the MMA two kept tiles back has read it), and
        // this tile's V and S landed
        const bool okp = mbar_wait(&pfree[slot], ((kc >> 1) & 1) ^ 1, limit) &&
                         mbar_wait(&vfull[b], (kc / kStages) & 1, limit);
        if (bar_red_or(!okp, 1, kEpi)) {
          stop = true;
          break;
        }
        const float *Ss = reinterpret_cast<const float *>(ring + b * kStage + kTileBytes);
        uint8_t *pb = pbuf + slot * kPBytes;
#pragma unroll
        for (int r = 0; r < N; ++r) {
          float pv = 0.f;
          if (r < RB && r < R) {
            const bool on = (act >> (r / it.Lq)) & 1u;
            const float mnew = on ? fmaxf(mref[r], rmj[r]) : mref[r];
            alpha[r] = mnew == -INFINITY ? 1.f : ex2_approx(mref[r] - mnew);
            mref[r] = mnew;
            pv = (on && mnew != -INFINITY) ? ex2_approx(Ss[r * kTile + t] - mnew) : 0.f;
            lsum[r] = fmaf(lsum[r], alpha[r], pv);
          } else if (r < RB) {
            alpha[r] = 1.f;
          }
          // key t of row r: box t/64, 16-byte chunk (t%64)/8 swizzled by row
          *reinterpret_cast<__nv_bfloat16 *>(pb + (t >> 6) * (N * 128) + r * 128 +
                                             ((((t >> 3) & 7) ^ (r & 7)) << 4) + (t & 7) * 2) =
              __float2bfloat16_rn(pv);
        }
        fence_proxy_async_smem();
        named_bar_sync(1, kEpi);
        if (t == 0) {
          mbar_arrive(&pready[slot]);
          mbar_arrive(&vempty[b]);   // S of this stage has been read
        }
        if (u > 0 && !take_d(kc - 1)) {
          stop = true;
          break;
        }
#pragma unroll
        for (int r = 0; r < RB; ++r) alpha_prev[r] = alpha[r];
      }
      if (!stop && n > 0 && !take_d(kc - 1)) stop = true;
      if (stop) break;
      // ---- write the split: O (thread t = column), the row sums, the reference max
#pragma unroll
      for (int r = 0; r < RB; ++r) {
        float x = lsum[r];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
        if (lane == 0) lred[warp][r] = x;
      }
      named_bar_sync(1, kEpi);
      const int64_t prow = (int64_t)item * p.rows;
#pragma unroll
      for (int r = 0; r < RB; ++r)
        if (r < R) p.pO[(prow + r) * kTile + t] = O[r];
      if (t < R) {
        p.pl[prow + t] = (lred[0][t] + lred[1][t]) + (lred[2][t] + lred[3][t]);
#pragma unroll
        for (int r = 0; r < RB; ++r)
          if (r == t) p.pm[prow + t] = mref[r];
      }
    }
    if (stop) abort_sh = 1;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (abort_sh && t == 0) atomicOr(&p.ws->status, kStatusTimeout);
  if (warp == 5) tmem_dealloc(tmem, 2 * N < 32 ? 32 : 2 * N);
}

// ============================================================ 3: merge

// One CTA per (sequence, query slot, query head); thread t = column t%128 of
// the splits q with q%4 == t/128, the four groups added at the end.
__global__ void __launch_bounds__(4 * kTile) dec_combine_kernel(const __grid_constant__ DecParams p) {
  __shared__ float red[4 * kTile / 32];
  __shared__ float part[3][kTile], lpart[4];
  grid_dep_wait();
  if (p.dw->total_items == 0) return;
  const int per_seq = p.max_q * p.Hq;
  const int s = blockIdx.x / per_seq, rem = blockIdx.x - s * per_seq;
  const int qi = rem / p.Hq, h = rem - qi * p.Hq;
  const int aq = p.cu_q[s], Lq = p.cu_q[s + 1] - aq;
  if (qi >= Lq) return;
  const int t = threadIdx.x, c = t & (kTile - 1), grp = t >> 7, lane = t & 31, warp = t >> 5;
  const int Lk = p.cu_k[s + 1] - p.cu_k[s];
  const int nk = (Lk + kTile - 1) / kTile, ns = (nk + p.split - 1) / p.split;
  const int kvh = h / p.group, r = (h - kvh * p.group) * Lq + qi;
  const int64_t it0 = (int64_t)p.item_off[s] + kvh;   // split q is item it0 + q * Hkv
  const int64_t H = p.Hkv;
  float m = -INFINITY;
  for (int q = t; q < ns; q += 4 * kTile) m = fmaxf(m, p.pm[(it0 + q * H) * p.rows + r]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) red[warp] = m;
  __syncthreads();
  m = red[0];
#pragma unroll
  for (int w = 1; w < 4 * kTile / 32; ++w) m = fmaxf(m, red[w]);
  float acc = 0.f, l = 0.f;
#pragma unroll 4
  for (int q = grp; q < ns; q += 4) {
    const int64_t ii = it0 + q * H;
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
// V ring with the staged scores, then two P buffers (N = RB rounded up to 16)
size_t pv_smem_bytes(int RB) {
  const int N = RB < 16 ? 16 : RB;
  return (size_t)kStages * (kTileBytes + RB * kTile * 4) + 1024 + 2 * (size_t)N * 256;
}
}  // namespace

cudaError_t launch_decode(const DecParams &p, const CUtensorMap &tk, const CUtensorMap &tv,
                          int sm_count, cudaStream_t stream) {
  const int64_t max_tiles = p.total_k / kTile + p.n_seqs;
  const int64_t max_items = (int64_t)p.Hkv * (max_tiles / p.split + p.n_seqs);
  const int grid = (int)(max_items < 4LL * sm_count ? max_items : 4LL * sm_count);
  const int block = kDecScoreThreads + 64;
  dec_prologue_kernel<<<1, 1024, 0, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (p.rows <= 16)
    e = launch_dependent(dec_scores_kernel<16>, grid, block, dec_smem_bytes(16), stream, p, tk);
  else
    e = launch_dependent(dec_scores_kernel<32>, grid, block, dec_smem_bytes(32), stream, p, tk);
  if (e != cudaSuccess) return e;
  if (p.rows <= 4)
    e = launch_dependent(dec_pv_kernel<4>, grid, block, pv_smem_bytes(4), stream, p, tv);
  else if (p.rows <= 8)
    e = launch_dependent(dec_pv_kernel<8>, grid, block, pv_smem_bytes(8), stream, p, tv);
  else if (p.rows <= 16)
    e = launch_dependent(dec_pv_kernel<16>, grid, block, pv_smem_bytes(16), stream, p, tv);
  else
    e = launch_dependent(dec_pv_kernel<32>, grid, block, pv_smem_bytes(32), stream, p, tv);
  if (e != cudaSuccess) return e;
  return launch_dependent(dec_combine_kernel, p.n_seqs * p.max_q * p.Hq, 4 * kTile, 0, stream, p);
}

cudaError_t prepare_decode() {
  const int smem = (int)dec_smem_bytes(kDecMaxRows);
  cudaError_t e =
      cudaFuncSetAttribute(dec_scores_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(dec_scores_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(dec_pv_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)pv_smem_bytes(4));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(dec_pv_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)pv_smem_bytes(8));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(dec_pv_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)pv_smem_bytes(16));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(dec_pv_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)pv_smem_bytes(32));
  return e;
}

}  // namespace bsa
