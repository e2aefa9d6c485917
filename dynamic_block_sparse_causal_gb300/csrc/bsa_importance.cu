// Token-block importance and top-p block selection on sm_103a.
//
// Operation: "UniPrefill：通过分块动态稀疏化实现通用长上下文预填充加速",
// §3.2 Eq. (3)-(4): per query head, the attention weights of the last n query
// positions over all N keys, normalised over the whole key range, averaged
// over the n rows and summed over blocks of G = 128 keys (divided by G);
// §3.3: the shortest prefix of the blocks, by descending score, whose scores
// reach p times their total. Readings: window rows attend causally (keys up
// to their own position) unless causal = 0; the selection score of a block is
// the mean of its per-head scores; ties in the sort keep ascending block order.
//
// Kernels, in stream order:
//  * imp_prologue_kernel (1 CTA): validates cu_seqlens against the caller's
//    block count, writes block and work-item offsets, patches the token
//    extent of the two TMA tensor maps.
//  * imp_tiles_kernel (persistent, 192 threads): work item = (sequence,
//    16-block chunk, query head), consecutive items = the query heads of one
//    chunk, so the CTAs running together share K tiles through L2. The last
//    128 query positions of the sequence are one Q tile (rows before the
//    window are ignored); each key block is one K tile. For a window of at
//    most 64 rows and an even group, an item takes two query heads of the
//    group instead: the last 64 positions of each fill the tile's two halves,
//    so every MMA row and every epilogue lane carries a window row.
//    S = Q K^T goes to one of four TMEM buffers (128 columns each), so the
//    MMAs run up to three tiles ahead of the epilogue reducing the oldest:
//    per row, a reference t and e = sum exp2(S c - t) over the keys the row
//    may see, written to a [head][block][row] table. t is the running max
//    of the chunk's earlier tiles (e 2^t does not depend on t), or the
//    tile's own max for a chunk's first tile and for a tile whose sum would
//    overflow against the running max.
//      warp 0 lane 0   TMA producer (Q double buffer, 4-stage K ring)
//      warp 1          TMEM allocation; lane 0 issues tcgen05.mma
//      warps 2-5       epilogue, TMEM lane quarter = warp % 4
//    Each item also leaves the pair combined over its 16 blocks.
//  * imp_lse_kernel (one CTA per sequence and head): each window row's
//    log-sum-exp over the chunk pairs.
//  * imp_block_kernel (head x 32 blocks per CTA): per block,
//    sum over window rows of e exp2(t - lse), divided by n G.
//  * imp_mean_kernel: mean of the per-head scores.
// topp_kernel (its own entry point): one CTA per sequence sorts the block
// scores (bitonic), takes running sums in double precision and writes the
// order, k* and the keep flags.
#include <cuda_bf16.h>

#include <climits>
#include <cmath>

#include "bsa_importance.h"
#include "ptx.cuh"

namespace bsa {

namespace {

constexpr uint32_t kTileBytes = 32768;   // 128 rows x 128 bf16
constexpr uint32_t kBoxBytes = 16384;    // one 128-row x 128-byte TMA box
constexpr int kKStages = 4;
constexpr int kSBufs = 4;   // S buffers in TMEM (128 columns each): the MMA runs 3 tiles ahead
constexpr uint32_t SM_Q = 0, SM_K = 2 * kTileBytes, SM_BYTES = SM_K + kKStages * kTileBytes;
constexpr uint32_t kIdesc = IDesc<1, false, 128, 128>::value;   // bf16 x bf16 -> f32, M = N = 128

enum : int {
  I_QF = 0,                 // Q tile landed (per buffer)
  I_QE = I_QF + 2,          // Q tile no longer read by MMAs
  I_KF = I_QE + 2,          // K ring
  I_KE = I_KF + kKStages,
  I_SF = I_KE + kKStages,   // S buffer written by the MMA
  I_SE = I_SF + kSBufs,     // S buffer read by the four epilogue warps
  I_DRAIN = I_SE + kSBufs,
  I_COUNT
};

struct Item {
  int s, h, kvh, chunk, g0, g1, a, L;   // h: the item's (first) query head
};

// items per chunk of a sequence: its query heads, or pairs of them
__device__ __forceinline__ int heads_per_chunk(const ImpParams &p) { return p.Hq / p.pair; }

__device__ __forceinline__ void decode_item(const ImpParams &p, int item, Item &it) {
  int lo = 0, hi = p.n_seqs;   // largest s with item_off[s] <= item
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (p.item_off[mid] <= item) lo = mid; else hi = mid;
  }
  const int local = item - p.item_off[lo];
  const int hpc = heads_per_chunk(p);
  const int chunk = local / hpc;
  it.s = lo;
  it.chunk = chunk;
  it.h = (local - chunk * hpc) * p.pair;
  it.kvh = it.h / p.group;
  it.a = p.cu[lo];
  it.L = p.cu[lo + 1] - it.a;
  const int nb = (it.L + kTile - 1) / kTile;
  it.g0 = chunk * kImpChunk;
  it.g1 = min(nb, it.g0 + kImpChunk);
}

}  // namespace

// ============================================================ prologue

__global__ void __launch_bounds__(1024)
imp_prologue_kernel(const int32_t *__restrict__ cu, int n_seqs, int hpc, int64_t total_blocks,
                    ImpWorkspace *iw, int64_t *blk_off, int32_t *item_off, Workspace *ws,
                    const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk) {
  __shared__ int s_bad;
  const int tid = threadIdx.x;
  grid_dep_launch();   // the tile kernel may start; it waits for this grid
  if (tid == 0) s_bad = cu[0] != 0;
  __syncthreads();
  for (int s = tid; s < n_seqs; s += blockDim.x)
    if (cu[s + 1] < cu[s]) atomicOr(&s_bad, 1);
  __syncthreads();
  if (tid == 0) {
    bool bad = s_bad != 0;
    long long blocks = 0, items = 0;
    for (int s = 0; s < n_seqs && !bad; ++s) {
      blk_off[s] = blocks;
      item_off[s] = (int32_t)min(items, (long long)INT_MAX);
      const long long nb = (cu[s + 1] - cu[s] + kTile - 1) / kTile;
      blocks += nb;
      items += (long long)hpc * ((nb + kImpChunk - 1) / kImpChunk);
    }
    blk_off[n_seqs] = blocks;
    item_off[n_seqs] = (int32_t)min(items, (long long)INT_MAX);
    if (blocks != total_blocks || items > INT_MAX) bad = true;
    iw->total_items = bad ? 0 : (int32_t)items;
    if (bad) atomicOr(&ws->status, kStatusBadSeqlens);
  }
  if (tid < 2) {
    const CUtensorMap *src = tid == 0 ? &tq : &tk;
    CUtensorMap *dst = &iw->tmap[tid];
    const uint64_t *s64 = reinterpret_cast<const uint64_t *>(src);
    uint64_t *d64 = reinterpret_cast<uint64_t *>(dst);
#pragma unroll
    for (int w = 0; w < 16; ++w) d64[w] = s64[w];
    const int T = max(cu[n_seqs], 1);
    asm volatile("tensormap.replace.tile.global_dim.global.b1024.b32 [%0], 2, %1;" ::"l"(dst),
                 "r"(T)
                 : "memory");
    asm volatile("fence.proxy.tensormap::generic.release.gpu;" ::: "memory");
  }
}

// ============================================================ score tiles

__global__ void __launch_bounds__(kImpThreads, 1) imp_tiles_kernel(const __grid_constant__ ImpParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar[I_COUNT];
  __shared__ uint32_t tmem_sh;
  __shared__ volatile int abort_sh;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t *sptr = smem_raw + (sbase - raw);
  grid_dep_wait();   // the prologue's tables and tensor maps
  grid_dep_launch();
  const int total = p.iw->total_items;
  const uint64_t limit = p.wait_limit_ns;

  if (threadIdx.x == 0) {
    for (int b = 0; b < I_COUNT; ++b) mbar_init(&bar[b], (b >= I_SE && b < I_SE + kSBufs) ? 4 : 1);
    fence_mbar_init();
    abort_sh = 0;
  }
  if (warp == 1) {
    tmem_alloc(&tmem_sh, 128 * kSBufs);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tensormap_acquire(&p.iw->tmap[0]);
    tensormap_acquire(&p.iw->tmap[1]);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_sh;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      const void *tq = &p.iw->tmap[0], *tk = &p.iw->tmap[1];
      uint32_t qi = 0, kc = 0;
      int q_last[2] = {-1, -1}, k_last[kKStages];
      for (int st = 0; st < kKStages; ++st) k_last[st] = -1;
      for (int item = blockIdx.x; item < total && !abort_sh; item += gridDim.x) {
        Item it;
        decode_item(p, item, it);
        const uint32_t qb = qi & 1;
        if (!mbar_wait(&bar[I_QE + qb], ((qi >> 1) & 1) ^ 1, limit)) {
          abort_sh = 1;
          break;
        }
        mbar_expect_tx(&bar[I_QF + qb], kTileBytes);
        // 64-row boxes. One head: its last 128 positions (rows before the
        // sequence start, or before token 0: zero fill, are never used). Two
        // heads: the last 64 positions of each, head h in rows 0-63.
        const int tok = it.a + it.L - kTile / 2;
        for (int b = 0; b < 2; ++b) {
          uint8_t *dst = sptr + SM_Q + qb * kTileBytes + b * kBoxBytes;
          if (p.pair == 2) {
            tma_load_3d(dst, tq, &bar[I_QF + qb], b * 64, it.h, tok);
            tma_load_3d(dst + kBoxBytes / 2, tq, &bar[I_QF + qb], b * 64, it.h + 1, tok);
          } else {
            tma_load_3d(dst, tq, &bar[I_QF + qb], b * 64, it.h, tok - kTile / 2);
            tma_load_3d(dst + kBoxBytes / 2, tq, &bar[I_QF + qb], b * 64, it.h, tok);
          }
        }
        q_last[qb] = (int)qi++;
        for (int g = it.g0; g < it.g1; ++g) {
          const uint32_t st = kc % kKStages;
          if (!mbar_wait(&bar[I_KE + st], ((kc / kKStages) & 1) ^ 1, limit)) {
            abort_sh = 1;
            break;
          }
          if ((int)kc != p.debug_drop_k_load) {
            mbar_expect_tx(&bar[I_KF + st], kTileBytes);
            for (int b = 0; b < 2; ++b)
              tma_load_3d(sptr + SM_K + st * kTileBytes + b * kBoxBytes, tk, &bar[I_KF + st],
                          b * 64, it.kvh, it.a + g * kTile);
            k_last[st] = (int)kc;
          }
          ++kc;
        }
      }
      if (abort_sh) {   // bounded wait for this CTA's copies still in flight
        for (int b = 0; b < 2; ++b)
          if (q_last[b] >= 0) mbar_wait(&bar[I_QF + b], (q_last[b] >> 1) & 1, limit);
        for (int st = 0; st < kKStages; ++st)
          if (k_last[st] >= 0) mbar_wait(&bar[I_KF + st], (k_last[st] / kKStages) & 1, limit);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuer
      uint32_t qi = 0, kc = 0, sc = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < total && ok && !abort_sh; item += gridDim.x) {
        Item it;
        decode_item(p, item, it);
        const uint32_t qb = qi & 1;
        if (!(ok = mbar_wait(&bar[I_QF + qb], (qi >> 1) & 1, limit))) break;
        tc_fence_after();
        const uint32_t qs = sbase + SM_Q + qb * kTileBytes;
        for (int g = it.g0; g < it.g1; ++g) {
          const uint32_t st = kc % kKStages, sb = sc % kSBufs;
          if (!(ok = mbar_wait(&bar[I_KF + st], (kc / kKStages) & 1, limit))) break;
          if (!(ok = mbar_wait(&bar[I_SE + sb], ((sc / kSBufs) & 1) ^ 1, limit))) break;
          tc_fence_after();
          const uint32_t ks = sbase + SM_K + st * kTileBytes;
          // K-major A and B, 128-byte swizzle: a K step of 16 is 32 bytes
          // inside a box, the second 64 columns are the next box
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
            mma_f16_ss(tmem + sb * 128, sdesc_sw128(qs + off, 16, 1024),
                       sdesc_sw128(ks + off, 16, 1024), kIdesc, kk > 0);
          }
          mma_commit(&bar[I_SF + sb]);
          mma_commit(&bar[I_KE + st]);
          ++kc;
          ++sc;
        }
        if (!ok) break;
        mma_commit(&bar[I_QE + qb]);
        ++qi;
      }
      if (!ok) abort_sh = 1;
      if (abort_sh) {   // let this thread's MMAs finish before TMEM is freed
        mma_commit(&bar[I_DRAIN]);
        mbar_wait(&bar[I_DRAIN], 0, limit);
      }
    }
  } else {
    // -------------------------------------------------- epilogue warps
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    uint32_t sc = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < total && ok && !abort_sh; item += gridDim.x) {
      Item it;
      decode_item(p, item, it);
      // this lane's query head and window row (row r of a head's table is
      // position L - 128 + r)
      const int hh = (p.pair == 2 && row >= kTile / 2) ? it.h + 1 : it.h;
      const int wrow = p.pair == 2 ? kTile / 2 + (row & (kTile / 2 - 1)) : row;
      const int pos = it.L - kTile + wrow;
      const int last_key = p.causal ? min(pos, it.L - 1) : it.L - 1;
      float *tt = p.stat_t + ((int64_t)hh * p.total_blocks + p.blk_off[it.s]) * kTile + wrow;
      float *te = p.stat_e + ((int64_t)hh * p.total_blocks + p.blk_off[it.s]) * kTile + wrow;
      float cm = -INFINITY, cl = 0.f;   // (t, e) combined over this chunk
      for (int g = it.g0; g < it.g1; ++g) {
        const uint32_t sb = sc % kSBufs;
        // warp-uniform outcome: the TMEM loads below are warp-collective
        ok = __all_sync(0xffffffffu, mbar_wait(&bar[I_SF + sb], (sc / kSBufs) & 1, limit));
        if (!ok) break;
        tc_fence_after();
        uint32_t v[4][32];
        const uint32_t ta = tmem + lane_off + sb * 128;
        tmem_ld32(ta, v[0]);
        tmem_ld32(ta + 32, v[1]);
        tmem_ld32(ta + 64, v[2]);
        tmem_ld32(ta + 96, v[3]);
        tmem_wait_ld(v[0]);
        reg_fence(v[1]);
        reg_fence(v[2]);
        reg_fence(v[3]);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar[I_SE + sb]);
        ++sc;
        // keys this row may see in block g: columns [0, ncol)
        const int ncol = last_key - g * kTile + 1;
        if (ncol < kTile) {
#pragma unroll
          for (int ch = 0; ch < 4; ++ch)
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (ch * 32 + e >= ncol) v[ch][e] = __float_as_uint(-INFINITY);
        }
        // (t, e) of the tile against a reference t: the chunk's running max
        // once it has one (any reference gives the same e 2^t; a tile more
        // than 2^127 above it overflows and is redone against its own max),
        // else the tile's own max
        auto exp_sum = [&](float tref) -> float {
          // two columns per instruction: packed f32x2 scale-and-subtract and
          // sums (eight partial sums), the exponentials one by one
          const uint64_t c2 = f2_pack(p.c, p.c), nt2 = f2_pack(-tref, -tref);
          uint64_t s2[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) s2[k] = f2_pack(0.f, 0.f);
#pragma unroll
          for (int ch = 0; ch < 4; ++ch)
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              float y0, y1;
              f2_unpack(f2_fma(f2_pack(__uint_as_float(v[ch][e]), __uint_as_float(v[ch][e + 1])), c2, nt2),
                        y0, y1);
              s2[(e >> 1) & 3] = f2_add(s2[(e >> 1) & 3], f2_pack(ex2_approx(y0), ex2_approx(y1)));
            }
          float s8[8];
#pragma unroll
          for (int k = 0; k < 4; ++k) f2_unpack(s2[k], s8[2 * k], s8[2 * k + 1]);
          return ((s8[0] + s8[1]) + (s8[2] + s8[3])) + ((s8[4] + s8[5]) + (s8[6] + s8[7]));
        };
        float t = -INFINITY, sum = 0.f;
        bool own = !(cm > -INFINITY);
        if (!own) {
          t = cm;
          sum = exp_sum(t);
          own = !(sum < INFINITY);
        }
        if (own) {
          float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int ch = 0; ch < 4; ++ch)
#pragma unroll
            for (int e = 0; e < 32; e += 2)
              m4[(e >> 1) & 3] = max3f(m4[(e >> 1) & 3], __uint_as_float(v[ch][e]),
                                       __uint_as_float(v[ch][e + 1]));
          const float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
          t = -INFINITY;
          sum = 0.f;
          if (mx > -INFINITY) {
            t = mx * p.c;
            sum = exp_sum(t);
          }
        }
        tt[(int64_t)g * kTile] = t;
        te[(int64_t)g * kTile] = sum;
        if (sum > 0.f) {
          const float mn = fmaxf(cm, t);
          cl = cl * ex2_approx(cm - mn) + sum * ex2_approx(t - mn);
          cm = mn;
        }
      }
      if (!ok) break;
      const int64_t ci =
          ((int64_t)hh * p.max_chunks + p.item_off[it.s] / heads_per_chunk(p) + it.chunk) * kTile + wrow;
      p.chunk_m[ci] = cm;
      p.chunk_l[ci] = cl;
    }
    if (!ok) abort_sh = 1;
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (abort_sh && threadIdx.x == 0) atomicOr(&p.ws->status, kStatusTimeout);
  if (warp == 1) tmem_dealloc(tmem, 128 * kSBufs);
}

// ============================================================ reductions

// One CTA per (sequence, head), thread r = window row r of the Q tile: the
// row's log2-sum-exp2 over the sequence's chunks. Rows before the window (or
// without any key) get +inf, so that they weigh nothing below.
__global__ void __launch_bounds__(kTile) imp_lse_kernel(const __grid_constant__ ImpParams p) {
  grid_dep_wait();
  grid_dep_launch();
  if (p.iw->total_items == 0) return;   // rejected, or nothing to do
  const int s = blockIdx.x / p.Hq, h = blockIdx.x - s * p.Hq;
  const int L = p.cu[s + 1] - p.cu[s];
  const int r = threadIdx.x;
  float *out = p.row_lse + ((int64_t)h * p.n_seqs + s) * kTile + r;
  if (L <= 0) {
    *out = INFINITY;
    return;
  }
  const int nch = ((L + kTile - 1) / kTile + kImpChunk - 1) / kImpChunk;
  const int ne = min(p.n_window, L);
  const int64_t base = ((int64_t)h * p.max_chunks + p.item_off[s] / heads_per_chunk(p)) * kTile + r;
  float m = -INFINITY, l = 0.f;
  for (int c0 = 0; c0 < nch; c0 += 8) {
    float cm[8], cl[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {   // eight loads in flight
      const bool in = c0 + u < nch;
      cm[u] = in ? p.chunk_m[base + (int64_t)(c0 + u) * kTile] : -INFINITY;
      cl[u] = in ? p.chunk_l[base + (int64_t)(c0 + u) * kTile] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (cl[u] > 0.f) {
        const float mn = fmaxf(m, cm[u]);
        l = l * ex2_approx(m - mn) + cl[u] * ex2_approx(cm[u] - mn);
        m = mn;
      }
    }
  }
  *out = (r >= kTile - ne && l > 0.f) ? m + log2f(l) : INFINITY;
}

// Per head, 32 consecutive blocks of the packed block axis per CTA, four per
// warp: score = sum over window rows of e exp2(t - lse), divided by n G.
__global__ void __launch_bounds__(256) imp_block_kernel(const __grid_constant__ ImpParams p) {
  grid_dep_wait();
  grid_dep_launch();
  if (p.iw->total_items == 0) return;
  const int h = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int u = 0; u < 4; ++u) {
    const int64_t b = (int64_t)blockIdx.x * 32 + warp * 4 + u;
    if (b >= p.total_blocks) return;
    int lo = 0, hi = p.n_seqs;   // sequence of block b: largest s with blk_off[s] <= b
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (p.blk_off[mid] <= b) lo = mid; else hi = mid;
    }
    const int L = p.cu[lo + 1] - p.cu[lo];
    const int ne = min(p.n_window, L);
    const float *lse = p.row_lse + ((int64_t)h * p.n_seqs + lo) * kTile;
    const float *T = p.stat_t + ((int64_t)h * p.total_blocks + b) * kTile;
    const float *E = p.stat_e + ((int64_t)h * p.total_blocks + b) * kTile;
    float acc = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {   // window rows only: the others may never be written
      const int rr = lane + 32 * k;
      if (rr >= kTile - ne) acc += E[rr] * ex2_approx(T[rr] - lse[rr]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) p.scores[(int64_t)h * p.total_blocks + b] = acc / ((float)ne * (float)kTile);
  }
}

__global__ void imp_mean_kernel(const __grid_constant__ ImpParams p) {
  grid_dep_wait();
  if (p.iw->total_items == 0) return;
  const float inv = 1.f / (float)p.Hq;
  for (int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; b < p.total_blocks;
       b += (int64_t)gridDim.x * blockDim.x) {
    float acc = 0.f;
    for (int h = 0; h < p.Hq; ++h) acc += p.scores[(int64_t)h * p.total_blocks + b];
    p.mean_scores[b] = acc * inv;
  }
}

// ============================================================ top-p

// Sorted position a comes before b: larger score first, then smaller index.
__device__ __forceinline__ bool before(float ka, int ia, float kb, int ib) {
  return ka > kb || (ka == kb && ia < ib);
}

__global__ void __launch_bounds__(kTopPThreads)
topp_kernel(const float *__restrict__ scores, const int32_t *__restrict__ cu, int n_seqs,
            int64_t total_blocks, float p, int32_t *order, int32_t *n_selected, uint8_t *keep,
            Workspace *ws) {
  extern __shared__ uint8_t smem_raw[];
  float *key = reinterpret_cast<float *>(smem_raw);
  int *idx = reinterpret_cast<int *>(smem_raw + kTopPMaxBlocks * 4);
  __shared__ unsigned long long s_off, s_total;
  __shared__ int s_bad, s_k;
  __shared__ double s_run_last, s_warp[kTopPThreads / 32];
  const int s = blockIdx.x, tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;

  // validate the whole batch and find this sequence's first block
  if (tid == 0) {
    s_off = 0;
    s_total = 0;
    s_bad = cu[0] != 0;
    s_k = INT_MAX;
  }
  __syncthreads();
  for (int t = tid; t < n_seqs; t += blockDim.x) {
    const int L = cu[t + 1] - cu[t];
    if (L < 0) {
      atomicOr(&s_bad, 1);
      continue;
    }
    const unsigned long long nb = (unsigned long long)((L + kTile - 1) / kTile);
    if (nb > (unsigned long long)kTopPMaxBlocks) atomicOr(&s_bad, 1);
    atomicAdd(&s_total, nb);
    if (t < s) atomicAdd(&s_off, nb);
  }
  __syncthreads();
  if (s_bad || (long long)s_total != total_blocks) {
    if (s == 0 && tid == 0) atomicOr(&ws->status, kStatusBadSeqlens);
    return;
  }
  const int L = cu[s + 1] - cu[s];
  const int nb = (L + kTile - 1) / kTile;
  const long long off = (long long)s_off;
  if (nb == 0) {
    if (tid == 0) n_selected[s] = 0;
    return;
  }
  int P2 = 1;
  while (P2 < nb) P2 <<= 1;
  for (int i = tid; i < P2; i += blockDim.x) {
    key[i] = i < nb ? scores[off + i] : -INFINITY;
    idx[i] = i < nb ? i : INT_MAX;
  }
  __syncthreads();
  // bitonic sort into the "before" order
  for (int k = 2; k <= P2; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = tid; i < P2; i += blockDim.x) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const bool fwd = (i & k) == 0;
          const float ka = key[i], kb = key[ixj];
          const int ia = idx[i], ib = idx[ixj];
          if (fwd != before(ka, ia, kb, ib)) {
            key[i] = kb;
            key[ixj] = ka;
            idx[i] = ib;
            idx[ixj] = ia;
          }
        }
      }
      __syncthreads();
    }
  }
  // running sums in double precision: thread t owns positions [t*w, t*w + w)
  const int w = (nb + blockDim.x - 1) / blockDim.x;
  const int b0 = min(nb, tid * w), b1 = min(nb, b0 + w);
  double loc = 0.0;
  for (int i = b0; i < b1; ++i) loc += (double)key[i];
  // exclusive scan of the per-thread sums
  double inc = loc;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += y;
  }
  if (lane == 31) s_warp[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    double x = lane < (int)(blockDim.x / 32) ? s_warp[lane] : 0.0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    s_warp[lane] = x;   // inclusive over warps
  }
  __syncthreads();
  const double excl = (warp > 0 ? s_warp[warp - 1] : 0.0) + (inc - loc);
  // the total is the running sum at the last position, formed the same way
  if (b0 < nb && b1 == nb) {
    double run = excl;
    for (int i = b0; i < b1; ++i) run += (double)key[i];
    s_run_last = run;
  }
  __syncthreads();
  const double thr = (double)p * s_run_last;
  {
    double run = excl;
    for (int i = b0; i < b1; ++i) {
      run += (double)key[i];
      if (run >= thr) {
        atomicMin(&s_k, i + 1);
        break;
      }
    }
  }
  __syncthreads();
  const int kstar = s_k;
  for (int i = tid; i < nb; i += blockDim.x) {
    order[off + i] = idx[i];
    if (keep) keep[off + idx[i]] = i < kstar ? 1 : 0;
  }
  if (tid == 0) n_selected[s] = kstar;
}

// ============================================================ launchers

size_t importance_smem_bytes() { return SM_BYTES + 1024; }
size_t topp_smem_bytes() { return (size_t)kTopPMaxBlocks * 8; }

cudaError_t launch_importance(const ImpParams &p, const CUtensorMap tmpl[2], int num_ctas,
                              cudaStream_t stream) {
  imp_prologue_kernel<<<1, 1024, 0, stream>>>(p.cu, p.n_seqs, p.Hq / p.pair, p.total_blocks, p.iw,
                                               const_cast<int64_t *>(p.blk_off),
                                               const_cast<int32_t *>(p.item_off), p.ws, tmpl[0],
                                               tmpl[1]);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if ((e = launch_dependent(imp_tiles_kernel, num_ctas, kImpThreads, importance_smem_bytes(), stream,
                            p)) != cudaSuccess)
    return e;
  if ((e = launch_dependent(imp_lse_kernel, p.n_seqs * p.Hq, kTile, 0, stream, p)) != cudaSuccess)
    return e;
  if (p.total_blocks > 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((p.total_blocks + 31) / 32), (unsigned)p.Hq);
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if ((e = cudaLaunchKernelEx(&cfg, imp_block_kernel, p)) != cudaSuccess) return e;
  }
  if (p.mean_scores && p.total_blocks > 0) {
    const int64_t want = (p.total_blocks + 255) / 256;
    const int grid = (int)(want < 4096 ? want : 4096);
    if ((e = launch_dependent(imp_mean_kernel, grid, 256, 0, stream, p)) != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

cudaError_t launch_top_p(const float *scores, const int32_t *cu, int n_seqs, int64_t total_blocks,
                         float p, int32_t *order, int32_t *n_selected, uint8_t *keep,
                         Workspace *ws, cudaStream_t stream) {
  topp_kernel<<<n_seqs, kTopPThreads, topp_smem_bytes(), stream>>>(
      scores, cu, n_seqs, total_blocks, p, order, n_selected, keep, ws);
  return cudaGetLastError();
}

cudaError_t prepare_importance() {
  cudaError_t e = cudaFuncSetAttribute(imp_tiles_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)importance_smem_bytes());
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(topp_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)topp_smem_bytes());
}

}  // namespace bsa
