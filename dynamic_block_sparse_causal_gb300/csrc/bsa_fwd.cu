// Causal prefill attention, device code for sm_103a: the per-call prologue
// and the dense forward kernel (lambda = 0; the skipping kernel for
// lambda > 0 is in bsa_skip.cu).
//
// Operation: dynamic sparse attention deployment guide
// ("长上下文推理加速方案部署实战：基于动态稀疏注意力机制的推理服务优化指南"),
// §3.2 -- online softmax over key blocks in order; with lambda = 0 the skip
// rule never fires and the pass is exact dense causal attention.
//
// Two kernels:
//  * prologue_kernel (1 CTA): validates cu_seqlens, orders sequences longest
//    first, builds the work-item level table and the skip-bitmap offsets,
//    and writes the TMA tensor maps with the token extent patched in. Both
//    forward kernels consume its tables.
//  * fwd_kernel<FP8> (persistent, one CTA per SM, 384 threads):
//      warp 0  lane 0   TMA producer: Q tiles, the K ring (3 stages) and V
//                       with every K (2-stage ring)
//      warp 1  lane 0   tcgen05 MMA issuer
//      warp 2  lane 0   fetches the next work item (atomic counter)
//      warps 4-7        softmax warpgroup of query slot 0 (TMEM lanes 0-127)
//      warps 8-11       softmax warpgroup of query slot 1
//    A work item is (sequence, KV head, two query heads of that group, query
//    tile i): both query tiles need exactly the key tiles 0..i, so each K
//    tile loaded feeds two QK^T MMAs.
//
// TMEM (512 columns): S0 [0,128) S1 [128,256) O0 [256,384) O1 [384,512),
// fp32, lane = query row; P_s (bf16 / e4m3) is written over the first
// columns of S_s and read from there by the P.V MMA. Shared memory
// (1024-aligned, 128-byte swizzle), 32 KiB regions: Q0 Q1, K[3], V[2].
//
// Pipeline counters live in registers within a work item and in shared
// memory between items, one set per role, so that no role's registers carry
// another role's counters through the item loop (register pressure in the
// softmax warpgroups sets the length of the per-tile chain).
//
// Per key tile j and query slot s the softmax warpgroup loads S_s from TMEM,
// masks the diagonal / tail and computes P = exp2(S c - m_ref) into TMEM:
// on the first tile after the row max, later in one pass against the current
// reference (scale-and-subtract and the row sum on pairs of scores with the
// packed f32x2 FMA / add), with a lazy O rescale (and a second pass) only for
// a row whose max grows by more than 2^8; then each warp posts its 32 rows
// to the P-ready barrier. The MMA warp issues O_s += P_s V_j before the next
// S_s, so the tensor pipe's in-order execution protects P until it has been
// read.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include <climits>
#include <cmath>

#include "bsa_internal.h"
#include "ptx.cuh"
#include "bsa_tile.cuh"

namespace bsa {

using namespace tile;

// ============================================================ prologue

// Query-tile count of sequence s (tiles of its queries) and key-tile count.
__device__ __forceinline__ int q_tiles(const int32_t *cu, int s) {
  return (cu[s + 1] - cu[s] + kTile - 1) / kTile;
}

__global__ void __launch_bounds__(1024)
prologue_kernel(const int32_t *__restrict__ cu, const int32_t *__restrict__ cuk, int n_seqs,
                int Hq, int Hkv, int items_per_group, int causal, const int32_t *__restrict__ page_table,
                int max_pages, int num_pages, Workspace *ws, int32_t *seq_sorted,
                int64_t *seq_bitmap_off, int32_t *level_start,
                const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                const __grid_constant__ CUtensorMap tv) {
  __shared__ int s_bad, s_maxn;
  const int tid = threadIdx.x;
  if (tid == 0) {
    s_bad = (cu[0] != 0) || (cuk[0] != 0);
    s_maxn = 0;
  }
  __syncthreads();
  for (int s = tid; s < n_seqs; s += blockDim.x) {
    const int Lq = cu[s + 1] - cu[s], Lk = cuk[s + 1] - cuk[s];
    // queries are the last Lq positions of a sequence of Lk keys
    if (Lq < 0 || Lk < 0 || (causal && Lk < Lq) || (Lq > 0 && Lk == 0)) atomicOr(&s_bad, 1);
    // query and key tiles per sequence are bounded by the level table and the
    // skipping kernel's on-chip keep bits (one per key tile)
    atomicMax(&s_maxn, max((Lq + kTile - 1) / kTile, (Lk + kTile - 1) / kTile));
    if (page_table && Lk > 0) {   // every page a sequence reads must exist
      const int nk = (Lk + kTile - 1) / kTile;
      if (nk > max_pages) {
        atomicOr(&s_bad, 1);
      } else {
        for (int j = 0; j < nk; ++j) {
          const int pg = page_table[(size_t)s * max_pages + j];
          if (pg < 0 || pg >= num_pages) atomicOr(&s_bad, 1);
        }
      }
    }
  }
  __syncthreads();
  const int maxn = s_maxn;
  // work items are ordered KV head by KV head (so CTAs running at the same time
  // stream the same head's K tiles through L2), and within a head longest
  // query tile first; U = items per (sequence, query tile) within one head
  const long long U = items_per_group;
  bool bad = s_bad || maxn > kMaxLevels;
  if (!bad) {
    // longest first (query tiles), ties by sequence index
    for (int s = tid; s < n_seqs; s += blockDim.x) {
      const int ns = q_tiles(cu, s);
      int rank = 0;
      for (int t = 0; t < n_seqs; ++t) {
        const int nt = q_tiles(cu, t);
        rank += (nt > ns) || (nt == ns && t < s);
      }
      seq_sorted[rank] = s;
    }
    // level_start[i] = first item of query-tile level i; items run from the
    // deepest level (longest causal rows) down to level 0.
    for (int i = tid; i < maxn; i += blockDim.x) {
      long long acc = 0;
      for (int t = 0; t < n_seqs; ++t) acc += max(0, q_tiles(cu, t) - 1 - i);
      level_start[i] = (int32_t)min(U * acc, (long long)INT_MAX);
    }
  }
  __syncthreads();
  if (tid == 0) {
    long long items = 0, words = 0;
    for (int s = 0; s < n_seqs && !bad; ++s) {
      const int nq = q_tiles(cu, s), nk = q_tiles(cuk, s);
      seq_bitmap_off[s] = words;
      words += (long long)Hq * nq * ((nk + 31) / 32);
      items += U * nq;
    }
    items *= Hkv;
    if (items > INT_MAX) bad = true;
    ws->counter = 0;
    ws->total_items = bad ? 0 : (int32_t)items;
    ws->max_tiles = maxn;
    ws->total_tokens = cu[n_seqs];
    if (bad) atomicOr(&ws->status, kStatusBadSeqlens);
  }
  if (tid < 3) {   // paged K/V maps already span the whole page pool
    const CUtensorMap *src = tid == 0 ? &tq : (tid == 1 ? &tk : &tv);
    CUtensorMap *dst = &ws->tmap[tid];
    const uint64_t *s64 = reinterpret_cast<const uint64_t *>(src);
    uint64_t *d64 = reinterpret_cast<uint64_t *>(dst);
#pragma unroll
    for (int w = 0; w < 16; ++w) d64[w] = s64[w];
    // token extent: query tokens for the Q map, key tokens for K and V
    if (tid == 0 || !page_table) {
      const int T = max(tid == 0 ? cu[n_seqs] : cuk[n_seqs], 1);
      asm volatile("tensormap.replace.tile.global_dim.global.b1024.b32 [%0], 2, %1;" ::"l"(dst),
                   "r"(T)
                   : "memory");
    }
    asm volatile("fence.proxy.tensormap::generic.release.gpu;" ::: "memory");
  }
}

cudaError_t launch_prologue(const int32_t *cu_seqlens, const int32_t *cu_seqlens_k, int n_seqs,
                            int Hq, int Hkv, int items_per_group, int causal,
                            const int32_t *page_table,
                            int max_pages, int num_pages, Workspace *ws,
                            const WorkspaceLayout &layout, const CUtensorMap tmpl[3],
                            cudaStream_t stream) {
  char *base = reinterpret_cast<char *>(ws);
  prologue_kernel<<<1, 1024, 0, stream>>>(
      cu_seqlens, cu_seqlens_k, n_seqs, Hq, Hkv, items_per_group, causal, page_table, max_pages, num_pages, ws,
      reinterpret_cast<int32_t *>(base + layout.seq_sorted),
      reinterpret_cast<int64_t *>(base + layout.seq_bitmap_off),
      reinterpret_cast<int32_t *>(base + layout.level_start), tmpl[0], tmpl[1], tmpl[2]);
  return cudaGetLastError();
}

// ============================================================ forward

namespace {

// K and V rings share five 32 KiB regions after the two Q tiles: 3 K + 2 V
// stages (V streams with every K)
constexpr int KST = 3, VST = 2;
constexpr uint32_t SM_Q0 = 0, SM_Q1 = kRegion, SM_K = 2 * kRegion, SM_BYTES = SM_K + 5 * kRegion;
constexpr float kRescaleLog2 = 8.0f;  // lazy O rescale once m grows by 2^8
constexpr uint32_t kColS = 0, kColO = 256;   // TMEM: S_s at s*128, O_s at 256 + s*128
// warp roles: TMA producer, MMA issuer, item fetch, then (from warp 4) the
// softmax warpgroups of query slots 0 and 1 (warp w reaches TMEM lanes 32 (w % 4) ..)
constexpr int kWarpProd = 0, kWarpMma = 1, kWarpFetch = 2, kWarpSoftmax = 4;

// barrier slots
enum : int {
  B_Q = 0,
  B_KF = 1,
  B_KE = B_KF + KST,
  B_VF = B_KE + KST,
  B_VE = B_VF + VST,
  B_SF = B_VE + VST,        // S_s computed (per slot)
  B_PRDY = B_SF + 2,        // P_s written to TMEM (S_s consumed)
  B_PV = B_PRDY + 2,        // O_s += P_s V done
  B_DRAIN = B_PV + 2,
  B_COUNT
};

// 2^x on the FMA pipe, used for part of the exponentials so that they do not
// all queue on the MUFU unit. Cody-Waite reduction to the nearest integer n
// (adding and subtracting 1.5 * 2^23), a degree-3 polynomial for 2^f on
// [-1/2, 1/2] minimising the relative error (Remez exchange, coefficients
// from fit_exp2_poly.py; at most 7.5e-5 relative error on [-125, 8]), and
// n added to the exponent field. Arguments are clamped at -126, where the
// result is a non-negative denormal below 2^-125.
constexpr float kExp2C0 = 0.9999280571937561f, kExp2C1 = 0.6932609677314758f,
                kExp2C2 = 0.2426111251115799f, kExp2C3 = 0.0551716685295105f;

__device__ __forceinline__ float exp2_fma(float x) {
  x = fmaxf(x, -126.f);
  const float t = __fadd_rn(x, 12582912.f);
  const float f = __fsub_rn(x, __fsub_rn(t, 12582912.f));
  float p = fmaf(kExp2C3, f, kExp2C2);
  p = fmaf(p, f, kExp2C1);
  p = fmaf(p, f, kExp2C0);
  return __int_as_float(__float_as_int(p) + (__float_as_int(t) << 23));
}

// Polling budget of the pipeline waits before they start to suspend: the
// single-thread MMA issuer / TMA producer, and the softmax warpgroups.
#ifndef BSA_SPIN_ISSUER
#define BSA_SPIN_ISSUER 0
#endif
#ifndef BSA_SPIN_SOFTMAX
#define BSA_SPIN_SOFTMAX 0
#endif
constexpr int kSpinIssuer = BSA_SPIN_ISSUER;

// Pass 1 loads all 128 score columns before a single TMEM wait (1), or in
// two halves of 64 with a wait each (0).
#ifndef BSA_PASS1_ONE_WAIT
#define BSA_PASS1_ONE_WAIT 0
#endif
constexpr int kSpinSoftmax = BSA_SPIN_SOFTMAX;

// One in kFmaExpEvery exponentials of a row goes to exp2_fma (0: none).
#ifndef BSA_FMA_EXP_EVERY
#define BSA_FMA_EXP_EVERY 0
#endif
constexpr int kFmaExpEvery = BSA_FMA_EXP_EVERY;

}  // namespace

template <bool FP8>
__global__ void __launch_bounds__(kFwdThreads, 1) fwd_kernel(const __grid_constant__ FwdParams p) {
  using C = Cfg<FP8>;
  constexpr uint32_t SM_V = SM_K + KST * kRegion;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar[B_COUNT];
  __shared__ uint32_t tmem_sh;
  __shared__ int item_sh[2][10];
  __shared__ volatile int abort_sh;
  // last load issued into each K stage, V stage and the Q slot (-1: none), for
  // the bounded drain after a time-out
  __shared__ int kc_last[KST], vc_last[VST], qc_last;
  // Pipeline counters, persistent across items: each role keeps its own here
  // between items and in registers within one, so that no role carries another
  // role's counters in its registers.
  //   [0, 3)    producer: Q, K, V loads
  //   [3, 6), [8, 10)  MMA warp: Q, K, V, P-ready of slots 0 / 1
  //   [12 + 4 s, 14 + 4 s)  softmax slot s: S tiles, P.V waits
  __shared__ uint32_t ctr_sh[20];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t *sptr = smem_raw + (sbase - raw);
  Workspace *ws = p.ws;
  const uint64_t limit = p.wait_limit_ns;

  if (threadIdx.x == 0) {
    for (int b = 0; b < B_COUNT; ++b)
      mbar_init(&bar[b], (b == B_PRDY || b == B_PRDY + 1) ? 4 : 1);   // P-ready: one arrival per warp
    fence_mbar_init();
    abort_sh = 0;
    for (int k = 0; k < 20; ++k) ctr_sh[k] = 0u;
    for (int st = 0; st < KST; ++st) kc_last[st] = -1;
    for (int st = 0; st < VST; ++st) vc_last[st] = -1;
    qc_last = -1;
  }
  if (threadIdx.x == kWarpFetch * 32) fetch_item(p, ws->total_items, ws->max_tiles, item_sh[0]);
  if (warp == kWarpMma) {
    tmem_alloc(&tmem_sh, 512);
    tmem_relinquish();
  }
  if ((warp == kWarpProd || warp == kWarpMma) && lane == 0) {
    tensormap_acquire(&ws->tmap[0]);
    tensormap_acquire(&ws->tmap[1]);
    tensormap_acquire(&ws->tmap[2]);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_sh;


  for (int it = 0;; ++it) {
    const int *I = item_sh[it & 1];
    if (!I[0] || abort_sh) break;
    const int s = I[1], kvh = I[2], h0 = I[3], h1 = I[4], qi = I[5], a = I[6], L = I[7];
    const int ak = I[8], Lk = I[9];
    // queries are the last L of Lk positions: query row r sits at key position off + r
    const int off = Lk - L;
    const int nq = (L + kTile - 1) / kTile, nk = (Lk + kTile - 1) / kTile;
    const int qlast = min(qi * kTile + kTile, L) - 1;   // last valid row of the query tile
    const int last = p.causal ? min((off + qlast) / kTile, nk - 1) : nk - 1;
    const bool has1 = h1 >= 0;
    // first token row of key tile j: packed K/V, or its page of the pool
    auto kv_row = [&](int j) -> int {
      return p.page_table ? p.page_table[(size_t)s * p.max_pages + j] * kTile : ak + j * kTile;
    };
    bool ok = true;

    if (warp == kWarpProd) {
      if (lane == 0) {
        // ------------------------------------------------ TMA producer
        uint32_t qc = ctr_sh[0], kc = ctr_sh[1], vc = ctr_sh[2];
        const void *tq = &ws->tmap[0], *tk = &ws->tmap[1], *tv = &ws->tmap[2];
        mbar_expect_tx(&bar[B_Q], (has1 ? 2 : 1) * C::kTileBytes);
        for (int b = 0; b < C::kBoxes; ++b) {
          tma_load_3d(sptr + SM_Q0 + b * kBox, tq, &bar[B_Q], b * C::kBoxCols, h0, a + qi * kTile);
          if (has1)
            tma_load_3d(sptr + SM_Q1 + b * kBox, tq, &bar[B_Q], b * C::kBoxCols, h1,
                        a + qi * kTile);
        }
        qc_last = (int)qc++;
        for (int j = 0; j <= last && ok; ++j) {
          const uint32_t st = kc % KST;
          ok = mbar_wait(&bar[B_KE + st], ((kc / KST) & 1) ^ 1, limit, kSpinIssuer);
          if (!ok) break;
          if ((int)kc != p.debug_drop_k_load) {
            mbar_expect_tx(&bar[B_KF + st], C::kTileBytes);
            for (int b = 0; b < C::kBoxes; ++b)
              tma_load_3d(sptr + SM_K + st * kRegion + b * kBox, tk, &bar[B_KF + st],
                          b * C::kBoxCols, kvh, kv_row(j));
            kc_last[st] = (int)kc;
          }
          ++kc;
          const uint32_t vs = vc % VST;   // V streams with K: every tile is kept
          ok = mbar_wait(&bar[B_VE + vs], ((vc / VST) & 1) ^ 1, limit, kSpinIssuer);
          if (!ok) break;
          mbar_expect_tx(&bar[B_VF + vs], C::kTileBytes);
          for (int b = 0; b < C::kBoxes; ++b)
            tma_load_3d(sptr + SM_V + vs * kRegion + b * kBox, tv, &bar[B_VF + vs],
                        b * C::kBoxCols, kvh, kv_row(j));
          vc_last[vs] = (int)vc;
          ++vc;
        }
        ctr_sh[0] = qc;
        ctr_sh[1] = kc;
        ctr_sh[2] = vc;
      }
    } else if (warp == kWarpMma) {
      if (lane == 0) {
        // ------------------------------------------------ MMA issuer
        uint32_t qc = ctr_sh[3], kc = ctr_sh[4], vc = ctr_sh[5];
        uint32_t pr0 = ctr_sh[8], pr1 = ctr_sh[9];
        const uint32_t S0 = tmem + kColS, S1 = tmem + kColS + 128;
        const uint32_t O0 = tmem + kColO, O1 = tmem + kColO + 128;
        const uint32_t q0s = sbase + SM_Q0, q1s = sbase + SM_Q1;
        do {
          ok = mbar_wait(&bar[B_Q], qc & 1, limit, kSpinIssuer);
          ++qc;
          if (!ok) break;
          uint32_t st = kc % KST;
          ok = mbar_wait(&bar[B_KF + st], (kc / KST) & 1, limit, kSpinIssuer);
          if (!ok) break;
          tc_fence_after();
          uint32_t ks = sbase + SM_K + st * kRegion;
          issue_qk<FP8>(S0, q0s, ks);
          mma_commit(&bar[B_SF + 0]);
          if (has1) {
            issue_qk<FP8>(S1, q1s, ks);
            mma_commit(&bar[B_SF + 1]);
          }
          mma_commit(&bar[B_KE + st]);
          ++kc;
          bool oinit0 = false, oinit1 = false;
          for (int j = 0; j <= last && ok; ++j) {
            bool vready = false;   // V_j landed (waited)
            const uint32_t vs = vc % VST;
            auto wait_v = [&]() -> bool {
              if (vready) return true;
              if (!mbar_wait(&bar[B_VF + vs], (vc / VST) & 1, limit, kSpinIssuer)) return false;
              tc_fence_after();
              vready = true;
              return true;
            };
            // ---- slot 0: P.V before the next S overwrites P
            {
              ok = mbar_wait(&bar[B_PRDY + 0], pr0 & 1, limit, kSpinIssuer);
              ++pr0;
              if (!ok || !(ok = wait_v())) break;
              tc_fence_after();
              issue_pv<FP8>(O0, S0, sbase + SM_V + vs * kRegion, oinit0);
              oinit0 = true;
              mma_commit(&bar[B_PV + 0]);
            }
            if (j < last) {
              st = kc % KST;
              ok = mbar_wait(&bar[B_KF + st], (kc / KST) & 1, limit, kSpinIssuer);
              if (!ok) break;
              tc_fence_after();
              ks = sbase + SM_K + st * kRegion;
              issue_qk<FP8>(S0, q0s, ks);
              mma_commit(&bar[B_SF + 0]);
            }
            // ---- slot 1
            if (has1) {
              {
                ok = mbar_wait(&bar[B_PRDY + 1], pr1 & 1, limit, kSpinIssuer);
                ++pr1;
                if (!ok || !(ok = wait_v())) break;
                tc_fence_after();
                issue_pv<FP8>(O1, S1, sbase + SM_V + vs * kRegion, oinit1);
                oinit1 = true;
                mma_commit(&bar[B_PV + 1]);
              }
              if (j < last) {
                issue_qk<FP8>(S1, q1s, ks);
                mma_commit(&bar[B_SF + 1]);
              }
            }
            if (j < last) {
              mma_commit(&bar[B_KE + st]);
              ++kc;
            }
            if (!(ok = wait_v())) break;
            mma_commit(&bar[B_VE + vs]);
            ++vc;
          }
        } while (false);
        ctr_sh[3] = qc;
        ctr_sh[4] = kc;
        ctr_sh[5] = vc;
        ctr_sh[8] = pr0;
        ctr_sh[9] = pr1;
      }
    } else if (warp == kWarpFetch) {
      if (lane == 0) fetch_item(p, ws->total_items, ws->max_tiles, item_sh[(it + 1) & 1]);
    } else if (warp >= kWarpSoftmax) {
      // -------------------------------------------------- softmax warpgroups
      const int slot = (warp - kWarpSoftmax) >> 2;
      const int h = slot ? h1 : h0;
      if (h >= 0) {
        const int row = threadIdx.x & 127;   // = TMEM lane
        uint32_t sc = ctr_sh[12 + 4 * slot], pvc = ctr_sh[13 + 4 * slot];
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + kColS + slot * 128 + lane_off;
        const uint32_t tO = tmem + kColO + slot * 128 + lane_off;
        const bool valid = qi * kTile + row < L;
        const bool tail = !p.causal && (Lk % kTile) != 0;
        float c = p.c;
        if (FP8) c *= p.q_scale[h] * p.k_scale[kvh];
        const int W = (nk + 31) >> 5;
        // this row's skip-bitmap words
        uint32_t *const brow =
            p.bitmap ? p.bitmap + p.seq_bitmap_off[s] + ((long long)h * nq + qi) * W : nullptr;
        const int doff0 = off + qi * kTile;   // row r of key tile j sees columns <= r + doff0 - 128 j
        float m2 = -INFINITY, mref = 0.f, l = 0.f;
        uint32_t word = 0;
        bool have_kept = false;

        for (int j = 0; j <= last; ++j) {
          if (!abort_sh && !mbar_wait(&bar[B_SF + slot], sc & 1, limit, kSpinSoftmax)) abort_sh = 1;
          ++sc;
          tc_fence_after();
          const int doff = doff0 - j * kTile;   // row r sees columns <= r + doff
          const bool diag = p.causal && doff < kTile - 1;
          const bool tailt = tail && j == nk - 1;
          if (have_kept) {
            // ---- after the first tile: one pass over S. P is
            // computed against the current reference max while the row max is
            // taken; only when a row's max outgrows the reference by more than
            // 2^8 is O rescaled and the tile's P recomputed (S is still intact:
            // P is stored at the end).
            if (!abort_sh && !mbar_wait(&bar[B_PV + slot], pvc & 1, limit)) abort_sh = 1;
            ++pvc;
            tc_fence_after();
            constexpr int kPk = FP8 ? 8 : 16;   // packed words per 32-key chunk
            uint32_t pk[4][kPk];
            float psum[8];
            auto exp_pass = [&](float nm, bool track, float &tm) {
              uint32_t vnext[32];
#pragma unroll
              for (int k = 0; k < 8; ++k) psum[k] = 0.f;
              float tmx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
              for (int ch = 0; ch < 4; ++ch) {
                uint32_t v[32];
                if ((ch & 1) == 0) {   // chunks 2h, 2h + 1 in one 64-column load
                  tmem_ld64(tS + ch * 32, v, vnext);
                  tmem_wait_ld(v);
                  reg_fence(vnext);
                } else {
#pragma unroll
                  for (int e = 0; e < 32; ++e) v[e] = vnext[e];
                }
                if (diag || tailt) mask_chunk(v, ch, diag, tailt, row, doff, j * kTile, Lk);
                float pv[32];
                const uint64_t c2 = f2_pack(c, c), nm2 = f2_pack(nm, nm);
                uint64_t ps2[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) ps2[k] = f2_pack(psum[2 * k], psum[2 * k + 1]);
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                  const float x0 = __uint_as_float(v[e]), x1 = __uint_as_float(v[e + 1]);
                  if (track) tmx[(e >> 1) & 3] = max3f(tmx[(e >> 1) & 3], x0, x1);
                  float y0, y1;
                  f2_unpack(f2_fma(f2_pack(x0, x1), c2, nm2), y0, y1);
                  pv[e] = ex2_approx(y0);
                  pv[e + 1] = ex2_approx(y1);
                  ps2[(e >> 1) & 3] = f2_add(ps2[(e >> 1) & 3], f2_pack(pv[e], pv[e + 1]));
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) f2_unpack(ps2[k], psum[2 * k], psum[2 * k + 1]);
#pragma unroll
                for (int k = 0; k < kPk; ++k) {
                  if (FP8)
                    pk[ch][k] = (uint32_t)pack_e4m3x2(pv[4 * k], pv[4 * k + 1]) |
                                ((uint32_t)pack_e4m3x2(pv[4 * k + 2], pv[4 * k + 3]) << 16);
                  else
                    pk[ch][k] = pack_bf16x2(pv[2 * k], pv[2 * k + 1]);
                }
              }
              if (track) tm = fmaxf(fmaxf(tmx[0], tmx[1]), fmaxf(tmx[2], tmx[3]));
            };
            float rmax = -INFINITY;
            exp_pass(valid ? -mref : -INFINITY, true, rmax);
            const float mnew = valid ? fmaxf(m2, rmax * c) : 0.f;
            const bool need = valid && (mnew - mref > kRescaleLog2);
            if (__any_sync(0xffffffffu, need)) {
              const float alpha = need ? ex2_approx(mref - mnew) : 1.f;
              l *= alpha;
              if (need) mref = mnew;
#pragma unroll
              for (int ch = 0; ch < 4; ++ch) {
                uint32_t v[32];
                tmem_ld32(tO + ch * 32, v);
                tmem_wait_ld(v);
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
                tmem_st32(tO + ch * 32, v);
              }
              float unused;
              exp_pass(valid ? -mref : -INFINITY, false, unused);
            }
            m2 = mnew;
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) {
              if (FP8)
                tmem_st8(tS + ch * 8, reinterpret_cast<const uint32_t(&)[8]>(pk[ch]));
              else
                tmem_st16(tS + ch * 16, reinterpret_cast<const uint32_t(&)[16]>(pk[ch]));
            }
            tmem_wait_st();
            l += ((psum[0] + psum[1]) + (psum[2] + psum[3])) + ((psum[4] + psum[5]) + (psum[6] + psum[7]));
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[B_PRDY + slot]);   // this warp's 32 rows of P
            if (abort_sh) {
              ok = false;
              break;
            }
            if (row == 0 && brow && (((j & 31) == 31) || j == last)) {
              brow[j >> 5] = word;
              word = 0;
            }
            continue;
          }
          float rm;
          {
            float acc[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) acc[k] = -INFINITY;
#if BSA_PASS1_ONE_WAIT
            uint32_t v0[32], v1[32], v2[32], v3[32];
            tmem_ld32(tS + 0, v0);
            tmem_ld32(tS + 32, v1);
            tmem_ld32(tS + 64, v2);
            tmem_ld32(tS + 96, v3);
            tmem_wait_ld(v0);
            reg_fence(v1);
            reg_fence(v2);
            reg_fence(v3);
            if (diag || tailt) {
              mask_chunk(v0, 0, diag, tailt, row, doff, j * kTile, Lk);
              mask_chunk(v1, 1, diag, tailt, row, doff, j * kTile, Lk);
              mask_chunk(v2, 2, diag, tailt, row, doff, j * kTile, Lk);
              mask_chunk(v3, 3, diag, tailt, row, doff, j * kTile, Lk);
            }
            row_max64(acc, v0, v1);
            row_max64(acc, v2, v3);
#else
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              uint32_t v0[32], v1[32];
              tmem_ld64(tS + half * 64, v0, v1);
              tmem_wait_ld(v0);
              reg_fence(v1);
              if (diag || tailt) {
                mask_chunk(v0, 2 * half, diag, tailt, row, doff, j * kTile, Lk);
                mask_chunk(v1, 2 * half + 1, diag, tailt, row, doff, j * kTile, Lk);
              }
              row_max64(acc, v0, v1);
            }
#endif
            rm = max3f(max3f(acc[0], acc[1], acc[2]), max3f(acc[3], acc[4], acc[5]),
                       fmaxf(acc[6], acc[7]));
          }
          // ---- the first tile: the row max first, then P against it
          {
            const float mnew = valid ? rm * c : 0.f;
            mref = mnew;
            m2 = mnew;
            // P = exp2(S c - m_ref), written over the S columns already read:
            // chunk ch (keys 32ch..32ch+31) goes to columns 16ch.. (bf16) or 8ch.. (e4m3)
            // rows past the end of the queries: scores of -inf give P = 0
            const float nm = valid ? -mref : -INFINITY;
            float psum[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) psum[k] = 0.f;
            {
              uint32_t va[32], vb[32];
              tmem_ld32(tS, va);
              tmem_wait_ld(va);
#pragma unroll
              for (int ch = 0; ch < 4; ++ch) {
                uint32_t(&v)[32] = (ch & 1) ? vb : va;
                uint32_t(&nxt)[32] = (ch & 1) ? va : vb;
                if (ch < 3) tmem_ld32(tS + (ch + 1) * 32, nxt);   // overlaps this chunk's math
                if (diag || tailt) mask_chunk(v, ch, diag, tailt, row, doff, j * kTile, Lk);
                // p = exp2(s c - m_ref), packed as it is produced
                auto pexp = [&](int e) -> float {
                  const float xe = fmaf(__uint_as_float(v[e]), c, nm);
                  const bool on_fma = kFmaExpEvery > 0 && (e % (kFmaExpEvery > 0 ? kFmaExpEvery : 1)) ==
                                                              (kFmaExpEvery > 0 ? kFmaExpEvery - 1 : 0);
                  const float pv = on_fma ? exp2_fma(xe) : ex2_approx(xe);
                  psum[e & 7] += pv;
                  return pv;
                };
                if (FP8) {
                  uint32_t w8[8];
#pragma unroll
                  for (int k = 0; k < 8; ++k) {
                    const float p0 = pexp(4 * k), p1 = pexp(4 * k + 1);
                    const float p2 = pexp(4 * k + 2), p3 = pexp(4 * k + 3);
                    w8[k] = (uint32_t)pack_e4m3x2(p0, p1) | ((uint32_t)pack_e4m3x2(p2, p3) << 16);
                  }
                  tmem_st8(tS + ch * 8, w8);
                } else {
                  uint32_t w2[16];
#pragma unroll
                  for (int k = 0; k < 16; ++k) {
                    const float p0 = pexp(2 * k), p1 = pexp(2 * k + 1);
                    w2[k] = pack_bf16x2(p0, p1);
                  }
                  tmem_st16(tS + ch * 16, w2);
                }
                if (ch < 3) tmem_wait_ld(nxt);
              }
            }
            const float sum = ((psum[0] + psum[1]) + (psum[2] + psum[3])) +
                              ((psum[4] + psum[5]) + (psum[6] + psum[7]));
            tmem_wait_st();
            l += sum;
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[B_PRDY + slot]);
            if (abort_sh) {
              ok = false;
              break;
            }
            have_kept = true;
          }
          if (row == 0 && brow && (((j & 31) == 31) || j == last)) {
            brow[j >> 5] = word;
            word = 0;
          }
        }
        // ------------------------------------------------ epilogue
        if (ok && have_kept) {
          if (!mbar_wait(&bar[B_PV + slot], pvc & 1, limit)) abort_sh = 1;
          ++pvc;
          tc_fence_after();
          // the item's fields again from shared memory (not kept in registers
          // through the tile loop)
          const volatile int *Iv = item_sh[it & 1];
          const int ea = Iv[6], eh = Iv[3 + slot], ekvh = Iv[2];
          const int tok = ea + Iv[5] * kTile + row;   // this row's query token
          float inv = 0.f;
          if (valid && l > 0.f) inv = (FP8 ? p.v_scale[ekvh] : 1.f) / l;
          __nv_bfloat16 *orow = reinterpret_cast<__nv_bfloat16 *>(p.out) +
                                ((size_t)tok * p.Hq + eh) * kHeadDim;
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            uint32_t v[32];
            tmem_ld32(tO + ch * 32, v);
            tmem_wait_ld(v);
            uint32_t w2[16];
#pragma unroll
            for (int k = 0; k < 16; ++k)
              w2[k] = pack_bf16x2(__uint_as_float(v[2 * k]) * inv,
                                  __uint_as_float(v[2 * k + 1]) * inv);
            if (valid) {
              uint4 *dst = reinterpret_cast<uint4 *>(orow + ch * 32);
#pragma unroll
              for (int q = 0; q < 4; ++q)
                dst[q] = make_uint4(w2[4 * q], w2[4 * q + 1], w2[4 * q + 2], w2[4 * q + 3]);
            }
          }
          if (valid && p.lse) p.lse[(size_t)eh * ws->total_tokens + tok] = (mref + log2f(l)) * kLn2;
          if (row == 0 && brow)
            for (int w = (last >> 5) + 1; w < W; ++w) brow[w] = 0u;
        }
        if (row == 0) {   // uniform over the warpgroup; read by all at the next item's start
          ctr_sh[12 + 4 * slot] = sc;
          ctr_sh[13 + 4 * slot] = pvc;
        }
      }
    }
    if (!ok) abort_sh = 1;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (abort_sh && threadIdx.x == 0) atomicOr(&ws->status, kStatusTimeout);
  }

  // Normal exit: every item ended fully drained. After a time-out, wait
  // (bounded) for this CTA's own copies and MMAs before giving TMEM back.
  if (abort_sh) {
    if ((warp == kWarpProd || warp == kWarpMma) && lane == 0) {
      for (int st = 0; st < KST; ++st)
        if (warp == kWarpProd && kc_last[st] >= 0)
          mbar_wait(&bar[B_KF + st], (kc_last[st] / KST) & 1, limit);
      for (int st = 0; st < VST; ++st)
        if (vc_last[st] >= 0) mbar_wait(&bar[B_VF + st], (vc_last[st] / VST) & 1, limit);
      if (warp == kWarpProd && qc_last >= 0) mbar_wait(&bar[B_Q], qc_last & 1, limit);
    }
    if (warp == kWarpMma && lane == 0) {
      mma_commit(&bar[B_DRAIN]);
      mbar_wait(&bar[B_DRAIN], 0, limit);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpMma) tmem_dealloc(tmem, 512);
}

size_t forward_smem_bytes() { return SM_BYTES + 1024; }

cudaError_t launch_forward(const FwdParams &p, bool fp8, int num_ctas, cudaStream_t stream) {
  const size_t smem = forward_smem_bytes();
  if (fp8)
    fwd_kernel<true><<<num_ctas, kFwdThreads, smem, stream>>>(p);
  else
    fwd_kernel<false><<<num_ctas, kFwdThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t prepare_forward() {
  const int smem = (int)forward_smem_bytes();
  const cudaFuncAttribute a = cudaFuncAttributeMaxDynamicSharedMemorySize;
  cudaError_t e = cudaFuncSetAttribute(fwd_kernel<false>, a, smem);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(fwd_kernel<true>, a, smem);
  return e;
}

}  // namespace bsa
