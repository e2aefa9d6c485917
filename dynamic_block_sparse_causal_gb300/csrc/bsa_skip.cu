// Block-skipping causal prefill attention with lambda > 0: two-phase kernel
// for sm_103a.
//
// Operation: dynamic sparse attention deployment guide
// ("长上下文推理加速方案部署实战：基于动态稀疏注意力机制的推理服务优化指南"),
// §3.2 -- key blocks in order, a block whose local max score falls below the
// running max by more than the threshold gets no exponentials, no V load and
// no P.V product; read as tile_max < running_max + ln(lambda) per row, AND-ed
// over the 128 rows of the query tile (§3.3 / §6.1 fix the direction).
//
// For lambda < 1 a skipped tile never raises the running max
// (tile_max < m + ln lambda < m), so the running max before key tile j is the
// prefix max of the earlier tiles' row maxima, whatever was skipped, and
// every decision follows from the row maxima alone. A work item (sequence,
// KV head, two query heads of the group, query tile i) therefore runs in two
// phases on one CTA:
//
//  1. scan: S = Q K^T for every causal key tile, two key tiles per MMA
//     (M = 128, N = 256), the masked row max, the prefix max and the vote.
//     The MMA issuer waits only for S to have been read, never for a vote,
//     so the tensor pipe streams QK^T back to back. Keep bits go to shared
//     memory (and to the caller's skip bitmap).
//  2. kept tiles, in order: S again, P = exp2(S c - m) against the final row
//     max m of phase 1 (the largest kept tile max, so there is never a
//     rescale), l += sum P, O += P V with P read from TMEM; then out = O / l
//     and lse = ln 2 (m + log2 l). V is loaded for kept tiles only.
//
// Roles (384 threads): warp 0 lane 0 TMA producer, warp 1 lane 0 MMA
// issuer, warp 2 lane 0 work-item fetch, warps 4-7 / 8-11 the warpgroups of
// query slots 0 / 1 (TMEM lane = query row). The control warpgroup hands
// registers to the slot warpgroups (setmaxnreg).
//
// TMEM: slot s owns columns [256 s, 256 s + 256): the two scanned S tiles in
// phase 1; S (first 128, P written over it) and O (last 128) in phase 2.
// Shared memory: Q0, Q1, a ring of stages (two key tiles in phase 1, one K
// and one V tile in phase 2; 2 stages bf16, 5 stages FP8) and the keep
// words of both slots (one bit per key tile, up to 65536 tiles).
#include <cuda_bf16.h>

#include <climits>
#include <cmath>

#include "bsa_internal.h"
#include "bsa_tile.cuh"
#include "ptx.cuh"

namespace bsa {

using namespace tile;

namespace {

constexpr int kKeepWords = kMaxLevels / 32;   // keep bits of one slot: a bit per key tile

template <bool FP8>
struct SkipCfg {
  static constexpr uint32_t kQBytes = Cfg<FP8>::kTileBytes;     // one Q tile
  static constexpr uint32_t kStageBytes = 2 * Cfg<FP8>::kTileBytes;  // 2 K tiles, or K + V
  static constexpr int kStages = FP8 ? 5 : 2;
  static constexpr uint32_t kSmStage = 2 * kQBytes;
  static constexpr uint32_t kSmKeep = kSmStage + kStages * kStageBytes;
  static constexpr uint32_t kSmBytes = kSmKeep + 2 * kKeepWords * 4;
  static constexpr uint32_t kIdescPair = IDesc<FP8 ? 0 : 1, false, 128, 256>::value;
};
constexpr int kMaxStages = 5;

enum : int {
  SB_Q = 0,
  SB_F = 1,                     // stage full (TMA bytes landed)
  SB_E = SB_F + kMaxStages,     // stage free (MMAs that read it done)
  SB_SF = SB_E + kMaxStages,    // S_s written (per slot)
  SB_SE = SB_SF + 2,            // scanned S_s read by the slot's warpgroup (4 arrivals)
  SB_DEC = SB_SE + 2,           // slot s's keep bits complete
  SB_PRDY = SB_DEC + 2,         // P_s in TMEM (4 arrivals)
  SB_OD = SB_PRDY + 2,          // the slot's last P.V done: O_s final
  SB_DRAIN = SB_OD + 2,
  SB_COUNT
};

// Warp roles: TMA producer, MMA issuer, item fetch (warp 3 idle), then the
// two slot warpgroups (warps 4-7 and 8-11; warp w reaches TMEM lanes
// 32 (w % 4) .. 32 (w % 4) + 31).
constexpr int kWarpProd = 0, kWarpMma = 1, kWarpFetch = 2, kWarpSoftmax = 4;
constexpr int kSkipThreads = 384;
// Register split: launched at 168 per thread (384 x 168 = 64512), the
// control warpgroup gives back down to 96 and the two slot warpgroups take
// 200 each: 128 x 96 + 256 x 200 = 63488 <= 64512, and per SM sub-partition
// (one control and two slot warps) 32 x (96 + 2 x 200) = 15872 <= 16384.
// prepare_skip() checks that the kernels were built with 168 per thread.
constexpr uint32_t kRegsLaunch = 168, kRegsControl = 96, kRegsSlot = 200;
static_assert(128 * kRegsControl + 256 * kRegsSlot <= kSkipThreads * kRegsLaunch,
              "register split exceeds the launch allocation");

// Phase 1 MMA: S (128 x 256) = Q K^T over a stage holding key tiles j, j + 1.
// bf16 stage: [box 0 of tile j][box 0 of tile j+1][box 1 of j][box 1 of j+1]
// (16 KiB boxes of 128 rows x 128 bytes), so K step kk reads the 256 key rows
// contiguously from half kk / 4. FP8 stage: [tile j][tile j+1]. A single last
// tile is an N = 128 MMA over the same addresses.
template <bool FP8>
__device__ __forceinline__ void issue_qk_pair(uint32_t d, uint32_t qs, uint32_t ks, bool two) {
  const uint32_t idesc = two ? SkipCfg<FP8>::kIdescPair : Cfg<FP8>::kIdescQK;
#pragma unroll
  for (int kk = 0; kk < Cfg<FP8>::kSteps; ++kk) {
    const uint32_t aoff = FP8 ? kk * 32 : (kk >> 2) * kBox + (kk & 3) * 32;
    const uint32_t boff = FP8 ? kk * 32 : (kk >> 2) * (2 * kBox) + (kk & 3) * 32;
    const uint64_t a = sdesc_sw128(qs + aoff, 16, 1024);
    const uint64_t b = sdesc_sw128(ks + boff, 16, 1024);
    if (FP8)
      mma_f8_ss(d, a, b, idesc, kk > 0);
    else
      mma_f16_ss(d, a, b, idesc, kk > 0);
  }
}

// Smallest key tile > j (and <= last) whose bit is set in `words`; last + 1
// if none.
__device__ __forceinline__ int next_set(const volatile uint32_t *words, int j, int last) {
  for (int t = j + 1; t <= last;) {
    const int w = t >> 5;
    const uint32_t m = words[w] & (~0u << (t & 31));
    if (m) {
      const int c = (w << 5) + __ffs(m) - 1;
      return c <= last ? c : last + 1;
    }
    t = (w + 1) << 5;
  }
  return last + 1;
}

// Same over the union of two slots' keep words.
__device__ __forceinline__ int next_union(const volatile uint32_t *a, const volatile uint32_t *b,
                                          int j, int last) {
  for (int t = j + 1; t <= last;) {
    const int w = t >> 5;
    const uint32_t m = (a[w] | b[w]) & (~0u << (t & 31));
    if (m) {
      const int c = (w << 5) + __ffs(m) - 1;
      return c <= last ? c : last + 1;
    }
    t = (w + 1) << 5;
  }
  return last + 1;
}

__device__ __forceinline__ bool bit_set(const volatile uint32_t *words, int j) {
  return (words[j >> 5] >> (j & 31)) & 1u;
}

// Masked row max of the 64 columns in (v0, v1) (chunks 2h, 2h + 1 of a key
// tile), folded into acc.
__device__ __forceinline__ void max_half(float (&acc)[8], uint32_t (&v0)[32], uint32_t (&v1)[32],
                                         int h, bool diag, bool tailt, int row, int doff, int key0,
                                         int Lk) {
  if (diag || tailt) {
    mask_chunk(v0, 2 * h, diag, tailt, row, doff, key0, Lk);
    mask_chunk(v1, 2 * h + 1, diag, tailt, row, doff, key0, Lk);
  }
  row_max64(acc, v0, v1);
}

__device__ __forceinline__ float fold8(const float (&a)[8]) {
  return max3f(max3f(a[0], a[1], a[2]), max3f(a[3], a[4], a[5]), fmaxf(a[6], a[7]));
}

}  // namespace

template <bool FP8>
__global__ void __launch_bounds__(kSkipThreads, 1) skip_kernel(const __grid_constant__ FwdParams p) {
  using C = Cfg<FP8>;
  using K = SkipCfg<FP8>;
  constexpr int ST = K::kStages;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar[SB_COUNT];
  __shared__ uint32_t tmem_sh;
  __shared__ int item_sh[2][10];
  __shared__ volatile int abort_sh;
  __shared__ int kc_last[kMaxStages], qc_last;   // last load into each stage / the Q slot
  // pipeline counters kept between work items, one set per role:
  //   [0, 4) producer: Q, stages, decision waits of slots 0 / 1
  //   [4, 12) MMA warp: Q, stages, scanned S of slots 0 / 1, P-ready of slots 0 / 1,
  //           decision waits of slots 0 / 1
  //   [12 + 2 s, 14 + 2 s) warpgroup s: S-full waits, O-done waits
  __shared__ uint32_t ctr_sh[16];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t *sptr = smem_raw + (sbase - raw);
  // keep words of slot s: keep_w + s * kKeepWords
  volatile uint32_t *const keep_w = reinterpret_cast<volatile uint32_t *>(sptr + K::kSmKeep);
  Workspace *ws = p.ws;
  const uint64_t limit = p.wait_limit_ns;

  if (threadIdx.x == 0) {
    for (int b = 0; b < SB_COUNT; ++b) {
      const bool four = (b == SB_SE || b == SB_SE + 1 || b == SB_PRDY || b == SB_PRDY + 1);
      mbar_init(&bar[b], four ? 4 : 1);   // one arrival per warp of a warpgroup
    }
    fence_mbar_init();
    abort_sh = 0;
    for (int k = 0; k < 16; ++k) ctr_sh[k] = 0u;
    for (int st = 0; st < kMaxStages; ++st) kc_last[st] = -1;
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
  // The control warpgroup and the slot warpgroups run the same item loop in
  // separate code, so each is register-allocated for its own budget.
  if (warp < kWarpSoftmax) {
    reg_dealloc<kRegsControl>();
  for (int it = 0;; ++it) {
    const int *I = item_sh[it & 1];
    if (!I[0] || abort_sh) break;
    const int s = I[1], kvh = I[2], h0 = I[3], h1 = I[4], qi = I[5], a = I[6], L = I[7];
    const int ak = I[8], Lk = I[9];
    const int off = Lk - L;   // query row r sits at key position off + r
    const int nk = (Lk + kTile - 1) / kTile;
    const int qlast = min(qi * kTile + kTile, L) - 1;
    const int last = p.causal ? min((off + qlast) / kTile, nk - 1) : nk - 1;
    const int npairs = (last + 2) >> 1;
    const bool has1 = h1 >= 0;
    auto kv_row = [&](int j) -> int {
      return p.page_table ? p.page_table[(size_t)s * p.max_pages + j] * kTile : ak + j * kTile;
    };
    bool ok = true;
    if (warp == kWarpProd) {
      if (lane == 0) {
        // ------------------------------------------------ TMA producer
        uint32_t qc = ctr_sh[0], kc = ctr_sh[1], dc0 = ctr_sh[2], dc1 = ctr_sh[3];
        const void *tq = &ws->tmap[0], *tk = &ws->tmap[1], *tv = &ws->tmap[2];
        mbar_expect_tx(&bar[SB_Q], (has1 ? 2 : 1) * K::kQBytes);
        for (int b = 0; b < C::kBoxes; ++b) {
          tma_load_3d(sptr + b * kBox, tq, &bar[SB_Q], b * C::kBoxCols, h0, a + qi * kTile);
          if (has1)
            tma_load_3d(sptr + K::kQBytes + b * kBox, tq, &bar[SB_Q], b * C::kBoxCols, h1,
                        a + qi * kTile);
        }
        qc_last = (int)qc++;
        // next stage, once the MMAs that read its previous contents are done
        auto acquire = [&](uint32_t &st) -> bool {
          st = kc % ST;
          return mbar_wait(&bar[SB_E + st], ((kc / ST) & 1) ^ 1, limit);
        };
        // phase 1: key tiles in pairs
        for (int pr = 0; pr < npairs && ok; ++pr) {
          uint32_t st;
          if (!(ok = acquire(st))) break;
          const int n = (2 * pr + 1 <= last) ? 2 : 1;
          if ((int)kc != p.debug_drop_k_load) {
            mbar_expect_tx(&bar[SB_F + st], n * C::kTileBytes);
            uint8_t *dst = sptr + K::kSmStage + st * K::kStageBytes;
            for (int t = 0; t < n; ++t)
              for (int b = 0; b < C::kBoxes; ++b)
                tma_load_3d(dst + b * 2 * kBox + t * (FP8 ? C::kTileBytes : kBox), tk,
                            &bar[SB_F + st], b * C::kBoxCols, kvh, kv_row(2 * pr + t));
            kc_last[st] = (int)kc;
          }
          ++kc;
        }
        // phase 2: K and V of the kept tiles. Tile 0 is kept by every row (the
        // running max starts at -inf), so it is loaded before the decisions.
        auto load_kv = [&](int j) -> bool {
          uint32_t st;
          if (!acquire(st)) return false;
          if ((int)kc != p.debug_drop_k_load) {
            mbar_expect_tx(&bar[SB_F + st], 2 * C::kTileBytes);
            uint8_t *dst = sptr + K::kSmStage + st * K::kStageBytes;
            for (int b = 0; b < C::kBoxes; ++b) {
              tma_load_3d(dst + b * kBox, tk, &bar[SB_F + st], b * C::kBoxCols, kvh, kv_row(j));
              tma_load_3d(dst + C::kTileBytes + b * kBox, tv, &bar[SB_F + st], b * C::kBoxCols,
                          kvh, kv_row(j));
            }
            kc_last[st] = (int)kc;
          }
          ++kc;
          return true;
        };
        if (ok) ok = load_kv(0);
        if (ok) ok = mbar_wait(&bar[SB_DEC + 0], dc0++ & 1, limit);
        if (ok && has1) ok = mbar_wait(&bar[SB_DEC + 1], dc1++ & 1, limit);
        const volatile uint32_t *k1w = has1 ? keep_w + kKeepWords : keep_w;
        for (int j = next_union(keep_w, k1w, 0, last); ok && j <= last;
             j = next_union(keep_w, k1w, j, last))
          ok = load_kv(j);
        ctr_sh[0] = qc;
        ctr_sh[1] = kc;
        ctr_sh[2] = dc0;
        ctr_sh[3] = dc1;
      }
    } else if (warp == kWarpMma) {
      if (lane == 0) {
        // ------------------------------------------------ MMA issuer
        uint32_t qc = ctr_sh[4], kc = ctr_sh[5], se0 = ctr_sh[6], se1 = ctr_sh[7];
        uint32_t pr0 = ctr_sh[8], pr1 = ctr_sh[9], dc0 = ctr_sh[10], dc1 = ctr_sh[11];
        const uint32_t q0s = sbase, q1s = sbase + K::kQBytes;
        const uint32_t T0 = tmem, T1 = tmem + 256;   // slot columns
        auto stage_addr = [&](uint32_t st) { return sbase + K::kSmStage + st * K::kStageBytes; };
        do {
          ok = mbar_wait(&bar[SB_Q], qc & 1, limit);
          ++qc;
          if (!ok) break;
          // ---- phase 1: every causal key tile, two per MMA
          for (int pr = 0; pr < npairs; ++pr) {
            const bool two = 2 * pr + 1 <= last;
            const uint32_t st = kc % ST;
            if (!(ok = mbar_wait(&bar[SB_F + st], (kc / ST) & 1, limit))) break;
            if (!(ok = mbar_wait(&bar[SB_SE + 0], (se0 & 1) ^ 1, limit))) break;
            tc_fence_after();
            issue_qk_pair<FP8>(T0, q0s, stage_addr(st), two);
            mma_commit(&bar[SB_SF + 0]);
            ++se0;
            if (has1) {
              if (!(ok = mbar_wait(&bar[SB_SE + 1], (se1 & 1) ^ 1, limit))) break;
              tc_fence_after();
              issue_qk_pair<FP8>(T1, q1s, stage_addr(st), two);
              mma_commit(&bar[SB_SF + 1]);
              ++se1;
            }
            mma_commit(&bar[SB_E + st]);
            ++kc;
          }
          if (!ok) break;
          // ---- phase 2: S of tile 0 (kept by every row) as soon as the last
          // scanned S of the slot has been read, then the kept tiles in order
          uint32_t st = kc % ST;
          if (!(ok = mbar_wait(&bar[SB_F + st], (kc / ST) & 1, limit))) break;
          if (!(ok = mbar_wait(&bar[SB_SE + 0], (se0 & 1) ^ 1, limit))) break;
          tc_fence_after();
          issue_qk<FP8>(T0, q0s, stage_addr(st));
          mma_commit(&bar[SB_SF + 0]);
          if (has1) {
            if (!(ok = mbar_wait(&bar[SB_SE + 1], (se1 & 1) ^ 1, limit))) break;
            tc_fence_after();
            issue_qk<FP8>(T1, q1s, stage_addr(st));
            mma_commit(&bar[SB_SF + 1]);
          }
          ok = mbar_wait(&bar[SB_DEC + 0], dc0++ & 1, limit);
          if (ok && has1) ok = mbar_wait(&bar[SB_DEC + 1], dc1++ & 1, limit);
          if (!ok) break;
          const volatile uint32_t *w0 = keep_w, *w1 = has1 ? keep_w + kKeepWords : keep_w;
          bool acc0 = false, acc1 = false;
          for (int j = 0; j <= last;) {
            const int jn = next_union(w0, w1, j, last);
            const bool more = jn <= last;
            const uint32_t vs = stage_addr(st) + C::kTileBytes;
            uint32_t st2 = 0;
            if (more) {   // the next kept tile's K (and V)
              st2 = (kc + 1) % ST;
              if (!(ok = mbar_wait(&bar[SB_F + st2], ((kc + 1) / ST) & 1, limit))) break;
            }
            // slot 0: P.V of tile j, then S of its next kept tile (in-order
            // execution: the P.V reads P before the new S overwrites it)
            if (bit_set(w0, j)) {
              if (!(ok = mbar_wait(&bar[SB_PRDY + 0], pr0 & 1, limit))) break;
              ++pr0;
              tc_fence_after();
              issue_pv<FP8>(T0 + 128, T0, vs, acc0);
              acc0 = true;
              if (next_set(w0, j, last) > last) mma_commit(&bar[SB_OD + 0]);
            }
            if (more && bit_set(w0, jn)) {
              tc_fence_after();
              issue_qk<FP8>(T0, q0s, stage_addr(st2));
              mma_commit(&bar[SB_SF + 0]);
            }
            if (has1) {
              if (bit_set(w1, j)) {
                if (!(ok = mbar_wait(&bar[SB_PRDY + 1], pr1 & 1, limit))) break;
                ++pr1;
                tc_fence_after();
                issue_pv<FP8>(T1 + 128, T1, vs, acc1);
                acc1 = true;
                if (next_set(w1, j, last) > last) mma_commit(&bar[SB_OD + 1]);
              }
              if (more && bit_set(w1, jn)) {
                tc_fence_after();
                issue_qk<FP8>(T1, q1s, stage_addr(st2));
                mma_commit(&bar[SB_SF + 1]);
              }
            }
            mma_commit(&bar[SB_E + st]);   // tile j's K and V are no longer read
            ++kc;
            st = st2;
            j = jn;
          }
        } while (false);
        ctr_sh[4] = qc;
        ctr_sh[5] = kc;
        ctr_sh[6] = se0;
        ctr_sh[7] = se1;
        ctr_sh[8] = pr0;
        ctr_sh[9] = pr1;
        ctr_sh[10] = dc0;
        ctr_sh[11] = dc1;
      }
    } else if (warp == kWarpFetch) {
      if (lane == 0) fetch_item(p, ws->total_items, ws->max_tiles, item_sh[(it + 1) & 1]);
    }
    if (!ok) abort_sh = 1;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (abort_sh && threadIdx.x == 0) atomicOr(&ws->status, kStatusTimeout);
  }
  } else {
    reg_alloc<kRegsSlot>();
  for (int it = 0;; ++it) {
    const int *I = item_sh[it & 1];
    if (!I[0] || abort_sh) break;
    const int s = I[1], kvh = I[2], h0 = I[3], h1 = I[4], qi = I[5], L = I[7];
    const int Lk = I[9];
    const int off = Lk - L;   // query row r sits at key position off + r
    const int nq = (L + kTile - 1) / kTile, nk = (Lk + kTile - 1) / kTile;
    const int qlast = min(qi * kTile + kTile, L) - 1;
    const int last = p.causal ? min((off + qlast) / kTile, nk - 1) : nk - 1;
    const int npairs = (last + 2) >> 1;
    bool ok = true;
    {
      // -------------------------------------------------- slot warpgroups
      const int slot = (warp - kWarpSoftmax) >> 2;
      const int h = slot ? h1 : h0;
      if (h >= 0) {
        const int row = ((warp & 3) << 5) | lane;   // = TMEM lane
        const uint32_t barid = 1 + slot;
        uint32_t sc = ctr_sh[12 + 2 * slot], odc = ctr_sh[13 + 2 * slot];
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + slot * 256 + lane_off;
        const uint32_t tO = tS + 128;
        volatile uint32_t *keep = keep_w + slot * kKeepWords;
        const bool valid = qi * kTile + row < L;
        const bool tail = !p.causal && (Lk % kTile) != 0;
        float c = p.c;
        if (FP8) c *= p.q_scale[h] * p.k_scale[kvh];
        const int W = (nk + 31) >> 5;
        uint32_t *const brow =
            p.bitmap ? p.bitmap + p.seq_bitmap_off[s] + ((long long)h * nq + qi) * W : nullptr;
        const int doff0 = off + qi * kTile;   // row r of key tile j sees columns <= r + doff0 - 128 j
        const float l2l = p.log2_lambda;
        auto wait_s = [&]() {
          if (!abort_sh && !mbar_wait(&bar[SB_SF + slot], sc & 1, limit)) abort_sh = 1;
          ++sc;
          tc_fence_after();
        };

        // ---- phase 1: row maxima, prefix max, votes
        for (int w = row; w <= (last >> 5); w += 128) keep[w] = 0u;
        named_bar_sync(barid, 128);
        float m = -INFINITY;   // running (prefix) max of S c, log2 units
        for (int pr = 0; pr < npairs; ++pr) {
          const int j0 = 2 * pr;
          const bool two = j0 + 1 <= last;
          wait_s();
          float rm0, rm1 = -INFINITY;
          {
            const int d0 = doff0 - j0 * kTile, d1 = d0 - kTile;
            const bool dg0 = p.causal && d0 < kTile - 1, dg1 = p.causal && d1 < kTile - 1;
            const bool tl0 = tail && j0 == nk - 1, tl1 = tail && j0 + 1 == nk - 1;
            float acc[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) acc[k] = -INFINITY;
            uint32_t a0[32], a1[32], b0[32], b1[32];
            tmem_ld64(tS, a0, a1);
            tmem_wait_ld(a0);
            reg_fence(a1);
            tmem_ld64(tS + 64, b0, b1);
            max_half(acc, a0, a1, 0, dg0, tl0, row, d0, j0 * kTile, Lk);
            tmem_wait_ld(b0);
            reg_fence(b1);
            if (two) {
              tmem_ld64(tS + 128, a0, a1);
              max_half(acc, b0, b1, 1, dg0, tl0, row, d0, j0 * kTile, Lk);
              rm0 = fold8(acc);
#pragma unroll
              for (int k = 0; k < 8; ++k) acc[k] = -INFINITY;
              tmem_wait_ld(a0);
              reg_fence(a1);
              tmem_ld64(tS + 192, b0, b1);
              max_half(acc, a0, a1, 0, dg1, tl1, row, d1, (j0 + 1) * kTile, Lk);
              tmem_wait_ld(b0);
              reg_fence(b1);
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&bar[SB_SE + slot]);   // S_s may be overwritten
              max_half(acc, b0, b1, 1, dg1, tl1, row, d1, (j0 + 1) * kTile, Lk);
              rm1 = fold8(acc);
            } else {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&bar[SB_SE + slot]);
              max_half(acc, b0, b1, 1, dg0, tl0, row, d0, j0 * kTile, Lk);
              rm0 = fold8(acc);
            }
          }
          // decisions of tiles j0 (and j0 + 1) against the running max before each
          const float t0 = rm0 * c;
          const bool p0 = !valid || t0 < m + l2l;
          m = fmaxf(m, t0);
          uint32_t bits = __all_sync(0xffffffffu, p0) ? 0u : 1u << (j0 & 31);
          if (two) {
            const float t1 = rm1 * c;
            const bool p1 = !valid || t1 < m + l2l;
            m = fmaxf(m, t1);
            if (!__all_sync(0xffffffffu, p1)) bits |= 1u << ((j0 + 1) & 31);
          }
          if (lane == 0 && bits) atomicOr(const_cast<uint32_t *>(&keep[j0 >> 5]), bits);
          const int jl = two ? j0 + 1 : j0;
          if ((jl & 31) == 31 || jl == last) {
            named_bar_sync(barid, 128);
            if (abort_sh) {   // read after the barrier: uniform over the warpgroup
              ok = false;
              break;
            }
            if (row == 0 && brow) {
              const uint32_t valid_bits = (jl == last && (last & 31) != 31)
                                              ? (1u << ((last & 31) + 1)) - 1u
                                              : 0xffffffffu;
              brow[jl >> 5] = ~keep[jl >> 5] & valid_bits;   // skip bit = no row kept
            }
          }
        }
        if (ok) {
          if (row == 0) {
            if (brow)
              for (int w = (last >> 5) + 1; w < W; ++w) brow[w] = 0u;
            mbar_arrive(&bar[SB_DEC + slot]);
          }
          // ---- phase 2: the kept tiles against the final row max
          const float nm = valid ? -m : -INFINITY;
          float l = 0.f;
          for (int j = 0; j <= last; j = next_set(keep, j, last)) {
            wait_s();
            const int doff = doff0 - j * kTile;
            const bool diag = p.causal && doff < kTile - 1;
            const bool tailt = tail && j == nk - 1;
            float psum[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) psum[k] = 0.f;
            uint32_t va[32], vb[32];
            tmem_ld32(tS, va);
            tmem_wait_ld(va);
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) {
              uint32_t(&v)[32] = (ch & 1) ? vb : va;
              uint32_t(&nxt)[32] = (ch & 1) ? va : vb;
              if (ch < 3) tmem_ld32(tS + (ch + 1) * 32, nxt);   // overlaps this chunk's math
              if (diag || tailt) mask_chunk(v, ch, diag, tailt, row, doff, j * kTile, Lk);
              auto pexp = [&](int e) -> float {
                const float pv = ex2_approx(fmaf(__uint_as_float(v[e]), c, nm));
                psum[e & 7] += pv;
                return pv;
              };
              if (FP8) {
                uint32_t w8[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                  const float q0 = pexp(4 * k), q1 = pexp(4 * k + 1);
                  const float q2 = pexp(4 * k + 2), q3 = pexp(4 * k + 3);
                  w8[k] = (uint32_t)pack_e4m3x2(q0, q1) | ((uint32_t)pack_e4m3x2(q2, q3) << 16);
                }
                tmem_st8(tS + ch * 8, w8);
              } else {
                uint32_t w2[16];
#pragma unroll
                for (int k = 0; k < 16; ++k) w2[k] = pack_bf16x2(pexp(2 * k), pexp(2 * k + 1));
                tmem_st16(tS + ch * 16, w2);
              }
              if (ch < 3) tmem_wait_ld(nxt);
            }
            l += ((psum[0] + psum[1]) + (psum[2] + psum[3])) +
                 ((psum[4] + psum[5]) + (psum[6] + psum[7]));
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[SB_PRDY + slot]);
          }
          // ---- epilogue: O / l, lse
          if (!abort_sh && !mbar_wait(&bar[SB_OD + slot], odc & 1, limit)) abort_sh = 1;
          ++odc;
          tc_fence_after();
          const volatile int *Iv = item_sh[it & 1];
          const int ea = Iv[6], eh = Iv[3 + slot], ekvh = Iv[2];
          const int tok = ea + Iv[5] * kTile + row;
          float inv = 0.f;
          if (valid && l > 0.f) inv = (FP8 ? p.v_scale[ekvh] : 1.f) / l;
          __nv_bfloat16 *orow =
              reinterpret_cast<__nv_bfloat16 *>(p.out) + ((size_t)tok * p.Hq + eh) * kHeadDim;
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            uint32_t v[32];
            tmem_ld32(tO + ch * 32, v);
            tmem_wait_ld(v);
            uint32_t w2[16];
#pragma unroll
            for (int k = 0; k < 16; ++k)
              w2[k] = pack_bf16x2(__uint_as_float(v[2 * k]) * inv, __uint_as_float(v[2 * k + 1]) * inv);
            if (valid) {
              uint4 *dst = reinterpret_cast<uint4 *>(orow + ch * 32);
#pragma unroll
              for (int q = 0; q < 4; ++q)
                dst[q] = make_uint4(w2[4 * q], w2[4 * q + 1], w2[4 * q + 2], w2[4 * q + 3]);
            }
          }
          if (valid && p.lse) p.lse[(size_t)eh * ws->total_tokens + tok] = (m + log2f(l)) * kLn2;
        }
        if (row == 0) {   // uniform over the warpgroup; read by all at the next item's start
          ctr_sh[12 + 2 * slot] = sc;
          ctr_sh[13 + 2 * slot] = odc;
        }
      }
    }
    if (!ok) abort_sh = 1;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (abort_sh && threadIdx.x == 0) atomicOr(&ws->status, kStatusTimeout);
  }
  }

  // Normal exit: every item ended drained. After a time-out, wait (bounded)
  // for this CTA's own copies and MMAs before giving TMEM back.
  if (abort_sh) {
    if (warp == kWarpProd && lane == 0) {
      for (int st = 0; st < ST; ++st)
        if (kc_last[st] >= 0) mbar_wait(&bar[SB_F + st], (kc_last[st] / ST) & 1, limit);
      if (qc_last >= 0) mbar_wait(&bar[SB_Q], qc_last & 1, limit);
    }
    if (warp == kWarpMma && lane == 0) {
      mma_commit(&bar[SB_DRAIN]);
      mbar_wait(&bar[SB_DRAIN], 0, limit);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpMma) tmem_dealloc(tmem, 512);
}

template <bool FP8>
static size_t skip_smem_bytes() {
  return SkipCfg<FP8>::kSmBytes + 1024;
}

cudaError_t launch_skip(const FwdParams &p, bool fp8, int num_ctas, cudaStream_t stream) {
  if (fp8)
    skip_kernel<true><<<num_ctas, kSkipThreads, skip_smem_bytes<true>(), stream>>>(p);
  else
    skip_kernel<false><<<num_ctas, kSkipThreads, skip_smem_bytes<false>(), stream>>>(p);
  return cudaGetLastError();
}

cudaError_t prepare_skip() {
  const cudaFuncAttribute a = cudaFuncAttributeMaxDynamicSharedMemorySize;
  cudaError_t e = cudaFuncSetAttribute(skip_kernel<false>, a, (int)skip_smem_bytes<false>());
  if (e == cudaSuccess) e = cudaFuncSetAttribute(skip_kernel<true>, a, (int)skip_smem_bytes<true>());
  // the register split hands out exactly the launch allocation: refuse a build
  // whose per-thread count differs (setmaxnreg.inc would wait for registers
  // that never come)
  cudaFuncAttributes fa;
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, skip_kernel<false>);
  if (e == cudaSuccess && fa.numRegs != (int)kRegsLaunch) e = cudaErrorInvalidKernelImage;
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, skip_kernel<true>);
  if (e == cudaSuccess && fa.numRegs != (int)kRegsLaunch) e = cudaErrorInvalidKernelImage;
  return e;
}

}  // namespace bsa
