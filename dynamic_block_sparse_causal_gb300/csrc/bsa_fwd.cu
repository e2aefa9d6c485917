// Block-skipping causal prefill attention: device code for sm_103a.
//
// Operation: dynamic sparse attention deployment guide
// ("长上下文推理加速方案部署实战：基于动态稀疏注意力机制的推理服务优化指南"),
// §3.2 -- online softmax over key blocks in order; a block whose local max
// score falls below the running max by more than the threshold skips the
// exponentials, its V load and its P.V product. Threshold read as
// tile_max < running_max + ln(lambda) per row, AND-ed over the 128 rows of
// the query tile (§3.3 and §6.1 fix the direction: larger lambda prunes more).
//
// Two kernels:
//  * prologue_kernel (1 CTA): validates cu_seqlens, orders sequences longest
//    first, builds the work-item level table and the skip-bitmap offsets,
//    and writes the TMA tensor maps with the token extent patched in.
//  * fwd_kernel<FP8> (persistent, one CTA per SM, 384 threads):
//      warp 0  lane 0   TMA producer: Q tiles, then the K ring (2 stages)
//      warp 1  lane 0   tcgen05 MMA issuer; also issues the V load of a tile
//                       once one of the two query tiles votes to keep it
//      warp 2  lane 0   fetches the next work item (atomic counter)
//      warps 4-7        softmax warpgroup of query slot 0 (TMEM lanes 0-127)
//      warps 8-11       softmax warpgroup of query slot 1
//    A work item is (sequence, KV head, two query heads of that group, query
//    tile i): both query tiles need exactly the key tiles 0..i, so each K
//    tile loaded feeds two QK^T MMAs.
//
// TMEM (512 columns): S0 [0,128) S1 [128,256) O0 [256,384) O1 [384,512),
// fp32, lane = query row. Shared memory (1024-aligned, 128-byte swizzle):
// Q0 Q1 K[2] V P0 P1, 32 KiB each.
//
// Per key tile j and query slot s the softmax warpgroup loads S_s from TMEM,
// masks the diagonal / tail, takes the row max, and votes with bar.red.and.
// A skipped tile releases S_s at once; a kept tile updates the running max
// (lazy rescale of O when the reference max grows by more than 2^8),
// writes P = exp2(S c - m_ref) as bf16 (e4m3) into shared memory and hands
// it to the MMA warp, which only then requests V_j.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include <climits>
#include <cmath>

#include "bsa_internal.h"
#include "ptx.cuh"

namespace bsa {

// ============================================================ prologue

__global__ void __launch_bounds__(1024)
prologue_kernel(const int32_t *__restrict__ cu, int n_seqs, int Hq, int Hkv, Workspace *ws,
                int32_t *seq_sorted, int64_t *seq_bitmap_off, int32_t *level_start,
                const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                const __grid_constant__ CUtensorMap tv) {
  __shared__ int s_bad, s_maxn;
  const int tid = threadIdx.x;
  if (tid == 0) {
    s_bad = (cu[0] != 0);
    s_maxn = 0;
  }
  __syncthreads();
  for (int s = tid; s < n_seqs; s += blockDim.x) {
    const int L = cu[s + 1] - cu[s];
    if (L < 0) atomicOr(&s_bad, 1);
    atomicMax(&s_maxn, (L + kTile - 1) / kTile);
  }
  __syncthreads();
  const int maxn = s_maxn;
  const int group = Hq / Hkv;
  const long long U = (long long)Hkv * ((group + 1) / 2);  // work items per (sequence, tile)
  bool bad = s_bad || maxn > kMaxLevels;
  if (!bad) {
    // longest first, ties by sequence index
    for (int s = tid; s < n_seqs; s += blockDim.x) {
      const int ns = (cu[s + 1] - cu[s] + kTile - 1) / kTile;
      int rank = 0;
      for (int t = 0; t < n_seqs; ++t) {
        const int nt = (cu[t + 1] - cu[t] + kTile - 1) / kTile;
        rank += (nt > ns) || (nt == ns && t < s);
      }
      seq_sorted[rank] = s;
    }
    // level_start[i] = first item of query-tile level i; items run from the
    // deepest level (longest causal rows) down to level 0.
    for (int i = tid; i < maxn; i += blockDim.x) {
      long long acc = 0;
      for (int t = 0; t < n_seqs; ++t) {
        const int nt = (cu[t + 1] - cu[t] + kTile - 1) / kTile;
        acc += max(0, nt - 1 - i);
      }
      level_start[i] = (int32_t)min(U * acc, (long long)INT_MAX);
    }
  }
  __syncthreads();
  if (tid == 0) {
    long long items = 0, words = 0;
    for (int s = 0; s < n_seqs && !bad; ++s) {
      const int ns = (cu[s + 1] - cu[s] + kTile - 1) / kTile;
      seq_bitmap_off[s] = words;
      words += (long long)Hq * ns * ((ns + 31) / 32);
      items += U * ns;
    }
    if (items > INT_MAX) bad = true;
    ws->counter = 0;
    ws->total_items = bad ? 0 : (int32_t)items;
    ws->max_tiles = maxn;
    ws->total_tokens = cu[n_seqs];
    if (bad) atomicOr(&ws->status, kStatusBadSeqlens);
  }
  if (tid < 3) {
    const CUtensorMap *src = tid == 0 ? &tq : (tid == 1 ? &tk : &tv);
    CUtensorMap *dst = &ws->tmap[tid];
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

cudaError_t launch_prologue(const int32_t *cu_seqlens, int n_seqs, int Hq, int Hkv, Workspace *ws,
                            const WorkspaceLayout &layout, const CUtensorMap tmpl[3],
                            cudaStream_t stream) {
  char *base = reinterpret_cast<char *>(ws);
  prologue_kernel<<<1, 1024, 0, stream>>>(
      cu_seqlens, n_seqs, Hq, Hkv, ws, reinterpret_cast<int32_t *>(base + layout.seq_sorted),
      reinterpret_cast<int64_t *>(base + layout.seq_bitmap_off),
      reinterpret_cast<int32_t *>(base + layout.level_start), tmpl[0], tmpl[1], tmpl[2]);
  return cudaGetLastError();
}

// ============================================================ forward

namespace {

constexpr uint32_t kRegion = 32768;   // one tile slot in shared memory
constexpr uint32_t kBox = 16384;      // one 128-row x 128-byte TMA box
constexpr uint32_t SM_Q0 = 0, SM_Q1 = kRegion, SM_K = 2 * kRegion, SM_V = 4 * kRegion,
                   SM_P0 = 5 * kRegion, SM_P1 = 6 * kRegion, SM_BYTES = 7 * kRegion;
constexpr int kStages = 2;
constexpr float kRescaleLog2 = 8.0f;  // lazy O rescale once m grows by 2^8
constexpr float kLn2 = 0.6931471805599453f;

// barrier slots
enum : int {
  B_Q = 0, B_KF = 1, B_KE = B_KF + kStages, B_VF = B_KE + kStages, B_VE, B_SF, B_DEC = B_SF + 2,
  B_PV = B_DEC + 2, B_DRAIN = B_PV + 2, B_COUNT
};

template <bool FP8>
struct Cfg {
  static constexpr uint32_t kTileBytes = FP8 ? 16384 : 32768;
  static constexpr int kBoxCols = FP8 ? 128 : 64;   // elements per 128-byte row
  static constexpr int kBoxes = FP8 ? 1 : 2;        // boxes along the head dim
  static constexpr int kSteps = FP8 ? 4 : 8;        // MMA K steps over 128
  static constexpr uint32_t kIdescQK = IDesc<FP8 ? 0 : 1, false, 128, 128>::value;
  static constexpr uint32_t kIdescPV = IDesc<FP8 ? 0 : 1, true, 128, 128>::value;
};

// S = Q K^T: A = Q (K-major), B = K (K-major), both 128-byte swizzled; each
// K step advances 32 bytes inside the swizzle atom.
template <bool FP8>
__device__ __forceinline__ void issue_qk(uint32_t d, uint32_t qs, uint32_t ks) {
#pragma unroll
  for (int kk = 0; kk < Cfg<FP8>::kSteps; ++kk) {
    const uint32_t off = FP8 ? kk * 32 : (kk >> 2) * kBox + (kk & 3) * 32;
    const uint64_t a = sdesc_sw128(qs + off, 16, 1024);
    const uint64_t b = sdesc_sw128(ks + off, 16, 1024);
    if (FP8)
      mma_f8_ss(d, a, b, Cfg<FP8>::kIdescQK, kk > 0);
    else
      mma_f16_ss(d, a, b, Cfg<FP8>::kIdescQK, kk > 0);
  }
}

// O += P V: A = P (K-major over keys), B = V as stored (keys x head dim,
// head dim contiguous) = MN-major; 8-row groups of keys 1024 bytes apart,
// the two 64-column halves of a bf16 V tile 16 KiB apart.
template <bool FP8>
__device__ __forceinline__ void issue_pv(uint32_t d, uint32_t ps, uint32_t vs, bool acc) {
#pragma unroll
  for (int kk = 0; kk < Cfg<FP8>::kSteps; ++kk) {
    const uint32_t aoff = FP8 ? kk * 32 : (kk >> 2) * kBox + (kk & 3) * 32;
    const uint32_t boff = FP8 ? kk * 4096 : kk * 2048;
    const uint64_t a = sdesc_sw128(ps + aoff, 16, 1024);
    const uint64_t b = sdesc_sw128(vs + boff, kBox, 1024);
    if (FP8)
      mma_f8_ss(d, a, b, Cfg<FP8>::kIdescPV, (kk > 0 || acc) ? 1u : 0u);
    else
      mma_f16_ss(d, a, b, Cfg<FP8>::kIdescPV, (kk > 0 || acc) ? 1u : 0u);
  }
}

struct Item {
  int valid, s, kvh, h0, h1, qi, a, L;
};

__device__ void fetch_item(const FwdParams &p, int total_items, int maxn, int *dst) {
  const int k = atomicAdd(&p.ws->counter, 1);
  if (k >= total_items) {
    dst[0] = 0;
    return;
  }
  int lo = 0, hi = maxn - 1;   // smallest level whose first item is <= k
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (p.level_start[mid] <= k)
      hi = mid;
    else
      lo = mid + 1;
  }
  const int U = p.Hkv * p.pairs_per_group;
  const int r = k - p.level_start[lo];
  const int s = p.seq_sorted[r / U];
  const int pidx = r % U;
  const int kvh = pidx / p.pairs_per_group, pp = pidx % p.pairs_per_group;
  const int h0 = kvh * p.group + 2 * pp;
  const int a = p.cu_seqlens[s];
  dst[0] = 1;
  dst[1] = s;
  dst[2] = kvh;
  dst[3] = h0;
  dst[4] = (2 * pp + 1 < p.group) ? h0 + 1 : -1;
  dst[5] = lo;
  dst[6] = a;
  dst[7] = p.cu_seqlens[s + 1] - a;
}

}  // namespace

template <bool FP8>
__global__ void __launch_bounds__(kFwdThreads, 1) fwd_kernel(const __grid_constant__ FwdParams p) {
  using C = Cfg<FP8>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar[B_COUNT];
  __shared__ uint32_t tmem_sh;
  __shared__ int item_sh[2][8];
  __shared__ volatile int dec_sh[2];
  __shared__ int abort_sh;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t *sptr = smem_raw + (sbase - raw);
  Workspace *ws = p.ws;
  const int total_items = ws->total_items, maxn = ws->max_tiles, T = ws->total_tokens;
  const uint64_t limit = p.wait_limit_ns;

  if (threadIdx.x == 0) {
    for (int b = 0; b < B_COUNT; ++b) mbar_init(&bar[b], 1);
    fence_mbar_init();
    abort_sh = 0;
  }
  if (threadIdx.x == 64) fetch_item(p, total_items, maxn, item_sh[0]);
  if (warp == 1) {
    tmem_alloc(&tmem_sh, 512);
    tmem_relinquish();
  }
  if ((warp == 0 || warp == 1) && lane == 0) {
    tensormap_acquire(&ws->tmap[0]);
    tensormap_acquire(&ws->tmap[1]);
    tensormap_acquire(&ws->tmap[2]);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_sh;

  // pipeline counters, persistent across items (each role keeps its own)
  uint32_t kc = 0, vc = 0, qc = 0, dc0 = 0, dc1 = 0, sc = 0, pvc = 0;
  int kc_last[kStages] = {-1, -1};
  int vc_last = -1, qc_last = -1;

  for (int it = 0;; ++it) {
    const int *I = item_sh[it & 1];
    if (!I[0] || abort_sh) break;
    const int kvh = I[2], h0 = I[3], h1 = I[4], qi = I[5], a = I[6], L = I[7];
    const int s = I[1];
    const int n = (L + kTile - 1) / kTile;
    const int last = p.causal ? qi : n - 1;
    const bool has1 = h1 >= 0;
    bool ok = true;

    if (warp == 0) {
      if (lane == 0) {
        // ------------------------------------------------ TMA producer
        const void *tq = &ws->tmap[0], *tk = &ws->tmap[1];
        mbar_expect_tx(&bar[B_Q], (has1 ? 2 : 1) * C::kTileBytes);
        for (int b = 0; b < C::kBoxes; ++b) {
          tma_load_3d(sptr + SM_Q0 + b * kBox, tq, &bar[B_Q], b * C::kBoxCols, h0, a + qi * kTile);
          if (has1)
            tma_load_3d(sptr + SM_Q1 + b * kBox, tq, &bar[B_Q], b * C::kBoxCols, h1,
                        a + qi * kTile);
        }
        qc_last = (int)qc++;
        for (int j = 0; j <= last && ok; ++j) {
          const uint32_t st = kc % kStages;
          ok = mbar_wait(&bar[B_KE + st], ((kc / kStages) & 1) ^ 1, limit);
          if (!ok) break;
          if ((int)kc != p.debug_drop_k_load) {
            mbar_expect_tx(&bar[B_KF + st], C::kTileBytes);
            for (int b = 0; b < C::kBoxes; ++b)
              tma_load_3d(sptr + SM_K + st * kRegion + b * kBox, tk, &bar[B_KF + st],
                          b * C::kBoxCols, kvh, a + j * kTile);
            kc_last[st] = (int)kc;
          }
          ++kc;
        }
      }
    } else if (warp == 1) {
      if (lane == 0) {
        // ------------------------------------------------ MMA issuer
        const void *tv = &ws->tmap[2];
        const uint32_t S0 = tmem, S1 = tmem + 128, O0 = tmem + 256, O1 = tmem + 384;
        const uint32_t q0s = sbase + SM_Q0, q1s = sbase + SM_Q1, vs = sbase + SM_V;
        const uint32_t p0s = sbase + SM_P0, p1s = sbase + SM_P1;
        auto issue_v = [&](int j) -> bool {
          if (!mbar_wait(&bar[B_VE], (vc & 1) ^ 1, limit)) return false;
          mbar_expect_tx(&bar[B_VF], C::kTileBytes);
          for (int b = 0; b < C::kBoxes; ++b)
            tma_load_3d(sptr + SM_V + b * kBox, tv, &bar[B_VF], b * C::kBoxCols, kvh,
                        a + j * kTile);
          vc_last = (int)vc;
          return true;
        };
        do {
          ok = mbar_wait(&bar[B_Q], qc & 1, limit);
          ++qc;
          if (!ok) break;
          uint32_t st = kc % kStages;
          ok = mbar_wait(&bar[B_KF + st], (kc / kStages) & 1, limit);
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
            bool v_issued = false;
            ok = mbar_wait(&bar[B_DEC + 0], dc0 & 1, limit);
            ++dc0;
            if (!ok) break;
            tc_fence_after();
            const bool skip0 = dec_sh[0] != 0;
            if (!skip0) {
              if (!(ok = issue_v(j))) break;
              v_issued = true;
            }
            if (j < last) {
              st = kc % kStages;
              ok = mbar_wait(&bar[B_KF + st], (kc / kStages) & 1, limit);
              if (!ok) break;
              tc_fence_after();
              ks = sbase + SM_K + st * kRegion;
              issue_qk<FP8>(S0, q0s, ks);
              mma_commit(&bar[B_SF + 0]);
            }
            bool skip1 = true;
            if (has1) {
              ok = mbar_wait(&bar[B_DEC + 1], dc1 & 1, limit);
              ++dc1;
              if (!ok) break;
              tc_fence_after();
              skip1 = dec_sh[1] != 0;
              if (!skip1 && !v_issued) {
                if (!(ok = issue_v(j))) break;
                v_issued = true;
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
            if (v_issued) {
              ok = mbar_wait(&bar[B_VF], vc & 1, limit);
              if (!ok) break;
              tc_fence_after();
              if (!skip0) {
                issue_pv<FP8>(O0, p0s, vs, oinit0);
                oinit0 = true;
                mma_commit(&bar[B_PV + 0]);
              }
              if (!skip1) {
                issue_pv<FP8>(O1, p1s, vs, oinit1);
                oinit1 = true;
                mma_commit(&bar[B_PV + 1]);
              }
              mma_commit(&bar[B_VE]);
              ++vc;
            }
          }
        } while (false);
      }
    } else if (warp == 2) {
      if (lane == 0) fetch_item(p, total_items, maxn, item_sh[(it + 1) & 1]);
    } else if (warp >= 4) {
      // -------------------------------------------------- softmax warpgroups
      const int slot = (warp - 4) >> 2;
      const int h = slot ? h1 : h0;
      if (h >= 0) {
        const int row = threadIdx.x - 128 * (slot + 1);   // 0..127 = TMEM lane
        const uint32_t barid = 1 + slot;
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + slot * 128 + lane_off;
        const uint32_t tO = tmem + 256 + slot * 128 + lane_off;
        const uint32_t ps = sbase + (slot ? SM_P1 : SM_P0);
        const int qpos = qi * kTile + row;
        const bool valid = qpos < L;
        const bool tail = !p.causal && (L % kTile) != 0;
        float c = p.c;
        if (FP8) c *= p.q_scale[h] * p.k_scale[kvh];
        const int W = (n + 31) >> 5;
        const long long boff = p.seq_bitmap_off[s] + ((long long)h * n + qi) * W;
        float m2 = -INFINITY, mref = 0.f, l = 0.f;
        uint32_t word = 0;
        bool pv_pending = false, have_kept = false;

        for (int j = 0; j <= last; ++j) {
          bool wok = true;
          if (row == 0) wok = mbar_wait(&bar[B_SF + slot], sc & 1, limit);
          ++sc;
          if (bar_red_or(!wok, barid, 128)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const bool diag = p.causal && j == qi;
          const bool tailt = tail && j == n - 1;
          const bool masked_tile = diag || tailt;
          float rm = -INFINITY;
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            uint32_t v[32];
            tmem_ld32(tS + ch * 32, v);
            tmem_wait_ld(v);
            if (masked_tile) {
#pragma unroll
              for (int e = 0; e < 32; ++e) {
                const int col = ch * 32 + e;
                const bool msk = (diag && col > row) || (tailt && j * kTile + col >= L);
                rm = fmaxf(rm, msk ? -INFINITY : __uint_as_float(v[e]));
              }
            } else {
#pragma unroll
              for (int e = 0; e < 32; ++e) rm = fmaxf(rm, __uint_as_float(v[e]));
            }
          }
          const float trm = rm * c;
          const bool pred = !valid || (trm < m2 + p.log2_lambda);
          tc_fence_before();
          const bool skip = bar_red_and(pred, barid, 128);
          if (skip) {
            if (row == 0) {
              word |= 1u << (j & 31);
              dec_sh[slot] = 1;
              mbar_arrive(&bar[B_DEC + slot]);
            }
          } else {
            const float mnew = valid ? fmaxf(m2, trm) : 0.f;
            if (pv_pending) {  // P buffer and O are still in use by the last P.V
              bool pok = true;
              if (row == 0) pok = mbar_wait(&bar[B_PV + slot], pvc & 1, limit);
              ++pvc;
              pv_pending = false;
              if (bar_red_or(!pok, barid, 128)) {
                ok = false;
                break;
              }
              tc_fence_after();
            }
            if (!have_kept) {
              mref = mnew;
            } else {
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
                  for (int e = 0; e < 32; ++e)
                    v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
                  tmem_st32(tO + ch * 32, v);
                }
                tmem_wait_st();
              }
            }
            m2 = mnew;
            float sum = 0.f;
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) {
              uint32_t v[32];
              tmem_ld32(tS + ch * 32, v);
              tmem_wait_ld(v);
              float pe[32];
#pragma unroll
              for (int e = 0; e < 32; ++e) {
                const int col = ch * 32 + e;
                const bool msk = !valid || (masked_tile && ((diag && col > row) ||
                                                           (tailt && j * kTile + col >= L)));
                pe[e] = msk ? 0.f : ex2_approx(fmaf(__uint_as_float(v[e]), c, -mref));
                sum += pe[e];
              }
              if (FP8) {
                uint32_t w8[8];
#pragma unroll
                for (int k = 0; k < 8; ++k)
                  w8[k] = (uint32_t)pack_e4m3x2(pe[4 * k], pe[4 * k + 1]) |
                          ((uint32_t)pack_e4m3x2(pe[4 * k + 2], pe[4 * k + 3]) << 16);
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                  const uint32_t u = 2 * ch + q;
                  st_shared_v4(ps + row * 128 + ((u ^ (row & 7)) << 4), w8[4 * q], w8[4 * q + 1],
                               w8[4 * q + 2], w8[4 * q + 3]);
                }
              } else {
                uint32_t w2[16];
#pragma unroll
                for (int k = 0; k < 16; ++k) w2[k] = pack_bf16x2(pe[2 * k], pe[2 * k + 1]);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                  const uint32_t u = (ch & 1) * 4 + q;
                  st_shared_v4(ps + (ch >> 1) * kBox + row * 128 + ((u ^ (row & 7)) << 4),
                               w2[4 * q], w2[4 * q + 1], w2[4 * q + 2], w2[4 * q + 3]);
                }
              }
            }
            l += sum;
            fence_proxy_async_smem();
            tc_fence_before();
            named_bar_sync(barid, 128);
            if (row == 0) {
              dec_sh[slot] = 0;
              mbar_arrive(&bar[B_DEC + slot]);
            }
            pv_pending = true;
            have_kept = true;
          }
          if (row == 0 && p.bitmap && (((j & 31) == 31) || j == last)) {
            p.bitmap[boff + (j >> 5)] = word;
            word = 0;
          }
        }
        // ------------------------------------------------ epilogue
        if (ok && pv_pending) {
          bool pok = true;
          if (row == 0) pok = mbar_wait(&bar[B_PV + slot], pvc & 1, limit);
          ++pvc;
          if (bar_red_or(!pok, barid, 128)) ok = false;
        }
        if (ok) {
          tc_fence_after();
          float inv = 0.f;
          if (valid && l > 0.f) inv = (FP8 ? p.v_scale[kvh] : 1.f) / l;
          __nv_bfloat16 *orow = reinterpret_cast<__nv_bfloat16 *>(p.out) +
                                ((size_t)(a + qpos) * p.Hq + h) * kHeadDim;
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
          if (valid && p.lse) p.lse[(size_t)h * T + a + qpos] = (mref + log2f(l)) * kLn2;
          if (row == 0 && p.bitmap)
            for (int w = (last >> 5) + 1; w < W; ++w) p.bitmap[boff + w] = 0u;
        }
      }
    }
    if (!ok) {
      abort_sh = 1;
      atomicOr(&ws->status, kStatusTimeout);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  }

  // Normal exit: every item ended fully drained. After a time-out, wait
  // (bounded) for this CTA's own copies and MMAs before giving TMEM back.
  if (abort_sh) {
    if (warp == 0 && lane == 0) {
      for (int st = 0; st < kStages; ++st)
        if (kc_last[st] >= 0) mbar_wait(&bar[B_KF + st], (kc_last[st] / kStages) & 1, limit);
      if (qc_last >= 0) mbar_wait(&bar[B_Q], qc_last & 1, limit);
    }
    if (warp == 1 && lane == 0) {
      if (vc_last >= 0) mbar_wait(&bar[B_VF], vc_last & 1, limit);
      mma_commit(&bar[B_DRAIN]);
      mbar_wait(&bar[B_DRAIN], 0, limit);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

size_t forward_smem_bytes() { return SM_BYTES + 1024; }

cudaError_t launch_forward(const FwdParams &p, bool fp8, int num_ctas, cudaStream_t stream) {
  const size_t smem = forward_smem_bytes();
  if (fp8) {
    fwd_kernel<true><<<num_ctas, kFwdThreads, smem, stream>>>(p);
  } else {
    fwd_kernel<false><<<num_ctas, kFwdThreads, smem, stream>>>(p);
  }
  return cudaGetLastError();
}

cudaError_t prepare_forward() {
  const int smem = (int)forward_smem_bytes();
  cudaError_t e = cudaFuncSetAttribute(fwd_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(fwd_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}

}  // namespace bsa
