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
//  * fwd_kernel<FP8, SKIP> (persistent, one CTA per SM, 384 threads):
//      warp 0  lane 0   TMA producer: Q tiles, the K ring (4 stages with
//                       skipping on, 3 with it off), and, when skipping is off,
//                       V with every K (2-stage ring)
//      warp 1  lane 0   tcgen05 MMA issuer; with skipping on it also requests
//                       V_j (one stage) as soon as a query tile votes to keep j
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
// (1024-aligned, 128-byte swizzle), 32 KiB regions: Q0 Q1, then K[4] V[1]
// with skipping on or K[3] V[2] with it off.
//
// Pipeline counters live in registers within a work item and in shared
// memory between items, one set per role, so that no role's registers carry
// another role's counters through the item loop (register pressure in the
// softmax warpgroups sets the length of the per-tile chain).
//
// Per key tile j and query slot s the softmax warpgroup loads S_s from TMEM,
// masks the diagonal / tail, takes the row max, and votes with one
// bar.red.and. The vote is posted at once: a skipped tile frees S_s for the
// next QK^T; a kept tile lets the MMA warp request V_j while the warpgroup
// computes P = exp2(S c - m_ref) (lazy O rescale when the reference max
// grows by more than 2^8) into TMEM and then posts P-ready. The MMA warp
// issues O_s += P_s V_j before the next S_s, so the tensor pipe's in-order
// execution protects P until it has been read.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include <climits>
#include <cmath>

#include "bsa_internal.h"
#include "ptx.cuh"

namespace bsa {

// ============================================================ prologue

// Query-tile count of sequence s (tiles of its queries) and key-tile count.
__device__ __forceinline__ int q_tiles(const int32_t *cu, int s) {
  return (cu[s + 1] - cu[s] + kTile - 1) / kTile;
}

__global__ void __launch_bounds__(1024)
prologue_kernel(const int32_t *__restrict__ cu, const int32_t *__restrict__ cuk, int n_seqs,
                int Hq, int Hkv, int causal, const int32_t *__restrict__ page_table,
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
    atomicMax(&s_maxn, (Lq + kTile - 1) / kTile);
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
  const int group = Hq / Hkv;
  // work items are ordered KV head by KV head (so CTAs running at the same time
  // stream the same head's K tiles through L2), and within a head longest
  // query tile first; U = items per (sequence, query tile) within one head
  const long long U = (group + 1) / 2;
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
                            int Hq, int Hkv, int causal, const int32_t *page_table,
                            int max_pages, int num_pages, Workspace *ws,
                            const WorkspaceLayout &layout, const CUtensorMap tmpl[3],
                            cudaStream_t stream) {
  char *base = reinterpret_cast<char *>(ws);
  prologue_kernel<<<1, 1024, 0, stream>>>(
      cu_seqlens, cu_seqlens_k, n_seqs, Hq, Hkv, causal, page_table, max_pages, num_pages, ws,
      reinterpret_cast<int32_t *>(base + layout.seq_sorted),
      reinterpret_cast<int64_t *>(base + layout.seq_bitmap_off),
      reinterpret_cast<int32_t *>(base + layout.level_start), tmpl[0], tmpl[1], tmpl[2]);
  return cudaGetLastError();
}

// ============================================================ forward

namespace {

constexpr uint32_t kRegion = 32768;   // one bf16 tile slot in shared memory
constexpr uint32_t kBox = 16384;      // one 128-row x 128-byte TMA box
// K and V rings share five 32 KiB regions after the two Q tiles: 3 K + 2 V
// stages with skipping off (V streams with every K), 4 K + 1 V with it on
// (V is loaded only for kept tiles, K for every tile)
constexpr int kKStages = 4, kVStages = 2;   // the deeper of the two, for barrier slots
template <bool SKIP>
struct Ring {
  static constexpr int K = SKIP ? 4 : 3, V = SKIP ? 1 : 2;
};
constexpr uint32_t SM_Q0 = 0, SM_Q1 = kRegion, SM_K = 2 * kRegion, SM_BYTES = SM_K + 5 * kRegion;
constexpr float kRescaleLog2 = 8.0f;  // lazy O rescale once m grows by 2^8
constexpr float kLn2 = 0.6931471805599453f;
constexpr uint32_t kColS = 0, kColO = 256;   // TMEM: S_s at s*128, O_s at 256 + s*128
// warp roles: TMA producer, MMA issuer, item fetch, then (from warp 4) the
// softmax warpgroups of query slots 0 and 1 (warp w reaches TMEM lanes 32 (w % 4) ..)
constexpr int kWarpProd = 0, kWarpMma = 1, kWarpFetch = 2, kWarpSoftmax = 4;

// barrier slots
enum : int {
  B_Q = 0,
  B_KF = 1,
  B_KE = B_KF + kKStages,
  B_VF = B_KE + kKStages,
  B_VE = B_VF + kVStages,
  B_SF = B_VE + kVStages,   // S_s computed (per slot)
  B_VOTE = B_SF + 2,        // slot s voted on the tile (S_s free if skipped)
  B_PRDY = B_VOTE + 2,      // P_s written to TMEM (S_s consumed)
  B_PV = B_PRDY + 2,        // O_s += P_s V done
  B_DRAIN = B_PV + 2,
  B_COUNT
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

// O += P V: A = P from TMEM (row = lane, two bf16 or four e4m3 keys per
// 32-bit column, so every K step is 8 columns), B = V as stored (keys x head
// dim, head dim contiguous) = MN-major; 8-row key groups 1024 bytes apart,
// the two 64-column halves of a bf16 V tile 16 KiB apart.
template <bool FP8>
__device__ __forceinline__ void issue_pv(uint32_t d, uint32_t p_tmem, uint32_t vs, bool acc) {
#pragma unroll
  for (int kk = 0; kk < Cfg<FP8>::kSteps; ++kk) {
    const uint32_t boff = FP8 ? kk * 4096 : kk * 2048;
    const uint64_t b = sdesc_sw128(vs + boff, kBox, 1024);
    if (FP8)
      mma_f8_ts(d, p_tmem + kk * 8, b, Cfg<FP8>::kIdescPV, (kk > 0 || acc) ? 1u : 0u);
    else
      mma_f16_ts(d, p_tmem + kk * 8, b, Cfg<FP8>::kIdescPV, (kk > 0 || acc) ? 1u : 0u);
  }
}

__device__ void fetch_item(const FwdParams &p, int total_items, int maxn, int *dst) {
  const int k = atomicAdd(&p.ws->counter, 1);
  if (k >= total_items) {
    dst[0] = 0;
    return;
  }
  // KV head major: items [g * per_head, (g + 1) * per_head) belong to head g
  const int per_head = total_items / p.Hkv;
  const int kvh = k / per_head;
  const int kr = k - kvh * per_head;
  int lo = 0, hi = maxn - 1;   // smallest level whose first item is <= kr
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (p.level_start[mid] <= kr)
      hi = mid;
    else
      lo = mid + 1;
  }
  const int U = p.pairs_per_group;
  const int r = kr - p.level_start[lo];
  const int s = p.seq_sorted[r / U];
  const int pp = r % U;
  const int h0 = kvh * p.group + 2 * pp;
  const int a = p.cu_seqlens[s], ak = p.cu_seqlens_k[s];
  dst[0] = 1;
  dst[1] = s;
  dst[2] = kvh;
  dst[3] = h0;
  dst[4] = (2 * pp + 1 < p.group) ? h0 + 1 : -1;
  dst[5] = lo;
  dst[6] = a;
  dst[7] = p.cu_seqlens[s + 1] - a;
  dst[8] = ak;
  dst[9] = p.cu_seqlens_k[s + 1] - ak;
}

// 32 lanes x 64 consecutive 32-bit columns in one load (two 32-register halves).
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&a)[32], uint32_t (&b)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];"
      : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(a[4]), "=r"(a[5]), "=r"(a[6]), "=r"(a[7]), "=r"(a[8]), "=r"(a[9]), "=r"(a[10]), "=r"(a[11]), "=r"(a[12]), "=r"(a[13]), "=r"(a[14]), "=r"(a[15]), "=r"(a[16]), "=r"(a[17]), "=r"(a[18]), "=r"(a[19]), "=r"(a[20]), "=r"(a[21]), "=r"(a[22]), "=r"(a[23]), "=r"(a[24]), "=r"(a[25]), "=r"(a[26]), "=r"(a[27]), "=r"(a[28]), "=r"(a[29]), "=r"(a[30]), "=r"(a[31]),
        "=r"(b[0]), "=r"(b[1]), "=r"(b[2]), "=r"(b[3]), "=r"(b[4]), "=r"(b[5]), "=r"(b[6]), "=r"(b[7]), "=r"(b[8]), "=r"(b[9]), "=r"(b[10]), "=r"(b[11]), "=r"(b[12]), "=r"(b[13]), "=r"(b[14]), "=r"(b[15]), "=r"(b[16]), "=r"(b[17]), "=r"(b[18]), "=r"(b[19]), "=r"(b[20]), "=r"(b[21]), "=r"(b[22]), "=r"(b[23]), "=r"(b[24]), "=r"(b[25]), "=r"(b[26]), "=r"(b[27]), "=r"(b[28]), "=r"(b[29]), "=r"(b[30]), "=r"(b[31])
      : "r"(taddr));
}

// Running row max over two 32-register chunks (three-input max, eight
// independent chains).
__device__ __forceinline__ void row_max64(float (&a)[8], const uint32_t (&v0)[32],
                                          const uint32_t (&v1)[32]) {
#pragma unroll
  for (int i = 0; i < 32; i += 16) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      a[k] = max3f(a[k], __uint_as_float(v0[i + 2 * k]), __uint_as_float(v0[i + 2 * k + 1]));
      a[k] = max3f(a[k], __uint_as_float(v1[i + 2 * k]), __uint_as_float(v1[i + 2 * k + 1]));
    }
  }
}

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

// -inf on the masked columns of one 32-column chunk: keys past the query
// (row r of the query tile sees columns up to r + doff of this key tile) or
// past the end of the keys (tail tile, non-causal).
__device__ __forceinline__ void mask_chunk(uint32_t (&v)[32], int ch, bool diag, bool tailt,
                                           int row, int doff, int key0, int Lk) {
#pragma unroll
  for (int e = 0; e < 32; ++e) {
    const int col = ch * 32 + e;
    if ((diag && col > row + doff) || (tailt && key0 + col >= Lk))
      v[e] = __float_as_uint(-INFINITY);
  }
}

}  // namespace

// SKIP: the skip rule is on (lambda > 0). Each mode is its own instantiation,
// so the code generated for one carries no branch of the other.
template <bool FP8, bool SKIP>
__global__ void __launch_bounds__(kFwdThreads, 1) fwd_kernel(const __grid_constant__ FwdParams p) {
  using C = Cfg<FP8>;
  constexpr int KST = Ring<SKIP>::K, VST = Ring<SKIP>::V;
  constexpr uint32_t SM_V = SM_K + KST * kRegion;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar[B_COUNT];
  __shared__ uint32_t tmem_sh;
  __shared__ int item_sh[2][10];
  // keep_sh[s][j & 1] != 0: some row of slot s keeps key tile j (one bit per warp
  // that keeps it); the MMA warp reads it after the slot's four vote arrivals
  __shared__ volatile uint32_t keep_sh[2][2];
  __shared__ volatile int abort_sh;
  // last load issued into each K stage, V stage and the Q slot (-1: none), for
  // the bounded drain after a time-out
  __shared__ int kc_last[kKStages], vc_last[kVStages], qc_last;   // sized for the deeper ring
  // Pipeline counters, persistent across items: each role keeps its own here
  // between items and in registers within one, so that no role carries another
  // role's counters in its registers.
  //   [0, 3)    producer: Q, K, V loads
  //   [3, 9)    MMA warp: Q, K, V, votes of slots 0 / 1, P-ready of slots 0 / 1
  //   [12 + 4 s, 14 + 4 s)  softmax slot s: S tiles, P.V waits
  __shared__ uint32_t ctr_sh[20];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t *sptr = smem_raw + (sbase - raw);
  Workspace *ws = p.ws;
  const uint64_t limit = p.wait_limit_ns;
  constexpr bool v_prefetch = !SKIP;   // no skipping: V streams with K

  if (threadIdx.x == 0) {
    for (int b = 0; b < B_COUNT; ++b)
      mbar_init(&bar[b], (b == B_VOTE || b == B_VOTE + 1) ? 4 : 1);   // a vote: one arrival per warp
    keep_sh[0][0] = keep_sh[0][1] = keep_sh[1][0] = keep_sh[1][1] = 0u;
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
          if (v_prefetch) {
            const uint32_t vs = vc % VST;
            ok = mbar_wait(&bar[B_VE + vs], ((vc / VST) & 1) ^ 1, limit, kSpinIssuer);
            if (!ok) break;
            mbar_expect_tx(&bar[B_VF + vs], C::kTileBytes);
            for (int b = 0; b < C::kBoxes; ++b)
              tma_load_3d(sptr + SM_V + vs * kRegion + b * kBox, tv, &bar[B_VF + vs],
                          b * C::kBoxCols, kvh, kv_row(j));
            vc_last[vs] = (int)vc;
            ++vc;
          }
        }
        ctr_sh[0] = qc;
        ctr_sh[1] = kc;
        ctr_sh[2] = vc;
      }
    } else if (warp == kWarpMma) {
      if (lane == 0) {
        // ------------------------------------------------ MMA issuer
        uint32_t qc = ctr_sh[3], kc = ctr_sh[4], vc = ctr_sh[5];
        uint32_t vt0 = ctr_sh[6], vt1 = ctr_sh[7], pr0 = ctr_sh[8], pr1 = ctr_sh[9];
        const void *tv = &ws->tmap[2];
        const uint32_t S0 = tmem + kColS, S1 = tmem + kColS + 128;
        const uint32_t O0 = tmem + kColO, O1 = tmem + kColO + 128;
        const uint32_t q0s = sbase + SM_Q0, q1s = sbase + SM_Q1;
        // V_j request from this thread (skipping on): only kept tiles are loaded
        auto issue_v = [&](int j) -> bool {
          const uint32_t vs = vc % VST;
          if (!mbar_wait(&bar[B_VE + vs], ((vc / VST) & 1) ^ 1, limit, kSpinIssuer)) return false;
          mbar_expect_tx(&bar[B_VF + vs], C::kTileBytes);
          for (int b = 0; b < C::kBoxes; ++b)
            tma_load_3d(sptr + SM_V + vs * kRegion + b * kBox, tv, &bar[B_VF + vs],
                        b * C::kBoxCols, kvh, kv_row(j));
          vc_last[vs] = (int)vc;
          return true;
        };
        do {
          // no vote of this item is in flight yet (the item started after a CTA barrier)
          keep_sh[0][0] = keep_sh[0][1] = keep_sh[1][0] = keep_sh[1][1] = 0u;
          // key tile 0 is never skipped: request its V before anything else
          if (!v_prefetch && !(ok = issue_v(0))) break;
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
            bool vload = v_prefetch || j == 0;   // V_j requested
            bool vready = false;                 // V_j landed (waited)
            const uint32_t vs = vc % VST;
            auto wait_v = [&]() -> bool {
              if (vready) return true;
              if (!mbar_wait(&bar[B_VF + vs], (vc / VST) & 1, limit, kSpinIssuer)) return false;
              tc_fence_after();
              vready = true;
              return true;
            };
            // ---- slot 0: vote, then P.V (if kept) before the next S overwrites P
            bool keep0 = true;   // with skipping off every tile is kept
            if (!v_prefetch) {
              ok = mbar_wait(&bar[B_VOTE + 0], vt0 & 1, limit, kSpinIssuer);
              ++vt0;
              if (!ok) break;
              keep0 = keep_sh[0][j & 1] != 0;
              keep_sh[0][(j + 1) & 1] = 0u;   // tile j - 1's entry: read, and reused by j + 1
            }
            if (keep0) {
              if (!vload && !(ok = issue_v(j))) break;
              vload = true;
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
              bool keep1 = true;
              if (!v_prefetch) {
                ok = mbar_wait(&bar[B_VOTE + 1], vt1 & 1, limit, kSpinIssuer);
                ++vt1;
                if (!ok) break;
                keep1 = keep_sh[1][j & 1] != 0;
                keep_sh[1][(j + 1) & 1] = 0u;
              }
              if (keep1) {
                if (!vload && !(ok = issue_v(j))) break;
                vload = true;
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
            if (vload) {   // keep the V ring in step even if nobody used the tile
              if (!(ok = wait_v())) break;
              mma_commit(&bar[B_VE + vs]);
              ++vc;
            }
          }
        } while (false);
        ctr_sh[3] = qc;
        ctr_sh[4] = kc;
        ctr_sh[5] = vc;
        ctr_sh[6] = vt0;
        ctr_sh[7] = vt1;
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
        const uint32_t barid = 1 + slot;
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
          if (!mbar_wait(&bar[B_SF + slot], sc & 1, limit, kSpinSoftmax)) abort_sh = 1;
          ++sc;
          tc_fence_after();
          const int doff = doff0 - j * kTile;   // row r sees columns <= r + doff
          const bool diag = p.causal && doff < kTile - 1;
          const bool tailt = tail && j == nk - 1;
          if (v_prefetch && have_kept) {
            // ---- skipping off, after the first tile: one pass over S. P is
            // computed against the current reference max while the row max is
            // taken; only when a row's max outgrows the reference by more than
            // 2^8 is O rescaled and the tile's P recomputed (S is still intact:
            // P is stored at the end).
            if (!mbar_wait(&bar[B_PV + slot], pvc & 1, limit)) abort_sh = 1;
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
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                  const float x = __uint_as_float(v[e]);
                  if (track) tmx[e & 3] = fmaxf(tmx[e & 3], x);
                  pv[e] = ex2_approx(fmaf(x, c, nm));
                  psum[e & 7] += pv[e];
                }
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
            named_bar_sync(barid, 128);
            if (abort_sh) {   // read after the barrier: uniform over the warpgroup
              ok = false;
              break;
            }
            if (row == 0) mbar_arrive(&bar[B_PRDY + slot]);
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
          const float trm = rm * c;
          const bool pred = !valid || (trm < m2 + p.log2_lambda);
          tc_fence_before();
          // each warp posts its vote as soon as it has it (the MMA warp acts on
          // all four arrivals); the warpgroup's own decision is the barrier's
          if (!v_prefetch) {   // with skipping off there is nothing to vote on
            const bool wkeep = !__all_sync(0xffffffffu, pred);
            if (lane == 0) {
              if (wkeep) atomicOr(const_cast<uint32_t *>(&keep_sh[slot][j & 1]), 1u);
              mbar_arrive(&bar[B_VOTE + slot]);
            }
          }
          const bool skip = bar_red_and(pred, barid, 128);
          if (abort_sh) {   // read after the barrier: uniform over the warpgroup
            ok = false;
            break;
          }
          if (skip) {
            if (row == 0) word |= 1u << (j & 31);
          } else {
            const float mnew = valid ? fmaxf(m2, trm) : 0.f;
            if (have_kept) {
              // the previous P.V of this slot is complete by now (it was issued
              // before this tile's S); waiting keeps the phase count exact and
              // orders the O rescale after it
              if (!mbar_wait(&bar[B_PV + slot], pvc & 1, limit)) abort_sh = 1;
              ++pvc;
              tc_fence_after();
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
              }
            } else {
              mref = mnew;
            }
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
            named_bar_sync(barid, 128);
            if (abort_sh) {
              ok = false;
              break;
            }
            if (row == 0) mbar_arrive(&bar[B_PRDY + slot]);
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
  const bool skip = p.log2_lambda > -INFINITY;
  if (fp8) {
    if (skip)
      fwd_kernel<true, true><<<num_ctas, kFwdThreads, smem, stream>>>(p);
    else
      fwd_kernel<true, false><<<num_ctas, kFwdThreads, smem, stream>>>(p);
  } else {
    if (skip)
      fwd_kernel<false, true><<<num_ctas, kFwdThreads, smem, stream>>>(p);
    else
      fwd_kernel<false, false><<<num_ctas, kFwdThreads, smem, stream>>>(p);
  }
  return cudaGetLastError();
}

cudaError_t prepare_forward() {
  const int smem = (int)forward_smem_bytes();
  const cudaFuncAttribute a = cudaFuncAttributeMaxDynamicSharedMemorySize;
  cudaError_t e = cudaFuncSetAttribute(fwd_kernel<false, true>, a, smem);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(fwd_kernel<false, false>, a, smem);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(fwd_kernel<true, true>, a, smem);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(fwd_kernel<true, false>, a, smem);
  return e;
}

}  // namespace bsa
