// Device helpers shared by the prefill kernels (the dense forward and the
// two-phase skipping kernel): tile geometry, the QK^T and P.V MMA issue
// sequences, the work-item fetch, TMEM row loads, the row max and the
// causal / tail masks.
#pragma once

#include <cmath>
#include <cstdint>

#include "bsa_internal.h"
#include "ptx.cuh"

namespace bsa {
namespace tile {

constexpr uint32_t kRegion = 32768;   // one bf16 tile slot in shared memory
constexpr uint32_t kBox = 16384;      // one 128-row x 128-byte TMA box
constexpr float kLn2 = 0.6931471805599453f;

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

__device__ __forceinline__ void fetch_item(const FwdParams &p, int total_items, int maxn, int *dst) {
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
  const int U = p.items_per_group;
  const int r = kr - p.level_start[lo];
  const int s = p.seq_sorted[r / U];
  const int pp = r % U;
  const int h0 = kvh * p.group + p.heads_per_item * pp;
  const int a = p.cu_seqlens[s], ak = p.cu_seqlens_k[s];
  dst[0] = 1;
  dst[1] = s;
  dst[2] = kvh;
  dst[3] = h0;
  dst[4] = (p.heads_per_item == 2 && 2 * pp + 1 < p.group) ? h0 + 1 : -1;
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

}  // namespace tile
}  // namespace bsa
