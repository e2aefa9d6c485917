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
// every decision depends on the tile maxima alone.
//
// One persistent kernel, one CTA per SM, takes work items (sequence, KV head,
// split of 8 or 4 key tiles) from an atomic counter in index order. Per item:
//   scores   S^T = K Q^T on the tensor cores for the split's tiles (K streamed
//            by TMA through a 4-stage ring), kept in TMEM (three items' worth,
//            so that P V work of a split does not hold up the K stream); their
//            per-tile row maxima go to shared memory and the split's row
//            maxima are published;
//   decide   the prefix max before the split, from the published maxima of
//            the earlier splits of the same (sequence, KV head) (a look-back
//            that stops at the nearest split that has published its inclusive
//            prefix), then the split's tiles in order, per query row; the AND
//            over each query head's rows gives its skip bits;
//   P V      for the kept tiles only: V by TMA (all of them prefetched into
//            L2 once the decisions are out), P from the S still in TMEM,
//            O^T = V^T P^T on the tensor cores, an online softmax with the
//            split's own reference max;
//   merge    the item of a (sequence, KV head) that finishes last (a counter)
//            merges the partial results of the splits that kept a tile; no
//            item waits for that.
// Published maxima need no fences: each is one relaxed 64-bit store of the
// value and the call's epoch (a per-stream count of calls), and a reader polls
// until it reads its own call's epoch. The first CTA to arrive writes the
// call's tables (a block-wide scan over the sequences) while the others wait
// for it; nothing else needs clearing between calls. An item waits only for
// items of lower index; those were claimed earlier by CTAs that are running
// and publish their maxima before they wait for anything outside their CTA,
// so the waits end; each is bounded by the wait limit all the same.
// Decisions equal the sequential walk's; outputs equal the online softmax
// over the kept tiles up to rounding order. The work is bound by reading K
// once and the kept V once from DRAM.
#include <cuda_bf16.h>

#include <climits>
#include <cmath>

#include "bsa_decode.h"
#include "ptx.cuh"

namespace bsa {

namespace {

constexpr uint32_t kTileBytes = 32768;   // 128 keys x 128 bf16
constexpr uint32_t kBoxBytes = 16384;    // one 128-row x 128-byte TMA box
constexpr float kLn2 = 0.6931471805599453f;

struct DecItem {
  int s, kvh, q, j0, j1, aq, Lq, ak, Lk, ns;
};

// item_off: the call's per-sequence first work items (shared memory or scratch)
__device__ __forceinline__ void decode_item(const DecParams &p, const int32_t *item_off, int item,
                                            DecItem &it) {
  int lo = 0, hi = p.n_seqs;   // largest s with item_off[s] <= item
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (item_off[mid] <= item) lo = mid; else hi = mid;
  }
  it.s = lo;
  it.aq = p.cu_q[lo];
  it.Lq = p.cu_q[lo + 1] - it.aq;
  it.ak = p.cu_k[lo];
  it.Lk = p.cu_k[lo + 1] - it.ak;
  const int nk = (it.Lk + kTile - 1) / kTile;
  it.ns = (nk + p.split - 1) / p.split;
  // the KV heads of one split are neighbours: CTAs running together read
  // whole token rows of K and V (all heads) from DRAM
  const int local = item - item_off[lo];
  it.q = local / p.Hkv;
  it.kvh = local - it.q * p.Hkv;
  it.j0 = it.q * p.split;
  it.j1 = min(nk, it.j0 + p.split);
}

// Run by one warp before the kernel waits for the previous kernel on the
// stream: the K tiles of work item blockIdx.x, the item this CTA most likely
// claims first, for L2, while the previous kernel's last CTAs finish. The
// lengths are read before they are guaranteed to be final, so a stale value
// only misplaces a prefetch (the TMA bounds its coordinates; the real tables
// are computed after the wait). Batches of at most 32 sequences.
__device__ __forceinline__ void prefetch_first_item(const DecParams &p, const CUtensorMap *tk,
                                                    int lane) {
  if (p.n_seqs > 32) return;
  int ni = 0, ak = 0, nk = 0;   // lane s: sequence s's items, first key, key tiles
  if (lane < p.n_seqs) {
    const int q0 = __ldcv(p.cu_q + lane), q1 = __ldcv(p.cu_q + lane + 1);
    ak = __ldcv(p.cu_k + lane);
    const int lk = __ldcv(p.cu_k + lane + 1) - ak;
    if (q1 > q0 && lk > 0) {
      nk = (lk + kTile - 1) / kTile;
      ni = p.Hkv * ((nk + p.split - 1) / p.split);
    }
  }
  int incl = ni;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int x = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += x;
  }
  const int b = blockIdx.x;
  if (ni > 0 && incl - ni <= b && b < incl) {   // at most one lane: the item's sequence
    const int local = b - (incl - ni);
    const int q = local / p.Hkv, kvh = local - q * p.Hkv;
    const int j0 = q * p.split, j1 = min(nk, j0 + p.split);
    for (int j = j0; j < j1; ++j) {
      tma_prefetch_3d(tk, 0, kvh, ak + j * kTile);
      tma_prefetch_3d(tk, 64, kvh, ak + j * kTile);
    }
  }
}

// One 128-key tile of K or V (both 64-column boxes); K and V are read once,
// so their lines leave L2 first and the per-item tables stay.
__device__ __forceinline__ void load_tile(uint8_t *dst, const CUtensorMap *map, uint64_t *bar,
                                          int head, int row, uint64_t policy) {
  mbar_expect_tx(bar, kTileBytes);
  tma_load_3d_hint(dst, map, bar, 0, head, row, policy);
  tma_load_3d_hint(dst + kBoxBytes, map, bar, 64, head, row, policy);
}

// Two published (epoch, value) words at once (16-byte aligned); several can
// be in flight.
__device__ __forceinline__ void ld_volatile_pair(const uint64_t *a, uint64_t &x, uint64_t &y) {
  asm volatile("ld.volatile.global.v2.u64 {%0,%1}, [%2];" : "=l"(x), "=l"(y) : "l"(a));
}
// Publish a maximum: one relaxed 64-bit store of (epoch, f32 bits).
__device__ __forceinline__ void publish(uint64_t *a, uint32_t epoch, float v) {
  const uint64_t w = ((uint64_t)epoch << 32) | __float_as_uint(v);
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(a), "l"(w) : "memory");
}
__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t *a) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(a) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_u32(uint32_t *a, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(a), "r"(v) : "memory");
}
// Epoch-tagged counters (epoch << 32 | count): lift a word an earlier call
// left to (epoch, 0) -- epochs only grow -- then count; same thread, same
// word, so the add sees the lift.
__device__ __forceinline__ void counter_enter(uint64_t *a, uint32_t epoch) {
  asm volatile("red.relaxed.gpu.global.max.u64 [%0], %1;" ::"l"(a), "l"((uint64_t)epoch << 32)
               : "memory");
}
__device__ __forceinline__ uint32_t counter_add(uint64_t *a) {
  uint64_t old;
  asm volatile("atom.relaxed.gpu.global.add.u64 %0, [%1], 1;" : "=l"(old) : "l"(a) : "memory");
  return (uint32_t)old;
}
__device__ __forceinline__ uint32_t counter_add_acq_rel(uint64_t *a) {
  uint64_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u64 %0, [%1], 1;" : "=l"(old) : "l"(a) : "memory");
  return (uint32_t)old;
}
__device__ __forceinline__ uint32_t counter_add_acquire(uint64_t *a) {
  uint64_t old;
  asm volatile("atom.acquire.gpu.global.add.u64 %0, [%1], 1;" : "=l"(old) : "l"(a) : "memory");
  return (uint32_t)old;
}

// Wait for a phase of an mbarrier; false when the CTA is aborting or the wait
// ran past the limit (then the CTA aborts).
__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, uint64_t limit,
                                         volatile int *abort) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 16; ++i)
      if (mbar_try_wait(a, parity)) return true;
    if (*abort) return false;
    if (globaltimer_ns() - t0 > limit) {
      *abort = 1;
      return false;
    }
  }
}

// The first R of RB published (epoch, value) words at a (16-byte aligned, RB
// even) into w, loads in flight together.
template <int RB>
__device__ __forceinline__ void load_maxima(const uint64_t *a, int R, uint64_t (&w)[RB]) {
#pragma unroll
  for (int r = 0; r < RB; r += 2) {
    w[r] = w[r + 1] = 0;
    if (r < R) ld_volatile_pair(a + r, w[r], w[r + 1]);
  }
}
template <int RB>
__device__ __forceinline__ bool all_published(const uint64_t (&w)[RB], int R, uint32_t epoch) {
  bool ok = true;
#pragma unroll
  for (int r = 0; r < RB; ++r) ok = ok && (r >= R || (uint32_t)(w[r] >> 32) == epoch);
  return ok;
}
__device__ __forceinline__ float value_of(uint64_t w) { return __uint_as_float((uint32_t)w); }

// Wait until the first R maxima at a carry this call's epoch; false on a CTA
// or grid abort, or past the limit.
template <int RB>
__device__ __forceinline__ bool wait_maxima(const uint64_t *a, int R, uint64_t (&w)[RB], uint32_t epoch,
                                            uint64_t limit, volatile int *abort,
                                            const volatile uint32_t *gabort) {
  load_maxima<RB>(a, R, w);
  if (all_published<RB>(w, R, epoch)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    __nanosleep(64);
    load_maxima<RB>(a, R, w);
    if (all_published<RB>(w, R, epoch)) return true;
    if (*abort || *gabort == epoch) return false;
    if (globaltimer_ns() - t0 > limit) return false;
  }
}

// Maximum over the warp in one redux: floats map to int32 keys that compare
// in the same order (negative floats have their magnitude bits flipped).
__device__ __forceinline__ float warp_max(float x) {
  const int i = __float_as_int(x);
  const int k = __reduce_max_sync(0xffffffffu, i >= 0 ? i : i ^ 0x7FFFFFFF);
  return __int_as_float(k >= 0 ? k : k ^ 0x7FFFFFFF);
}



}  // namespace

// ============================================================ decode

namespace {

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

// N TMEM columns (N = 16 or 32) of this warp's 32 lanes into v.
template <int N>
__device__ __forceinline__ void tmem_ldN(uint32_t taddr, uint32_t (&v)[N]) {
  tmem_ld16(taddr, *reinterpret_cast<uint32_t(*)[16]>(&v[0]));
  if constexpr (N > 16) tmem_ld16(taddr + 16, *reinterpret_cast<uint32_t(*)[16]>(&v[16]));
  tmem_wait_ld16(*reinterpret_cast<uint32_t(*)[16]>(&v[0]));
  if constexpr (N > 16) tmem_wait_ld16(*reinterpret_cast<uint32_t(*)[16]>(&v[16]));
}

// RB >= group x Lq query rows; N = RB rounded up to 16 is the MMA width; an
// item's scores take 128 TMEM columns (kSplit tiles x N), three items' worth,
// then two N-column P V accumulators.
template <int RB>
struct DecCfg {
  static constexpr int N = RB < 16 ? 16 : RB;
  static constexpr int kSplit = 128 / N;
  static constexpr int KST = N == 16 ? 4 : 3;   // K ring stages
  static constexpr int VST = 2;                 // V ring stages
  static constexpr uint32_t kQBytes = N * 256;  // query rows, bf16, 128-byte swizzled
  static constexpr uint32_t kPBytes = N * 256;  // P, bf16, 128-byte swizzled
  static constexpr uint32_t kVOff = KST * kTileBytes;
  static constexpr uint32_t kQOff = kVOff + VST * kTileBytes;
  static constexpr uint32_t kPOff = kQOff + 2 * kQBytes;
  static constexpr size_t kSmem = 1024 + kPOff + 2 * kPBytes;
  static constexpr int kSBufs = 3;              // items whose scores TMEM holds
  static constexpr uint32_t kDCol = kSBufs * 128;   // first P V accumulator column
};

constexpr int kGroup = 128;          // threads of the score group and of the P V group
constexpr int kDecThreadsAll = 384;  // two groups + K producer, V producer, two MMA warps
// Registers per thread: the launch gives every thread kRegsLaunch; the
// producer / MMA warpgroup gives most of its share to the two groups.
constexpr uint32_t kRegsLaunch = 168, kRegsIssue = 64, kRegsScore = 184, kRegsPV = 256;
static_assert(kGroup * (kRegsScore + kRegsPV + kRegsIssue) <= kDecThreadsAll * kRegsLaunch,
              "register split above the launch allocation");
constexpr int kMaxSplitRB = 128;     // kSplit x RB: tile-max entries of one item

}  // namespace

// The call's tables, written by all NT threads of a CTA: per sequence its
// first work item and first skip-bitmap word (a block-wide scan over the
// sequences, NT at a time) into item_off / bm_off, the checks of the lengths
// on the device, and the item count into items_sh (0 when rejected).
// bad_sh and carry start at zero (set with the barriers at kernel start), so
// the first loads of the lengths are also the first memory round trip.
template <int NT>
__device__ void dec_tables(const DecParams &p, long long (&wsum)[NT / 32][2], long long (&carry)[2],
                           int &bad_sh, int32_t *item_off, int64_t *bm_off, int &items_sh) {
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  if (t == 0 && (p.cu_q[0] != 0 || p.cu_k[0] != 0 || (int64_t)p.cu_k[p.n_seqs] != p.total_k))
    atomicOr(&bad_sh, 1);
  for (int b0 = 0; b0 < p.n_seqs; b0 += NT) {
    const int s = b0 + t;
    long long ni = 0, nw = 0;   // this sequence's work items and bitmap words
    if (s < p.n_seqs) {
      const int Lq = p.cu_q[s + 1] - p.cu_q[s], Lk = p.cu_k[s + 1] - p.cu_k[s];
      if (Lq < 0 || Lk < 0 || Lq > p.max_q || (p.causal && Lk < Lq) || (Lq > 0 && Lk == 0)) {
        atomicOr(&bad_sh, 1);
      } else {
        const long long nk = (Lk + kTile - 1) / kTile, nq = (Lq + kTile - 1) / kTile;
        if (Lq > 0) ni = (long long)p.Hkv * ((nk + p.split - 1) / p.split);
        nw = (long long)p.Hq * nq * ((nk + 31) / 32);
      }
    }
    long long si = ni, sw = nw;   // inclusive scans within the warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long xi = __shfl_up_sync(0xffffffffu, si, o);
      const long long xw = __shfl_up_sync(0xffffffffu, sw, o);
      if (lane >= o) {
        si += xi;
        sw += xw;
      }
    }
    if (lane == 31) {
      wsum[warp][0] = si;
      wsum[warp][1] = sw;
    }
    __syncthreads();
    long long oi = carry[0], ow = carry[1];
    for (int w = 0; w < warp; ++w) {
      oi += wsum[w][0];
      ow += wsum[w][1];
    }
    if (s < p.n_seqs) {
      item_off[s] = (int32_t)min(oi + si - ni, (long long)INT_MAX);
      bm_off[s] = ow + sw - nw;
    }
    __syncthreads();
    if (t == 0)
      for (int w = 0; w < NT / 32; ++w) {
        carry[0] += wsum[w][0];
        carry[1] += wsum[w][1];
      }
    __syncthreads();
  }
  if (t == 0) {
    const long long items = carry[0];
    item_off[p.n_seqs] = (int32_t)min(items, (long long)INT_MAX);
    bm_off[p.n_seqs] = carry[1];
    const bool bad = bad_sh != 0 || items > p.max_items;
    items_sh = bad ? 0 : (int32_t)items;
    if (bad) atomicOr(&p.ws->status, kStatusBadSeqlens);
  }
  __syncthreads();
}

// Roles:
//   warps 0-3   score group: the scores of the split from TMEM (thread =
//               key), per-tile row maxima, the split maxima published; the
//               look-back, the decisions, the kept list and the skip bits
//   warps 4-7   P V group: P of the kept tiles (thread = key), O (thread =
//               head-dim column), partial results, the merge
//   warp 8      claims items, stages their query rows (the score MMA's B
//               operand); lane 0: TMA producer of the K ring
//   warp 9      lane 0: TMA producer of the V ring (kept tiles only)
//   warp 10     TMEM allocation; lane 0 issues the score MMAs
//   warp 11     lane 0 issues the P V MMAs
template <int RB>
__global__ void __launch_bounds__(kDecThreadsAll, 1)
dec_kernel(const __grid_constant__ DecParams p, const __grid_constant__ CUtensorMap tk,
           const __grid_constant__ CUtensorMap tv) {
  using C = DecCfg<RB>;
  constexpr int N = C::N, KST = C::KST, VST = C::VST, SPL = C::kSplit;
  // scores: bf16 x bf16 -> f32, both K-major, M = 128 keys, N rows
  constexpr uint32_t kIdescS = IDesc<1, false, 128, N>::value;
  // P V: A (V) MN-major (bit 15), B (P) K-major, M = 128 head-dim columns
  constexpr uint32_t kIdescO = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 15) |
                               ((uint32_t)(N >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
  extern __shared__ uint8_t smem_raw[];
  __shared__ float red[4][kMaxSplitRB];   // per warp: max over its 32 keys, [tile][row]
  __shared__ float tmax[3][kMaxSplitRB];  // per score buffer: tile row maxima, [tile][row]
  __shared__ float mred[4][RB], lred[4][RB];
  __shared__ int klist[2][SPL];
  __shared__ uint32_t kact[2][SPL];
  __shared__ int nkept_sh[2];
  __shared__ int it_sh[4];
  __shared__ int wmin[4], wcnt[4], clist[kGroup];
  __shared__ int merge_sh;
  __shared__ float pmsh[16][RB], plsh[16][RB], wsh[16][RB];
  __shared__ float msh[RB], lsh[RB], scsh[RB];
  __shared__ uint64_t itfull[4], itempty[4], kfull[KST], kempty[KST], vfull[VST], vempty[VST],
      qready[2], qfree[2], sfull[3], sfree[3], lready[2], lfree[2], pready[2], pfree[2],
      dfull[2], dempty[2], drain[2];
  __shared__ long long wsum[kDecThreadsAll / 32][2], carry[2];
  __shared__ int bad_sh, owner_sh, items_sh;
  __shared__ int32_t s_iofs[kDecLocalSeqs + 1];
  __shared__ int64_t s_bofs[kDecLocalSeqs + 1];
  __shared__ uint32_t tmem_sh;
  __shared__ volatile int abort_sh;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t *base = smem_raw + (sbase - raw);
  if (t == 0) {
    for (int b = 0; b < 4; ++b) {
      mbar_init(&itfull[b], 1);
      mbar_init(&itempty[b], 5);   // score MMA, score group, P V group, V producer, P V MMA
    }
    for (int b = 0; b < KST; ++b) {
      mbar_init(&kfull[b], 1);
      mbar_init(&kempty[b], 1);
    }
    for (int b = 0; b < VST; ++b) {
      mbar_init(&vfull[b], 1);
      mbar_init(&vempty[b], 1);
    }
    for (int b = 0; b < 3; ++b) {
      mbar_init(&sfull[b], 1);
      mbar_init(&sfree[b], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&qready[b], 1);
      mbar_init(&qfree[b], 1);
      mbar_init(&lready[b], 1);
      mbar_init(&lfree[b], 3);   // V producer, P V MMA, P V group
      mbar_init(&pready[b], 1);
      mbar_init(&pfree[b], 1);
      mbar_init(&dfull[b], 1);
      mbar_init(&dempty[b], kGroup / 32);
      mbar_init(&drain[b], 1);
    }
    fence_mbar_init();
    abort_sh = 0;
    bad_sh = 0;
    carry[0] = carry[1] = 0;
  }
  if (warp == 10) {
    tmem_alloc(&tmem_sh, 512);
    tmem_relinquish();
  }
  // the P buffers start zeroed: rows past RB are never written again
  for (uint32_t x = t; x < 2 * C::kPBytes / 16; x += kDecThreadsAll)
    reinterpret_cast<uint4 *>(base + C::kPOff)[x] = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_sh;
  if (warp == 8) prefetch_first_item(p, &tk, lane);
  grid_dep_wait();     // the previous kernel on the stream is done
  grid_dep_launch();
  const uint64_t limit = p.wait_limit_ns;
  const volatile uint32_t *gabort = &p.dw->abort;   // == epoch: a CTA gave up
  // the first claim goes out now: its round trip overlaps the tables
  uint32_t first_claim = 0;
  if (warp == 8 && lane == 0) {
    counter_enter(&p.dw->claim, p.epoch);
    first_claim = counter_add(&p.dw->claim);
  }
  // the call's tables: a batch of at most kDecLocalSeqs sequences in every
  // CTA's shared memory; a larger one once, by the first CTA to arrive, in the
  // scratch, while the others wait for it
  const bool local_tables = p.n_seqs <= kDecLocalSeqs;
  if (local_tables) {
    dec_tables<kDecThreadsAll>(p, wsum, carry, bad_sh, s_iofs, s_bofs, items_sh);
  } else {
    if (t == 0) owner_sh = atomicExch(&p.dw->setup_owner, p.epoch) != p.epoch;
    __syncthreads();
    if (owner_sh) {
      dec_tables<kDecThreadsAll>(p, wsum, carry, bad_sh, const_cast<int32_t *>(p.item_off),
                                 const_cast<int64_t *>(p.bm_off), items_sh);
      if (t == 0) {
        p.dw->total_items = items_sh;
        __threadfence();
        st_release_u32(&p.dw->setup_done, p.epoch);
      }
    } else if (t == 0) {
      bool ok = ld_acquire_u32(&p.dw->setup_done) == p.epoch;
      const uint64_t t0 = globaltimer_ns();
      while (!ok && globaltimer_ns() - t0 <= limit) {
        __nanosleep(100);
        ok = ld_acquire_u32(&p.dw->setup_done) == p.epoch;
      }
      items_sh = ok ? __ldcg(&p.dw->total_items) : 0;
      if (!ok) abort_sh = 1;
    }
  }
  __syncthreads();
  const int total = abort_sh ? 0 : items_sh;
  const int32_t *iofs = local_tables ? s_iofs : p.item_off;
  const int64_t *bofs = local_tables ? s_bofs : p.bm_off;

  if (warp >= 8) {
    reg_dealloc<kRegsIssue>();
    const uint64_t pol = policy_evict_first();
    if (warp == 8) {
      // ---------------------------------------------------- claims, Q rows, K producer
      const __nv_bfloat16 *q = static_cast<const __nv_bfloat16 *>(p.q);
      uint32_t kc = 0;
      int last_issue[KST];
  #pragma unroll
      for (int b = 0; b < KST; ++b) last_issue[b] = -1;
      for (uint32_t i = 0;; ++i) {
        const uint32_t slot = i & 3, par = i & 1;
        int item = -1;
        bool ok = true;
        if (lane == 0) {
          ok = wait_bar(&itempty[slot], ((i >> 2) & 1) ^ 1, limit, &abort_sh);
          // claims only (never a fixed item per CTA): every claimed item then
          // belongs to a CTA that is running, even when other grids hold SMs
          if (ok && !abort_sh && *gabort != p.epoch) {
            const uint32_t c = i == 0 ? first_claim : counter_add(&p.dw->claim);
            item = c >= (uint32_t)total ? -1 : (int)c;
          }
          if (ok) {
            it_sh[slot] = item;
            mbar_arrive(&itfull[slot]);
          }
          // the score MMAs of the item two back have read this query buffer
          if (ok && item >= 0 && i >= 2) ok = wait_bar(&qfree[par], ((i >> 1) - 1) & 1, limit, &abort_sh);
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        item = __shfl_sync(0xffffffffu, item, 0);
        if (!ok || item < 0) break;
        DecItem it;
        decode_item(p, iofs, item, it);
        // K loads into ring stages that are free right now go first (at the
        // start, the whole ring), the rest after the query rows are staged
        int jn = it.j0;
        if (lane == 0) {
          for (; jn < it.j1; ++jn, ++kc) {
            const uint32_t b = kc % KST;
            if (!mbar_test_wait(smem_u32(&kempty[b]), ((kc / KST) & 1) ^ 1)) break;
            if ((int)kc != p.debug_drop_k_load) {
              load_tile(base + b * kTileBytes, &tk, &kfull[b], it.kvh, it.ak + jn * kTile, pol);
              last_issue[b] = (int)kc;
            }
          }
        }
        // B operand: query row r at its 128-byte-swizzled K-major position
        const int R = p.group * it.Lq;
        uint8_t *qb = base + C::kQOff + par * C::kQBytes;
        for (int c = lane; c < N * 16; c += 32) {
          const int r = c >> 4, ch = c & 15;
          uint4 w = make_uint4(0u, 0u, 0u, 0u);
          if (r < R) {
            const int h = it.kvh * p.group + r / it.Lq, qi = r % it.Lq;
            w = *reinterpret_cast<const uint4 *>(q + ((size_t)(it.aq + qi) * p.Hq + h) * kTile + ch * 8);
          }
          *reinterpret_cast<uint4 *>(qb + (ch >> 3) * (N * 128) + r * 128 + (((ch & 7) ^ (r & 7)) << 4)) = w;
        }
        fence_proxy_async_smem();
        __syncwarp();
        bool okk = true;
        if (lane == 0) {
          mbar_arrive(&qready[par]);
          for (int j = jn; j < it.j1; ++j, ++kc) {
            const uint32_t b = kc % KST;
            if (!(okk = wait_bar(&kempty[b], ((kc / KST) & 1) ^ 1, limit, &abort_sh))) break;
            if ((int)kc != p.debug_drop_k_load) {
              load_tile(base + b * kTileBytes, &tk, &kfull[b], it.kvh, it.ak + j * kTile, pol);
              last_issue[b] = (int)kc;
            }
          }
        }
        if (!__shfl_sync(0xffffffffu, okk, 0)) break;
      }
      if (lane == 0 && abort_sh)   // bounded wait for the copies still in flight
        for (int b = 0; b < KST; ++b)
          if (last_issue[b] >= 0) mbar_wait(&kfull[b], (last_issue[b] / KST) & 1, limit);
    } else if (warp == 9) {
      // ---------------------------------------------------- V producer
      if (lane == 0) {
        uint32_t vc = 0;
        int last_issue[VST];
  #pragma unroll
        for (int b = 0; b < VST; ++b) last_issue[b] = -1;
        for (uint32_t i = 0;; ++i) {
          const uint32_t slot = i & 3, par = i & 1;
          if (!wait_bar(&itfull[slot], (i >> 2) & 1, limit, &abort_sh)) break;
          const int item = it_sh[slot];
          mbar_arrive(&itempty[slot]);
          if (item < 0) break;
          DecItem it;
          decode_item(p, iofs, item, it);
          if (!wait_bar(&lready[par], (i >> 1) & 1, limit, &abort_sh)) break;
          const int n = nkept_sh[par];
          // every kept tile's V heads for L2 at once; the two ring stages then
          // fill from L2 instead of waiting out DRAM latency tile by tile
          for (int u = VST; u < n; ++u) {
            tma_prefetch_3d(&tv, 0, it.kvh, it.ak + klist[par][u] * kTile);
            tma_prefetch_3d(&tv, 64, it.kvh, it.ak + klist[par][u] * kTile);
          }
          bool ok = true;
          for (int u = 0; u < n; ++u, ++vc) {
            const uint32_t b = vc % VST;
            if (!(ok = wait_bar(&vempty[b], ((vc / VST) & 1) ^ 1, limit, &abort_sh))) break;
            load_tile(base + C::kVOff + b * kTileBytes, &tv, &vfull[b], it.kvh,
                      it.ak + klist[par][u] * kTile, pol);
            last_issue[b] = (int)vc;
          }
          if (!ok) break;
          mbar_arrive(&lfree[par]);
        }
        if (abort_sh)
          for (int b = 0; b < VST; ++b)
            if (last_issue[b] >= 0) mbar_wait(&vfull[b], (last_issue[b] / VST) & 1, limit);
      }
    } else if (warp == 10) {
      // ---------------------------------------------------- score MMAs
      if (lane == 0) {
        uint32_t kc = 0;
        for (uint32_t i = 0;; ++i) {
          const uint32_t slot = i & 3, par = i & 1;
          if (!wait_bar(&itfull[slot], (i >> 2) & 1, limit, &abort_sh)) break;
          const int item = it_sh[slot];
          mbar_arrive(&itempty[slot]);
          if (item < 0) break;
          DecItem it;
          decode_item(p, iofs, item, it);
          // the query rows are staged, and the P V group is done with the S
          // columns of the item three back
          const uint32_t sb = i % 3;
          if (!wait_bar(&qready[par], (i >> 1) & 1, limit, &abort_sh)) break;
          if (!wait_bar(&sfree[sb], ((i / 3) & 1) ^ 1, limit, &abort_sh)) break;
          tc_fence_after();
          const uint32_t qs = sbase + C::kQOff + par * C::kQBytes;
          bool ok = true;
          for (int j = it.j0; j < it.j1; ++j, ++kc) {
            const uint32_t b = kc % KST;
            if (!(ok = wait_bar(&kfull[b], (kc / KST) & 1, limit, &abort_sh))) break;
            tc_fence_after();
            const uint32_t ks = sbase + b * kTileBytes;
            const uint32_t dcol = sb * 128 + (j - it.j0) * N;
  #pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint32_t ka = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
              const uint32_t kb = (kk >> 2) * (N * 128) + (kk & 3) * 32;
              mma_f16_ss(tmem + dcol, sdesc_sw128(ks + ka, 16, 1024), sdesc_sw128(qs + kb, 16, 1024),
                         kIdescS, kk > 0);
            }
            mma_commit(&kempty[b]);
          }
          if (!ok) break;
          mma_commit(&sfull[sb]);
          mma_commit(&qfree[par]);
        }
        if (abort_sh) {   // this thread's MMAs finish before TMEM is freed
          mma_commit(&drain[0]);
          mbar_wait(&drain[0], 0, limit);
        }
      }
    } else {   // warp 11
      // ---------------------------------------------------- P V MMAs
      if (lane == 0) {
        uint32_t vc = 0;
        for (uint32_t i = 0;; ++i) {
          const uint32_t slot = i & 3, par = i & 1;
          if (!wait_bar(&itfull[slot], (i >> 2) & 1, limit, &abort_sh)) break;
          const int item = it_sh[slot];
          mbar_arrive(&itempty[slot]);
          if (item < 0) break;
          if (!wait_bar(&lready[par], (i >> 1) & 1, limit, &abort_sh)) break;
          const int n = nkept_sh[par];
          mbar_arrive(&lfree[par]);
          bool ok = true;
          for (int u = 0; u < n; ++u, ++vc) {
            const uint32_t b = vc % VST, ps = vc & 1;
            if (!(ok = wait_bar(&vfull[b], (vc / VST) & 1, limit, &abort_sh))) break;
            if (!(ok = wait_bar(&pready[ps], (vc >> 1) & 1, limit, &abort_sh))) break;
            if (!(ok = wait_bar(&dempty[ps], ((vc >> 1) & 1) ^ 1, limit, &abort_sh))) break;
            tc_fence_after();
            const uint32_t vs = sbase + C::kVOff + b * kTileBytes;
            const uint32_t pb = sbase + C::kPOff + ps * C::kPBytes;
  #pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              // A: 16 keys = two 8-key swizzle atoms (2048 bytes); the two 64-wide
              // halves of the head dim are one box apart. B: 32 bytes per K step.
              const uint64_t ad = sdesc_sw128(vs + kk * 2048, kBoxBytes, 1024);
              const uint64_t bd = sdesc_sw128(pb + (kk >> 2) * (N * 128) + (kk & 3) * 32, 16, 1024);
              mma_f16_ss(tmem + C::kDCol + ps * N, ad, bd, kIdescO, kk > 0);
            }
            mma_commit(&dfull[ps]);
            mma_commit(&vempty[b]);
            mma_commit(&pfree[ps]);
          }
          if (!ok) break;
        }
        if (abort_sh) {
          mma_commit(&drain[1]);
          mbar_wait(&drain[1], 0, limit);
        }
      }
    }
  } else if (warp < 4) {
    reg_alloc<kRegsScore>();
    // ---------------------------------------------------- score group
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    for (uint32_t i = 0;; ++i) {
      const uint32_t slot = i & 3, par = i & 1, sb = i % 3;
      // control flow follows barrier reductions only, so the four warps agree
      bool ok = wait_bar(&itfull[slot], (i >> 2) & 1, limit, &abort_sh);
      const int item = ok ? it_sh[slot] : -1;
      if (bar_red_or(!ok, 1, kGroup)) break;
      if (t == 0) mbar_arrive(&itempty[slot]);
      if (item < 0) break;
      DecItem it;
      decode_item(p, iofs, item, it);
      const int R = p.group * it.Lq, nt = it.j1 - it.j0;
      const int64_t first = (int64_t)iofs[it.s] + it.kvh;   // split qq is first + qq * Hkv
      const int64_t bmo = p.bitmap ? bofs[it.s] : 0;
      // key position of each row's query (rows past R: unused)
      int pos[RB];
#pragma unroll
      for (int r = 0; r < RB; ++r) pos[r] = it.Lk - it.Lq + (r < R ? r % it.Lq : 0);
      // the look-back's first window (the nearest 128 earlier splits): loads
      // issued now, while this split's K tiles still stream in
      uint64_t a[RB], c[RB];
      if (t < it.q) {
        const int64_t prow = (first + (int64_t)(it.q - 1 - t) * p.Hkv) * p.mpitch;
        load_maxima<RB>(p.incl + prow, R, c);
        load_maxima<RB>(p.agg + prow, R, a);
      }
      ok = wait_bar(&sfull[sb], (i / 3) & 1, limit, &abort_sh);
      if (bar_red_or(!ok, 1, kGroup)) break;
      tc_fence_after();
      for (int u = 0; u < nt; ++u) {
        uint32_t v[N];
        tmem_ldN<N>(tmem + lane_off + sb * 128 + u * N, v);
        const int kpos = (it.j0 + u) * kTile + t;
        const bool out = kpos >= it.Lk;
#pragma unroll
        for (int r = 0; r < RB; ++r) {
          const bool masked = out || (p.causal && kpos > pos[r]);
          const float m = warp_max(masked ? -INFINITY : __uint_as_float(v[r]) * p.c);
          if (lane == 0) red[warp][u * RB + r] = m;
        }
      }
      tc_fence_before();
      named_bar_sync(1, kGroup);
      for (int x = t; x < nt * RB; x += kGroup)
        tmax[sb][x] = fmaxf(fmaxf(red[0][x], red[1][x]), fmaxf(red[2][x], red[3][x]));
      if (t < R) {   // the split's row maxima, for the look-back of later splits
        float m = -INFINITY;
        for (int u = 0; u < nt; ++u)
          m = fmaxf(m, fmaxf(fmaxf(red[0][u * RB + t], red[1][u * RB + t]),
                             fmaxf(red[2][u * RB + t], red[3][u * RB + t])));
        publish(p.agg + (int64_t)item * p.mpitch + t, p.epoch, m);
      }
      named_bar_sync(1, kGroup);   // tmax and the split maxima are out

      // ---- running max before the split (after this split's own maxima are
      // out, so that no split waits for one that waits for it): nearest
      // earlier splits first, 128 at a time, down to the nearest one with an
      // inclusive prefix; values the prefetch found unpublished are waited for
      float mp[RB];
#pragma unroll
      for (int r = 0; r < RB; ++r) mp[r] = -INFINITY;
      bool fail = false, anyfail = false;
      for (int hi = it.q; hi > 0; hi -= kGroup) {
        // thread t: split qq; its row maxima (waited for) and, if every
        // row's inclusive prefix is out already, those
        const int qq = hi - 1 - t;
        const bool mine = t < hi;   // qq >= 0; the window is hi-128 .. hi-1
        const int64_t prow = (first + (int64_t)qq * p.Hkv) * p.mpitch;
        bool incl_ok = false;
        if (mine) {
          if (hi != it.q) {
            load_maxima<RB>(p.incl + prow, R, c);
            load_maxima<RB>(p.agg + prow, R, a);
          }
          incl_ok = all_published<RB>(c, R, p.epoch);
          if (!all_published<RB>(a, R, p.epoch) &&
              !wait_maxima<RB>(p.agg + prow, R, a, p.epoch, limit, &abort_sh, gabort))
            fail = true;
        }
        if (bar_red_or(fail, 1, kGroup)) {
          anyfail = true;
          break;
        }
        const unsigned bal = __ballot_sync(0xffffffffu, incl_ok);
        if (lane == 0) wmin[warp] = bal ? warp * 32 + __ffs(bal) - 1 : INT_MAX;
        named_bar_sync(1, kGroup);
        const int tmin = min(min(wmin[0], wmin[1]), min(wmin[2], wmin[3]));
        if (mine && t <= tmin) {
#pragma unroll
          for (int r = 0; r < RB; ++r)
            if (r < R) mp[r] = fmaxf(mp[r], value_of(t == tmin ? c[r] : a[r]));
        }
        named_bar_sync(1, kGroup);   // wmin is rewritten by the next window
        if (tmin != INT_MAX) break;
      }
      if (anyfail) {
        abort_sh = 1;
        break;
      }
#pragma unroll
      for (int r = 0; r < RB; ++r) {
        const float m = warp_max(mp[r]);
        if (lane == 0) mred[warp][r] = m;
      }

      // the kept lists of the item two back are no longer read
      ok = wait_bar(&lfree[par], ((i >> 1) & 1) ^ 1, limit, &abort_sh);
      if (bar_red_or(!ok, 1, kGroup)) break;

      // ---- decisions, in the group's first warp (R <= 32 rows): walk the
      // split's tiles in order per row; a head skips a tile when all its rows
      // do; the kept list and the skip bits follow from ballots
      if (warp == 0) {
        uint32_t bits = 0;   // bit u: row lane would skip tile j0 + u
        if (lane < R) {
          float mr = fmaxf(fmaxf(mred[0][lane], mred[1][lane]), fmaxf(mred[2][lane], mred[3][lane]));
          for (int u = 0; u < nt; ++u) {
            const float x = tmax[sb][u * RB + lane];
            if (x < mr + p.log2_lambda) bits |= 1u << u;
            mr = fmaxf(mr, x);
          }
          // max over every tile up to the split's end: the later splits' look-back
          publish(p.incl + (int64_t)item * p.mpitch + lane, p.epoch, mr);
        }
        // lane g < group: the tiles head g skips (the AND over its query rows)
        uint32_t hs = nt >= 32 ? 0xFFFFFFFFu : ((1u << nt) - 1u);
        for (int qi = 0; qi < it.Lq; ++qi) {
          const uint32_t b = __shfl_sync(0xffffffffu, bits, (lane * it.Lq + qi) & 31);
          hs &= b;
        }
        const bool head = lane < p.group;
        int n = 0;
        for (int u = 0; u < nt; ++u) {
          const uint32_t act = __ballot_sync(0xffffffffu, head && !((hs >> u) & 1u));
          if (act) {
            if (lane == 0) {
              klist[par][n] = it.j0 + u;
              kact[par][n] = act;
            }
            ++n;
          }
        }
        if (lane == 0) {
          nkept_sh[par] = n;
          mbar_arrive(&lready[par]);
        }
        if (p.bitmap && head) {   // this split's bits of each head's row: its range
          // of the word cleared (the last split's reaches the word's end), then set
          const int nk = (it.Lk + kTile - 1) / kTile, W = (nk + 31) / 32;
          uint32_t *word = p.bitmap + bmo + (int64_t)(it.kvh * p.group + lane) * W + (it.j0 >> 5);
          const uint32_t sh = it.j0 & 31;
          const uint32_t range = it.q == it.ns - 1 ? 0xFFFFFFFFu << sh
                                                   : (nt >= 32 ? 0xFFFFFFFFu : ((1u << nt) - 1u)) << sh;
          atomicAnd(word, ~range);
          if (hs) atomicOr(word, hs << sh);
        }
      }
      named_bar_sync(1, kGroup);   // mred is rewritten by the next item
    }
    if (abort_sh && t == 0) atomicExch(const_cast<uint32_t *>(gabort), p.epoch);
  } else {
    reg_alloc<kRegsPV>();
    // ---------------------------------------------------- P V group
    const int tp = t - kGroup, wp = warp - 4;   // key, head-dim column; warp in group
    const uint32_t lane_off = (uint32_t)(wp * 32) << 16;
    uint32_t kc = 0;
    bool stop = false;
    for (uint32_t i = 0; !stop; ++i) {
      const uint32_t slot = i & 3, par = i & 1, sb = i % 3;
      bool ok = wait_bar(&itfull[slot], (i >> 2) & 1, limit, &abort_sh);
      const int item = ok ? it_sh[slot] : -1;
      if (bar_red_or(!ok, 2, kGroup)) break;
      if (tp == 0) mbar_arrive(&itempty[slot]);
      if (item < 0) break;
      DecItem it;
      decode_item(p, iofs, item, it);
      const int R = p.group * it.Lq;
      const int64_t first = (int64_t)iofs[it.s] + it.kvh;   // split qq is first + qq * Hkv

      // the decisions of this split (the score group's)
      ok = wait_bar(&lready[par], (i >> 1) & 1, limit, &abort_sh);
      if (bar_red_or(!ok, 2, kGroup)) break;
      tc_fence_after();
      const int n = nkept_sh[par];

      // ---- kept tiles
      float O[RB], mref[RB], lsum[RB], alpha[RB], alpha_prev[RB];
      int hrow[RB], posr[RB];   // head (in the group) and query key position of each row
#pragma unroll
      for (int r = 0; r < RB; ++r) {
        O[r] = 0.f;
        mref[r] = -INFINITY;
        lsum[r] = 0.f;
        alpha[r] = alpha_prev[r] = 1.f;
        hrow[r] = r < R ? r / it.Lq : 31;
        posr[r] = it.Lk - it.Lq + (r < R ? r % it.Lq : 0);
      }
      // O = alpha_prev O + D of kept tile number kd
      auto take_d = [&](uint32_t kd) -> bool {
        const uint32_t ps = kd & 1;
        const bool okd = wait_bar(&dfull[ps], (kd >> 1) & 1, limit, &abort_sh);
        if (bar_red_or(!okd, 2, kGroup)) return false;
        tc_fence_after();
        uint32_t v[N];
        tmem_ldN<N>(tmem + lane_off + C::kDCol + ps * N, v);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&dempty[ps]);
#pragma unroll
        for (int r = 0; r < RB; ++r) O[r] = fmaf(O[r], alpha_prev[r], __uint_as_float(v[r]));
        return true;
      };
      for (int u = 0; u < n && !stop; ++u, ++kc) {
        const int j = klist[par][u];
        const uint32_t act = kact[par][u], ps = kc & 1;
        const float *tm = tmax[sb] + (j - it.j0) * RB;
        // P buffer free: the MMA two kept tiles back has read it
        ok = wait_bar(&pfree[ps], ((kc >> 1) & 1) ^ 1, limit, &abort_sh);
        if (bar_red_or(!ok, 2, kGroup)) {
          stop = true;
          break;
        }
        uint32_t v[N];
        tmem_ldN<N>(tmem + lane_off + sb * 128 + (j - it.j0) * N, v);
        const int kpos = j * kTile + tp;
        const bool outside = kpos >= it.Lk;
        uint8_t *pb = base + C::kPOff + ps * C::kPBytes;
        // rows past RB stay zero from the start of the kernel
#pragma unroll
        for (int r = 0; r < RB; ++r) {
          float pv = 0.f;
          if (r < R) {
            const bool on = (act >> hrow[r]) & 1u;
            const float mnew = on ? fmaxf(mref[r], tm[r]) : mref[r];
            alpha[r] = mnew == -INFINITY ? 1.f : ex2_approx(mref[r] - mnew);
            mref[r] = mnew;
            const bool masked = outside || (p.causal && kpos > posr[r]);
            const float s2 = masked ? -INFINITY : __uint_as_float(v[r]) * p.c;
            pv = (on && mnew != -INFINITY) ? ex2_approx(s2 - mnew) : 0.f;
            lsum[r] = fmaf(lsum[r], alpha[r], pv);
          } else {
            alpha[r] = 1.f;
          }
          // key tp of row r: box tp/64, 16-byte chunk (tp%64)/8 swizzled by row
          *reinterpret_cast<__nv_bfloat16 *>(pb + (tp >> 6) * (N * 128) + r * 128 +
                                             ((((tp >> 3) & 7) ^ (r & 7)) << 4) + (tp & 7) * 2) =
              __float2bfloat16_rn(pv);
        }
        fence_proxy_async_smem();
        named_bar_sync(2, kGroup);
        if (tp == 0) mbar_arrive(&pready[ps]);
        if (u > 0 && !take_d(kc - 1)) {
          stop = true;
          break;
        }
#pragma unroll
        for (int r = 0; r < RB; ++r) alpha_prev[r] = alpha[r];
      }
      if (!stop && n > 0 && !take_d(kc - 1)) stop = true;
      if (stop) break;
      // the item's score columns are free for the item three ahead, its kept
      // list for the item two ahead
      tc_fence_before();
      named_bar_sync(2, kGroup);
      if (tp == 0) {
        mbar_arrive(&sfree[sb]);
        mbar_arrive(&lfree[par]);
      }

      // ---- partial result of the split (only if it kept a tile)
      if (n > 0) {
#pragma unroll
        for (int r = 0; r < RB; ++r) {
          float x = lsum[r];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
          if (lane == 0) lred[wp][r] = x;
        }
        named_bar_sync(2, kGroup);
        const int64_t prow = (int64_t)item * p.rows;
#pragma unroll
        for (int r = 0; r < RB; ++r)
          if (r < R) p.pO[(prow + r) * kTile + tp] = O[r];
        if (tp < R) {
          p.pl[prow + tp] = (lred[0][tp] + lred[1][tp]) + (lred[2][tp] + lred[3][tp]);
#pragma unroll
          for (int r = 0; r < RB; ++r)
            if (r == tp) p.pm[prow + tp] = mref[r];
        }
      }
      // The group's writes of the partial result are ordered before thread
      // 0's count by the barrier, and the count (acq_rel, gpu scope) releases
      // them with it: the CTA whose count completes the (sequence, KV head)
      // acquires every earlier count's writes, and its barrier hands them to
      // its whole group, which reads them from L2. A split without a partial
      // result counts with acquire only: it has nothing to release, and its
      // read-modify-write still continues the release sequences of the
      // counts before it.
      named_bar_sync(2, kGroup);
      if (tp == 0) {   // the last of the splits of this (sequence, KV head) merges
        if (n > 0) p.flags[item] = p.epoch;
        uint64_t *done = p.done + it.s * p.Hkv + it.kvh;
        counter_enter(done, p.epoch);
        const uint32_t before = n > 0 ? counter_add_acq_rel(done) : counter_add_acquire(done);
        merge_sh = before == (uint32_t)(it.ns - 1);
      }
      named_bar_sync(2, kGroup);
      if (!merge_sh) continue;

      // ---- merge: the splits of this (sequence, KV head) that kept a tile,
      // in split order: 128 candidates at a time, their list taken in batches
      // of kE. Thread tp owns column quads g = tp + 128 k (row g / 32,
      // columns 4 (g % 32) .. +3). Per batch all loads (maxima and sums into
      // shared memory, the quads' partial outputs into registers) are in
      // flight together; the running max, the rescale of the accumulators
      // and the weights are then computed once per row.
      constexpr int kQ = RB / 4;              // column quads per thread
      constexpr int kE = 16 / kQ;             // batch: partial results whose loads overlap
      float4 acc[kQ];
#pragma unroll
      for (int k = 0; k < kQ; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (tp < RB) {
        msh[tp] = -INFINITY;
        lsh[tp] = 0.f;
      }
      for (int b0 = 0; b0 < it.ns; b0 += kGroup) {
        const int qq = b0 + tp;
        const int64_t x = first + (int64_t)qq * p.Hkv;
        const bool has = qq < it.ns && __ldcg(p.flags + x) == p.epoch;
        const unsigned bal = __ballot_sync(0xffffffffu, has);
        if (lane == 0) wcnt[wp] = __popc(bal);
        named_bar_sync(2, kGroup);
        int off = 0;
        for (int w = 0; w < wp; ++w) off += wcnt[w];
        const int cnt = (wcnt[0] + wcnt[1]) + (wcnt[2] + wcnt[3]);
        if (has) clist[off + __popc(bal & ((1u << lane) - 1u))] = (int)(x - first);
        named_bar_sync(2, kGroup);
        for (int e0 = 0; e0 < cnt; e0 += kE) {
          const int E = min(kE, cnt - e0);
          // the batch's maxima, sums and partial outputs, all loads in flight
          for (int y = tp; y < E * R; y += kGroup) {
            const int e = y / R, r = y - e * R;
            const int64_t prow = (first + clist[e0 + e]) * p.rows;
            pmsh[e][r] = __ldcg(p.pm + prow + r);
            plsh[e][r] = __ldcg(p.pl + prow + r);
          }
          float4 v[kE][kQ];
#pragma unroll
          for (int e = 0; e < kE; ++e) {
            const int64_t prow = (first + clist[e0 + (e < E ? e : 0)]) * p.rows;
#pragma unroll
            for (int k = 0; k < kQ; ++k) {
              const int g = tp + kGroup * k, r = g >> 5;
              v[e][k] = make_float4(0.f, 0.f, 0.f, 0.f);
              if (e < E && r < R)
                v[e][k] = __ldcg(reinterpret_cast<const float4 *>(p.pO + (prow + r) * kTile) + (g & 31));
            }
          }
          named_bar_sync(2, kGroup);
          if (tp < R) {   // running max, rescale, sum and weights of row tp
            const float mo = msh[tp];
            float mn = mo;
            for (int e = 0; e < E; ++e) mn = fmaxf(mn, pmsh[e][tp]);
            const float sc = mo == -INFINITY ? 0.f : ex2_approx(mo - mn);
            float l = lsh[tp] * sc;
            for (int e = 0; e < E; ++e) {
              const float w = pmsh[e][tp] == -INFINITY ? 0.f : ex2_approx(pmsh[e][tp] - mn);
              wsh[e][tp] = w;
              l = fmaf(plsh[e][tp], w, l);
            }
            msh[tp] = mn;
            lsh[tp] = l;
            scsh[tp] = sc;
          }
          named_bar_sync(2, kGroup);
#pragma unroll
          for (int k = 0; k < kQ; ++k) {
            const int g = tp + kGroup * k, r = g >> 5;
            if (r < R) {
              const float sc = scsh[r];
              float4 a = make_float4(acc[k].x * sc, acc[k].y * sc, acc[k].z * sc, acc[k].w * sc);
#pragma unroll
              for (int e = 0; e < kE; ++e) {
                const float w = e < E ? wsh[e][r] : 0.f;
                a.x = fmaf(v[e][k].x, w, a.x);
                a.y = fmaf(v[e][k].y, w, a.y);
                a.z = fmaf(v[e][k].z, w, a.z);
                a.w = fmaf(v[e][k].w, w, a.w);
              }
              acc[k] = a;
            }
          }
          named_bar_sync(2, kGroup);   // the staged batch is rewritten next
        }
      }
      __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(p.out);
      const int total_q = p.cu_q[p.n_seqs];
#pragma unroll
      for (int k = 0; k < kQ; ++k) {
        const int g = tp + kGroup * k, r = g >> 5;
        if (r < R) {
          const int h = it.kvh * p.group + r / it.Lq, qi = r % it.Lq;
          const float l = lsh[r], inv = l > 0.f ? 1.f / l : 0.f;
          uint2 o;
          o.x = pack_bf16x2(acc[k].x * inv, acc[k].y * inv);
          o.y = pack_bf16x2(acc[k].z * inv, acc[k].w * inv);
          *reinterpret_cast<uint2 *>(out + ((size_t)(it.aq + qi) * p.Hq + h) * kTile + 4 * (g & 31)) = o;
        }
      }
      if (p.lse && tp < R) {
        const int h = it.kvh * p.group + tp / it.Lq, qi = tp % it.Lq;
        p.lse[(size_t)h * total_q + it.aq + qi] = (msh[tp] + log2f(lsh[tp])) * kLn2;
      }
      named_bar_sync(2, kGroup);   // msh / lsh are reset by the next merge
    }
    if (stop) abort_sh = 1;
    if (abort_sh && tp == 0) atomicExch(const_cast<uint32_t *>(gabort), p.epoch);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (abort_sh && t == 0) atomicOr(&p.ws->status, kStatusTimeout);
  if (warp == 10) tmem_dealloc(tmem, 512);
}

// ============================================================ launchers

cudaError_t launch_decode(const DecParams &p, const CUtensorMap &tk, const CUtensorMap &tv,
                          int sm_count, cudaStream_t stream) {
  const int grid = (int)(p.max_items < sm_count ? p.max_items : sm_count);
  if (p.rows <= 4)
    return launch_dependent(dec_kernel<4>, grid, kDecThreadsAll, DecCfg<4>::kSmem, stream, p, tk, tv);
  if (p.rows <= 8)
    return launch_dependent(dec_kernel<8>, grid, kDecThreadsAll, DecCfg<8>::kSmem, stream, p, tk, tv);
  if (p.rows <= 16)
    return launch_dependent(dec_kernel<16>, grid, kDecThreadsAll, DecCfg<16>::kSmem, stream, p, tk, tv);
  return launch_dependent(dec_kernel<32>, grid, kDecThreadsAll, DecCfg<32>::kSmem, stream, p, tk, tv);
}

int decode_split(int rows) { return rows <= 16 ? DecCfg<16>::kSplit : DecCfg<32>::kSplit; }

namespace {
// The register split adds up only if every thread starts with kRegsLaunch.
template <int RB>
cudaError_t prepare_one() {
  cudaError_t e = cudaFuncSetAttribute(dec_kernel<RB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)DecCfg<RB>::kSmem);
  cudaFuncAttributes fa{};
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, dec_kernel<RB>);
  if (e == cudaSuccess && fa.numRegs != (int)kRegsLaunch) e = cudaErrorInvalidKernelImage;
  return e;
}
}  // namespace

cudaError_t prepare_decode() {
  cudaError_t e = prepare_one<4>();
  if (e == cudaSuccess) e = prepare_one<8>();
  if (e == cudaSuccess) e = prepare_one<16>();
  if (e == cudaSuccess) e = prepare_one<32>();
  return e;
}

}  // namespace bsa
