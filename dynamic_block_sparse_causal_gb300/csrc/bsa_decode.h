// Internal declarations of the split-KV decode path: a few new queries per
// sequence against a long key range, with the block-skipping rule.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "bsa_internal.h"

namespace bsa {

constexpr int kDecSplit = 16;      // most key tiles per work item of the split passes
constexpr int kDecMaxRows = 32;    // query rows per (sequence, KV head): group x Lq
constexpr int kDecThreads = 256;       // P V pass
constexpr int kDecScoreThreads = 128;  // score pass: one thread per key of a tile

// Per-stream scratch of the decode path. Tables follow the header:
//   int64 tile_off[n_seqs + 1]   first key tile of every sequence (packed)
//   int32 item_off[n_seqs + 1]   first work item (KV head x split) of every sequence;
//                                a split is 8 or 16 key tiles (the host picks 8 when
//                                16-tile splits would leave SMs idle)
//   int64 bm_off[n_seqs + 1]     first skip-bitmap word of every sequence
//   float S[tiles][Hkv][rows][128]  scaled scores (log2 units), -inf where masked
//   float rm[Hkv][tiles][rows]      their row maxima per tile
//   float smax[Hkv][splits][rows]   and per split (splits = items / Hkv)
//   float pO[items][rows][128], pm[items][rows], pl[items][rows]
//                                   per-split output, reference max, sum
// with tiles <= total_k / 128 + n_seqs and items <= Hkv (tiles / split + n_seqs).
struct alignas(128) DecWorkspace {
  int32_t total_items;   // 0 when the arguments were rejected on the device
  int32_t pad_[31];
};

struct DecLayout {
  size_t tile_off, item_off, bm_off, S, rm, smax, pO, pm, pl, bytes;
  int64_t max_tiles, max_items;
  static DecLayout make(int n_seqs, int Hq, int Hkv, int rows, int64_t total_k, int split) {
    DecLayout l;
    l.max_tiles = total_k / kTile + n_seqs;
    l.max_items = (int64_t)Hkv * (l.max_tiles / split + n_seqs);
    auto up = [](size_t x) { return (x + 127) / 128 * 128; };
    size_t off = sizeof(DecWorkspace);
    l.tile_off = off;
    off += up((size_t)(n_seqs + 1) * 8);
    l.item_off = off;
    off += up((size_t)(n_seqs + 1) * 4);
    l.bm_off = off;
    off += up((size_t)(n_seqs + 1) * 8);
    l.S = off;
    off += up((size_t)l.max_tiles * Hkv * rows * kTile * 4);
    l.rm = off;
    off += up((size_t)l.max_tiles * Hkv * rows * 4);
    l.smax = off;
    off += up((size_t)l.max_items * rows * 4);
    l.pO = off;
    off += up((size_t)l.max_items * rows * kTile * 4);
    l.pm = off;
    off += up((size_t)l.max_items * rows * 4);
    l.pl = off;
    off += up((size_t)l.max_items * rows * 4);
    l.bytes = off;
    return l;
  }
};

struct DecParams {
  DecWorkspace *dw;
  Workspace *ws;              // status word
  const void *q;              // bf16 [total_q, Hq, 128]
  const int32_t *cu_q, *cu_k;
  const int64_t *tile_off, *bm_off;
  const int32_t *item_off;
  float *S, *rm, *smax, *pO, *pm, *pl;
  void *out;                  // bf16 [total_q, Hq, 128]
  float *lse;                 // [Hq, total_q] or null
  uint32_t *bitmap;           // or null
  int64_t total_k;
  int64_t max_tiles;          // rows of the rm table per KV head
  int64_t max_splits;         // rows of the smax table per KV head
  int32_t n_seqs, Hq, Hkv, group, rows, max_q, causal;
  int32_t split;              // key tiles per split: 8 or 16
  float c, log2_lambda;
  uint64_t wait_limit_ns;
  int32_t debug_drop_k_load;  // >= 0: the score producer omits that K load (fault drill)
};

cudaError_t launch_decode(const DecParams &p, const CUtensorMap &tk, const CUtensorMap &tv,
                          int sm_count, cudaStream_t stream);
cudaError_t prepare_decode();

}  // namespace bsa
