// Internal declarations of the block-importance and top-p selection path
// (UniPrefill page, §3.2 Eq. 3-4 and §3.3).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "bsa_internal.h"

namespace bsa {

constexpr int kImpChunk = 16;           // key blocks per work item of the score kernel
constexpr int kImpMaxWindow = 128;      // window rows: one 128-row MMA tile
constexpr int kImpThreads = 192;        // producer, MMA, 4 epilogue warps
constexpr int kTopPMaxBlocks = 16384;   // blocks per sequence the selection sorts (2M tokens)
constexpr int kTopPThreads = 1024;

// Per-stream scratch of the importance path. Tables follow the header:
//   int64 blk_off[n_seqs + 1]            first block of every sequence
//   int32 item_off[n_seqs + 1]           first work item of every sequence
//                                        (= Hq / pair x first 16-block chunk)
//   float stat_t[Hq][total_blocks][128]  per window row and key block:
//   float stat_e[Hq][total_blocks][128]  t = max of S c, e = sum of exp2(S c - t)
//   float chunk_m[Hq][chunks][128]       the same pair combined over a chunk
//   float chunk_l[Hq][chunks][128]        (chunks <= total_blocks/16 + n_seqs)
//   float row_lse[Hq][n_seqs][128]       log2-sum-exp2 of each window row
struct alignas(128) ImpWorkspace {
  CUtensorMap tmap[2];   // q (Hq heads), k (Hkv heads); token extent patched on device
  int32_t total_items;   // 0 when cu_seqlens or total_blocks was rejected
  int32_t pad_[31];
};

struct ImpLayout {
  size_t blk_off, item_off, stat_t, stat_e, chunk_m, chunk_l, row_lse, bytes;
  int64_t max_chunks;
  static ImpLayout make(int n_seqs, int Hq, int64_t total_blocks) {
    ImpLayout l;
    size_t off = sizeof(ImpWorkspace);
    l.blk_off = off;
    off += ((size_t)(n_seqs + 1) * 8 + 127) / 128 * 128;
    l.item_off = off;
    off += ((size_t)(n_seqs + 1) * 4 + 127) / 128 * 128;
    const size_t stat = (size_t)Hq * (size_t)total_blocks * kTile * 4;
    l.stat_t = off;
    off += stat;
    l.stat_e = off;
    off += stat;
    l.max_chunks = total_blocks / kImpChunk + n_seqs;
    const size_t chunk = (size_t)Hq * (size_t)l.max_chunks * kTile * 4;
    l.chunk_m = off;
    off += chunk;
    l.chunk_l = off;
    off += chunk;
    l.row_lse = off;
    off += (size_t)Hq * n_seqs * kTile * 4;
    l.bytes = off;
    return l;
  }
};

struct ImpParams {
  ImpWorkspace *iw;
  Workspace *ws;             // status word
  const int32_t *cu;
  const int64_t *blk_off;
  const int32_t *item_off;
  float *stat_t, *stat_e;
  float *chunk_m, *chunk_l;  // [Hq][max_chunks][128]
  float *row_lse;            // [Hq][n_seqs][128]
  int64_t max_chunks;
  float *scores;             // [Hq, total_blocks]
  float *mean_scores;        // [total_blocks] or null
  int64_t total_blocks;
  int32_t n_seqs, Hq, Hkv, group, n_window, causal;
  int32_t pair;              // query heads per work item: 2 for a window of <= 64 rows and an even group
  float c;                   // softmax scale * log2(e)
  uint64_t wait_limit_ns;
  int32_t debug_drop_k_load;  // >= 0: the tile producer omits that K load (fault drill)
};

// Prologue, score tiles, per-head reduction and head mean, in stream order.
cudaError_t launch_importance(const ImpParams &p, const CUtensorMap tmpl[2], int num_ctas,
                              cudaStream_t stream);
// Top-p selection over per-sequence block scores.
cudaError_t launch_top_p(const float *scores, const int32_t *cu, int n_seqs, int64_t total_blocks,
                         float p, int32_t *order, int32_t *n_selected, uint8_t *keep,
                         Workspace *ws, cudaStream_t stream);
cudaError_t prepare_importance();   // per device: opt in to the shared-memory sizes

}  // namespace bsa
