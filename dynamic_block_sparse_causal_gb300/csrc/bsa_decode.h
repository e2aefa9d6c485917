// Internal declarations of the split-KV decode path: a few new queries per
// sequence against a long key range, with the block-skipping rule.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "bsa_internal.h"

namespace bsa {

constexpr int kDecMaxRows = 32;    // query rows per (sequence, KV head): group x Lq

// Per-call counters of the decode kernel (zeroed by its prologue).
struct alignas(128) DecWorkspace {
  int32_t total_items;   // 0 when the arguments were rejected on the device
  int32_t next_item;     // work-item counter the CTAs claim from
  int32_t abort;         // set by a CTA that gave up a wait: the others stop
  int32_t pad_[29];
};

// Per-stream scratch of the decode path. Tables follow the header:
//   int32 item_off[n_seqs + 1]   first work item (KV head x split) of every sequence
//   int64 bm_off[n_seqs + 1]     first skip-bitmap word of every sequence
//   uint32 flags[items]          per work item: maxima / inclusive prefix
//                                published, partial result written
//   int32 done[n_seqs x Hkv]     finished work items per (sequence, KV head)
//   float agg[items][mpitch]     the split's row maxima (log2 units)
//   float incl[items][mpitch]    row maxima over every tile up to the split's end
//                                (mpitch = rows rounded up to a multiple of 4)
//   float pO[items][rows][128], pm[items][rows], pl[items][rows]
//                                per-split output, reference max, sum
// with items <= Hkv (tiles / split + n_seqs), tiles <= total_k / 128 + n_seqs.
struct DecLayout {
  size_t item_off, bm_off, flags, done, agg, incl, pO, pm, pl, bytes;
  int64_t max_items;
  static DecLayout make(int n_seqs, int Hkv, int rows, int64_t total_k, int split) {
    DecLayout l;
    const int64_t max_tiles = total_k / kTile + n_seqs;
    l.max_items = (int64_t)Hkv * (max_tiles / split + n_seqs);
    auto up = [](size_t x) { return (x + 127) / 128 * 128; };
    size_t off = sizeof(DecWorkspace);
    l.item_off = off;
    off += up((size_t)(n_seqs + 1) * 4);
    l.bm_off = off;
    off += up((size_t)(n_seqs + 1) * 8);
    l.flags = off;
    off += up((size_t)l.max_items * 4);
    l.done = off;
    off += up((size_t)n_seqs * Hkv * 4);
    const size_t mpitch = (size_t)(rows + 3) / 4 * 4;
    l.agg = off;
    off += up((size_t)l.max_items * mpitch * 4);
    l.incl = off;
    off += up((size_t)l.max_items * mpitch * 4);
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
  const int64_t *bm_off;
  const int32_t *item_off;
  uint32_t *flags;
  int32_t *done;
  float *agg, *incl, *pO, *pm, *pl;
  void *out;                  // bf16 [total_q, Hq, 128]
  float *lse;                 // [Hq, total_q] or null
  uint32_t *bitmap;           // or null
  int64_t total_k;
  int64_t max_items;          // rows of the per-item tables
  int32_t n_seqs, Hq, Hkv, group, rows, max_q, causal;
  int32_t mpitch;             // row pitch of agg and incl: rows rounded up to a multiple of 4
  int32_t split;              // key tiles per work item (decode_split(rows))
  float c, log2_lambda;
  uint64_t wait_limit_ns;
  int32_t debug_drop_k_load;  // >= 0: the K producer omits that load (fault drill)
};

// Key tiles per work item for `rows` query rows per (sequence, KV head).
int decode_split(int rows);
cudaError_t launch_decode(const DecParams &p, const CUtensorMap &tk, const CUtensorMap &tv,
                          int sm_count, cudaStream_t stream);
cudaError_t prepare_decode();

}  // namespace bsa
