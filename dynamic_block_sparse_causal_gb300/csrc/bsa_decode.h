// Internal declarations of the split-KV decode path: a few new queries per
// sequence against a long key range, with the block-skipping rule.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "bsa_internal.h"

namespace bsa {

constexpr int kDecMaxRows = 32;    // query rows per (sequence, KV head): group x Lq

// Per-call words of the decode kernel. Each call carries an epoch (a per
// stream count of calls, never 0): per-call state is either written by the
// call's set-up CTA before any item starts, or tagged with the epoch, so no
// call has to clear what the one before left.
struct alignas(128) DecWorkspace {
  int32_t total_items;   // set-up: work items (0 when the arguments were rejected)
  int32_t next_item;     // set-up zeroes it; the CTAs claim work items from it
  uint32_t abort;        // the epoch, once a CTA of that call gave up a wait
  uint32_t setup_owner;  // the epoch, once a CTA of that call has taken the set-up
  uint32_t setup_done;   // the epoch, once that call's tables are written
  int32_t pad_[27];
};

// Per-stream scratch of the decode path (zero-filled when allocated). Tables
// follow the header:
//   int32 item_off[n_seqs + 1]   set-up: first work item (KV head x split) of every sequence
//   int64 bm_off[n_seqs + 1]     set-up: first skip-bitmap word of every sequence
//   uint32 flags[items]          the epoch once the item's partial result is written
//   int32 done[n_seqs x Hkv]     set-up zeroes them: finished items per (sequence, KV head)
//   uint64 agg[items][mpitch]    (epoch << 32) | the split's row maxima (f32 bits, log2 units)
//   uint64 incl[items][mpitch]   (epoch << 32) | row maxima over every tile up to the split's end
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
    off += up((size_t)l.max_items * mpitch * 8);
    l.incl = off;
    off += up((size_t)l.max_items * mpitch * 8);
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
  uint64_t *agg, *incl;
  float *pO, *pm, *pl;
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
  uint32_t epoch;             // this call's number on the stream (never 0)
  int32_t debug_drop_k_load;  // >= 0: the K producer omits that load (fault drill)
};

// Key tiles per work item for `rows` query rows per (sequence, KV head).
int decode_split(int rows);
cudaError_t launch_decode(const DecParams &p, const CUtensorMap &tk, const CUtensorMap &tv,
                          int sm_count, cudaStream_t stream);
cudaError_t prepare_decode();

}  // namespace bsa
