// Internal declarations of the split-KV decode path: a few new queries per
// sequence against a long key range, with the block-skipping rule.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "bsa_internal.h"

namespace bsa {

constexpr int kDecMaxRows = 32;    // query rows per (sequence, KV head): group x Lq
constexpr int kDecLocalSeqs = 256; // batches up to this size: per-sequence tables in each CTA

// Per-call words of the decode kernel. Each call carries an epoch (a per
// stream count of calls, never 0): per-call state is tagged with it, so no
// call has to clear what the one before left. A counter is a 64-bit word
// (epoch << 32 | count): an atomic max with (epoch << 32) first lifts a word
// left by an earlier call to (epoch, 0), then the atomic add counts.
struct alignas(128) DecWorkspace {
  uint64_t claim;        // work items claimed by the call (epoch-tagged counter)
  int32_t total_items;   // set-up of a large batch: work items (0: arguments rejected)
  uint32_t abort;        // the epoch, once a CTA of that call gave up a wait
  uint32_t setup_owner;  // the epoch, once a CTA of that call has taken the set-up
  uint32_t setup_done;   // the epoch, once that call's tables are written
  int32_t pad_[26];
};

// Per-stream scratch of the decode path. Its layout follows per-stream
// capacities that only grow (DecCaps); when one grows the whole area is laid
// out again and zero-filled, so each address only ever holds values of its
// own table, and the epoch-tagged words never meet another table's bytes.
// Tables follow the header:
//   int32 item_off[n_seqs + 1]   first work item (KV head x split) of every sequence, and
//   int64 bm_off[n_seqs + 1]     first skip-bitmap word (written by a set-up CTA for
//                                batches above kDecLocalSeqs; smaller ones keep them in
//                                every CTA's shared memory)
//   uint32 flags[items]          the epoch once the item's partial result is written
//   uint64 done[n_seqs x Hkv]    finished items per (sequence, KV head), epoch-tagged
//   uint64 agg[items][mpitch]    (epoch << 32) | the split's row maxima (f32 bits, log2 units)
//   uint64 incl[items][mpitch]   (epoch << 32) | row maxima over every tile up to the split's end
//                                (mpitch = rows rounded up to a multiple of 4)
//   float pO[items][rows][128], pm[items][rows], pl[items][rows]
//                                per-split output, reference max, sum
// A call needs items <= Hkv (tiles / split + n_seqs), tiles <= total_k / 128 +
// n_seqs.
struct DecCaps {
  int64_t n_seqs = 0, seq_heads = 0, rows = 0, items = 0;
  bool covers(const DecCaps &c) const {
    return c.n_seqs <= n_seqs && c.seq_heads <= seq_heads && c.rows <= rows && c.items <= items;
  }
  DecCaps grown_to(const DecCaps &c) const {
    DecCaps g;
    g.n_seqs = c.n_seqs > n_seqs ? c.n_seqs : n_seqs;
    g.seq_heads = c.seq_heads > seq_heads ? c.seq_heads : seq_heads;
    g.rows = c.rows > rows ? c.rows : rows;
    g.items = c.items > items ? c.items : items;
    return g;
  }
};

struct DecLayout {
  size_t item_off, bm_off, flags, done, agg, incl, pO, pm, pl, bytes;
  int64_t mpitch;   // row pitch of agg and incl: rows rounded up to a multiple of 4
  static DecLayout make(const DecCaps &c) {
    DecLayout l;
    auto up = [](size_t x) { return (x + 127) / 128 * 128; };
    size_t off = sizeof(DecWorkspace);
    l.item_off = off;
    off += up((size_t)(c.n_seqs + 1) * 4);
    l.bm_off = off;
    off += up((size_t)(c.n_seqs + 1) * 8);
    l.flags = off;
    off += up((size_t)c.items * 4);
    l.done = off;
    off += up((size_t)c.seq_heads * 8);
    l.mpitch = (c.rows + 3) / 4 * 4;
    l.agg = off;
    off += up((size_t)c.items * l.mpitch * 8);
    l.incl = off;
    off += up((size_t)c.items * l.mpitch * 8);
    l.pO = off;
    off += up((size_t)c.items * c.rows * kTile * 4);
    l.pm = off;
    off += up((size_t)c.items * c.rows * 4);
    l.pl = off;
    off += up((size_t)c.items * c.rows * 4);
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
  uint64_t *done;
  uint64_t *agg, *incl;
  float *pO, *pm, *pl;
  void *out;                  // bf16 [total_q, Hq, 128]
  float *lse;                 // [Hq, total_q] or null
  uint32_t *bitmap;           // or null
  int64_t total_k;
  int64_t max_items;          // most work items this call can have (bounds the tables)
  int32_t n_seqs, Hq, Hkv, group, rows, max_q, causal;
  int32_t mpitch;             // row pitch of agg and incl (of the layout: >= rows, a multiple of 4)
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
