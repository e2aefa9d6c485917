// Internal structures shared by the host interface and the kernels.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <utility>

namespace bsa {

constexpr int kTile = 128;          // query / key tile edge (block_size)
constexpr int kHeadDim = 128;       // the only supported head dimension
constexpr int kMaxLevels = 65536;   // longest sequence: 65536 tiles = 8M tokens
constexpr int kFwdThreads = 384;    // 4 control warps + 2 softmax warpgroups

// Bits of the device status word.
constexpr int kStatusBadSeqlens = 1 << 0;
constexpr int kStatusTimeout = 1 << 1;

// Per-stream scratch area, written by the prologue kernel and read by the
// forward kernel. Variable-length tables follow the header:
//   int32 seq_sorted[n_seqs]      sequences by tile count, longest first
//   int64 seq_bitmap_off[n_seqs]  first skip-bitmap word of each sequence
//   int32 level_start[kMaxLevels] first work item of each query-tile level
struct alignas(128) Workspace {
  CUtensorMap tmap[3];   // q, k, v tile maps; token extent patched on device
  int32_t counter;       // next work item (atomic)
  int32_t status;        // kStatus* bits, sticky until read by the host
  int32_t total_items;   // 0 when cu_seqlens was rejected
  int32_t max_tiles;     // longest sequence, in tiles
  int32_t total_tokens;  // cu_seqlens[n_seqs] (query tokens)
  int32_t pad_[27];
};

struct WorkspaceLayout {
  size_t seq_sorted, seq_bitmap_off, level_start, bytes;
  static WorkspaceLayout make(int n_seqs) {
    WorkspaceLayout l;
    size_t off = sizeof(Workspace);
    l.seq_sorted = off;
    off += ((size_t)n_seqs * 4 + 127) / 128 * 128;
    l.seq_bitmap_off = off;
    off += ((size_t)n_seqs * 8 + 127) / 128 * 128;
    l.level_start = off;
    off += (size_t)kMaxLevels * 4;
    l.bytes = off;
    return l;
  }
};

struct FwdParams {
  Workspace *ws;
  const int32_t *seq_sorted;
  const int64_t *seq_bitmap_off;
  const int32_t *level_start;
  const int32_t *cu_seqlens;     // query boundaries
  const int32_t *cu_seqlens_k;   // key/value boundaries (== cu_seqlens unless chunked)
  const int32_t *page_table;     // paged KV: [n_seqs, max_pages] physical page of key tile j
  int32_t max_pages;             // row length of page_table (0: K/V are packed, not paged)
  void *out;                 // bf16 [T, Hq, d]
  float *lse;                // [Hq, T] or null
  uint32_t *bitmap;          // or null
  const float *q_scale;      // fp8 only
  const float *k_scale;
  const float *v_scale;
  int32_t Hq, Hkv, group;    // group = Hq / Hkv
  int32_t heads_per_item;    // query heads of one group per work item (2: they share K tiles)
  int32_t items_per_group;   // ceil(group / heads_per_item)
  int32_t causal;
  float c;                   // softmax scale * log2(e)
  float log2_lambda;         // -inf when skipping is off
  uint64_t wait_limit_ns;    // bound on every pipeline wait
  int32_t debug_drop_k_load; // >= 0: the producer omits that K load (fault drill)
};

// Host-side launchers (bsa_fwd.cu).
// page_table / max_pages / num_pages: paged K/V (page = one 128-token tile);
// page_table == nullptr for packed K/V, whose token extent the prologue patches.
// items_per_group: work items per (sequence, KV head, query tile).
cudaError_t launch_prologue(const int32_t *cu_seqlens, const int32_t *cu_seqlens_k, int n_seqs,
                            int Hq, int Hkv, int items_per_group, int causal,
                            const int32_t *page_table,
                            int max_pages, int num_pages, Workspace *ws,
                            const WorkspaceLayout &layout, const CUtensorMap tmpl[3],
                            cudaStream_t stream);
// Dense forward (lambda = 0): one online-softmax pass over every causal tile.
cudaError_t launch_forward(const FwdParams &p, bool fp8, int num_ctas, cudaStream_t stream);
size_t forward_smem_bytes();
cudaError_t prepare_forward();   // per device: opt in to the shared-memory size
// Skipping forward (lambda > 0, bsa_skip.cu): scan of every causal tile for the
// decisions, then the kept tiles.
cudaError_t launch_skip(const FwdParams &p, bool fp8, int num_ctas, cudaStream_t stream);
cudaError_t prepare_skip();


// FP8 scales registered on the calling thread (bsa_api.cu).
void current_fp8_scales(const float **q, const float **k, const float **v);

// FP8 quantiser (bsa_quant.cu).
cudaError_t launch_quantize_fp8(const void *x, int64_t tokens, int H, int d, uint8_t *codes,
                                float *scale, cudaStream_t stream);

// Launch with programmatic stream serialisation: the kernel may start while
// the previous one on the stream finishes, and waits for it in grid_dep_wait.
template <typename... Params, typename... Args>
cudaError_t launch_dependent(void (*kernel)(Params...), int grid, int block, size_t smem,
                             cudaStream_t stream, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3((unsigned)block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace bsa
