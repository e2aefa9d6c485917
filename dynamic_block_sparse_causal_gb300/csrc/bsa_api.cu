// C interface of libbsa (declared in include/bsa.h): argument checks,
// per-stream scratch areas, TMA tensor-map templates, launches.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <climits>
#include <cmath>
#include <cstring>
#include <map>
#include <memory>
#include <mutex>
#include <utility>

#include "bsa.h"
#include "bsa_decode.h"
#include "bsa_importance.h"
#include "bsa_internal.h"

namespace {

using bsa::Workspace;
using bsa::WorkspaceLayout;

struct DeviceInfo {
  bool ready = false;
  bool supported = false;
  int sm_count = 0;
};

// A growable device buffer, grown stream-ordered.
struct Buffer {
  void *ptr = nullptr;
  size_t bytes = 0;
};

// Everything the library keeps for one (device, stream): the scratch area of
// the prefill and top-p calls (work queue, tensor maps, status word, tables),
// the block-importance tables and the decode tables. Calls on one stream
// share it, so `mu` serialises them from enqueue to the last launch; calls on
// different streams only meet briefly on g_mu, for the lookup.
struct StreamState {
  std::mutex mu;
  Buffer ws, imp, dec;
  uint32_t dec_epoch = 0;   // decode calls on this stream (tags their per-call state)
  bsa::DecCaps dec_caps;    // sizes the decode tables are laid out for
};

std::mutex g_mu;   // guards g_streams, g_devices and g_encode
std::map<std::pair<int, cudaStream_t>, std::unique_ptr<StreamState>> g_streams;
std::map<int, DeviceInfo> g_devices;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

thread_local const float *t_q_scale = nullptr;
thread_local const float *t_k_scale = nullptr;
thread_local const float *t_v_scale = nullptr;
thread_local int32_t t_drop_k_load = -1;
thread_local uint64_t t_wait_limit_ns = 2000000000ull;  // 2 s

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Resolve the driver's tensor-map encoder once (no link-time libcuda). Under g_mu.
bool encoder() {
  if (g_encode) return true;
  void *fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn)
    return false;
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return true;
}

// Per-device set-up (capability, SM count, kernel attributes) and the
// tensor-map encoder, once; the returned record is not modified afterwards.
bsa_status_t device_info(int dev, DeviceInfo **out) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (!encoder()) return BSA_ERR_CUDA;
  DeviceInfo &d = g_devices[dev];
  if (!d.ready) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return BSA_ERR_CUDA;
    d.supported = (major == 10 && minor == 3);
    if (d.supported &&
        (bsa::prepare_forward() != cudaSuccess || bsa::prepare_skip() != cudaSuccess ||
         bsa::prepare_importance() != cudaSuccess || bsa::prepare_decode() != cudaSuccess))
      return BSA_ERR_CUDA;
    d.ready = true;
  }
  *out = &d;
  return BSA_OK;
}

// The state of (device, stream), created on first use. The caller locks its mu.
StreamState *stream_state(int dev, cudaStream_t stream) {
  std::lock_guard<std::mutex> lock(g_mu);
  std::unique_ptr<StreamState> &p = g_streams[{dev, stream}];
  if (!p) p.reset(new StreamState);
  return p.get();
}

// Scratch area of a stream, grown stream-ordered when n_seqs grows. Under ss->mu.
bsa_status_t scratch_for(StreamState *ss, cudaStream_t stream, size_t bytes, Workspace **out) {
  Buffer &s = ss->ws;
  if (s.bytes < bytes) {
    void *p = nullptr;
    if (cudaMallocAsync(&p, bytes, stream) != cudaSuccess) return BSA_ERR_NO_MEMORY;
    if (cudaMemsetAsync(p, 0, sizeof(Workspace), stream) != cudaSuccess) return BSA_ERR_CUDA;
    if (s.ptr) {  // keep the sticky status word
      if (cudaMemcpyAsync(&static_cast<Workspace *>(p)->status,
                          &static_cast<Workspace *>(s.ptr)->status, sizeof(int32_t),
                          cudaMemcpyDeviceToDevice, stream) != cudaSuccess ||
          cudaFreeAsync(s.ptr, stream) != cudaSuccess)
        return BSA_ERR_CUDA;
    }
    s.ptr = p;
    s.bytes = bytes;
  }
  *out = static_cast<Workspace *>(s.ptr);
  return BSA_OK;
}

// Block-importance or decode tables of a stream, grown stream-ordered. Under ss->mu.
bsa_status_t table_for(Buffer &s, cudaStream_t stream, size_t bytes, void **out,
                       bool *grown = nullptr) {
  if (grown) *grown = false;
  if (s.bytes < bytes) {
    void *p = nullptr;
    if (cudaMallocAsync(&p, bytes, stream) != cudaSuccess) return BSA_ERR_NO_MEMORY;
    if (s.ptr && cudaFreeAsync(s.ptr, stream) != cudaSuccess) return BSA_ERR_CUDA;
    s.ptr = p;
    s.bytes = bytes;
    if (grown) *grown = true;
  }
  *out = s.ptr;
  return BSA_OK;
}

// [tokens, H, 128] tiles of 128 rows (or box_rows) x 128 bytes, 128-byte swizzle. The token
// extent is a placeholder (1) that the prologue replaces with cu[n_seqs],
// except for a paged K/V pool, whose extent (pages x 128) is known here.
bool encode_tile_map(CUtensorMap *m, const void *base, int H, bool fp8, uint64_t tokens = 1,
                     uint32_t box_rows = bsa::kTile) {
  const cuuint64_t elem = fp8 ? 1 : 2;
  cuuint64_t dims[3] = {(cuuint64_t)bsa::kHeadDim, (cuuint64_t)H, (cuuint64_t)tokens};
  cuuint64_t strides[2] = {bsa::kHeadDim * elem, (cuuint64_t)H * bsa::kHeadDim * elem};
  cuuint32_t box[3] = {(cuuint32_t)(128 / elem), 1, (cuuint32_t)box_rows};
  cuuint32_t estride[3] = {1, 1, 1};
  const CUresult r =
      g_encode(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
               const_cast<void *>(base), dims, strides, box, estride,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace

namespace bsa {
// FP8 scales set on the calling thread (for other translation units).
void current_fp8_scales(const float **q, const float **k, const float **v) {
  *q = t_q_scale;
  *k = t_k_scale;
  *v = t_v_scale;
}
}  // namespace bsa

namespace {

// Shared body of bsa_prefill_fwd (cu_k == cu_q) and bsa_prefill_fwd_chunked.
bsa_status_t prefill(const void *q, const void *k, const void *v, const int32_t *cu_seqlens,
                     const int32_t *cu_seqlens_k, int32_t n_seqs, int32_t Hq, int32_t Hkv,
                     int32_t d, int32_t causal, float lambda, bsa_dtype_t dtype, void *out,
                     float *lse, uint32_t *skip_bitmap, bsa_stream_t stream_,
                     const int32_t *page_table = nullptr, int32_t max_pages = 0,
                     int32_t num_pages = 0) {
  // ---- host-only checks: nothing is enqueued on failure
  if (!q || !k || !v || !cu_seqlens || !cu_seqlens_k || !out) return BSA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) ||
      !aligned(cu_seqlens, 4) || !aligned(cu_seqlens_k, 4) || !aligned(lse, 4) ||
      !aligned(skip_bitmap, 4))
    return BSA_ERR_INVALID_ARG;
  if (n_seqs < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || Hq > 65535) return BSA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return BSA_ERR_INVALID_ARG;
  if (!(lambda >= 0.0f && lambda < 1.0f)) return BSA_ERR_INVALID_ARG;  // also rejects NaN
  if (dtype != BSA_BF16 && dtype != BSA_FP8_E4M3) return BSA_ERR_INVALID_ARG;
  const bool fp8 = dtype == BSA_FP8_E4M3;
  if (fp8 && (!t_q_scale || !t_k_scale || !t_v_scale)) return BSA_ERR_INVALID_ARG;
  if (d != bsa::kHeadDim) return BSA_ERR_UNSUPPORTED;

  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return BSA_ERR_CUDA;
  DeviceInfo *info = nullptr;
  bsa_status_t st = device_info(dev, &info);
  if (st != BSA_OK) return st;
  if (!info->supported) return BSA_ERR_UNSUPPORTED;

  CUtensorMap tmpl[3];
  const uint64_t kv_tokens = page_table ? (uint64_t)num_pages * bsa::kTile : 1;
  if (!encode_tile_map(&tmpl[0], q, Hq, fp8) || !encode_tile_map(&tmpl[1], k, Hkv, fp8, kv_tokens) ||
      !encode_tile_map(&tmpl[2], v, Hkv, fp8, kv_tokens))
    return BSA_ERR_INVALID_ARG;

  const WorkspaceLayout layout = WorkspaceLayout::make(n_seqs);
  StreamState *ss = stream_state(dev, stream);
  std::lock_guard<std::mutex> lock(ss->mu);
  Workspace *ws = nullptr;
  if ((st = scratch_for(ss, stream, layout.bytes, &ws)) != BSA_OK) return st;
  // two query heads of a group per work item (they share every K tile)
  const bool skip = lambda > 0.f;
  const int heads = 2;
  const int group = Hq / Hkv, items_per_group = (group + heads - 1) / heads;
  if (bsa::launch_prologue(cu_seqlens, cu_seqlens_k, n_seqs, Hq, Hkv, items_per_group, causal,
                           page_table, max_pages, num_pages, ws, layout, tmpl, stream) !=
      cudaSuccess)
    return BSA_ERR_CUDA;

  char *base = reinterpret_cast<char *>(ws);
  bsa::FwdParams p{};
  p.ws = ws;
  p.seq_sorted = reinterpret_cast<const int32_t *>(base + layout.seq_sorted);
  p.seq_bitmap_off = reinterpret_cast<const int64_t *>(base + layout.seq_bitmap_off);
  p.level_start = reinterpret_cast<const int32_t *>(base + layout.level_start);
  p.cu_seqlens = cu_seqlens;
  p.cu_seqlens_k = cu_seqlens_k;
  p.page_table = page_table;
  p.max_pages = page_table ? max_pages : 0;
  p.out = out;
  p.lse = lse;
  p.bitmap = skip_bitmap;
  p.q_scale = fp8 ? t_q_scale : nullptr;
  p.k_scale = fp8 ? t_k_scale : nullptr;
  p.v_scale = fp8 ? t_v_scale : nullptr;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.group = group;
  p.heads_per_item = heads;
  p.items_per_group = items_per_group;
  p.causal = causal;
  p.c = (float)(1.0 / std::sqrt((double)d) * 1.4426950408889634);
  p.log2_lambda = lambda > 0.f ? (float)std::log2((double)lambda) : -INFINITY;
  p.wait_limit_ns = t_wait_limit_ns;
  p.debug_drop_k_load = t_drop_k_load;
  // lambda > 0: decisions first, then the kept tiles; lambda = 0: one dense pass
  const cudaError_t e = skip ? bsa::launch_skip(p, fp8, info->sm_count, stream)
                             : bsa::launch_forward(p, fp8, info->sm_count, stream);
  if (e != cudaSuccess) return BSA_ERR_CUDA;
  return BSA_OK;
}

}  // namespace

extern "C" {

bsa_status_t bsa_prefill_fwd(const void *q, const void *k, const void *v,
                             const int32_t *cu_seqlens, int32_t n_seqs, int32_t Hq, int32_t Hkv,
                             int32_t d, int32_t causal, float lambda, bsa_dtype_t dtype,
                             void *out, float *lse, uint32_t *skip_bitmap,
                             bsa_stream_t stream) {
  return prefill(q, k, v, cu_seqlens, cu_seqlens, n_seqs, Hq, Hkv, d, causal, lambda, dtype, out,
                 lse, skip_bitmap, stream);
}

bsa_status_t bsa_prefill_fwd_chunked(const void *q, const void *k, const void *v,
                                     const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                                     int32_t n_seqs, int32_t Hq, int32_t Hkv, int32_t d,
                                     int32_t causal, float lambda, bsa_dtype_t dtype, void *out,
                                     float *lse, uint32_t *skip_bitmap, bsa_stream_t stream) {
  return prefill(q, k, v, cu_seqlens_q, cu_seqlens_k, n_seqs, Hq, Hkv, d, causal, lambda, dtype,
                 out, lse, skip_bitmap, stream);
}

bsa_status_t bsa_prefill_fwd_paged(const void *q, const void *k_cache, const void *v_cache,
                                   const int32_t *page_table, int32_t max_pages_per_seq,
                                   int32_t num_pages, const int32_t *cu_seqlens_q,
                                   const int32_t *cu_seqlens_k, int32_t n_seqs, int32_t Hq,
                                   int32_t Hkv, int32_t d, int32_t causal, float lambda,
                                   bsa_dtype_t dtype, void *out, float *lse,
                                   uint32_t *skip_bitmap, bsa_stream_t stream) {
  if (!page_table || !aligned(page_table, 4) || max_pages_per_seq < 1 || num_pages < 1 ||
      (int64_t)num_pages * bsa::kTile > INT32_MAX)
    return BSA_ERR_INVALID_ARG;
  return prefill(q, k_cache, v_cache, cu_seqlens_q, cu_seqlens_k, n_seqs, Hq, Hkv, d, causal,
                 lambda, dtype, out, lse, skip_bitmap, stream, page_table, max_pages_per_seq,
                 num_pages);
}

bsa_status_t bsa_decode_fwd(const void *q, const void *k, const void *v,
                            const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                            int32_t n_seqs, int32_t max_seqlen_q, int64_t total_k, int32_t Hq,
                            int32_t Hkv, int32_t d, int32_t causal, float lambda, void *out,
                            float *lse, uint32_t *skip_bitmap, bsa_stream_t stream_) {
  if (!q || !k || !v || !cu_seqlens_q || !cu_seqlens_k || !out) return BSA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) ||
      !aligned(cu_seqlens_q, 4) || !aligned(cu_seqlens_k, 4) || !aligned(lse, 4) ||
      !aligned(skip_bitmap, 4))
    return BSA_ERR_INVALID_ARG;
  if (n_seqs < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || Hq > 65535) return BSA_ERR_INVALID_ARG;
  const int group = Hq / Hkv;
  if (group > 16 || max_seqlen_q < 1 || (int64_t)group * max_seqlen_q > bsa::kDecMaxRows)
    return BSA_ERR_INVALID_ARG;
  if ((int64_t)n_seqs * max_seqlen_q * Hq > INT_MAX || (int64_t)n_seqs * Hkv > INT_MAX)
    return BSA_ERR_INVALID_ARG;
  if (total_k < 0 || total_k > INT_MAX - 2 * bsa::kTile) return BSA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return BSA_ERR_INVALID_ARG;
  if (!(lambda >= 0.0f && lambda < 1.0f)) return BSA_ERR_INVALID_ARG;
  if (d != bsa::kHeadDim) return BSA_ERR_UNSUPPORTED;

  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return BSA_ERR_CUDA;
  DeviceInfo *info = nullptr;
  bsa_status_t st = device_info(dev, &info);
  if (st != BSA_OK) return st;
  if (!info->supported) return BSA_ERR_UNSUPPORTED;
  CUtensorMap tk, tv;
  const uint64_t extent = total_k > 0 ? (uint64_t)total_k : 1;
  if (!encode_tile_map(&tk, k, Hkv, false, extent) || !encode_tile_map(&tv, v, Hkv, false, extent))
    return BSA_ERR_INVALID_ARG;
  StreamState *ss = stream_state(dev, stream);
  std::lock_guard<std::mutex> lock(ss->mu);
  Workspace *ws = nullptr;
  if ((st = scratch_for(ss, stream, sizeof(Workspace), &ws)) != BSA_OK) return st;
  const int rows = group * max_seqlen_q;
  const int split = bsa::decode_split(rows);
  bsa::DecCaps need;
  need.n_seqs = n_seqs;
  need.seq_heads = (int64_t)n_seqs * Hkv;
  need.rows = rows;
  need.items = (int64_t)Hkv * ((total_k / bsa::kTile + n_seqs) / split + n_seqs);
  // the tables keep their layout while it covers the call; a new layout (or a
  // new buffer, or the count of calls wrapping) starts from zeroes
  bool reset = !ss->dec_caps.covers(need);
  if (reset) ss->dec_caps = ss->dec_caps.grown_to(need);
  const bsa::DecLayout layout = bsa::DecLayout::make(ss->dec_caps);
  void *buf = nullptr;
  bool grown = false;
  if ((st = table_for(ss->dec, stream, layout.bytes, &buf, &grown)) != BSA_OK) return st;
  if (++ss->dec_epoch == 0) {
    ss->dec_epoch = 1;
    reset = true;
  }
  if ((reset || grown) && cudaMemsetAsync(buf, 0, ss->dec.bytes, stream) != cudaSuccess)
    return BSA_ERR_CUDA;
  char *base = static_cast<char *>(buf);
  bsa::DecParams p{};
  p.dw = static_cast<bsa::DecWorkspace *>(buf);
  p.epoch = ss->dec_epoch;
  p.ws = ws;
  p.q = q;
  p.cu_q = cu_seqlens_q;
  p.cu_k = cu_seqlens_k;
  p.item_off = reinterpret_cast<const int32_t *>(base + layout.item_off);
  p.bm_off = reinterpret_cast<const int64_t *>(base + layout.bm_off);
  p.flags = reinterpret_cast<uint32_t *>(base + layout.flags);
  p.done = reinterpret_cast<uint64_t *>(base + layout.done);
  p.agg = reinterpret_cast<uint64_t *>(base + layout.agg);
  p.incl = reinterpret_cast<uint64_t *>(base + layout.incl);
  p.pO = reinterpret_cast<float *>(base + layout.pO);
  p.pm = reinterpret_cast<float *>(base + layout.pm);
  p.pl = reinterpret_cast<float *>(base + layout.pl);
  p.out = out;
  p.lse = lse;
  p.bitmap = skip_bitmap;
  p.total_k = total_k;
  p.max_items = need.items;
  p.n_seqs = n_seqs;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.group = group;
  p.rows = rows;
  p.mpitch = (int32_t)layout.mpitch;
  p.max_q = max_seqlen_q;
  p.split = split;
  p.causal = causal;
  p.c = (float)(1.0 / std::sqrt((double)d) * 1.4426950408889634);
  p.log2_lambda = lambda > 0.f ? (float)std::log2((double)lambda) : -INFINITY;
  p.wait_limit_ns = t_wait_limit_ns;
  p.debug_drop_k_load = t_drop_k_load;
  if (bsa::launch_decode(p, tk, tv, info->sm_count, stream) != cudaSuccess) return BSA_ERR_CUDA;
  return BSA_OK;
}

int64_t bsa_importance_blocks(const int32_t *cu, int32_t n_seqs) {
  if (!cu || n_seqs < 1 || cu[0] != 0) return -1;
  int64_t blocks = 0;
  for (int32_t s = 0; s < n_seqs; ++s) {
    const int64_t L = (int64_t)cu[s + 1] - cu[s];
    if (L < 0) return -1;
    blocks += (L + bsa::kTile - 1) / bsa::kTile;
  }
  return blocks;
}

bsa_status_t bsa_block_importance(const void *q, const void *k, const int32_t *cu_seqlens,
                                  int32_t n_seqs, int32_t Hq, int32_t Hkv, int32_t d,
                                  int32_t n_window, int32_t causal, int64_t total_blocks,
                                  float *scores, float *mean_scores, bsa_stream_t stream_) {
  if (!q || !k || !cu_seqlens || !scores) return BSA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(cu_seqlens, 4) || !aligned(scores, 4) ||
      !aligned(mean_scores, 4))
    return BSA_ERR_INVALID_ARG;
  if (n_seqs < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || Hq > 65535 ||
      (int64_t)n_seqs * Hq > INT_MAX)
    return BSA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return BSA_ERR_INVALID_ARG;
  if (n_window < 1 || n_window > bsa::kImpMaxWindow) return BSA_ERR_INVALID_ARG;
  if (total_blocks < 0 || total_blocks > ((int64_t)1 << 40) / Hq) return BSA_ERR_INVALID_ARG;
  if (d != bsa::kHeadDim) return BSA_ERR_UNSUPPORTED;

  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return BSA_ERR_CUDA;
  DeviceInfo *info = nullptr;
  bsa_status_t st = device_info(dev, &info);
  if (st != BSA_OK) return st;
  if (!info->supported) return BSA_ERR_UNSUPPORTED;

  CUtensorMap tmpl[2];
  // Q in 64-row boxes: a tile is one head's last 128 positions or the last
  // 64 of two heads
  if (!encode_tile_map(&tmpl[0], q, Hq, false, 1, bsa::kTile / 2) ||
      !encode_tile_map(&tmpl[1], k, Hkv, false))
    return BSA_ERR_INVALID_ARG;
  StreamState *ss = stream_state(dev, stream);
  std::lock_guard<std::mutex> lock(ss->mu);
  Workspace *ws = nullptr;   // holds the status word
  if ((st = scratch_for(ss, stream, sizeof(Workspace), &ws)) != BSA_OK) return st;
  const bsa::ImpLayout layout = bsa::ImpLayout::make(n_seqs, Hq, total_blocks);
  void *buf = nullptr;
  if ((st = table_for(ss->imp, stream, layout.bytes, &buf)) != BSA_OK) return st;
  char *base = static_cast<char *>(buf);

  bsa::ImpParams p{};
  p.iw = static_cast<bsa::ImpWorkspace *>(buf);
  p.ws = ws;
  p.cu = cu_seqlens;
  p.blk_off = reinterpret_cast<const int64_t *>(base + layout.blk_off);
  p.item_off = reinterpret_cast<const int32_t *>(base + layout.item_off);
  p.stat_t = reinterpret_cast<float *>(base + layout.stat_t);
  p.stat_e = reinterpret_cast<float *>(base + layout.stat_e);
  p.chunk_m = reinterpret_cast<float *>(base + layout.chunk_m);
  p.chunk_l = reinterpret_cast<float *>(base + layout.chunk_l);
  p.row_lse = reinterpret_cast<float *>(base + layout.row_lse);
  p.max_chunks = layout.max_chunks;
  p.scores = scores;
  p.mean_scores = mean_scores;
  p.total_blocks = total_blocks;
  p.n_seqs = n_seqs;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.group = Hq / Hkv;
  p.n_window = n_window;
  p.causal = causal;
  p.pair = (n_window <= bsa::kTile / 2 && p.group % 2 == 0) ? 2 : 1;
  p.c = (float)(1.0 / std::sqrt((double)d) * 1.4426950408889634);
  p.wait_limit_ns = t_wait_limit_ns;
  p.debug_drop_k_load = t_drop_k_load;
  if (bsa::launch_importance(p, tmpl, info->sm_count, stream) != cudaSuccess) return BSA_ERR_CUDA;
  return BSA_OK;
}

bsa_status_t bsa_top_p_select(const float *scores, const int32_t *cu_seqlens, int32_t n_seqs,
                              int64_t total_blocks, float p, int32_t *order, int32_t *n_selected,
                              uint8_t *keep, bsa_stream_t stream_) {
  if (!scores || !cu_seqlens || !order || !n_selected) return BSA_ERR_INVALID_ARG;
  if (!aligned(scores, 4) || !aligned(cu_seqlens, 4) || !aligned(order, 4) ||
      !aligned(n_selected, 4))
    return BSA_ERR_INVALID_ARG;
  if (n_seqs < 1 || total_blocks < 0) return BSA_ERR_INVALID_ARG;
  if (!(p > 0.0f && p <= 1.0f)) return BSA_ERR_INVALID_ARG;   // also rejects NaN
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return BSA_ERR_CUDA;
  DeviceInfo *info = nullptr;
  bsa_status_t st = device_info(dev, &info);
  if (st != BSA_OK) return st;
  if (!info->supported) return BSA_ERR_UNSUPPORTED;
  StreamState *ss = stream_state(dev, stream);
  std::lock_guard<std::mutex> lock(ss->mu);
  Workspace *ws = nullptr;
  if ((st = scratch_for(ss, stream, sizeof(Workspace), &ws)) != BSA_OK) return st;
  if (bsa::launch_top_p(scores, cu_seqlens, n_seqs, total_blocks, p, order, n_selected, keep, ws,
                        stream) != cudaSuccess)
    return BSA_ERR_CUDA;
  return BSA_OK;
}

bsa_status_t bsa_set_fp8_scales(const float *q_scale, const float *k_scale,
                                const float *v_scale) {
  const int nulls = !q_scale + !k_scale + !v_scale;
  if (nulls != 0 && nulls != 3) return BSA_ERR_INVALID_ARG;
  if (!aligned(q_scale, 4) || !aligned(k_scale, 4) || !aligned(v_scale, 4))
    return BSA_ERR_INVALID_ARG;
  t_q_scale = q_scale;
  t_k_scale = k_scale;
  t_v_scale = v_scale;
  return BSA_OK;
}

bsa_status_t bsa_quantize_fp8(const void *x_bf16, int64_t tokens, int32_t H, int32_t d,
                              uint8_t *x_e4m3, float *scale, bsa_stream_t stream) {
  if (!x_bf16 || !x_e4m3 || !scale) return BSA_ERR_INVALID_ARG;
  if (!aligned(x_bf16, 16) || !aligned(x_e4m3, 8) || !aligned(scale, 4)) return BSA_ERR_INVALID_ARG;
  if (tokens < 0 || H < 1 || H > 1024 || d < 8 || d % 8 != 0) return BSA_ERR_INVALID_ARG;
  if (bsa::launch_quantize_fp8(x_bf16, tokens, H, d, x_e4m3, scale,
                               reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return BSA_ERR_CUDA;
  return BSA_OK;
}

int64_t bsa_skip_bitmap_words(const int32_t *cu, int32_t n_seqs, int32_t Hq) {
  if (!cu || n_seqs < 1 || Hq < 1 || cu[0] != 0) return -1;
  int64_t words = 0;
  for (int32_t s = 0; s < n_seqs; ++s) {
    const int64_t L = (int64_t)cu[s + 1] - cu[s];
    if (L < 0) return -1;
    const int64_t n = (L + bsa::kTile - 1) / bsa::kTile;
    words += (int64_t)Hq * n * ((n + 31) / 32);
  }
  return words;
}

int64_t bsa_skip_bitmap_words_chunked(const int32_t *cu_q, const int32_t *cu_k, int32_t n_seqs,
                                      int32_t Hq) {
  if (!cu_q || !cu_k || n_seqs < 1 || Hq < 1 || cu_q[0] != 0 || cu_k[0] != 0) return -1;
  int64_t words = 0;
  for (int32_t s = 0; s < n_seqs; ++s) {
    const int64_t Lq = (int64_t)cu_q[s + 1] - cu_q[s], Lk = (int64_t)cu_k[s + 1] - cu_k[s];
    if (Lq < 0 || Lk < 0) return -1;
    const int64_t nq = (Lq + bsa::kTile - 1) / bsa::kTile, nk = (Lk + bsa::kTile - 1) / bsa::kTile;
    words += (int64_t)Hq * nq * ((nk + 31) / 32);
  }
  return words;
}

bsa_status_t bsa_get_device_status(bsa_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (cudaStreamSynchronize(stream) != cudaSuccess) return BSA_ERR_CUDA;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return BSA_ERR_CUDA;
  StreamState *ss = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    auto it = g_streams.find({dev, stream});
    if (it == g_streams.end()) return BSA_OK;
    ss = it->second.get();
  }
  std::lock_guard<std::mutex> lock(ss->mu);
  if (!ss->ws.ptr) return BSA_OK;
  int32_t *word = &static_cast<Workspace *>(ss->ws.ptr)->status;
  int32_t status = 0;
  if (cudaMemcpy(&status, word, sizeof(status), cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemset(word, 0, sizeof(status)) != cudaSuccess)
    return BSA_ERR_CUDA;
  if (status & bsa::kStatusBadSeqlens) return BSA_ERR_BAD_SEQLENS;
  if (status & bsa::kStatusTimeout) return BSA_ERR_TIMEOUT;
  return BSA_OK;
}

const char *bsa_status_string(bsa_status_t s) {
  switch (s) {
    case BSA_OK: return "ok";
    case BSA_ERR_INVALID_ARG: return "invalid argument";
    case BSA_ERR_UNSUPPORTED: return "unsupported device or head dimension";
    case BSA_ERR_CUDA: return "CUDA error";
    case BSA_ERR_TIMEOUT: return "device pipeline wait timed out";
    case BSA_ERR_NO_MEMORY: return "scratch allocation failed";
    case BSA_ERR_BAD_SEQLENS: return "cu_seqlens is not a valid prefix sum";
  }
  return "unknown status";
}

int32_t bsa_version(void) { return 200; }

void bsa_release(void) {
  std::lock_guard<std::mutex> lock(g_mu);
  int cur = 0;
  cudaGetDevice(&cur);
  for (auto &kv : g_streams) {
    std::lock_guard<std::mutex> slock(kv.second->mu);
    cudaSetDevice(kv.first.first);
    for (Buffer *b : {&kv.second->ws, &kv.second->imp, &kv.second->dec})
      if (b->ptr) cudaFree(b->ptr);
  }
  g_streams.clear();
  cudaSetDevice(cur);
}

bsa_status_t bsa_release_stream(bsa_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return BSA_ERR_CUDA;
  std::unique_ptr<StreamState> ss;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    auto it = g_streams.find({dev, stream});
    if (it == g_streams.end()) return BSA_OK;
    ss = std::move(it->second);
    g_streams.erase(it);
  }
  std::lock_guard<std::mutex> slock(ss->mu);   // a call still enqueueing on it finishes first
  bsa_status_t st = BSA_OK;
  for (Buffer *b : {&ss->ws, &ss->imp, &ss->dec})
    if (b->ptr && cudaFreeAsync(b->ptr, stream) != cudaSuccess) st = BSA_ERR_CUDA;
  return st;
}

bsa_status_t bsa_debug_fault_drill(int32_t drop_k_load, int64_t wait_limit_ns) {
  if (wait_limit_ns <= 0 || drop_k_load < -1) return BSA_ERR_INVALID_ARG;
  t_drop_k_load = drop_k_load;
  t_wait_limit_ns = (uint64_t)wait_limit_ns;
  return BSA_OK;
}

}  // extern "C"
