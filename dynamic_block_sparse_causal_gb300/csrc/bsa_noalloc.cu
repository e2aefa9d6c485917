// bsa_prefill_fwd_noalloc: the same forward pass as bsa_prefill_fwd for
// callers that are not allowed to allocate device memory.
//
// Who needs it: a serving engine that reserves (nearly) all of HBM up front
// for its weights and KV-cache pool and hands out memory only from that
// pool, or a caller whose attention call must never enter the CUDA
// allocator (an allocation can fail under such a budget, and a first-time
// cudaMalloc can synchronise the device). bsa_prefill_fwd keeps a small
// per-stream scratch area that it grows with cudaMallocAsync; this entry
// point instead uses a fixed scratch array compiled into the library.
//
// The scratch array (kNoAllocScratchBytes, about 270 KiB) lives in device
// global memory of every GPU that loads the library, for the life of the
// process. Its address is looked up with cudaGetSymbolAddress by the first
// call made in each device context (a new context after cudaDeviceReset
// gets its own look-up). Every call shares the array, so calls whose work
// overlaps on the GPU (for example on two streams at once) race on it;
// calls on one stream are ordered. Device-side errors accumulate in the
// array's status word until bsa_get_noalloc_status() reads and clears it.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <mutex>

#include "bsa.h"
#include "bsa_internal.h"

namespace {

// Largest batch the fixed scratch area holds.
constexpr int kNoAllocMaxSeqs = 1024;

const bsa::WorkspaceLayout kLayout = bsa::WorkspaceLayout::make(kNoAllocMaxSeqs);
constexpr size_t kNoAllocScratchBytes =
    sizeof(bsa::Workspace) + kNoAllocMaxSeqs * 4 + kNoAllocMaxSeqs * 8 + bsa::kMaxLevels * 4;

// Work queue, tensor maps, sequence order, bitmap offsets and level table of
// the no-allocation path. Zero at load; the prologue rewrites what it uses.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

struct DeviceSetup {
  bool done = false;
  bool supported = false;
  int sm_count = 0;
  CUcontext ctx = nullptr;  // the context the address below belongs to
  void *scratch = nullptr;  // device address of g_noalloc_scratch in that context
};

constexpr int kMaxDevices = 64;
std::mutex g_mu;
DeviceSetup g_setup[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;

template <typename F>
bool driver_entry(const char *name, int version, F *fn) {
  void *p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &p, version, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !p)
    return false;
  *fn = reinterpret_cast<F>(p);
  return true;
}

// Set-up for the current device and its current context, once per context:
// the context's address of the scratch array, the SM count and the forward
// kernels' shared-memory opt-in. Under g_mu.
bsa_status_t setup_device(int dev, DeviceSetup **out) {
  if (dev < 0 || dev >= kMaxDevices) return BSA_ERR_UNSUPPORTED;
  if (kLayout.bytes > kNoAllocScratchBytes) return BSA_ERR_UNSUPPORTED;
  if (!g_ctx_current && !driver_entry("cuCtxGetCurrent", 4000, &g_ctx_current)) return BSA_ERR_CUDA;
  // null before the runtime has made a context current on this thread
  CUcontext ctx = nullptr;
  if (g_ctx_current(&ctx) != CUDA_SUCCESS) return BSA_ERR_CUDA;
  DeviceSetup &s = g_setup[dev];
  if (s.done && (!ctx || s.ctx != ctx)) s = DeviceSetup{};   // a new context (e.g. after a reset)
  if (!s.done) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&s.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return BSA_ERR_CUDA;
    s.supported = (major == 10 && minor == 3);
    if (s.supported) {
      void *ptr = nullptr;
      if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return BSA_ERR_CUDA;
      if (bsa::prepare_forward() != cudaSuccess || bsa::prepare_skip() != cudaSuccess)
        return BSA_ERR_CUDA;
      // the symbol look-up made the device's primary context current
      if (g_ctx_current(&ctx) != CUDA_SUCCESS || !ctx) return BSA_ERR_CUDA;
      s.scratch = ptr;
    }
    if (!g_encode && !driver_entry("cuTensorMapEncodeTiled", 12000, &g_encode)) return BSA_ERR_CUDA;
    s.ctx = ctx;
    s.done = true;
  }
  *out = &s;
  return BSA_OK;
}

bool encode(CUtensorMap *m, const void *base, int H, bool fp8) {
  const cuuint64_t elem = fp8 ? 1 : 2;
  cuuint64_t dims[3] = {(cuuint64_t)bsa::kHeadDim, (cuuint64_t)H, 1};
  cuuint64_t strides[2] = {bsa::kHeadDim * elem, (cuuint64_t)H * bsa::kHeadDim * elem};
  cuuint32_t box[3] = {(cuuint32_t)(128 / elem), 1, (cuuint32_t)bsa::kTile};
  cuuint32_t estride[3] = {1, 1, 1};
  return g_encode(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                  const_cast<void *>(base), dims, strides, box, estride,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" bsa_status_t bsa_prefill_fwd_noalloc(
    const void *q, const void *k, const void *v, const int32_t *cu_seqlens, int32_t n_seqs,
    int32_t Hq, int32_t Hkv, int32_t d, int32_t causal, float lambda, bsa_dtype_t dtype,
    void *out, float *lse, uint32_t *skip_bitmap, bsa_stream_t stream_) {
  if (!q || !k || !v || !cu_seqlens || !out) return BSA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) ||
      !aligned(cu_seqlens, 4) || !aligned(lse, 4) || !aligned(skip_bitmap, 4))
    return BSA_ERR_INVALID_ARG;
  if (n_seqs < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || Hq > 65535) return BSA_ERR_INVALID_ARG;
  if (n_seqs > kNoAllocMaxSeqs) return BSA_ERR_INVALID_ARG;  // beyond the fixed scratch area
  if (causal != 0 && causal != 1) return BSA_ERR_INVALID_ARG;
  if (!(lambda >= 0.0f && lambda < 1.0f)) return BSA_ERR_INVALID_ARG;
  if (dtype != BSA_BF16 && dtype != BSA_FP8_E4M3) return BSA_ERR_INVALID_ARG;
  const bool fp8 = dtype == BSA_FP8_E4M3;
  const float *qs = nullptr, *ks = nullptr, *vs = nullptr;
  if (fp8) {
    bsa::current_fp8_scales(&qs, &ks, &vs);
    if (!qs || !ks || !vs) return BSA_ERR_INVALID_ARG;
  }
  if (d != bsa::kHeadDim) return BSA_ERR_UNSUPPORTED;

  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return BSA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceSetup *s = nullptr;
  bsa_status_t st = setup_device(dev, &s);
  if (st != BSA_OK) return st;
  if (!s->supported) return BSA_ERR_UNSUPPORTED;

  CUtensorMap tmpl[3];
  if (!encode(&tmpl[0], q, Hq, fp8) || !encode(&tmpl[1], k, Hkv, fp8) ||
      !encode(&tmpl[2], v, Hkv, fp8))
    return BSA_ERR_INVALID_ARG;

  // the status word keeps its bits until bsa_get_noalloc_status reads them;
  // everything else the prologue rewrites
  bsa::Workspace *ws = static_cast<bsa::Workspace *>(s->scratch);
  // the same kernels as bsa_prefill_fwd (two query heads per work item)
  const bool skip = lambda > 0.f;
  const int heads = 2;
  const int group = Hq / Hkv, items_per_group = (group + heads - 1) / heads;
  if (bsa::launch_prologue(cu_seqlens, cu_seqlens, n_seqs, Hq, Hkv, items_per_group, causal,
                           nullptr, 0, 0, ws, kLayout, tmpl, stream) != cudaSuccess)
    return BSA_ERR_CUDA;

  char *base = static_cast<char *>(s->scratch);
  bsa::FwdParams p{};
  p.ws = ws;
  p.seq_sorted = reinterpret_cast<const int32_t *>(base + kLayout.seq_sorted);
  p.seq_bitmap_off = reinterpret_cast<const int64_t *>(base + kLayout.seq_bitmap_off);
  p.level_start = reinterpret_cast<const int32_t *>(base + kLayout.level_start);
  p.cu_seqlens = cu_seqlens;
  p.cu_seqlens_k = cu_seqlens;
  p.page_table = nullptr;
  p.max_pages = 0;
  p.out = out;
  p.lse = lse;
  p.bitmap = skip_bitmap;
  p.q_scale = qs;
  p.k_scale = ks;
  p.v_scale = vs;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.group = group;
  p.heads_per_item = heads;
  p.items_per_group = items_per_group;
  p.causal = causal;
  p.c = (float)(1.0 / std::sqrt((double)d) * 1.4426950408889634);
  p.log2_lambda = lambda > 0.f ? (float)std::log2((double)lambda) : -INFINITY;
  p.wait_limit_ns = 2000000000ull;
  p.debug_drop_k_load = -1;
  const cudaError_t e = skip ? bsa::launch_skip(p, fp8, s->sm_count, stream)
                             : bsa::launch_forward(p, fp8, s->sm_count, stream);
  if (e != cudaSuccess) return BSA_ERR_CUDA;
  return BSA_OK;
}

extern "C" bsa_status_t bsa_get_noalloc_status(bsa_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (cudaStreamSynchronize(stream) != cudaSuccess) return BSA_ERR_CUDA;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return BSA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (dev < 0 || dev >= kMaxDevices || !g_setup[dev].done || !g_setup[dev].scratch) return BSA_OK;
  CUcontext ctx = nullptr;
  if (!g_ctx_current || g_ctx_current(&ctx) != CUDA_SUCCESS) return BSA_ERR_CUDA;
  if (ctx != g_setup[dev].ctx) return BSA_OK;   // no call in this context yet
  int32_t *word = &static_cast<bsa::Workspace *>(g_setup[dev].scratch)->status;
  int32_t status = 0;
  if (cudaMemcpy(&status, word, sizeof(status), cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemset(word, 0, sizeof(status)) != cudaSuccess)
    return BSA_ERR_CUDA;
  if (status & bsa::kStatusBadSeqlens) return BSA_ERR_BAD_SEQLENS;
  if (status & bsa::kStatusTimeout) return BSA_ERR_TIMEOUT;
  return BSA_OK;
}
