// Per-head FP8 E4M3 quantisation of bf16 Q/K/V for the FP8 attention path.
//
// FP8 prefill is the precision behind the best speedups the block-sparse
// prefill monitoring page reports (FlashPrefill V2 at 128K); the page gives
// no quantisation recipe, so this follows the plainest one: one scale per
// head, scale = absmax / 448 (the largest finite E4M3 magnitude), codes =
// E4M3(x / scale) rounded to nearest even and saturated. Division is IEEE
// float32 (round to nearest) so the codes are reproducible bit for bit.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "bsa_internal.h"

namespace bsa {
namespace {

constexpr int kMaxHeadsSmem = 1024;

__global__ void absmax_kernel(const uint4 *__restrict__ x, int64_t nvec, int H, int vec_per_head,
                              unsigned *__restrict__ absmax_bits) {
  __shared__ unsigned sm[kMaxHeadsSmem];
  for (int h = threadIdx.x; h < H; h += blockDim.x) sm[h] = 0u;
  __syncthreads();
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < nvec;
       i += (int64_t)gridDim.x * blockDim.x) {
    const uint4 w = x[i];
    const int h = (int)((i / vec_per_head) % H);
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
    unsigned m = 0u;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      // |bf16| widened to float32 bits: drop the sign, keep the order
      m = max(m, (u[k] & 0x7FFFu) << 16);
      m = max(m, (u[k] >> 16 & 0x7FFFu) << 16);
    }
    atomicMax(&sm[h], m);
  }
  __syncthreads();
  for (int h = threadIdx.x; h < H; h += blockDim.x)
    if (sm[h]) atomicMax(&absmax_bits[h], sm[h]);
}

__global__ void scale_kernel(float *scale, int H) {
  const int h = blockIdx.x * blockDim.x + threadIdx.x;
  if (h < H) {
    const float a = __uint_as_float(reinterpret_cast<unsigned *>(scale)[h]);
    scale[h] = a > 0.f ? __fdiv_rn(a, 448.f) : 1.f;
  }
}

__global__ void cast_kernel(const uint4 *__restrict__ x, int64_t nvec, int H, int vec_per_head,
                            const float *__restrict__ scale, uint2 *__restrict__ out) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < nvec;
       i += (int64_t)gridDim.x * blockDim.x) {
    const uint4 w = x[i];
    const float s = scale[(i / vec_per_head) % H];
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
    uint32_t r[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const float a0 = __fdiv_rn(__uint_as_float(u[2 * k] << 16), s);
      const float a1 = __fdiv_rn(__uint_as_float(u[2 * k] & 0xFFFF0000u), s);
      const float a2 = __fdiv_rn(__uint_as_float(u[2 * k + 1] << 16), s);
      const float a3 = __fdiv_rn(__uint_as_float(u[2 * k + 1] & 0xFFFF0000u), s);
      const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a0, a1), __NV_SATFINITE, __NV_E4M3);
      const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(make_float2(a2, a3), __NV_SATFINITE, __NV_E4M3);
      r[k] = (uint32_t)lo | ((uint32_t)hi << 16);
    }
    out[i] = make_uint2(r[0], r[1]);
  }
}

}  // namespace

cudaError_t launch_quantize_fp8(const void *x, int64_t tokens, int H, int d, uint8_t *codes,
                                float *scale, cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(scale, 0, sizeof(float) * H, stream);
  if (e != cudaSuccess) return e;
  const int64_t nvec = tokens * H * (d / 8);
  const int vph = d / 8;
  if (nvec > 0) {
    const int blocks = (int)((nvec + 255) / 256 < 152 * 8 ? (nvec + 255) / 256 : 152 * 8);
    absmax_kernel<<<blocks, 256, 0, stream>>>(reinterpret_cast<const uint4 *>(x), nvec, H, vph,
                                              reinterpret_cast<unsigned *>(scale));
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  scale_kernel<<<(H + 127) / 128, 128, 0, stream>>>(scale, H);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (nvec > 0) {
    const int blocks = (int)((nvec + 255) / 256 < 152 * 8 ? (nvec + 255) / 256 : 152 * 8);
    cast_kernel<<<blocks, 256, 0, stream>>>(reinterpret_cast<const uint4 *>(x), nvec, H, vph,
                                            scale, reinterpret_cast<uint2 *>(codes));
    e = cudaGetLastError();
  }
  return e;
}

}  // namespace bsa
