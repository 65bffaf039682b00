// E4M3 (FP8) drafter weights: quantization from bf16 and the check
// dflash_create runs over given codes and scales.
//
// Format (the library's reading; the pages serve their models in FP8 without
// fixing a scheme): E4M3 with no infinities (largest finite 448), one float32
// scale per output row, weight = code * scale.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "common.cuh"
#include "rowops.h"

namespace dfl {
namespace {

constexpr int kQuantThreads = 256;
constexpr float kE4M3Max = 448.0f;

// One CTA per row: the row's largest magnitude, its scale amax / 448 (1 for a
// row of zeros), then every pair of weights divided by the scale (float32,
// round to nearest) and rounded to E4M3 (nearest, ties to even, saturating).
__global__ void __launch_bounds__(kQuantThreads)
    quantize_e4m3_kernel(const __nv_bfloat16* __restrict__ w, int cols, uint8_t* __restrict__ codes,
                         float* __restrict__ scales) {
  __shared__ float red[32];
  const size_t r = blockIdx.x;
  const __nv_bfloat162* row = reinterpret_cast<const __nv_bfloat162*>(w + r * (size_t)cols);
  const int pairs = cols / 2;
  float m = 0.0f;
  for (int c = threadIdx.x; c < pairs; c += kQuantThreads) {
    const float2 f = __bfloat1622float2(row[c]);
    m = fmaxf(m, fmaxf(fabsf(f.x), fabsf(f.y)));
  }
  m = warp_max_f(m);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x < 32) {
    float t = threadIdx.x < kQuantThreads / 32 ? red[threadIdx.x] : 0.0f;
    t = warp_max_f(t);
    if (threadIdx.x == 0) red[0] = t;
  }
  __syncthreads();
  const float amax = red[0];
  const float s = amax > 0.0f ? __fdiv_rn(amax, kE4M3Max) : 1.0f;
  if (threadIdx.x == 0) scales[r] = s;
  __nv_fp8x2_storage_t* out = reinterpret_cast<__nv_fp8x2_storage_t*>(codes + r * (size_t)cols);
  for (int c = threadIdx.x; c < pairs; c += kQuantThreads) {
    const float2 f = __bfloat1622float2(row[c]);
    out[c] = __nv_cvt_float2_to_fp8x2(make_float2(__fdiv_rn(f.x, s), __fdiv_rn(f.y, s)), __NV_SATFINITE,
                                      __NV_E4M3);
  }
}

// *flag = 1 if a code is NaN (exponent and mantissa bits all set) or a scale
// is not finite and positive.
__global__ void __launch_bounds__(256)
    check_e4m3_kernel(const uint4* __restrict__ codes, size_t n16, const float* __restrict__ scales,
                      size_t rows, int* flag) {
  bool bad = false;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += stride) {
    const uint4 u = __ldg(codes + i);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      // a byte b is NaN iff (b & 0x7F) == 0x7F
      const uint32_t x = w[k] & 0x7F7F7F7Fu;
      const uint32_t eq = ~(x ^ 0x7F7F7F7Fu);  // bytes equal to 0x7F have all bits set
      bad |= ((eq & (eq >> 1) & (eq >> 2) & (eq >> 3) & (eq >> 4) & (eq >> 5) & (eq >> 6)) & 0x01010101u) != 0;
    }
  }
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < rows; i += stride) {
    const float s = __ldg(scales + i);
    bad |= !(s > 0.0f) || !(s <= 3.402823466e38f);
  }
  if (bad) atomicExch(flag, 1);
}

}  // namespace

int launch_quantize_e4m3(const void* w, int rows, int cols, void* codes, float* scales, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(rows);
  cfg.blockDim = dim3(kQuantThreads);
  cfg.stream = s;
  return cudaLaunchKernelEx(&cfg, quantize_e4m3_kernel, static_cast<const __nv_bfloat16*>(w), cols,
                            static_cast<uint8_t*>(codes), scales) == cudaSuccess
             ? DFLASH_OK
             : DFLASH_ERR_LAUNCH;
}

int launch_check_e4m3(const void* codes, size_t n, const float* scales, size_t rows, int* flag, int grid,
                      cudaStream_t s) {
  if (n % 16 || (reinterpret_cast<uintptr_t>(codes) & 15)) return DFLASH_ERR_ALIGN;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  return cudaLaunchKernelEx(&cfg, check_e4m3_kernel, static_cast<const uint4*>(codes), n / 16, scales, rows,
                            flag) == cudaSuccess
             ? DFLASH_OK
             : DFLASH_ERR_LAUNCH;
}

}  // namespace dfl
