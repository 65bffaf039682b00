// Small device helpers of the block-attention kernel (attention_tc.cu):
// swizzled tile offsets, bf16 -> fp16 widening, 16-bit packing, 2^x, and a
// warp-wide bounded wait.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "common.cuh"

namespace dfl {
namespace attn {

// Byte offset of element (row, col) in a [rows][64] bf16 tile with the
// 128-byte swizzle (16-byte chunk index XOR row % 8).
__device__ __forceinline__ uint32_t swz(int row, int col) {
  return (uint32_t)(row * 128 + ((((col >> 3) ^ row) & 7) << 4) + ((col & 7) << 1));
}

// Two bf16 values (one 32-bit register) as two fp16 values.  Ring keys (bf16)
// are widened to fp16 for the score MMAs: exact within the fp16
// range.  A key beyond +-65504 (a ring the caller filled itself; ctx_append
// reports what it would write out of range) becomes infinite rather than
// saturated: its scores and the head's attention output turn non-finite, and
// the next fp16 store of the pass reports DFLASH_ERR_RANGE.  Keys in slots
// outside the visible window are masked before the softmax and never matter.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
  const float lo = __uint_as_float(w << 16);
  const float hi = __uint_as_float(w & 0xFFFF0000u);
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void store_h2(__half* out, size_t o, float y0, float y1) {
  *reinterpret_cast<__half2*>(out + o) = __floats2half2_rn(y0, y1);
}

// 2^x by the special-function unit (ex2.approx: about 2 ulp; -inf gives +0).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void named_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Bounded wait taken by a whole warp: the warp goes on only if every lane saw
// the phase complete, so that the warp-collective instructions after it
// (tcgen05.ld/st) stay convergent even when a wait gives up.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          int* status) {
  const bool ok = mbar_wait_bounded(bar, parity, abort_flag, status);
  return __all_sync(0xffffffffu, ok);
}

}  // namespace attn
}  // namespace dfl
