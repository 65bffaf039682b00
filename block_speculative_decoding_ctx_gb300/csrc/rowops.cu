// Row-wise support kernels of the draft pass: block embedding + RMSNorm,
// RMSNorm (optionally gathering the MASK rows of each block), per-position
// top-k with log-sum-exp over the LM-head logits, and the context-length
// update of ctx_append.
//
// Sources: "DFlash vs DFlash 2" blog, section "DFlash: generate the block all
// at once" (draft input [anchor, MASK, MASK, ...]; shared embedding and LM
// head) and section "The candidate selector" (top-k candidates kept per
// position); product doc "Speculative decoding", section "How it works".
#include "common.cuh"
#include "rowops.h"

namespace dfl {
namespace {

constexpr int kNormThreads = 256;

// Two adjacent GEMM operand values as fp16 (range-checked).
__device__ __forceinline__ void store_h2(__half* out, size_t o, float y0, float y1, int* status) {
  *reinterpret_cast<__half2*>(out + o) =
      __halves2half2(to_f16_checked(y0, status), to_f16_checked(y1, status));
}

// One CTA per block row m = b * gamma + i: x[m] = embed[id] (fp32 residual
// stream), h[m] = RMSNorm(x[m]) * g in fp16, id = anchor[b] for i = 0, MASK
// after; and row m of the rotation table at position ctx_len[b] + i (shared
// by every head and layer of the pass).  The row is staged in shared memory
// (dynamic, 4 d bytes) with 16-byte loads issued together.
__global__ void __launch_bounds__(kNormThreads)
    embed_norm_kernel(const __nv_bfloat16* __restrict__ embed, const int32_t* __restrict__ anchor,
                      int gamma, int mask_id, int vocab, int d, const float* __restrict__ g, float eps,
                      float* __restrict__ x, __half* __restrict__ h, int* status,
                      const int64_t* __restrict__ ctx_len, float2* __restrict__ rope_cs, int half,
                      const RopeInv inv) {
  pdl_enter();
  extern __shared__ float row_s[];
  __shared__ float red[33];
  const int m = blockIdx.x;
  const int b = m / gamma, i = m % gamma;
  rope_table_row(rope_cs, m, half, (float)(ctx_len[b] + i), inv, threadIdx.x);
  int id = i == 0 ? anchor[b] : mask_id;
  if (id < 0 || id >= vocab) {
    if (threadIdx.x == 0) report_status(status, DFLASH_ERR_ARG);
    id = 0;
  }
  const uint4* e8 = reinterpret_cast<const uint4*>(embed + (size_t)id * d);
  float ss = 0.0f;
#pragma unroll 4
  for (int c = threadIdx.x; c < d / 8; c += kNormThreads) {
    const uint4 u = __ldg(e8 + c);
    const __nv_bfloat16* hv = reinterpret_cast<const __nv_bfloat16*>(&u);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float v = __bfloat162float(hv[k]);
      row_s[c * 8 + k] = v;
      ss += v * v;
    }
  }
  ss = block_sum(ss, red);
  const float rs = rsqrtf(ss / (float)d + eps);
  for (int c = threadIdx.x; c < d / 2; c += kNormThreads) {
    const float2 v = reinterpret_cast<const float2*>(row_s)[c];
    const float2 gg = reinterpret_cast<const float2*>(g)[c];
    reinterpret_cast<float2*>(x + (size_t)m * d)[c] = v;
    store_h2(h, (size_t)m * d + 2 * c, v.x * rs * gg.x, v.y * rs * gg.y, status);
  }
}

// out row r = RMSNorm(x[src(r)] (+ add[src(r)])) * g in fp16.  `add` is the
// fp32 output of the projection that feeds the residual stream (O or down):
// the residual add happens here, and with write_back the sum is stored to
// x[src(r)].  With rope_cs, also row r of the rotation table at position
// ctx_len[r / n_max] + r % n_max.
// gather_gamma = 0: src(r) = r; otherwise the MASK rows:
// src(r) = (r / (G - 1)) * G + r % (G - 1) + 1.  The row is staged in
// shared memory (dynamic, 4 d bytes) with 16-byte loads issued together.
__global__ void __launch_bounds__(kNormThreads)
    rmsnorm_kernel(float* x, const float* __restrict__ add, int write_back, int d,
                   const float* __restrict__ g, float eps,
                   int gather_gamma, __half* __restrict__ out, int* status,
                   const int64_t* __restrict__ ctx_len, int n_max, float2* __restrict__ rope_cs,
                   int half, const RopeInv inv) {
  pdl_enter();
  extern __shared__ float row_s[];
  __shared__ float red[33];
  const int r = blockIdx.x;
  if (rope_cs)
    rope_table_row(rope_cs, r, half, (float)(ctx_len[r / n_max] + r % n_max), inv, threadIdx.x);
  int src = r;
  if (gather_gamma > 0) src = (r / (gather_gamma - 1)) * gather_gamma + r % (gather_gamma - 1) + 1;
  float4* x4 = reinterpret_cast<float4*>(x + (size_t)src * d);
  const float4* a4 = add ? reinterpret_cast<const float4*>(add + (size_t)src * d) : nullptr;
  float ss = 0.0f;
#pragma unroll 4
  for (int c = threadIdx.x; c < d / 4; c += kNormThreads) {
    float4 v = __ldcg(x4 + c);
    if (a4) {
      const float4 y = __ldcg(a4 + c);
      v.x += y.x;
      v.y += y.y;
      v.z += y.z;
      v.w += y.w;
      if (write_back) x4[c] = v;
    }
    reinterpret_cast<float4*>(row_s)[c] = v;
    ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
  }
  ss = block_sum(ss, red);
  const float rs = rsqrtf(ss / (float)d + eps);
  for (int c = threadIdx.x; c < d / 2; c += kNormThreads) {
    const float2 v = reinterpret_cast<const float2*>(row_s)[c];
    const float2 gg = reinterpret_cast<const float2*>(g)[c];
    store_h2(out, (size_t)r * d + 2 * c, v.x * rs * gg.x, v.y * rs * gg.y, status);
  }
}

// dst = fp16(src) for a bf16 array of n8 * 8 elements (16-byte aligned);
// *flag = 1 if an element is NaN or beyond the fp16 range (+-65504).  Every
// other bf16 value is exactly an fp16 value, or (below 2^-14) rounds to an
// fp16 subnormal within 2^-25.
__global__ void __launch_bounds__(256)
    to_f16_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, size_t n8, int* flag) {
  bool bad = false;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8;
       i += (size_t)gridDim.x * blockDim.x) {
    const uint4 u = __ldg(src + i);
    const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&u);
    uint4 o;
    __half2* h = reinterpret_cast<__half2*>(&o);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 f = __bfloat1622float2(b[k]);
      bad |= !(fabsf(f.x) <= kF16Max) || !(fabsf(f.y) <= kF16Max);
      h[k] = __floats2half2_rn(f.x, f.y);
    }
    dst[i] = o;
  }
  if (bad) atomicExch(flag, 1);
}

// ------------------------------------------------------ top-k and LSE

constexpr int kTopkThreads = 256;

// Per-row top-k and log-sum-exp.  CTA (c, r) covers chunk c of row r: every
// thread keeps a sorted top-KT of its 32 values and a running (max, sum);
// warp tournaments reduce the lists to the CTA's top-k; the last CTA of the
// row (atomic ticket) merges the chunks' lists and (max, sum) pairs the same
// way, one chunk per lane (a row has at most 32 chunks: V <= 2^18).
template <int KT>
__global__ void __launch_bounds__(kTopkThreads)
    topk_lse_kernel(const float* __restrict__ logits, int V, int k, int chunks,
                    unsigned long long* __restrict__ part_keys, float* __restrict__ part_ml,
                    int* counters, int32_t* __restrict__ ids, float* __restrict__ vals,
                    float* __restrict__ lse, int32_t* __restrict__ draft) {
  pdl_enter();
  constexpr int kWarps = kTopkThreads / 32;
  __shared__ unsigned long long wsel[kWarps][KT];
  __shared__ float redm[kWarps], reds[kWarps];
  __shared__ int s_last;
  const int c = blockIdx.x, r = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float* row = logits + (size_t)r * V;
  const int v0 = c * kRowChunk, v1 = min(V, v0 + kRowChunk);

  unsigned long long top[KT];
#pragma unroll
  for (int j = 0; j < KT; ++j) top[j] = 0;
  // the thread's 32 elements of the chunk, loaded together
  constexpr int kPer = kRowChunk / kTopkThreads;
  float xv[kPer];
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int v = v0 + threadIdx.x + j * kTopkThreads;
    xv[j] = v < v1 ? __ldg(row + v) : -INFINITY;
  }
  float m = -INFINITY;
#pragma unroll
  for (int j = 0; j < kPer; ++j) m = fmaxf(m, xv[j]);
  float s = 0.0f;
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int v = v0 + threadIdx.x + j * kTopkThreads;
    if (v < v1) {
      s += expf(xv[j] - m);
      insert_key<KT>(top, vkey(xv[j], v));
    }
  }
  warp_lse(m, s);
#pragma unroll
  for (int j = 0; j < KT; ++j) {
    if (j < k) {
      const unsigned long long b = warp_pop_max(top);
      if (lane == 0) wsel[warp][j] = b;
    }
  }
  if (lane == 0) {
    redm[warp] = m;
    reds[warp] = s;
  }
  __syncthreads();
  if (warp == 0) {
    unsigned long long lst[KT];
#pragma unroll
    for (int j = 0; j < KT; ++j) lst[j] = (lane < kWarps && j < k) ? wsel[lane][j] : 0ull;
    float mm = lane < kWarps ? redm[lane] : -INFINITY;
    float ss = lane < kWarps ? reds[lane] : 0.0f;
    warp_lse(mm, ss);
    unsigned long long* pk = part_keys + ((size_t)r * chunks + c) * KT;
#pragma unroll
    for (int j = 0; j < KT; ++j) {
      if (j < k) {
        const unsigned long long b = warp_pop_max(lst);
        if (lane == 0) pk[j] = b;
      }
    }
    if (lane == 0) {
      part_ml[((size_t)r * chunks + c) * 2 + 0] = mm;
      part_ml[((size_t)r * chunks + c) * 2 + 1] = ss;
      __threadfence();
      s_last = (atomicAdd(&counters[r], 1) == chunks - 1);
    }
  }
  __syncthreads();
  if (!s_last || warp != 0) return;
  __threadfence();
  // merge the chunks of row r: lane cc holds chunk cc
  unsigned long long lst[KT];
  float M = -INFINITY, S = 0.0f;
#pragma unroll
  for (int j = 0; j < KT; ++j)
    lst[j] = (lane < chunks && j < k) ? __ldcg(part_keys + ((size_t)r * chunks + lane) * KT + j) : 0ull;
  if (lane < chunks) {
    M = __ldcg(part_ml + ((size_t)r * chunks + lane) * 2);
    S = __ldcg(part_ml + ((size_t)r * chunks + lane) * 2 + 1);
  }
  warp_lse(M, S);
#pragma unroll
  for (int j = 0; j < KT; ++j) {
    if (j < k) {
      const unsigned long long key = warp_pop_max(lst);
      if (lane == 0) {
        if (ids) ids[(size_t)r * k + j] = (int32_t)(~(uint32_t)(key & 0xFFFFFFFFull));
        if (vals) vals[(size_t)r * k + j] = key_to_float((uint32_t)(key >> 32));
        if (draft && j == 0) draft[r] = (int32_t)(~(uint32_t)(key & 0xFFFFFFFFull));
      }
    }
  }
  if (lane == 0) {
    if (lse) lse[r] = M + logf(S);
    atomicExch(&counters[r], 0);
  }
}

// Row r's top-k and log-sum-exp from the LM head's per-tile partials (the
// GEMM epilogue's top keys of each 128-row vocabulary tile, descending, and
// the tile's (max, sum of exp)).  Every thread merges the tiles t = tid, tid +
// 256, ... into a sorted top-KT and a running (max, sum); warp tournaments
// reduce those to the CTA's, and warp 0 merges the warps' lists.
template <int KT>
__global__ void __launch_bounds__(kTopkThreads)
    topk_merge_kernel(const unsigned long long* __restrict__ keys, const float2* __restrict__ ml, int tiles,
                      int slots, int k, int32_t* __restrict__ ids, float* __restrict__ vals,
                      float* __restrict__ lse, int32_t* __restrict__ draft) {
  pdl_enter();
  constexpr int kWarps = kTopkThreads / 32;
  __shared__ unsigned long long wsel[kWarps][KT];
  __shared__ float redm[kWarps], reds[kWarps];
  const int r = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  unsigned long long top[KT];
#pragma unroll
  for (int j = 0; j < KT; ++j) top[j] = 0;
  float m = -INFINITY, s = 0.0f;
  for (int t = threadIdx.x; t < tiles; t += kTopkThreads) {
    const unsigned long long* kp = keys + ((size_t)r * tiles + t) * slots;
    for (int j = 0; j < k; ++j) {
      const unsigned long long key = __ldcg(kp + j);
      if (key <= top[KT - 1]) break;  // the tile's keys are descending
      insert_key<KT>(top, key);
    }
    const float2 p = __ldcg(ml + (size_t)r * tiles + t);
    lse_merge(m, s, p.x, p.y);
  }
  warp_lse(m, s);
#pragma unroll
  for (int j = 0; j < KT; ++j) {
    if (j < k) {
      const unsigned long long b = warp_pop_max(top);
      if (lane == 0) wsel[warp][j] = b;
    }
  }
  if (lane == 0) {
    redm[warp] = m;
    reds[warp] = s;
  }
  __syncthreads();
  if (warp != 0) return;
  unsigned long long lst[KT];
#pragma unroll
  for (int j = 0; j < KT; ++j) lst[j] = (lane < kWarps && j < k) ? wsel[lane][j] : 0ull;
  float M = lane < kWarps ? redm[lane] : -INFINITY;
  float S = lane < kWarps ? reds[lane] : 0.0f;
  warp_lse(M, S);
#pragma unroll
  for (int j = 0; j < KT; ++j) {
    if (j < k) {
      const unsigned long long key = warp_pop_max(lst);
      if (lane == 0) {
        if (ids) ids[(size_t)r * k + j] = (int32_t)(~(uint32_t)(key & 0xFFFFFFFFull));
        if (vals) vals[(size_t)r * k + j] = key_to_float((uint32_t)(key >> 32));
        if (draft && j == 0) draft[r] = (int32_t)(~(uint32_t)(key & 0xFFFFFFFFull));
      }
    }
  }
  if (lane == 0 && lse) lse[r] = M + logf(S);
}

__global__ void add_lengths_kernel(int B, const int32_t* __restrict__ n_new, int64_t* ctx_len) {
  pdl_enter();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < B) ctx_len[b] += n_new[b];
}

}  // namespace

int launch_embed_norm(const void* embed, const int32_t* anchor, int B, int gamma, int mask_id,
                      int vocab, int d, const float* g, float eps, float* x, void* h, int* status,
                      const int64_t* ctx_len, float2* rope_cs, int half, const RopeInv& inv,
                      cudaStream_t s) {
  return launch_pdl(embed_norm_kernel, dim3(B * gamma), dim3(kNormThreads), (size_t)d * 4, s,
                    static_cast<const __nv_bfloat16*>(embed), anchor, gamma, mask_id, vocab, d, g, eps,
                    x, static_cast<__half*>(h), status, ctx_len, rope_cs, half, inv);
}

int launch_add_rmsnorm(float* x, const float* add, int write_back, int rows, int d, const float* g,
                       float eps, int gather_gamma, void* out, int* status, cudaStream_t s) {
  return launch_pdl(rmsnorm_kernel, dim3(rows), dim3(kNormThreads), (size_t)d * 4, s, x, add,
                    write_back, d, g, eps, gather_gamma, static_cast<__half*>(out), status,
                    (const int64_t*)nullptr, 1, (float2*)nullptr, 0, RopeInv{});
}

int launch_rmsnorm_rope(float* x, int rows, int d, const float* g, float eps, int gather_gamma,
                        void* out, int* status, const int64_t* ctx_len, int n_max, float2* rope_cs,
                        int half, const RopeInv& inv, cudaStream_t s) {
  return launch_pdl(rmsnorm_kernel, dim3(rows), dim3(kNormThreads), (size_t)d * 4, s, x,
                    (const float*)nullptr, 0, d, g, eps, gather_gamma, static_cast<__half*>(out), status,
                    ctx_len, n_max, rope_cs, half, inv);
}

int launch_to_f16(const void* src, void* dst, size_t n, int* flag, int grid, cudaStream_t s) {
  if (n % 8 || (reinterpret_cast<uintptr_t>(src) & 15) || (reinterpret_cast<uintptr_t>(dst) & 15))
    return DFLASH_ERR_ALIGN;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  return cudaLaunchKernelEx(&cfg, to_f16_kernel, static_cast<const uint4*>(src), static_cast<uint4*>(dst),
                            n / 8, flag) == cudaSuccess
             ? DFLASH_OK
             : DFLASH_ERR_LAUNCH;
}

int topk_slots(int k) { return k <= 4 ? 4 : 16; }

int launch_topk_lse(const float* logits, int rows, int V, int k, unsigned long long* part_keys,
                    float* part_ml, int* counters, int32_t* ids, float* vals, float* lse,
                    int32_t* draft, cudaStream_t s) {
  const int chunks = row_chunks(V);
  dim3 grid(chunks, rows);
  if (k <= 4)
    return launch_pdl(topk_lse_kernel<4>, grid, dim3(kTopkThreads), 0, s, logits, V, k, chunks,
                      part_keys, part_ml, counters, ids, vals, lse, draft);
  return launch_pdl(topk_lse_kernel<16>, grid, dim3(kTopkThreads), 0, s, logits, V, k, chunks,
                    part_keys, part_ml, counters, ids, vals, lse, draft);
}

int launch_topk_merge(int rows, int tiles, int slots, int k, const unsigned long long* keys, const float2* ml,
                      int32_t* ids, float* vals, float* lse, int32_t* draft, cudaStream_t s) {
  if (slots == 4)
    return launch_pdl(topk_merge_kernel<4>, dim3(rows), dim3(kTopkThreads), 0, s, keys, ml, tiles, slots, k, ids,
                      vals, lse, draft);
  return launch_pdl(topk_merge_kernel<16>, dim3(rows), dim3(kTopkThreads), 0, s, keys, ml, tiles, slots, k, ids,
                    vals, lse, draft);
}

int launch_add_lengths(int B, const int32_t* n_new, int64_t* ctx_len, cudaStream_t s) {
  return launch_pdl(add_lengths_kernel, dim3((B + 127) / 128), dim3(128), 0, s, B, n_new, ctx_len);
}

}  // namespace dfl
