// Internal interface of the row-wise support kernels (rowops.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "kernels.h"

namespace dfl {

// x: fp32 [B gamma, d] residual stream; h: fp16 [B gamma, d]; rope_cs:
// [B gamma][half] (cos, sin) rotation table of the block positions
int launch_embed_norm(const void* embed, const int32_t* anchor, int B, int gamma, int mask_id,
                      int vocab, int d, const float* g, float eps, float* x, void* h, int* status,
                      const int64_t* ctx_len, float2* rope_cs, int half, const RopeInv& inv,
                      cudaStream_t s);
// out: fp16 [rows, d] = RMSNorm(x + add) * g (rows gathered when
// gather_gamma > 0); with write_back, x += add in place.  status receives
// DFLASH_ERR_RANGE for values beyond fp16.
int launch_add_rmsnorm(float* x, const float* add, int write_back, int rows, int d, const float* g,
                       float eps, int gather_gamma, void* out, int* status, cudaStream_t s);
// out = RMSNorm(x) * g, and rope_cs [rows][half] for the positions
// ctx_len[r / n_max] + r % n_max
int launch_rmsnorm_rope(float* x, int rows, int d, const float* g, float eps, int gather_gamma,
                        void* out, int* status, const int64_t* ctx_len, int n_max, float2* rope_cs,
                        int half, const RopeInv& inv, cudaStream_t s);
// dst (fp16) = src (bf16), n elements (a multiple of 8, 16-byte aligned
// pointers); *flag = 1 if a value is NaN or beyond the fp16 range.
int launch_to_f16(const void* src, void* dst, size_t n, int* flag, int grid, cudaStream_t s);
// Slots per row and tile of the top-k partials (4 or 16).
int topk_slots(int k);
int launch_topk_lse(const float* logits, int rows, int V, int k, unsigned long long* part_keys,
                    float* part_ml, int* counters, int32_t* ids, float* vals, float* lse,
                    int32_t* draft, cudaStream_t s);
// Row r's top-k (ids, values; descending, ties to the lower id), log-sum-exp
// and top-1 draft from the LM head's per-tile partials (GemmEpi::tk_*):
// keys [rows][tiles][slots], ml [rows][tiles].  Any output may be nullptr.
int launch_topk_merge(int rows, int tiles, int slots, int k, const unsigned long long* keys, const float2* ml,
                      int32_t* ids, float* vals, float* lse, int32_t* draft, cudaStream_t s);
int launch_add_lengths(int B, const int32_t* n_new, int64_t* ctx_len, cudaStream_t s);
// quant.cu: E4M3 codes and per-row scales from bf16 weights [rows, cols]
// (cols even), and the check of given codes (n bytes, a multiple of 16) and
// scales (*flag = 1 on a NaN code or a scale that is not finite and positive).
int launch_quantize_e4m3(const void* w, int rows, int cols, void* codes, float* scales, cudaStream_t s);
int launch_check_e4m3(const void* codes, size_t n, const float* scales, size_t rows, int* flag, int grid,
                      cudaStream_t s);

}  // namespace dfl
