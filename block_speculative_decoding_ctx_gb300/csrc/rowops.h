// Internal interface of the row-wise support kernels (rowops.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "kernels.h"

namespace dfl {

int launch_embed_norm(const void* embed, const int32_t* anchor, int B, int gamma, int mask_id,
                      int vocab, int d, const float* g, float eps, float* x, void* h, void* h_lo,
                      int* status, cudaStream_t s);
// out (and out_lo, the bf16 remainder, when not null): [rows, d]
int launch_rmsnorm(const float* x, int rows, int d, const float* g, float eps, int gather_gamma,
                   void* out, void* out_lo, cudaStream_t s);
// Slots per row and chunk of the top-k partials (4 or 16).
int topk_slots(int k);
int launch_topk_lse(const float* logits, int rows, int V, int k, unsigned long long* part_keys,
                    float* part_ml, int* counters, int32_t* ids, float* vals, float* lse,
                    int32_t* draft, cudaStream_t s);
int launch_add_lengths(int B, const int32_t* n_new, int64_t* ctx_len, cudaStream_t s);

}  // namespace dfl
