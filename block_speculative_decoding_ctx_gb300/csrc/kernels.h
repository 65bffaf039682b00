// Internal launchers of libdflash (not part of the C ABI).  Every launcher
// validates nothing: the C-ABI layer has checked shapes and pointers.  Each
// returns DFLASH_OK or DFLASH_ERR_LAUNCH.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dflash.h"

namespace dfl {

// ---------------------------------------------------------------- verify.cu

// Elements of one vocabulary row handled by one CTA of the row kernels.
constexpr int kRowChunk = 8192;
inline int row_chunks(int V) { return (V + kRowChunk - 1) / kRowChunk; }

// Greedy verification.  counters [B] and keys [B * gamma] must be zero on
// entry and are zero again on exit.
int launch_verify_greedy(int B, int gamma, int V, const float* target, const int32_t* draft,
                         int32_t* accept_len, int32_t* tokens, int32_t* next_anchor,
                         int32_t* n_append, int* counters, unsigned long long* keys, int* status,
                         cudaStream_t s);

// Sampled verification.  counters [B] zero on entry and exit;
// zsum [B * row_chunks(V) * 2] scratch.
int launch_verify_sampled(int B, int gamma, int V, const float* p, const float* q,
                          const int32_t* draft, const uint64_t* seeds, uint64_t step,
                          int32_t* accept_len, int32_t* tokens, int32_t* next_anchor,
                          int32_t* n_append, int* counters, unsigned long long* zsum, int* status,
                          cudaStream_t s);

// out[r] ~ w[r, :] for rows r = b * rows_per_req + i with Philox
// (seeds[b], step, position = i, purpose).  counters [rows] zero on entry and
// exit; zsum [rows * row_chunks(V)] scratch.
int launch_sample_rows(int rows, int V, const float* w, long long row_stride, int rows_per_req,
                       const uint64_t* seeds, uint64_t step, uint32_t purpose, int32_t* out,
                       long long out_stride, int* counters, unsigned long long* zsum, int* status,
                       cudaStream_t s);

// probs[r] = top_p(softmax(logits[r] / T)), one CTA per row.
int launch_probs(int rows, int V, const float* logits, float temperature, float top_p,
                 float* probs, cudaStream_t s);

}  // namespace dfl
