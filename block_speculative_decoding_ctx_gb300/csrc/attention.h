// Internal interface of the block attention (launcher attention.cu, kernel
// attention_tc.cu).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace dfl {

struct AttnArgs {
  const __half* qkv;         // fp16 [B*gamma, (Hq + 2 Hkv) hd]: rotated q, rotated k, v
  long long ld_qkv;
  __half* out;               // fp16 [B*gamma, Hq hd]
  long long ld_out;
  const int64_t* ctx_len;    // [B] context lengths L
  const int32_t* req_slot;   // [B] ring rows or nullptr
  int gamma, n_q, n_kv, hd, window, ring_batch;
  int splits;                // key-range splits per (request, KV head): a power of two <= 16;
                             // the splits of one head run as a thread-block cluster
  float scale_log2;          // log2(e) / sqrt(hd)
  int* status;
};

// Largest number of query rows (query heads of a KV head's group x gamma).
int attn_max_rows();

// ring_*_layer: the layer's slice of the ring, bf16 [ring_batch, Hkv, W, hd].
// Runs the tensor-core kernel (attention_tc.cu); DFLASH_ERR_UNSUPPORTED for
// shapes it does not take (dflash_create rejects those configurations).
int launch_attention(const void* ring_k_layer, const void* ring_v_layer, const AttnArgs& a, int B,
                     cudaStream_t s);

// Head dim 64 or 128, at most 128 query rows (query heads of a group x
// gamma) and gamma <= 16.
bool attention_tc_supported(const AttnArgs& a);
int launch_attention_tc(const CUtensorMap& tk, const CUtensorMap& tv, const AttnArgs& a, int B,
                        cudaStream_t s);

}  // namespace dfl
