// C ABI: verification, sampling preparation, status and error strings.
// See include/dflash.h for the contract of every entry point.
#include <cstdint>

#include "common.cuh"
#include "kernels.h"

using namespace dfl;

namespace {

constexpr int kMaxVocab = 1 << 18;  // fixed-point row sums stay below 2^63

struct VerifyLayout {
  int* status;
  int* counters;
  unsigned long long* keys;
  unsigned long long* zsum;
  size_t bytes;
};

VerifyLayout verify_layout(void* base, int B, int gamma, int V) {
  Carve c(base, kWsHeader);
  VerifyLayout L;
  L.status = static_cast<int*>(base);
  L.counters = c.take<int>(B);
  L.keys = c.take<unsigned long long>((size_t)B * gamma);
  L.zsum = c.take<unsigned long long>((size_t)B * row_chunks(V) * 2);
  L.bytes = c.off;
  return L;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" {

size_t dflash_verify_workspace_bytes(int batch, int gamma, int vocab) {
  if (batch < 1 || gamma < 2 || vocab < 1) return 0;
  return verify_layout(nullptr, batch, gamma, vocab).bytes;
}

size_t dflash_probs_workspace_bytes(int rows, int vocab) {
  (void)rows;
  (void)vocab;
  return kWsHeader;
}

int dflash_verify(int mode, int B, int gamma, int vocab, const float* target, const float* q,
                  const int32_t* draft, const uint64_t* seeds, uint64_t step,
                  int32_t* accept_len, int32_t* tokens, int32_t* next_anchor, int32_t* n_append,
                  void* workspace, size_t ws_bytes, dflash_stream_t stream) {
  if (mode != DFLASH_VERIFY_GREEDY && mode != DFLASH_VERIFY_SAMPLED) return DFLASH_ERR_ARG;
  if (B < 1 || B > 65535 || gamma < 2 || gamma > 64 || vocab < 1 || vocab > kMaxVocab)
    return DFLASH_ERR_SHAPE;
  if (!target || !draft || !accept_len || !tokens) return DFLASH_ERR_ARG;
  if (mode == DFLASH_VERIFY_SAMPLED && (!q || !seeds)) return DFLASH_ERR_ARG;
  if (!aligned(target, 4) || !aligned(draft, 4) || !aligned(accept_len, 4) ||
      !aligned(tokens, 4) || (q && !aligned(q, 4)) || (seeds && !aligned(seeds, 8)) ||
      (next_anchor && !aligned(next_anchor, 4)) || (n_append && !aligned(n_append, 4)))
    return DFLASH_ERR_ALIGN;
  if (!workspace || !aligned(workspace, 256)) return DFLASH_ERR_WORKSPACE;
  VerifyLayout L = verify_layout(workspace, B, gamma, vocab);
  if (ws_bytes < L.bytes) return DFLASH_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (mode == DFLASH_VERIFY_GREEDY)
    return launch_verify_greedy(B, gamma, vocab, target, draft, accept_len, tokens, next_anchor,
                                n_append, L.counters, L.keys, L.status, s);
  return launch_verify_sampled(B, gamma, vocab, target, q, draft, seeds, step, accept_len, tokens,
                               next_anchor, n_append, L.counters, L.zsum, L.status, s);
}

int dflash_probs(int rows, int vocab, const float* logits, float temperature, float top_p,
                 float* probs, void* workspace, size_t ws_bytes, dflash_stream_t stream) {
  if (rows < 1 || rows > (1 << 30) || vocab < 1 || vocab > kMaxVocab) return DFLASH_ERR_SHAPE;
  if (!logits || !probs) return DFLASH_ERR_ARG;
  if (!(temperature > 0.0f) || !(top_p > 0.0f) || !(top_p <= 1.0f)) return DFLASH_ERR_ARG;
  if (logits == probs) return DFLASH_ERR_ARG;
  if (!aligned(logits, 4) || !aligned(probs, 4)) return DFLASH_ERR_ALIGN;
  if (!workspace || !aligned(workspace, 256) || ws_bytes < kWsHeader) return DFLASH_ERR_WORKSPACE;
  return launch_probs(rows, vocab, logits, temperature, top_p, probs,
                      reinterpret_cast<cudaStream_t>(stream));
}

size_t dflash_sample_workspace_bytes(int rows, int vocab) {
  if (rows < 1 || vocab < 1) return 0;
  Carve c(nullptr, kWsHeader);
  c.take<int>(rows);
  c.take<unsigned long long>((size_t)rows * row_chunks(vocab));
  return c.off;
}

int dflash_sample_draft(int B, int G, int vocab, const float* q, const uint64_t* seeds,
                        uint64_t step, int32_t* y, void* workspace, size_t ws_bytes,
                        dflash_stream_t stream) {
  if (B < 1 || G < 1 || (long long)B * G > 65535 || vocab < 1 || vocab > kMaxVocab)
    return DFLASH_ERR_SHAPE;
  if (!q || !seeds || !y) return DFLASH_ERR_ARG;
  if (!aligned(q, 4) || !aligned(seeds, 8) || !aligned(y, 4)) return DFLASH_ERR_ALIGN;
  if (!workspace || !aligned(workspace, 256)) return DFLASH_ERR_WORKSPACE;
  const int rows = B * G;
  if (ws_bytes < dflash_sample_workspace_bytes(rows, vocab)) return DFLASH_ERR_WORKSPACE;
  Carve c(workspace, kWsHeader);
  int* counters = c.take<int>(rows);
  unsigned long long* zsum = c.take<unsigned long long>((size_t)rows * row_chunks(vocab));
  return launch_sample_rows(rows, vocab, q, vocab, G, seeds, step, kPurposeDraft, y, G, counters,
                            zsum, static_cast<int*>(workspace), reinterpret_cast<cudaStream_t>(stream));
}

int dflash_read_status(const void* workspace, int32_t* status_host, dflash_stream_t stream) {
  if (!workspace || !status_host) return DFLASH_ERR_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  DFL_CUDA_TRY(cudaMemcpyAsync(status_host, workspace, sizeof(int32_t), cudaMemcpyDeviceToHost, s));
  DFL_CUDA_TRY(cudaStreamSynchronize(s));
  return DFLASH_OK;
}

const char* dflash_strerror(int code) {
  switch (code) {
    case DFLASH_OK: return "ok";
    case DFLASH_ERR_ARG: return "invalid argument";
    case DFLASH_ERR_SHAPE: return "sizes out of range or inconsistent";
    case DFLASH_ERR_ALIGN: return "pointer not suitably aligned";
    case DFLASH_ERR_UNSUPPORTED: return "configuration not supported by the kernels";
    case DFLASH_ERR_LAUNCH: return "kernel launch failed";
    case DFLASH_ERR_DEVICE_TIMEOUT: return "a bounded device-side wait gave up";
    case DFLASH_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case DFLASH_ERR_CUDA: return "CUDA runtime or driver call failed";
    case DFLASH_ERR_RANGE: return "a weight or an activation is beyond the fp16 range";
    default: return "unknown error code";
  }
}

}  // extern "C"
