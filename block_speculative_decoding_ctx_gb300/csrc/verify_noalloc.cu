// Verification without a caller-provided workspace.
//
// Some callers cannot hand the library any device memory of their own when
// they verify: a serving process whose device memory is reserved up front by
// another allocator (a further cudaMalloc fails, or fragments that
// reservation), or a host framework that does not let plug-ins allocate
// device memory behind its back (cudaMalloc also synchronises the device,
// which such callers avoid on the decode path).  dflash_verify_noalloc serves
// them: it runs the same kernels as dflash_verify, but their scratch (the
// status word, per-request tickets, argmax keys and chunk masses) lives in one
// file-scope __device__ array of kNoAllocScratchBytes that every GPU loading
// this library holds until the process exits.  The call allocates nothing.
//
// The array is shared by every call on a device and keeps what the last call
// left in it, so each call first clears the part that must start at zero
// (status, tickets, keys) on its stream.  Two calls whose work overlaps on the
// GPU (different streams, or graphs replayed concurrently) race on it.
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace {

constexpr size_t kNoAllocScratchBytes = 256 * 1024;

static __device__ __align__(256) unsigned char g_verify_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};
void* g_scratch_ctx[kMaxDevices] = {};

// The CUDA context current on this thread (driver entry point, so that the
// library needs no link to libcuda), or nullptr.
void* current_context() {
  using Fn = int (*)(void**);
  static Fn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<Fn>(f);
  }();
  void* ctx = nullptr;
  if (!fn || fn(&ctx) != 0) return nullptr;
  return ctx;
}

// Device address of g_verify_scratch on the current device.  In host code the
// symbol is only a host-side stand-in.  A call made outside a stream capture
// looks the address up afresh (cheap once the module is loaded, and right
// after a device reset has loaded the module again at another address) and
// remembers it with the context it belongs to.  A call made while `s` is
// being captured must not trigger a module load, so it uses the remembered
// address, and only if it belongs to the current context; otherwise it
// returns DFLASH_ERR_UNSUPPORTED and launches nothing.
int scratch_address(cudaStream_t s, void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DFLASH_ERR_CUDA;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) {
    (void)cudaGetLastError();
    return DFLASH_ERR_CUDA;
  }
  void* ctx = current_context();
  std::lock_guard<std::mutex> lock(g_mu);
  if (cs == cudaStreamCaptureStatusNone) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_verify_scratch) != cudaSuccess || !p) return DFLASH_ERR_CUDA;
    g_scratch_ptr[dev] = p;
    g_scratch_ctx[dev] = ctx;
  } else if (!g_scratch_ptr[dev] || !ctx || g_scratch_ctx[dev] != ctx) {
    return DFLASH_ERR_UNSUPPORTED;
  }
  *out = g_scratch_ptr[dev];
  return DFLASH_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" {

int dflash_verify_noalloc(int mode, int B, int gamma, int vocab, const float* target,
                          const float* q, const int32_t* draft, const uint64_t* seeds,
                          uint64_t step, int32_t* accept_len, int32_t* tokens,
                          int32_t* next_anchor, int32_t* n_append, dflash_stream_t stream) {
  using namespace dfl;
  if (mode != DFLASH_VERIFY_GREEDY && mode != DFLASH_VERIFY_SAMPLED) return DFLASH_ERR_ARG;
  if (B < 1 || B > 65535 || gamma < 2 || gamma > 64 || vocab < 1 || vocab > (1 << 18))
    return DFLASH_ERR_SHAPE;
  if (!target || !draft || !accept_len || !tokens) return DFLASH_ERR_ARG;
  if (mode == DFLASH_VERIFY_SAMPLED && (!q || !seeds)) return DFLASH_ERR_ARG;
  if (!aligned(target, 4) || !aligned(draft, 4) || !aligned(accept_len, 4) ||
      !aligned(tokens, 4) || (q && !aligned(q, 4)) || (seeds && !aligned(seeds, 8)) ||
      (next_anchor && !aligned(next_anchor, 4)) || (n_append && !aligned(n_append, 4)))
    return DFLASH_ERR_ALIGN;

  // same layout as the workspace of dflash_verify, inside the static array
  Carve measure(nullptr, kWsHeader);
  measure.take<int>(B);
  measure.take<unsigned long long>((size_t)B * gamma);
  const size_t zero_end = measure.off;  // status, tickets and keys start at zero
  measure.take<unsigned long long>((size_t)B * row_chunks(vocab) * 2);
  if (measure.off > kNoAllocScratchBytes) return DFLASH_ERR_SHAPE;  // beyond the fixed scratch

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  void* base = nullptr;
  int rc = scratch_address(s, &base);
  if (rc) return rc;
  Carve c(base, kWsHeader);
  int* counters = c.take<int>(B);
  unsigned long long* keys = c.take<unsigned long long>((size_t)B * gamma);
  unsigned long long* zsum = c.take<unsigned long long>((size_t)B * row_chunks(vocab) * 2);
  int* status = static_cast<int*>(base);

  if (cudaMemsetAsync(base, 0, zero_end, s) != cudaSuccess) return DFLASH_ERR_CUDA;
  if (mode == DFLASH_VERIFY_GREEDY)
    return launch_verify_greedy(B, gamma, vocab, target, draft, accept_len, tokens, next_anchor,
                                n_append, counters, keys, status, s);
  return launch_verify_sampled(B, gamma, vocab, target, q, draft, seeds, step, accept_len, tokens,
                               next_anchor, n_append, counters, zsum, status, s);
}

}  // extern "C"
