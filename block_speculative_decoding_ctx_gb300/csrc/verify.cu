// Verification and sampling kernels (greedy prefix match, rejection sampling
// with residual and bonus, row draws, temperature / top-p preparation).
//
// Method: "DFlash vs DFlash 2" (blog), section "The problem: one expensive
// token at a time" — accept y ~ q with probability min(1, p(y)/q(y)); at the
// first rejection draw from the normalised [p - q]+; if every draft survives
// draw a bonus token from the target's next distribution.  Sampling settings
// (temperature 0.7, top-p 0.99): model card "Beam-1.0-501B-A23B-DFlash2",
// section "Acceptance length".
//
// Design: every vocabulary row is split into chunks of kRowChunk floats, one
// CTA per (chunk, row), so that even one request keeps many SMs streaming.
// Each CTA reduces its chunk (a packed argmax key, or fixed-point masses) and
// the last CTA of a request — found with an atomic ticket after a memory
// fence — finishes the request: prefix match, or the integer inverse-CDF
// draw, which re-reads only the one chunk that holds the sampled index.  The
// tickets are reset by that last CTA, so the scratch needs no clearing
// between calls.  All draws are integer arithmetic on floor(w * 2^45), which
// makes them independent of summation order.  The temperature / top-p
// preparation of a row is in probs.cu.
#include "common.cuh"
#include "kernels.h"

namespace dfl {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ unsigned long long argmax_key(float v, int idx) {
  return ((unsigned long long)ordered_key(v) << 32) | (uint32_t)(~(uint32_t)idx);
}

// Fixed-point mass of `wfn(v)` over [v0, v1), strided by the block.
template <class WFn>
__device__ __forceinline__ unsigned long long chunk_mass(const WFn& wfn, int v0, int v1) {
  unsigned long long z = 0;
  int v = v0 + threadIdx.x;
  for (; v + 3 * kThreads < v1; v += 4 * kThreads) {
    const float a = wfn(v), b = wfn(v + kThreads), c = wfn(v + 2 * kThreads),
                d = wfn(v + 3 * kThreads);
    z += to_fixed45(a) + to_fixed45(b) + to_fixed45(c) + to_fixed45(d);
  }
  for (; v < v1; v += kThreads) z += to_fixed45(wfn(v));
  return z;
}

// Smallest v in [v0, v1) whose running fixed-point mass (from v0) exceeds T.
// Requires T < mass([v0, v1)).  Result on all threads (-1 if not found).
template <class WFn>
__device__ int find_in_chunk(const WFn& wfn, int v0, int v1, unsigned long long T,
                             unsigned long long* scratch, int* s_found) {
  const int len = v1 - v0;
  const int seg = (len + kThreads - 1) / kThreads;
  const int s0 = min(v1, v0 + (int)threadIdx.x * seg);
  const int s1 = min(v1, s0 + seg);
  unsigned long long local = 0;
  for (int v = s0; v < s1; ++v) local += to_fixed45(wfn(v));
  unsigned long long total;
  const unsigned long long excl = block_exclusive_scan(local, scratch, &total);
  if (threadIdx.x == 0) *s_found = -1;
  __syncthreads();
  if (local > 0 && T >= excl && T < excl + local) {
    unsigned long long acc = excl;
    for (int v = s0; v < s1; ++v) {
      acc += to_fixed45(wfn(v));
      if (acc > T) {
        *s_found = v;
        break;
      }
    }
  }
  __syncthreads();
  return *s_found;
}

// ------------------------------------------------------------------ greedy

__global__ void __launch_bounds__(kThreads)
    verify_greedy_kernel(const float* __restrict__ target, const int32_t* __restrict__ draft,
                         int gamma, int V, int chunks, int32_t* __restrict__ accept_len,
                         int32_t* __restrict__ tokens, int32_t* __restrict__ next_anchor,
                         int32_t* __restrict__ n_append, int* counters, unsigned long long* keys) {
  pdl_enter();
  __shared__ unsigned long long red[33];
  __shared__ int s_last;
  const int c = blockIdx.x;
  const int r = blockIdx.y;  // b * gamma + i
  const int b = r / gamma;
  const float* row = target + (size_t)r * V;
  const int v0 = c * kRowChunk;
  const int v1 = min(V, v0 + kRowChunk);

  // the thread's 32 elements of the chunk, loaded together
  constexpr int kPer = kRowChunk / kThreads;
  float xv[kPer];
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int v = v0 + threadIdx.x + j * kThreads;
    xv[j] = v < v1 ? __ldg(row + v) : -INFINITY;
  }
  unsigned long long best = 0ull;
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int v = v0 + threadIdx.x + j * kThreads;
    if (v < v1) {
      const unsigned long long k = argmax_key(xv[j], v);
      best = k > best ? k : best;
    }
  }
  best = block_max_u64(best, red);
  if (threadIdx.x == 0) {
    atomicMax(&keys[r], best);
    __threadfence();
    s_last = (atomicAdd(&counters[b], 1) == chunks * gamma - 1);
  }
  __syncthreads();
  if (!s_last) return;
  if (threadIdx.x == 0) {
    __threadfence();
    const int G = gamma - 1;
    int n = 0;
    bool match = true;
    int32_t last = -1;
    for (int i = 0; i < gamma; ++i) {
      const unsigned long long k = atomicExch(&keys[b * gamma + i], 0ull);
      const int a = (int)(~(uint32_t)(k & 0xFFFFFFFFull));
      int32_t t = -1;
      if (match) {
        t = a;
        if (i < G && draft[b * G + i] == a) {
          n = i + 1;
        } else {
          match = false;
          last = a;
        }
      }
      tokens[b * gamma + i] = t;
    }
    accept_len[b] = n;
    if (next_anchor) next_anchor[b] = last;
    if (n_append) n_append[b] = n + 1;
    atomicExch(&counters[b], 0);
  }
}

// ----------------------------------------------------------------- sampled

struct ResidW {
  const float* p;
  const float* q;
  __device__ __forceinline__ float operator()(int v) const {
    return fmaxf(__fsub_rn(__ldg(p + v), __ldg(q + v)), 0.0f);
  }
};
struct RowW {
  const float* p;
  __device__ __forceinline__ float operator()(int v) const { return __ldg(p + v); }
};

__global__ void __launch_bounds__(kThreads)
    verify_sampled_kernel(const float* __restrict__ p, const float* __restrict__ q,
                          const int32_t* __restrict__ draft, const uint64_t* __restrict__ seeds,
                          uint64_t step, int gamma, int V, int chunks,
                          int32_t* __restrict__ accept_len, int32_t* __restrict__ tokens,
                          int32_t* __restrict__ next_anchor, int32_t* __restrict__ n_append,
                          int* counters, unsigned long long* zsum, int* status) {
  pdl_enter();
  __shared__ unsigned long long red[33];
  __shared__ int s_n, s_last, s_chunk, s_use_resid, s_found;
  __shared__ unsigned long long s_T;
  const int c = blockIdx.x, b = blockIdx.y, G = gamma - 1;
  const uint64_t seed = seeds[b];

  // Accept tests: every CTA of the request derives the same n.
  if (threadIdx.x == 0) {
    int n = G;
    for (int i = 0; i < G; ++i) {
      const int y = draft[b * G + i];
      if (y < 0 || y >= V) {
        report_status(status, DFLASH_ERR_ARG);
        n = i;
        break;
      }
      const uint4 w = philox_draw(seed, step, (uint32_t)i, kPurposeAccept);
      const double u = (double)(w.x >> 8) * 0x1p-24;
      const double qy = (double)q[((size_t)b * G + i) * V + y];
      const double py = (double)p[((size_t)b * gamma + i) * V + y];
      if (!(u * qy < py)) {  // exact: 24-bit x 24-bit mantissas
        n = i;
        break;
      }
    }
    s_n = n;
  }
  __syncthreads();
  const int n = s_n;
  const bool rejected = n < G;
  const float* prow = p + ((size_t)b * gamma + n) * V;
  const float* qrow = q + ((size_t)b * G + (rejected ? n : 0)) * V;
  const int v0 = c * kRowChunk, v1 = min(V, v0 + kRowChunk);

  unsigned long long zr = 0, zp;
  zp = chunk_mass(RowW{prow}, v0, v1);
  if (rejected) zr = chunk_mass(ResidW{prow, qrow}, v0, v1);
  zp = block_sum(zp, red);
  zr = block_sum(zr, red);
  if (threadIdx.x == 0) {
    zsum[((size_t)b * chunks + c) * 2 + 0] = zr;
    zsum[((size_t)b * chunks + c) * 2 + 1] = zp;
    __threadfence();
    s_last = (atomicAdd(&counters[b], 1) == chunks - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (threadIdx.x == 0) {
    unsigned long long Zr = 0, Zp = 0;
    for (int k = 0; k < chunks; ++k) {
      Zr += __ldcg(&zsum[((size_t)b * chunks + k) * 2 + 0]);
      Zp += __ldcg(&zsum[((size_t)b * chunks + k) * 2 + 1]);
    }
    const int use_r = rejected && Zr > 0;
    const unsigned long long Z = use_r ? Zr : Zp;
    const uint4 w = philox_draw(seed, step, (uint32_t)n, kPurposeResidual);
    const unsigned long long u64 = ((unsigned long long)w.y << 32) | w.z;
    const unsigned long long T = __umul64hi(u64, Z);
    unsigned long long acc = 0;
    int ck = -1;
    for (int k = 0; k < chunks; ++k) {
      const unsigned long long z = __ldcg(&zsum[((size_t)b * chunks + k) * 2 + (use_r ? 0 : 1)]);
      if (T < acc + z) {
        ck = k;
        break;
      }
      acc += z;
    }
    if (Z == 0) report_status(status, DFLASH_ERR_ARG);
    s_use_resid = use_r;
    s_chunk = ck;
    s_T = T - acc;
  }
  __syncthreads();
  int tok = -1;
  if (s_chunk >= 0) {
    const int c0 = s_chunk * kRowChunk, c1 = min(V, c0 + kRowChunk);
    tok = s_use_resid ? find_in_chunk(ResidW{prow, qrow}, c0, c1, s_T, red, &s_found)
                      : find_in_chunk(RowW{prow}, c0, c1, s_T, red, &s_found);
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < gamma; ++i) {
      int32_t t = -1;
      if (i < n) t = draft[b * G + i];
      if (i == n) t = tok;
      tokens[b * gamma + i] = t;
    }
    accept_len[b] = n;
    if (next_anchor) next_anchor[b] = tok;
    if (n_append) n_append[b] = n + 1;
    atomicExch(&counters[b], 0);
  }
}

// --------------------------------------------------------------- row draws

__global__ void __launch_bounds__(kThreads)
    sample_rows_kernel(const float* __restrict__ w, long long row_stride, int V, int chunks,
                       int rows_per_req, const uint64_t* __restrict__ seeds, uint64_t step,
                       uint32_t purpose, int32_t* __restrict__ out, long long out_stride,
                       int* counters, unsigned long long* zsum, int* status) {
  pdl_enter();
  __shared__ unsigned long long red[33];
  __shared__ int s_last, s_chunk, s_found;
  __shared__ unsigned long long s_T;
  const int c = blockIdx.x, r = blockIdx.y;
  const float* row = w + (size_t)r * row_stride;
  const int v0 = c * kRowChunk, v1 = min(V, v0 + kRowChunk);
  unsigned long long z = block_sum(chunk_mass(RowW{row}, v0, v1), red);
  if (threadIdx.x == 0) {
    zsum[(size_t)r * chunks + c] = z;
    __threadfence();
    s_last = (atomicAdd(&counters[r], 1) == chunks - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const int b = r / rows_per_req, i = r % rows_per_req;
  if (threadIdx.x == 0) {
    unsigned long long Z = 0;
    for (int k = 0; k < chunks; ++k) Z += __ldcg(&zsum[(size_t)r * chunks + k]);
    const uint4 wd = philox_draw(seeds[b], step, (uint32_t)i, purpose);
    const unsigned long long u64 = ((unsigned long long)wd.y << 32) | wd.z;
    const unsigned long long T = __umul64hi(u64, Z);
    unsigned long long acc = 0;
    int ck = -1;
    for (int k = 0; k < chunks; ++k) {
      const unsigned long long zk = __ldcg(&zsum[(size_t)r * chunks + k]);
      if (T < acc + zk) {
        ck = k;
        break;
      }
      acc += zk;
    }
    if (Z == 0) report_status(status, DFLASH_ERR_ARG);
    s_chunk = ck;
    s_T = T - acc;
  }
  __syncthreads();
  int tok = -1;
  if (s_chunk >= 0) {
    const int c0 = s_chunk * kRowChunk, c1 = min(V, c0 + kRowChunk);
    tok = find_in_chunk(RowW{row}, c0, c1, s_T, red, &s_found);
  }
  if (threadIdx.x == 0) {
    out[(size_t)b * out_stride + i] = tok;
    atomicExch(&counters[r], 0);
  }
}

}  // namespace

int launch_verify_greedy(int B, int gamma, int V, const float* target, const int32_t* draft,
                         int32_t* accept_len, int32_t* tokens, int32_t* next_anchor,
                         int32_t* n_append, int* counters, unsigned long long* keys,
                         int* /*status*/, cudaStream_t s) {
  const int chunks = row_chunks(V);
  dim3 grid(chunks, B * gamma);
  return launch_pdl(verify_greedy_kernel, grid, dim3(kThreads), 0, s, target, draft, gamma, V, chunks,
                    accept_len, tokens, next_anchor, n_append, counters, keys);
}

int launch_verify_sampled(int B, int gamma, int V, const float* p, const float* q,
                          const int32_t* draft, const uint64_t* seeds, uint64_t step,
                          int32_t* accept_len, int32_t* tokens, int32_t* next_anchor,
                          int32_t* n_append, int* counters, unsigned long long* zsum, int* status,
                          cudaStream_t s) {
  const int chunks = row_chunks(V);
  dim3 grid(chunks, B);
  return launch_pdl(verify_sampled_kernel, grid, dim3(kThreads), 0, s, p, q, draft, seeds, step, gamma,
                    V, chunks, accept_len, tokens, next_anchor, n_append, counters, zsum, status);
}

int launch_sample_rows(int rows, int V, const float* w, long long row_stride, int rows_per_req,
                       const uint64_t* seeds, uint64_t step, uint32_t purpose, int32_t* out,
                       long long out_stride, int* counters, unsigned long long* zsum, int* status,
                       cudaStream_t s) {
  const int chunks = row_chunks(V);
  dim3 grid(chunks, rows);
  return launch_pdl(sample_rows_kernel, grid, dim3(kThreads), 0, s, w, row_stride, V, chunks,
                    rows_per_req, seeds, step, purpose, out, out_stride, counters, zsum, status);
}

}  // namespace dfl
