// Sampling distribution of raw logits: probs = top_p(softmax(logits / T)).
//
// Model card "Beam-1.0-501B-A23B-DFlash2", section "Acceptance length":
// temperature 0.7, top-p 0.99.  Nucleus (the library's reading): ids ordered
// by (probability desc, id asc), the shortest prefix whose mass reaches
// top_p, renormalised.
//
// Design: one thread-block cluster of kPC CTAs per row.  Each CTA keeps its
// contiguous slice of the row in shared memory (logits, then e = exp(l/T -
// M), then p = e / S), so the row is read from memory once and every later
// pass runs on shared memory.  Row-wide values are merged over distributed
// shared memory in rank order, so every CTA of the cluster derives the same
// bits: the maximum M, the sum S, the fixed-point mass Z = sum floor(p 2^45),
// and, for top-p, a radix select over the bit patterns of p (8 bits per pass;
// each pass merges the CTAs' 256-bin histograms of mass and count) for the
// smallest kept probability t* and the mass above it.  Ties at t* that the
// nucleus cannot all keep go to the lowest ids, counted across the cluster in
// id order.
#include <cooperative_groups.h>

#include "common.cuh"
#include "kernels.h"

namespace dfl {
namespace {

namespace cg = cooperative_groups;

constexpr int kPC = 8;           // CTAs per row (one cluster)
constexpr int kPThreads = 512;

// Warp-aggregated add of (mass, count) into a 256-bin shared histogram.
// Every lane of the warp calls it (a warp-uniform loop).
__device__ __forceinline__ void hist_add(unsigned long long* hist, unsigned* histc, bool active,
                                         uint32_t digit, unsigned long long mass) {
  const unsigned act = __ballot_sync(0xffffffffu, active);
  if (!active) return;
  const unsigned grp = __match_any_sync(act, digit);
  const unsigned lo = __reduce_add_sync(grp, (unsigned)(mass & 0x7FFFFFu));
  const unsigned hi = __reduce_add_sync(grp, (unsigned)(mass >> 23));
  if ((int)(threadIdx.x & 31) == __ffs(grp) - 1) {
    atomicAdd(&hist[digit], ((unsigned long long)hi << 23) + lo);
    atomicAdd(&histc[digit], (unsigned)__popc(grp));
  }
}

__global__ void __launch_bounds__(kPThreads)
    probs_cluster_kernel(const float* __restrict__ logits, int V, int chunk, float invT, float top_p,
                         float* __restrict__ probs) {
  pdl_enter();
  extern __shared__ float vals[];
  __shared__ float redf[33];
  __shared__ unsigned long long redu[33];
  __shared__ float s_max, s_sum;                  // this CTA's partials, read by the cluster
  __shared__ unsigned long long s_z, s_tie, s_before;
  __shared__ unsigned long long hist[2][256];
  __shared__ unsigned histc[2][256];
  __shared__ unsigned long long tot_m[256];     // the cluster's histogram, summed here
  __shared__ unsigned tot_c[256];
  __shared__ float s_part[kPC];                 // the CTAs' partials, gathered here
  __shared__ unsigned long long s_above, s_thr, s_ntie;
  __shared__ uint32_t s_prefix, s_mask;

  cg::cluster_group cl = cg::this_cluster();
  const int rank = (int)cl.block_rank();
  const int tid = threadIdx.x;
  const size_t r = blockIdx.x / kPC;
  const int v0 = min(V, rank * chunk), v1 = min(V, v0 + chunk), n = v1 - v0;
  const float* row = logits + r * (size_t)V + v0;
  float* out = probs + r * (size_t)V + v0;

  // ---- max of l / T over the row
  float m = -INFINITY;
  for (int i = tid; i < n; i += kPThreads) {
    const float l = __ldg(row + i);
    vals[i] = l;
    m = fmaxf(m, l * invT);
  }
  m = warp_max_f(m);
  if ((tid & 31) == 0) redf[tid >> 5] = m;
  __syncthreads();
  if (tid < 32) {
    float t = tid < kPThreads / 32 ? redf[tid] : -INFINITY;
    t = warp_max_f(t);
    if (tid == 0) s_max = t;
  }
  cl.sync();
  if (tid < kPC) s_part[tid] = *cl.map_shared_rank(&s_max, tid);
  __syncthreads();
  float M = -INFINITY;
  for (int k = 0; k < kPC; ++k) M = fmaxf(M, s_part[k]);

  // ---- e = exp(l / T - M) (one fused rounding inside), S in rank order
  float s = 0.0f;
  for (int i = tid; i < n; i += kPThreads) {
    const float e = expf(__fmaf_rn(vals[i], invT, -M));
    vals[i] = e;
    s += e;
  }
  s = block_sum(s, redf);
  if (tid == 0) s_sum = s;
  cl.sync();
  if (tid < kPC) s_part[tid] = *cl.map_shared_rank(&s_sum, tid);
  __syncthreads();
  float S = 0.0f;
  for (int k = 0; k < kPC; ++k) S += s_part[k];

  // ---- p = e / S
  unsigned long long z = 0;
  for (int i = tid; i < n; i += kPThreads) {
    const float p = __fdiv_rn(vals[i], S);
    vals[i] = p;
    z += to_fixed45(p);
  }
  if (!(top_p < 1.0f)) {
    for (int i = tid; i < n; i += kPThreads) out[i] = vals[i];
    cl.sync();  // no CTA leaves while another may read its partials
    return;
  }

  // ---- fixed-point total and the nucleus threshold thr = ceil(top_p * Z)
  z = block_sum(z, redu);
  if (tid == 0) s_z = z;
  cl.sync();
  if (tid == 0) {
    unsigned long long Z = 0;
    for (int k = 0; k < kPC; ++k) Z += *cl.map_shared_rank(&s_z, k);
    unsigned long long thr = (unsigned long long)ceil((double)top_p * (double)Z);
    if (thr == 0) thr = 1;
    if (thr > Z) thr = Z;
    s_thr = thr;
    s_above = 0;
    s_prefix = 0;
    s_mask = 0;
  }
  __syncthreads();

  // ---- radix select on the bit pattern of p (p >= 0 orders like its bits):
  // the largest key t* whose mass of {key >= t*} reaches thr; s_above ends as
  // the mass of {key > t*}, s_ntie as the count of {key == t*}
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass, buf = pass & 1;
    if (tid < 256) {
      hist[buf][tid] = 0;
      histc[buf][tid] = 0;
    }
    __syncthreads();
    const uint32_t prefix = s_prefix, mask = s_mask;
    for (int i0 = 0; i0 < n; i0 += kPThreads) {
      const int i = i0 + tid;
      const float p = i < n ? vals[i] : 0.0f;
      const uint32_t key = __float_as_uint(p);
      hist_add(hist[buf], histc[buf], i < n && (key & mask) == prefix, (key >> shift) & 255u, to_fixed45(p));
    }
    cl.sync();
    if (tid < 256) {
      // bin tid summed over the cluster (in rank order)
      unsigned long long a = 0;
      unsigned c = 0;
#pragma unroll
      for (int k = 0; k < kPC; ++k) {
        a += cl.map_shared_rank(&hist[buf][0], k)[tid];
        c += cl.map_shared_rank(&histc[buf][0], k)[tid];
      }
      tot_m[tid] = a;
      tot_c[tid] = c;
    }
    __syncthreads();
    if (tid < 32) {
      // lane l holds digits 255 - 8l - j, j = 0..7 (descending); find the
      // digit where the running mass from the top reaches thr
      unsigned long long mass[8], tot = 0;
      unsigned cnt[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int d = 255 - 8 * tid - j;
        mass[j] = tot_m[d];
        cnt[j] = tot_c[d];
        tot += mass[j];
      }
      unsigned long long incl = tot;  // inclusive scan over lanes (lane 0 = top digits)
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long nb = __shfl_up_sync(0xffffffffu, incl, o);
        if (tid >= o) incl += nb;
      }
      const unsigned long long base = s_above, thr = s_thr;
      const unsigned long long excl = incl - tot;
      const bool here = base + excl < thr && base + incl >= thr;
      const unsigned who = __ballot_sync(0xffffffffu, here);
      // thr <= the remaining mass, so some lane holds it; fall back to the
      // lowest digit otherwise
      const int lw = who ? __ffs(who) - 1 : 31;
      if (tid == lw) {
        unsigned long long cum = base + excl;
        int j = 0;
        for (; j < 7; ++j) {
          if (cum + mass[j] >= thr) break;
          cum += mass[j];
        }
        const int d = 255 - 8 * tid - j;
        s_above = cum;
        s_prefix = prefix | ((uint32_t)d << shift);
        s_mask = mask | (255u << shift);
        s_ntie = cnt[j];
      }
    }
    __syncthreads();
  }
  const uint32_t tstar = s_prefix;
  const unsigned long long above = s_above, thr = s_thr;
  const unsigned long long pstar = to_fixed45(__uint_as_float(tstar));
  const unsigned long long n_tie = s_ntie;
  unsigned long long k_tie = pstar ? (thr - above + pstar - 1) / pstar : n_tie;
  if (k_tie > n_tie) k_tie = n_tie;
  const unsigned long long kept = above + k_tie * pstar;
  const float Sk = (float)((double)kept * 0x1p-45);

  if (k_tie == n_tie) {
    for (int i = tid; i < n; i += kPThreads) {
      const float p = vals[i];
      out[i] = (__float_as_uint(p) >= tstar) ? __fdiv_rn(p, Sk) : 0.0f;
    }
    cl.sync();
    return;
  }
  // Some ties at t* are dropped: keep the lowest ids.  Contiguous segments
  // per thread give an id-ordered rank inside the CTA; the CTAs before this
  // one (lower ids) contribute their tie counts.
  const int seg = (n + kPThreads - 1) / kPThreads;
  const int s0 = min(n, tid * seg), s1 = min(n, s0 + seg);
  unsigned long long nt = 0;
  for (int i = s0; i < s1; ++i) nt += (__float_as_uint(vals[i]) == tstar);
  unsigned long long tot;
  unsigned long long rk = block_exclusive_scan(nt, redu, &tot);
  if (tid == 0) s_tie = tot;
  cl.sync();
  if (tid == 0) {
    unsigned long long b0 = 0;
    for (int k = 0; k < rank; ++k) b0 += *cl.map_shared_rank(&s_tie, k);
    s_before = b0;
  }
  __syncthreads();
  rk += s_before;
  for (int i = s0; i < s1; ++i) {
    const float p = vals[i];
    const uint32_t key = __float_as_uint(p);
    bool keep = key > tstar;
    if (key == tstar) keep = (rk++ < k_tie);
    out[i] = keep ? __fdiv_rn(p, Sk) : 0.0f;
  }
  cl.sync();
}

}  // namespace

int launch_probs(int rows, int V, const float* logits, float temperature, float top_p, float* probs,
                 cudaStream_t s) {
  const int chunk = ((V + kPC - 1) / kPC + 3) / 4 * 4;
  const size_t smem = (size_t)chunk * sizeof(float);
  static size_t smem_set = 0;
  if (smem > smem_set) {
    if (cudaFuncSetAttribute(probs_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
      return DFLASH_ERR_LAUNCH;
    smem_set = smem;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)rows * kPC);
  cfg.blockDim = dim3(kPThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kPC;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, probs_cluster_kernel, logits, V, chunk, 1.0f / temperature, top_p, probs) ==
                 cudaSuccess
             ? DFLASH_OK
             : DFLASH_ERR_LAUNCH;
}

}  // namespace dfl
