// Block attention of the drafter on mma.sync, and the launcher.  The
// tensor-core kernel (attention_tc.cu) takes every shape this one takes (head
// dims 64 and 128, gamma <= 16; up to 128 query rows per KV head against 96
// here) and runs by default; this one is built in for comparison and runs
// when the library is compiled with DFLASH_ATTN_TC=0.  The gamma block queries of every query
// head attend over [context window ; whole block], non-causally inside the
// block ("DFlash vs DFlash 2" blog, section "Conditioning on the target
// model": K_i = [W^K H_t ; W^K H_d], V_i = [W^V H_t ; W^V H_d]; block
// positions attend to one another non-causally; model card
// "Beam-1.0-501B-A23B-DFlash2", section "Model": 4,096-token sliding window,
// 40 query / 8 KV heads).
//
// One CTA serves one (request, KV head, key split).  The group of query heads
// that share the KV head times the gamma block positions (5 x 8 = 40 rows at
// the full size) is packed into 16-row MMA tiles, so every K/V byte read from
// HBM is used by all query heads of its group.  Each row tile has KW consumer
// warps that take alternate key tiles (more warps in flight per SM: one warp's
// chain of dependent MMAs, shuffles and exponentials leaves the SM idle) and
// merge their softmax states at the end.
// A producer warp streams 64-key K/V tiles of the context ring into shared
// memory with TMA (128-byte swizzle, evict-first), STAGES deep.  Scores run
// on mma.sync with fp16 operands (queries are fp16; ring keys, stored bf16,
// are widened to fp16 — exact in fp16's range — either in registers by each
// consumer or, with many row tiles, once per tile in place by a converter
// warp) and P.V on bf16
// operands against the bf16 ring values (fp16 for the block's own values),
// all with fp32 accumulation; the softmax is online
// (running max and sum per row, reduced with warp shuffles); the window and
// block masks are arithmetic (context slot j is visible iff j < min(L, W),
// every block key is visible).  Splits of the key range write unnormalised
// partials, and the last CTA of a (request, KV head) merges them in split
// order — deterministic.
#include <cooperative_groups.h>

#include <cmath>

#include "attention.h"
#include "attention_util.cuh"
#include "common.cuh"
#include "gemm.h"

namespace dfl {
namespace {

namespace cg = cooperative_groups;
using namespace attn;

// Largest thread-block cluster (key splits of one head) attention will use.
// (8 measured faster than 16 at batch 1 on GB300: a 16-CTA cluster waits for
// 16 free SMs of one GPC while the previous kernel drains.)
#ifndef DFLASH_ATTN_MAX_CLUSTER
#define DFLASH_ATTN_MAX_CLUSTER 8
#endif

constexpr int kKeys = 64;      // keys per context tile (both kernels)

// 1: attention runs on the tensor-core kernel (attention_tc.cu); 0: on the
// mma.sync kernel below (for comparison)
#ifndef DFLASH_ATTN_TC
#define DFLASH_ATTN_TC 1
#endif

// Stage buffers: each key-split group owns its own stages (2 each; 3 when
// there is one group), so every consumer waits on its stages' phases in
// order.  Key tile i goes to group i % KW, stage (i % KW) * SPG + (i / KW) % SPG.
__host__ __device__ constexpr int attn_spg(int KW) { return KW == 1 ? 3 : 2; }
__host__ __device__ constexpr int attn_stages(int KW) { return KW * attn_spg(KW); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_f16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
template <int HD>
struct WarpState {
  static constexpr int NT = HD / 8;  // output n-tiles of 8 dims
  float o[NT][4];
  float m[2], l[2];
  uint32_t qa[HD / 16][4];           // fp16 Q fragments (A operand), k-steps of 16 dims
};

// Scores, online softmax and P.V of one key tile held in shared memory as
// HD/64 swizzled halves [NK keys][64 dims] for K and for V: bf16 ring values
// (RING) or the block's own fp16 values.  Keys are fp16, or bf16 ring keys
// widened in registers here when WIDEN.
template <int HD, int NK, bool RING, bool WIDEN>
__device__ __forceinline__ void process_tile(WarpState<HD>& st, uint32_t k_base, uint32_t v_base,
                                             int n_valid, float scale_log2) {
  constexpr int NT_S = NK / 8;
  constexpr uint32_t kHalf = NK * 128;  // bytes of one 64-dim half
  const int lane = threadIdx.x & 31;
  float s[NT_S][4];
#pragma unroll
  for (int j = 0; j < NT_S; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.0f;

  // S = Q K^T on fp16 operands.  For each 16-dim k-step the K fragments of
  // all key n-tiles are loaded (and widened) first, then every accumulator
  // receives its MMA.
#pragma unroll
  for (int kk = 0; kk < HD / 16; ++kk) {
    uint32_t bk[NT_S / 2][4];
#pragma unroll
    for (int kp = 0; kp < NT_S / 2; ++kp) {
      const int key = kp * 16 + (lane & 7) + ((lane >> 4) << 3);
      const int dim = kk * 16 + (((lane >> 3) & 1) << 3);
      ldsm_x4(k_base + (dim >> 6) * kHalf + swz(key, dim & 63), bk[kp][0], bk[kp][1], bk[kp][2],
              bk[kp][3]);
      if (WIDEN) {
#pragma unroll
        for (int e = 0; e < 4; ++e) bk[kp][e] = bf16x2_to_f16x2(bk[kp][e]);
      }
    }
#pragma unroll
    for (int kp = 0; kp < NT_S / 2; ++kp) {
      mma_f16(s[2 * kp], st.qa[kk][0], st.qa[kk][1], st.qa[kk][2], st.qa[kk][3], bk[kp][0], bk[kp][1]);
      mma_f16(s[2 * kp + 1], st.qa[kk][0], st.qa[kk][1], st.qa[kk][2], st.qa[kk][3], bk[kp][2],
              bk[kp][3]);
    }
  }
  // mask and scale; rows r0 = lane/4 (regs 0,1) and r1 = lane/4 + 8 (regs 2,3)
  float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
  for (int j = 0; j < NT_S; ++j) {
    const int key = j * 8 + ((lane & 3) << 1);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const bool ok = (key + (e & 1)) < n_valid;
      s[j][e] = ok ? s[j][e] * scale_log2 : -INFINITY;
      mx[e >> 1] = fmaxf(mx[e >> 1], s[j][e]);
    }
  }
  float corr[2], mnew[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
    mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
    mnew[h] = fmaxf(st.m[h], mx[h]);
    const float base = mnew[h] == -INFINITY ? 0.0f : mnew[h];
    corr[h] = exp2f(st.m[h] - base);
    st.m[h] = mnew[h];
    mnew[h] = base;
    st.l[h] *= corr[h];
  }
#pragma unroll
  for (int t = 0; t < WarpState<HD>::NT; ++t) {
    st.o[t][0] *= corr[0];
    st.o[t][1] *= corr[0];
    st.o[t][2] *= corr[1];
    st.o[t][3] *= corr[1];
  }
#pragma unroll
  for (int j = 0; j < NT_S; ++j) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      s[j][e] = exp2f(s[j][e] - mnew[e >> 1]);
      st.l[e >> 1] += s[j][e];
    }
  }
  // O += P V: k-steps of 16 keys; V^T fragments through ldmatrix.trans; P in
  // the type of V (bf16 for ring tiles, fp16 for the block).  Keys past
  // n_valid have P = 0, and their V halves are zeroed in registers so that
  // whatever those slots hold cannot turn 0 * V into NaN.
  const int kq = (lane & 3) << 1;
#pragma unroll
  for (int ks = 0; ks < NK / 16; ++ks) {
    const uint32_t a0 = RING ? pack_bf16(s[2 * ks][0], s[2 * ks][1]) : pack_f16(s[2 * ks][0], s[2 * ks][1]);
    const uint32_t a1 = RING ? pack_bf16(s[2 * ks][2], s[2 * ks][3]) : pack_f16(s[2 * ks][2], s[2 * ks][3]);
    const uint32_t a2 = RING ? pack_bf16(s[2 * ks + 1][0], s[2 * ks + 1][1])
                             : pack_f16(s[2 * ks + 1][0], s[2 * ks + 1][1]);
    const uint32_t a3 = RING ? pack_bf16(s[2 * ks + 1][2], s[2 * ks + 1][3])
                             : pack_f16(s[2 * ks + 1][2], s[2 * ks + 1][3]);
    const int k0 = ks * 16 + kq;  // keys of the low (k0, k0+1) and high (k0+8, k0+9) halves
    const uint32_t m_lo = (k0 < n_valid ? 0x0000FFFFu : 0u) | (k0 + 1 < n_valid ? 0xFFFF0000u : 0u);
    const uint32_t m_hi = (k0 + 8 < n_valid ? 0x0000FFFFu : 0u) | (k0 + 9 < n_valid ? 0xFFFF0000u : 0u);
#pragma unroll
    for (int dp = 0; dp < HD / 16; ++dp) {
      const int key = ks * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
      const int dim = dp * 16 + ((lane >> 4) << 3);
      const uint32_t addr = v_base + (dim >> 6) * kHalf + swz(key, dim & 63);
      uint32_t b0, b1, b2, b3;
      ldsm_x4_t(addr, b0, b1, b2, b3);
      b0 &= m_lo;
      b2 &= m_lo;
      b1 &= m_hi;
      b3 &= m_hi;
      if (RING) {
        mma_bf16(st.o[2 * dp], a0, a1, a2, a3, b0, b1);
        mma_bf16(st.o[2 * dp + 1], a0, a1, a2, a3, b2, b3);
      } else {
        mma_f16(st.o[2 * dp], a0, a1, a2, a3, b0, b1);
        mma_f16(st.o[2 * dp + 1], a0, a1, a2, a3, b2, b3);
      }
    }
  }
}

// One CTA per (key split, KV head, request); the S splits of a (request, KV
// head) form one thread-block cluster and merge their partial softmax states
// through distributed shared memory.  Warp 0 produces; warp 1 + mt + MT * kw
// is the consumer of row tile mt taking key tiles kw, kw + KW, ...  With four
// or more row tiles one more warp widens each ring key tile to fp16 in place,
// once for all its consumers (measured: batch 32, gamma 16, 1.16 -> 0.94 ms
// per pass); with fewer, each consumer widens its fragments in registers (the
// extra handoff cost more than it saved at gamma 8 and batch 1).
template <int HD, int MT, int KW>
__host__ __device__ constexpr bool attn_conv_warp() { return MT >= 4; }

template <int HD, int MT, int KW>
__global__ void __launch_bounds__((MT * KW + 1 + (attn_conv_warp<HD, MT, KW>() ? 1 : 0)) * 32)
    attn_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                const AttnArgs a) {
  pdl_enter();
  constexpr int kTileBytes = kKeys * HD * 2;     // one of K or V, all halves
  constexpr int kStageBytes = 2 * kTileBytes;
  constexpr int kMq = MT * 16;
  constexpr int kBlkKeys = 16;
  constexpr int kConsumers = MT * KW * 32;
  constexpr int SPG = attn_spg(KW);
  constexpr int kStages = attn_stages(KW);
  static_assert((KW - 1) * kMq * (HD + 2) * 4 <= kStages * kStageBytes,
                "key-split states must fit the stage buffers");
  auto stage_of = [](int i) { return (i % KW) * SPG + (i / KW) % SPG; };
  auto phase_of = [](int i) { return (uint32_t)((i / KW) / SPG) & 1u; };
  static_assert(kMq * (HD + 2 + 16) * 4 <= kStages * kStageBytes, "partials must fit the stage buffers");
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[kStages], empty_bar[kStages], kready_bar[kStages];
  constexpr bool kHasConv = attn_conv_warp<HD, MT, KW>();
  constexpr int kConv = kHasConv ? MT * KW + 1 : 1 << 20;  // converter warp (if any)
  __shared__ int abort_sh;

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* q_s = smem + kStages * kStageBytes;            // fp16 [kMq][HD] swizzled halves
  uint8_t* bk_s = q_s + kMq * HD * 2;                     // block K, fp16 [16][HD]
  uint8_t* bv_s = bk_s + kBlkKeys * HD * 2;               // block V [16][HD]
  float* part_s = reinterpret_cast<float*>(smem);         // after the loop: [kMq][HD] partial O
  float* ml_s = part_s + kMq * HD;                        // [kMq][2] running max (log2) and sum
  float* w_s = ml_s + kMq * 2;                            // [rows of this CTA][16] merge weights

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int S = gridDim.x;
  const int group = a.n_q / a.n_kv;
  const int rows = group * a.gamma;                       // valid query rows
  const long long L = a.ctx_len[b];
  const int n_valid = (int)(L < (long long)a.window ? (L < 0 ? 0 : L) : a.window);
  const int tiles = (n_valid + kKeys - 1) / kKeys;
  const int t0 = (int)((long long)split * tiles / S), t1 = (int)((long long)(split + 1) * tiles / S);
  const int nt = t1 - t0;
  const bool do_block = split == S - 1;
  int slot_b = a.req_slot ? a.req_slot[b] : b;
  if (slot_b < 0 || slot_b >= a.ring_batch) {
    // reads then fall outside the ring and come back as zeros (TMA bounds check)
    if (threadIdx.x == 0 && split == 0) report_status(a.status, DFLASH_ERR_ARG);
    slot_b = a.ring_batch;
  }
  const int row_base = (slot_b * a.n_kv + g) * a.window;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], MT);
      mbar_init(&kready_bar[s], 1);
    }
    abort_sh = 0;
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && nt > 0) {
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      const uint64_t pol = policy_evict_first();
      int issued = 0;
      for (int i = 0; i < nt; ++i) {
        const int s = stage_of(i);
        const uint32_t ph = phase_of(i);
        if (!mbar_wait_bounded(&empty_bar[s], ph ^ 1u, &abort_sh, a.status)) break;
        uint8_t* ks = smem + s * kStageBytes;
        uint8_t* vs = ks + kTileBytes;
        mbar_arrive_expect_tx(&full_bar[s], kStageBytes);
        const int row = row_base + (t0 + i) * kKeys;
#pragma unroll
        for (int h = 0; h < HD / 64; ++h) {
          tma_load_2d(ks + h * (kKeys * 128), &tmK, &full_bar[s], h * 64, row, pol);
          tma_load_2d(vs + h * (kKeys * 128), &tmV, &full_bar[s], h * 64, row, pol);
        }
        issued = i + 1;
      }
      if (abort_sh) {
        // a wait gave up: let the copies in flight land before reusing the buffers
        int dummy = 0;
        for (int i = (issued > kStages ? issued - kStages : 0); i < issued; ++i)
          (void)mbar_wait_bounded(&full_bar[stage_of(i)], phase_of(i), &dummy, nullptr, 100000000ull);
      }
    }
  }

  if (kHasConv && warp == kConv) {
    // ------------------------------------------------------------- converter
    // ring keys are bf16: widen each tile's keys to fp16 in place, once
    for (int i = 0; i < nt; ++i) {
      const int s = stage_of(i);
      if (!warp_wait(&full_bar[s], phase_of(i), &abort_sh, a.status)) break;
      uint4* k4 = reinterpret_cast<uint4*>(smem + s * kStageBytes);
#pragma unroll 4
      for (int idx = lane; idx < kTileBytes / 16; idx += 32) {
        uint4 u = k4[idx];
        u.x = bf16x2_to_f16x2(u.x);
        u.y = bf16x2_to_f16x2(u.y);
        u.z = bf16x2_to_f16x2(u.z);
        u.w = bf16x2_to_f16x2(u.w);
        k4[idx] = u;
      }
      // these generic-proxy writes must be ordered before the TMA copy that
      // later refills the stage (an async-proxy write to the same bytes)
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&kready_bar[s]);
    }
  }

  WarpState<HD> st;
  if (warp > 0 && warp < kConv) {
    // ----------------------------------------------------------- consumers
    const int ctid = threadIdx.x - 32;
    // Q rows ri = hh * gamma + i  <-  qkv row b*gamma + i, column (g*group + hh) * hd,
    // and the block's own K/V rows: asynchronous 16-byte copies, all in flight
    // together (rows past the block are zero-filled).
    for (int idx = ctid; idx < kMq * (HD / 8); idx += kConsumers) {
      const int ri = idx / (HD / 8), ch = idx % (HD / 8);
      const bool ok = ri < rows;
      const int hh = ok ? ri / a.gamma : 0, i = ok ? ri % a.gamma : 0;
      const size_t src = (size_t)(b * a.gamma + i) * a.ld_qkv + (size_t)(g * group + hh) * HD + ch * 8;
      const int col = ch * 8;
      const uint32_t off = (col >> 6) * (kMq * 128) + swz(ri, col & 63);
      cp_async16(q_s + off, a.qkv + src, ok);
    }
    if (do_block) {
      const size_t kcol = (size_t)a.n_q * HD + (size_t)g * HD;
      const size_t vcol = (size_t)(a.n_q + a.n_kv) * HD + (size_t)g * HD;
      for (int idx = ctid; idx < kBlkKeys * (HD / 8); idx += kConsumers) {
        const int r = idx / (HD / 8), ch = idx % (HD / 8);
        const bool ok = r < a.gamma;
        const __half* row = a.qkv + (size_t)(b * a.gamma + (ok ? r : 0)) * a.ld_qkv;
        const int col = ch * 8;
        const uint32_t off = (col >> 6) * (kBlkKeys * 128) + swz(r, col & 63);
        cp_async16(bk_s + off, row + kcol + ch * 8, ok);
        cp_async16(bv_s + off, row + vcol + ch * 8, ok);
      }
    }
    cp_async_wait_all();
    named_sync(1, kConsumers);

    const int mt = (warp - 1) % MT, kw = (warp - 1) / MT;
    {
      const uint32_t qb = smem_u32(q_s);
#pragma unroll
      for (int kk = 0; kk < HD / 16; ++kk) {
        const int row = mt * 16 + (lane & 15);
        const int col = kk * 16 + ((lane >> 4) << 3);
        ldsm_x4(qb + (col >> 6) * (kMq * 128) + swz(row, col & 63), st.qa[kk][0], st.qa[kk][1],
                st.qa[kk][2], st.qa[kk][3]);
      }
    }
#pragma unroll
    for (int t = 0; t < WarpState<HD>::NT; ++t) st.o[t][0] = st.o[t][1] = st.o[t][2] = st.o[t][3] = 0.f;
    st.m[0] = st.m[1] = -INFINITY;
    st.l[0] = st.l[1] = 0.0f;

    // the block's own keys go to the key-split warp with the fewest ring tiles
    if (do_block && kw == (KW - 1 - (nt % KW)) % KW)
      process_tile<HD, kBlkKeys, false, false>(st, smem_u32(bk_s), smem_u32(bv_s), a.gamma, a.scale_log2);
    for (int i = kw; i < nt; i += KW) {
      const int s = stage_of(i);
      const uint32_t ph = phase_of(i);
      // K widened (or just landed), V landed
      if (!warp_wait(kHasConv ? &kready_bar[s] : &full_bar[s], ph, &abort_sh, a.status)) break;
      uint8_t* ks = smem + s * kStageBytes;
      uint8_t* vs = ks + kTileBytes;
      const int slot0 = (t0 + i) * kKeys;
      const int valid = n_valid - slot0 < kKeys ? n_valid - slot0 : kKeys;
      process_tile<HD, kKeys, true, !kHasConv>(st, smem_u32(ks), smem_u32(vs), valid, a.scale_log2);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[s]);
    }
    // full row sums
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      st.l[h] += __shfl_xor_sync(0xffffffffu, st.l[h], 1);
      st.l[h] += __shfl_xor_sync(0xffffffffu, st.l[h], 2);
    }
  }

  const int cw = (warp > 0 && warp < kConv) ? (warp - 1) % MT : 0;  // row tile of a consumer warp
  const bool lead = warp > 0 && warp <= MT;                // kw == 0: holds the merged state
  if (KW > 1) {
    // Merge the key-split states of each row tile into its kw == 0 warp,
    // through the stage buffers (every stage has been consumed, or the CTA
    // gave up).  State (o, m, l) of warp kw >= 1 sits at [kw - 1][row].
    __syncthreads();
    float* kst = reinterpret_cast<float*>(smem);
    constexpr int kRowF = HD + 2;                          // o[HD], m, l
    if (warp > MT && warp < kConv) {
      const int kw = (warp - 1) / MT;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float* row = kst + ((size_t)(kw - 1) * kMq + cw * 16 + (lane >> 2) + 8 * h) * kRowF;
#pragma unroll
        for (int t = 0; t < WarpState<HD>::NT; ++t)
          *reinterpret_cast<float2*>(row + t * 8 + ((lane & 3) << 1)) =
              make_float2(st.o[t][2 * h], st.o[t][2 * h + 1]);
        if ((lane & 3) == 0) {
          row[HD] = st.m[h];
          row[HD + 1] = st.l[h];
        }
      }
    }
    __syncthreads();
    if (lead) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float M = st.m[h];
        for (int k = 1; k < KW; ++k)
          M = fmaxf(M, kst[((size_t)(k - 1) * kMq + cw * 16 + (lane >> 2) + 8 * h) * kRowF + HD]);
        const float base = M == -INFINITY ? 0.0f : M;
        const float c0 = exp2f(st.m[h] - base);
        st.l[h] *= c0;
#pragma unroll
        for (int t = 0; t < WarpState<HD>::NT; ++t) {
          st.o[t][2 * h] *= c0;
          st.o[t][2 * h + 1] *= c0;
        }
        for (int k = 1; k < KW; ++k) {
          const float* row = kst + ((size_t)(k - 1) * kMq + cw * 16 + (lane >> 2) + 8 * h) * kRowF;
          const float ck = exp2f(row[HD] - base);
          st.l[h] += ck * row[HD + 1];
#pragma unroll
          for (int t = 0; t < WarpState<HD>::NT; ++t) {
            const float2 v = *reinterpret_cast<const float2*>(row + t * 8 + ((lane & 3) << 1));
            st.o[t][2 * h] += ck * v.x;
            st.o[t][2 * h + 1] += ck * v.y;
          }
        }
        st.m[h] = M;
      }
    }
  }

  const int r0 = cw * 16 + (lane >> 2), r1 = r0 + 8;
  if (S == 1) {
    if (lead) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int ri = h ? r1 : r0;
        if (ri < rows) {
          const float inv = 1.0f / st.l[h];
          const int hh = ri / a.gamma, i = ri % a.gamma;
          const size_t off = (size_t)(b * a.gamma + i) * a.ld_out + (size_t)(g * group + hh) * HD;
#pragma unroll
          for (int t = 0; t < WarpState<HD>::NT; ++t) {
            const int d = t * 8 + ((lane & 3) << 1);
            store_h2(a.out, off + d, st.o[t][2 * h] * inv, st.o[t][2 * h + 1] * inv);
          }
        }
      }
    }
    return;
  }

  // ------------------------------------------------ merge across the cluster
  // every stage buffer has been consumed (or the CTA gave up): reuse them
  __syncthreads();
  if (lead) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int ri = h ? r1 : r0;
#pragma unroll
      for (int t = 0; t < WarpState<HD>::NT; ++t) {
        const int d = t * 8 + ((lane & 3) << 1);
        *reinterpret_cast<float2*>(part_s + ri * HD + d) = make_float2(st.o[t][2 * h], st.o[t][2 * h + 1]);
      }
      if ((lane & 3) == 0) {
        ml_s[ri * 2 + 0] = st.m[h];
        ml_s[ri * 2 + 1] = st.l[h];
      }
    }
  }
  cg::cluster_group cluster = cg::this_cluster();
  cluster.sync();
  const int rank = (int)cluster.block_rank();
  const int my_rows = (rows - rank + S - 1) / S;           // rows rank, rank + S, ...
  if ((int)threadIdx.x < my_rows) {
    const int ri = rank + (int)threadIdx.x * S;
    float mv[16], lv[16];
#pragma unroll
    for (int s = 0; s < 16; ++s) {
      if (s < S) {
        const float* ml = cluster.map_shared_rank(ml_s, s);
        mv[s] = ml[ri * 2];
        lv[s] = ml[ri * 2 + 1];
      }
    }
    float M = -INFINITY;
#pragma unroll
    for (int s = 0; s < 16; ++s)
      if (s < S) M = fmaxf(M, mv[s]);
    float den = 0.0f;
#pragma unroll
    for (int s = 0; s < 16; ++s) {
      if (s < S) {
        mv[s] = mv[s] == -INFINITY ? 0.0f : exp2f(mv[s] - M);
        den += mv[s] * lv[s];
      }
    }
    const float inv = 1.0f / den;
#pragma unroll
    for (int s = 0; s < 16; ++s)
      if (s < S) w_s[threadIdx.x * 16 + s] = mv[s] * inv;
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < my_rows * (HD / 2); idx += blockDim.x) {
    const int k = idx / (HD / 2), d = (idx % (HD / 2)) * 2;
    const int ri = rank + k * S;
    float2 pv[16];
#pragma unroll
    for (int s = 0; s < 16; ++s)
      if (s < S) pv[s] = *reinterpret_cast<const float2*>(cluster.map_shared_rank(part_s, s) + ri * HD + d);
    float o0 = 0.0f, o1 = 0.0f;
#pragma unroll
    for (int s = 0; s < 16; ++s) {
      if (s < S) {
        o0 += w_s[k * 16 + s] * pv[s].x;
        o1 += w_s[k * 16 + s] * pv[s].y;
      }
    }
    const int hh = ri / a.gamma, i = ri % a.gamma;
    store_h2(a.out, (size_t)(b * a.gamma + i) * a.ld_out + (size_t)(g * group + hh) * HD + d, o0, o1);
  }
  // no CTA may leave while another still reads its shared memory
  cluster.sync();
}

// Key-split warps per row tile: 3 for up to 3 row tiles, 2 for 4-5, else 1
// (at most 10 consumer warps, so that the registers of one SM suffice).
#ifndef DFLASH_ATTN_KW_MAX
#define DFLASH_ATTN_KW_MAX 3
#endif
constexpr int attn_kw(int MT) {
  return MT <= 3 && DFLASH_ATTN_KW_MAX >= 3 ? 3 : (MT <= 5 && DFLASH_ATTN_KW_MAX >= 2 ? 2 : 1);
}

template <int HD, int MT>
int launch_t(const CUtensorMap& tk, const CUtensorMap& tv, const AttnArgs& a, int B, cudaStream_t s) {
  constexpr int KW = attn_kw(MT);
  constexpr int kThreadsT = (MT * KW + 1 + (attn_conv_warp<HD, MT, KW>() ? 1 : 0)) * 32;
  constexpr size_t smem = 1024 + (size_t)attn_stages(KW) * 2 * kKeys * HD * 2 +
                          (size_t)MT * 16 * HD * 2 + 2 * 16 * HD * 2;
  auto kern = attn_kernel<HD, MT, KW>;
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return DFLASH_ERR_LAUNCH;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
      return DFLASH_ERR_LAUNCH;
    attr = true;
  }
  // Largest power-of-two cluster (<= 16, the non-portable maximum) that the GPU
  // can co-schedule for this kernel; the key splits are capped to it.
  static int max_cluster = 0;
  if (max_cluster == 0) {
    max_cluster = 1;
    for (int c = DFLASH_ATTN_MAX_CLUSTER; c >= 2; c >>= 1) {
      cudaLaunchConfig_t q = {};
      q.gridDim = dim3(c, 1, 1);
      q.blockDim = dim3(kThreadsT);
      q.dynamicSmemBytes = smem;
      cudaLaunchAttribute qa[1];
      qa[0].id = cudaLaunchAttributeClusterDimension;
      qa[0].val.clusterDim.x = c;
      qa[0].val.clusterDim.y = 1;
      qa[0].val.clusterDim.z = 1;
      q.attrs = qa;
      q.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, kern, &q) == cudaSuccess && n > 0) {
        max_cluster = c;
        break;
      }
      (void)cudaGetLastError();
    }
  }
  // The key splits are capped to one cluster.  Splitting a head over two
  // 8-CTA clusters that meet through a ticket and merge partials from global
  // memory was measured slower at batch 1 (21 -> 35 us per layer).
  AttnArgs aa = a;
  while (aa.splits > max_cluster) aa.splits >>= 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(aa.splits, aa.n_kv, B);
  cfg.blockDim = dim3(kThreadsT);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr_c[2];
  attr_c[0].id = cudaLaunchAttributeClusterDimension;
  attr_c[0].val.clusterDim.x = aa.splits;
  attr_c[0].val.clusterDim.y = 1;
  attr_c[0].val.clusterDim.z = 1;
  attr_c[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr_c[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr_c;
  cfg.numAttrs = 2;
  if (cudaLaunchKernelEx(&cfg, kern, tk, tv, aa) != cudaSuccess) return DFLASH_ERR_LAUNCH;
  return DFLASH_OK;
}

}  // namespace

int attn_row_tiles(int n_q, int n_kv, int gamma) { return (n_q / n_kv * gamma + 15) / 16; }

int launch_attention(const void* ring_k_layer, const void* ring_v_layer, const AttnArgs& a, int B,
                     cudaStream_t s) {
  CUtensorMap tk, tv;
  const uint64_t rows = (uint64_t)a.ring_batch * a.n_kv * a.window;
  int rc = encode_2d(&tk, ring_k_layer, OPND_BF16, (uint64_t)a.hd, rows, 64, kKeys);
  if (rc) return rc;
  rc = encode_2d(&tv, ring_v_layer, OPND_BF16, (uint64_t)a.hd, rows, 64, kKeys);
  if (rc) return rc;
  if (DFLASH_ATTN_TC && attention_tc_supported(a)) return launch_attention_tc(tk, tv, a, B, s);
  const int mt = attn_row_tiles(a.n_q, a.n_kv, a.gamma);
  if (a.hd == 128) {
    switch (mt) {
      case 1: return launch_t<128, 1>(tk, tv, a, B, s);
      case 2: return launch_t<128, 2>(tk, tv, a, B, s);
      case 3: return launch_t<128, 3>(tk, tv, a, B, s);
      case 4: return launch_t<128, 4>(tk, tv, a, B, s);
      case 5: return launch_t<128, 5>(tk, tv, a, B, s);
      case 6: return launch_t<128, 6>(tk, tv, a, B, s);
      default: return DFLASH_ERR_UNSUPPORTED;
    }
  }
  switch (mt) {
    case 1: return launch_t<64, 1>(tk, tv, a, B, s);
    case 2: return launch_t<64, 2>(tk, tv, a, B, s);
    case 3: return launch_t<64, 3>(tk, tv, a, B, s);
    case 4: return launch_t<64, 4>(tk, tv, a, B, s);
    case 5: return launch_t<64, 5>(tk, tv, a, B, s);
    case 6: return launch_t<64, 6>(tk, tv, a, B, s);
    default: return DFLASH_ERR_UNSUPPORTED;
  }
}

}  // namespace dfl
