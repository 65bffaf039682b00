// Block attention of the drafter on the 5th-generation tensor cores: the
// same operation as attention.cu ("DFlash vs DFlash 2" blog, section
// "Conditioning on the target model": the gamma block queries of every head
// attend over [context window ; whole block], non-causally inside the block;
// model card "Beam-1.0-501B-A23B-DFlash2", section "Model": 4,096-token
// window, 40 query / 8 KV heads), for many requests at once.
//
// One CTA serves one (request, KV head, key split); the query group x gamma
// rows (40 or 80 at the full size) are the M = 128 rows of every MMA (rows
// past them are zero).  Per 64-key tile j:
//   S_j = Q K_j^T      tcgen05.mma, M 128 x N 64 x K hd, fp32 in TMEM (two
//                      buffers).  The ring holds bf16 keys, so Q enters as a
//                      bf16 value plus its bf16 remainder (two MMAs): about 16
//                      significant bits of the fp16 queries.
//   P_j = exp2(S_j - m) computed by four softmax warps, one thread per row
//                      (the whole row is in the thread: no shuffles), written
//                      to shared memory as bf16 in the MMA's K-major layout.
//                      The running max m moves only when a row's tile max
//                      exceeds it by more than 2^8; then the O row is rescaled
//                      in TMEM first.
//   O += P_j V_j       tcgen05.mma, M 128 x N hd x K 64.  V arrives from the
//                      ring key-major; four warps transpose each tile to the
//                      dimension-major layout the MMA reads as a K-major B
//                      operand.
// A producer warp streams K and V tiles with TMA (three stages); one thread
// issues every MMA, S_{j+1} before P_j V_j so that the softmax of tile j
// overlaps the next score MMA.  The block's own keys and values (from the
// QKV projection, fp16, rounded to bf16) form one more tile.  The key splits
// of a (request, KV head) run as a thread-block cluster and merge their
// partial states over distributed shared memory in split order, as in
// attention.cu.  Every wait is bounded (mbar_wait_bounded).
#include <cooperative_groups.h>

#include <cmath>

#include "attention.h"
#include "common.cuh"
#include "gemm.h"

namespace dfl {
namespace {

namespace cg = cooperative_groups;

#ifndef DFLASH_ATTN_MAX_CLUSTER
#define DFLASH_ATTN_MAX_CLUSTER 8
#endif

constexpr int kKeysT = 64;        // keys per tile
constexpr int kThreadsT = 320;    // warp 0 TMA, 1 MMA, 2-5 softmax, 6-9 V transpose
constexpr int kSt = 3;            // K/V stages
constexpr float kRescale = 8.0f;  // log2 headroom before the running max moves

// Byte offset of element (row, col) of a [rows][64] 16-bit tile stored with
// the 128-byte swizzle (16-byte chunk index XOR row % 8) — the layout TMA
// writes and the tcgen05 K-major descriptors read.
__device__ __forceinline__ uint32_t swz(int row, int col) {
  return (uint32_t)(row * 128 + ((((col >> 3) ^ row) & 7) << 4) + ((col & 7) << 1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void named_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Bounded wait taken by a whole warp: every lane waits, and the warp goes on
// only if every lane saw the phase complete (a warp-uniform outcome, so that
// warp-collective instructions and __syncwarp after it stay convergent).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          int* status) {
  const bool ok = mbar_wait_bounded(bar, parity, abort_flag, status);
  return __all_sync(0xffffffffu, ok);
}

// Shared memory: Q (bf16 value and remainder), kSt stages of (K, V), two P
// tiles, two transposed V tiles.  The block's own keys live in the second P tile: the softmax first
// writes it for tile 1, after the block tile's score MMA (tile 0) completed.
template <int HD>
struct TcLayout {
  static constexpr int kHalves = HD / 64;
  static constexpr int kQ = 128 * HD * 2;           // one of Q value / remainder
  static constexpr int kKV = kKeysT * HD * 2;       // one of K or V (one tile)
  static constexpr int kP = 128 * kKeysT * 2;       // P tile
  static constexpr int kVt = HD * kKeysT * 2;       // transposed V tile
  static constexpr int oQh = 0;
  static constexpr int oQl = oQh + kQ;
  static constexpr int oStage = oQl + kQ;
  static constexpr int oP = oStage + kSt * 2 * kKV;
  static constexpr int oVt = oP + 2 * kP;
  static constexpr int oKblk = oP + kP;             // aliases P[1]
  static constexpr int kBytes = oVt + 2 * kVt;
  static_assert(kKV <= kP, "the block's keys must fit a P tile");
};

template <int HD>
__global__ void __launch_bounds__(kThreadsT, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                   const AttnArgs a) {
  pdl_enter();
  using Lay = TcLayout<HD>;
  constexpr uint32_t kTmemCols = 256;  // S: cols 0-127 (two buffers), O: cols 128-(128+HD)
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[kSt], empty_bar[kSt], s_full[2], s_empty[2], p_full[2],
      vt_full[2], pv_done[2], pro_bar, o_bar;
  __shared__ uint32_t tmem_sh;
  __shared__ int abort_sh;

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int S = gridDim.x;
  const int group = a.n_q / a.n_kv;
  const int rows = group * a.gamma;                 // valid query rows (<= 96)
  // softmax warps whose 32 rows hold at least one query; the others (their
  // rows are padding) sit out the tile loop
  const int n_live = (rows + 31) / 32;
  const long long L = a.ctx_len[b];
  const int n_valid = (int)(L < (long long)a.window ? (L < 0 ? 0 : L) : a.window);
  const int tiles = (n_valid + kKeysT - 1) / kKeysT;
  const int t0 = (int)((long long)split * tiles / S), t1 = (int)((long long)(split + 1) * tiles / S);
  const int nt = t1 - t0;                           // ring tiles of this CTA
  const bool do_block = split == S - 1;
  const int NT = nt + (do_block ? 1 : 0);           // tile 0 is the block's own when do_block
  int slot_b = a.req_slot ? a.req_slot[b] : b;
  if (slot_b < 0 || slot_b >= a.ring_batch) {
    // reads then fall outside the ring and come back as zeros (TMA bounds check)
    if (threadIdx.x == 0 && split == 0) report_status(a.status, DFLASH_ERR_ARG);
    slot_b = a.ring_batch;
  }
  const int row_base = (slot_b * a.n_kv + g) * a.window;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kSt; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], 1 + 4);   // K read by the score MMA, V by the 4 transpose warps
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_empty[i], n_live);
      mbar_init(&p_full[i], n_live);
      mbar_init(&vt_full[i], 4);
      mbar_init(&pv_done[i], 1);
    }
    mbar_init(&pro_bar, 1);
    mbar_init(&o_bar, 1);
    abort_sh = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_sh, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_sh;

  auto ring_index = [&](int t) { return t - (do_block ? 1 : 0); };
  auto is_block = [&](int t) { return do_block && t == 0; };
  // keys of tile t that exist (the rest are masked)
  auto tile_keys = [&](int t) {
    if (is_block(t)) return a.gamma;
    const int slot0 = (t0 + ring_index(t)) * kKeysT;
    return n_valid - slot0 < kKeysT ? n_valid - slot0 : kKeysT;
  };

  if (warp == 0) {
    // -------------------------------------------------------------- producer
    if (lane == 0 && nt > 0) {
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      const uint64_t pol = policy_evict_first();
      int issued = 0;
      for (int i = 0; i < nt; ++i) {
        const int s = i % kSt;
        const uint32_t ph = (uint32_t)(i / kSt) & 1u;
        if (!mbar_wait_bounded(&empty_bar[s], ph ^ 1u, &abort_sh, a.status)) break;
        uint8_t* ks = smem + Lay::oStage + s * 2 * Lay::kKV;
        uint8_t* vs = ks + Lay::kKV;
        mbar_arrive_expect_tx(&full_bar[s], 2 * Lay::kKV);
        const int row = row_base + (t0 + i) * kKeysT;
#pragma unroll
        for (int h = 0; h < Lay::kHalves; ++h) {
          tma_load_2d(ks + h * (kKeysT * 128), &tmK, &full_bar[s], h * 64, row, pol);
          tma_load_2d(vs + h * (kKeysT * 128), &tmV, &full_bar[s], h * 64, row, pol);
        }
        issued = i + 1;
      }
      if (abort_sh) {
        int dummy = 0;
        for (int i = (issued > kSt ? issued - kSt : 0); i < issued; ++i)
          (void)mbar_wait_bounded(&full_bar[i % kSt], (uint32_t)(i / kSt) & 1u, &dummy, nullptr,
                                  100000000ull);
      }
    }
  } else if (warp == 1) {
    // -------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc_s = idesc_f32acc(128, kKeysT, true);   // bf16 Q parts and K
      const uint32_t idesc_o = idesc_f32acc(128, HD, true);       // bf16 P and V
      const uint32_t qh = smem_u32(smem + Lay::oQh), ql = smem_u32(smem + Lay::oQl);
      const uint32_t t_o = tmem + 128;
      auto issue_pv = [&](int u) -> bool {
        const int pb = u & 1;
        const uint32_t ph = (uint32_t)(u >> 1) & 1u;
        if (!mbar_wait_bounded(&p_full[pb], ph, &abort_sh, a.status)) return false;
        if (!mbar_wait_bounded(&vt_full[pb], ph, &abort_sh, a.status)) return false;
        tc_fence_after();
        const uint32_t pa = smem_u32(smem + Lay::oP + pb * Lay::kP);
        const uint32_t vb = smem_u32(smem + Lay::oVt + pb * Lay::kVt);
#pragma unroll
        for (int k = 0; k < kKeysT / 16; ++k)
          tc_mma_f16(t_o, smem_desc_sw128(pa + k * 32), smem_desc_sw128(vb + k * 32), idesc_o,
                     (u | k) ? 1u : 0u);
        tc_commit(&pv_done[pb]);
        return true;
      };
      bool ok = mbar_wait_bounded(&pro_bar, 0, &abort_sh, a.status);
      for (int t = 0; ok && t < NT; ++t) {
        const int sb = t & 1;
        if (t >= 2 && !mbar_wait_bounded(&s_empty[sb], (uint32_t)((t - 2) >> 1) & 1u, &abort_sh, a.status))
          break;
        uint32_t kaddr;
        int stage = -1;
        if (is_block(t)) {
          kaddr = smem_u32(smem + Lay::oKblk);
        } else {
          const int i = ring_index(t);
          stage = i % kSt;
          if (!mbar_wait_bounded(&full_bar[stage], (uint32_t)(i / kSt) & 1u, &abort_sh, a.status)) break;
          kaddr = smem_u32(smem + Lay::oStage + stage * 2 * Lay::kKV);
        }
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(sb * kKeysT);
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint32_t off = (uint32_t)((kk >> 2) * (128 * 128) + (kk & 3) * 32);
          const uint32_t koff = (uint32_t)((kk >> 2) * (kKeysT * 128) + (kk & 3) * 32);
          const uint64_t bd = smem_desc_sw128(kaddr + koff);
          tc_mma_f16(d, smem_desc_sw128(qh + off), bd, idesc_s, kk ? 1u : 0u);
          tc_mma_f16(d, smem_desc_sw128(ql + off), bd, idesc_s, 1u);
        }
        tc_commit(&s_full[sb]);
        if (stage >= 0) tc_commit(&empty_bar[stage]);
        if (t >= 1 && !issue_pv(t - 1)) break;
      }
      if (!abort_sh && NT > 0) (void)issue_pv(NT - 1);
      tc_commit(&o_bar);  // all MMAs issued by this thread, also on abort
    }
  }
  __syncwarp();  // lanes 1-31 of warps 0 and 1 wait here instead of spinning

  if (warp >= 2) {
    // -------------------------------------------------------------- prologue
    // warps 2-9: Q value / remainder, the block's keys and (transposed) values
    const int tid = threadIdx.x - 64;  // 0..255
    const size_t qrow0 = (size_t)b * a.gamma;
    // Q rows ri = hh * gamma + i <- qkv row b*gamma + i, columns of head g*group + hh
    for (int idx = tid; idx < 128 * (HD / 8); idx += 256) {
      const int ri = idx / (HD / 8), ch = idx % (HD / 8);
      uint4 hi = make_uint4(0, 0, 0, 0), lo = make_uint4(0, 0, 0, 0);
      if (ri < rows) {
        const int hh = ri / a.gamma, i = ri % a.gamma;
        const uint4 u = *reinterpret_cast<const uint4*>(a.qkv + (qrow0 + i) * a.ld_qkv +
                                                        (size_t)(g * group + hh) * HD + ch * 8);
        const __half* hv = reinterpret_cast<const __half*>(&u);
        uint32_t* ph = reinterpret_cast<uint32_t*>(&hi);
        uint32_t* pl = reinterpret_cast<uint32_t*>(&lo);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float x0 = __half2float(hv[2 * k]), x1 = __half2float(hv[2 * k + 1]);
          const __nv_bfloat162 h2 = __floats2bfloat162_rn(x0, x1);
          ph[k] = *reinterpret_cast<const uint32_t*>(&h2);
          pl[k] = pack_bf16(x0 - __low2float(h2), x1 - __high2float(h2));
        }
      }
      const int col = ch * 8;
      const uint32_t off = (col >> 6) * (128 * 128) + swz(ri, col & 63);
      *reinterpret_cast<uint4*>(smem + Lay::oQh + off) = hi;
      *reinterpret_cast<uint4*>(smem + Lay::oQl + off) = lo;
    }
    if (do_block) {
      const size_t kcol = (size_t)a.n_q * HD + (size_t)g * HD;
      const size_t vcol = (size_t)(a.n_q + a.n_kv) * HD + (size_t)g * HD;
      // block keys [64][HD], rounded to bf16 (keys past gamma zero)
      for (int idx = tid; idx < kKeysT * (HD / 8); idx += 256) {
        const int r = idx / (HD / 8), ch = idx % (HD / 8);
        uint4 kv = make_uint4(0, 0, 0, 0);
        if (r < a.gamma) {
          const uint4 u = *reinterpret_cast<const uint4*>(a.qkv + (qrow0 + r) * a.ld_qkv + kcol + ch * 8);
          const __half* hv = reinterpret_cast<const __half*>(&u);
          uint32_t* pk = reinterpret_cast<uint32_t*>(&kv);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            pk[k] = pack_bf16(__half2float(hv[2 * k]), __half2float(hv[2 * k + 1]));
        }
        const int col = ch * 8;
        *reinterpret_cast<uint4*>(smem + Lay::oKblk + (col >> 6) * (kKeysT * 128) + swz(r, col & 63)) = kv;
      }
      // block values, transposed: Vt[d][key] for 8 keys per item
      for (int idx = tid; idx < HD * (kKeysT / 8); idx += 256) {
        const int dd = idx / (kKeysT / 8), j = idx % (kKeysT / 8);
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int k0 = 8 * j + 2 * k, k1 = k0 + 1;
          const float v0 = k0 < a.gamma ? __half2float(a.qkv[(qrow0 + k0) * a.ld_qkv + vcol + dd]) : 0.0f;
          const float v1 = k1 < a.gamma ? __half2float(a.qkv[(qrow0 + k1) * a.ld_qkv + vcol + dd]) : 0.0f;
          w[k] = pack_bf16(v0, v1);
        }
        *reinterpret_cast<uint4*>(smem + Lay::oVt + dd * 128 + ((j ^ (dd & 7)) << 4)) =
            make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
    fence_proxy_async_smem();
    named_sync(1, 256);
    if (tid == 0) mbar_arrive(&pro_bar);
  }

  float m_run = -INFINITY, l_run = 0.0f;
  const int q = warp & 3;                 // TMEM lane quarter
  const int r = 32 * q + lane;            // softmax row
  if (warp >= 2 && warp < 6 && q < n_live) {
    // ------------------------------------------------------------- softmax
    // (P rows of the idle warps are never written: they only reach O rows
    // that are never read)
    const bool row_ok = r < rows;
    const uint32_t t_row = tmem + ((uint32_t)(32 * q) << 16);
    for (int t = 0; t < NT; ++t) {
      const int sb = t & 1;
      if (!warp_wait(&s_full[sb], (uint32_t)(t >> 1) & 1u, &abort_sh, a.status)) break;
      tc_fence_after();
      float s[kKeysT];
      {
        uint32_t raw[kKeysT / 16][16];
#pragma unroll
        for (int c = 0; c < kKeysT / 16; ++c) tmem_ld_x16(t_row + (uint32_t)(sb * kKeysT + c * 16), raw[c]);
        tc_wait_ld();  // one round trip for the whole row
#pragma unroll
        for (int c = 0; c < kKeysT / 16; ++c)
#pragma unroll
          for (int j = 0; j < 16; ++j) s[c * 16 + j] = __uint_as_float(raw[c][j]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_empty[sb]);
      const int nk = tile_keys(t);
      float mt = -INFINITY;
#pragma unroll
      for (int c = 0; c < kKeysT; ++c) {
        s[c] = (row_ok && c < nk) ? s[c] * a.scale_log2 : -INFINITY;
        mt = fmaxf(mt, s[c]);
      }
      const bool resc = mt > m_run + kRescale;  // also true when m_run is -inf and mt finite
      const float corr = resc ? exp2f(m_run - mt) : 1.0f;  // 0 when m_run is -inf
      if (__any_sync(0xffffffffu, resc) && t >= 1) {
        // O holds tiles < t: wait until P_{t-1} V_{t-1} is done, then rescale this warp's rows
        if (!warp_wait(&pv_done[(t - 1) & 1], (uint32_t)((t - 1) >> 1) & 1u, &abort_sh, a.status))
          break;
        tc_fence_after();
#pragma unroll
        for (int c0 = 0; c0 < HD / 16; c0 += 4) {
          uint32_t raw[4][16];
#pragma unroll
          for (int c = 0; c < 4; ++c) tmem_ld_x16(t_row + 128 + (c0 + c) * 16, raw[c]);
          tc_wait_ld();
#pragma unroll
          for (int c = 0; c < 4; ++c) {
#pragma unroll
            for (int j = 0; j < 16; ++j) raw[c][j] = __float_as_uint(__uint_as_float(raw[c][j]) * corr);
            tmem_st_x16(t_row + 128 + (c0 + c) * 16, raw[c]);
          }
        }
        tc_wait_st();
      }
      if (resc) {
        l_run *= corr;
        m_run = mt;
      }
      const float base = m_run == -INFINITY ? 0.0f : m_run;
      uint32_t pw[kKeysT / 2];
      float ls = 0.0f;
#pragma unroll
      for (int c = 0; c < kKeysT / 2; ++c) {
        const float p0 = exp2f(s[2 * c] - base), p1 = exp2f(s[2 * c + 1] - base);
        const __nv_bfloat162 h2 = __floats2bfloat162_rn(p0, p1);
        ls += __low2float(h2) + __high2float(h2);  // the sum of what P V adds up
        pw[c] = *reinterpret_cast<const uint32_t*>(&h2);
      }
      l_run += ls;
      const int pb = t & 1;
      if (t >= 2 && !warp_wait(&pv_done[pb], (uint32_t)((t - 2) >> 1) & 1u, &abort_sh, a.status))
        break;
      uint8_t* prow = smem + Lay::oP + pb * Lay::kP + r * 128;
#pragma unroll
      for (int j = 0; j < 8; ++j)
        *reinterpret_cast<uint4*>(prow + ((j ^ (r & 7)) << 4)) =
            make_uint4(pw[4 * j], pw[4 * j + 1], pw[4 * j + 2], pw[4 * j + 3]);
      tc_fence_before();
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[pb]);
    }
  } else if (warp >= 6) {
    // -------------------------------------------------- V transpose (ring tiles)
    const int tt = threadIdx.x - 192;  // 0..127
    for (int t = 0; t < NT; ++t) {
      if (is_block(t)) {
        // Vt[0] was written by the prologue
        __syncwarp();
        if (lane == 0) mbar_arrive(&vt_full[0]);
        continue;
      }
      const int i = ring_index(t), stage = i % kSt, vb = t & 1;
      if (!warp_wait(&full_bar[stage], (uint32_t)(i / kSt) & 1u, &abort_sh, a.status)) break;
      if (t >= 2 && !warp_wait(&pv_done[vb], (uint32_t)((t - 2) >> 1) & 1u, &abort_sh, a.status))
        break;
      const int nk = tile_keys(t);
      const uint8_t* vs = smem + Lay::oStage + stage * 2 * Lay::kKV + Lay::kKV;
      uint8_t* vt = smem + Lay::oVt + vb * Lay::kVt;
      for (int idx = tt; idx < HD * (kKeysT / 8); idx += 128) {
        const int dd = idx % HD, j = idx / HD;  // consecutive threads: consecutive dims
        const int hsel = dd >> 6, dc = dd & 63;
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int k0 = 8 * j + 2 * k;
          const uint16_t e0 = k0 < nk ? *reinterpret_cast<const uint16_t*>(vs + hsel * (kKeysT * 128) + swz(k0, dc)) : 0;
          const uint16_t e1 = k0 + 1 < nk ? *reinterpret_cast<const uint16_t*>(vs + hsel * (kKeysT * 128) + swz(k0 + 1, dc)) : 0;
          w[k] = (uint32_t)e0 | ((uint32_t)e1 << 16);
        }
        *reinterpret_cast<uint4*>(vt + dd * 128 + ((j ^ (dd & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&vt_full[vb]);
        mbar_arrive(&empty_bar[stage]);
      }
    }
  }

  // ------------------------------------------------------------- results
  // all MMAs complete (or the CTA gave up): O is final in TMEM
  (void)mbar_wait_bounded(&o_bar, 0, &abort_sh, a.status);  // a timeout sets abort_sh
  tc_fence_after();
  __syncthreads();
  const bool have_o = abort_sh == 0 && NT > 0;          // CTA-uniform
  float* part_s = reinterpret_cast<float*>(smem);      // [rows][HD] partial O (stage data is dead)
  float* ml_s = part_s + 96 * HD;                      // [rows][2] max (log2) and sum
  float* w_s = ml_s + 96 * 2;                          // [rows of this CTA][16] merge weights
  if (warp >= 2 && warp < 6) {
    // tcgen05.ld is warp-collective: every lane loads, the rows that exist store
    const uint32_t t_row = tmem + ((uint32_t)(32 * q) << 16);
    const bool mine = r < rows;
    const int hh = mine ? r / a.gamma : 0, i = mine ? r % a.gamma : 0;
    const size_t off = (size_t)(b * a.gamma + i) * a.ld_out + (size_t)(g * group + hh) * HD;
    const float inv = l_run > 0.0f ? 1.0f / l_run : 0.0f;
#pragma unroll
    for (int c = 0; c < HD / 16; ++c) {
      uint32_t raw[16];
      if (have_o) {
        tmem_ld_x16(t_row + 128 + c * 16, raw);
        tc_wait_ld();
      } else {
#pragma unroll
        for (int j2 = 0; j2 < 16; ++j2) raw[j2] = 0u;
      }
      if (!mine) continue;
      if (S == 1) {
        uint32_t hv[8];
#pragma unroll
        for (int j2 = 0; j2 < 8; ++j2) {
          const __half2 h2 = __floats2half2_rn(__uint_as_float(raw[2 * j2]) * inv,
                                               __uint_as_float(raw[2 * j2 + 1]) * inv);
          hv[j2] = *reinterpret_cast<const uint32_t*>(&h2);
        }
        *reinterpret_cast<uint4*>(a.out + off + c * 16) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
        *reinterpret_cast<uint4*>(a.out + off + c * 16 + 8) = make_uint4(hv[4], hv[5], hv[6], hv[7]);
      } else {
#pragma unroll
        for (int j2 = 0; j2 < 16; ++j2) part_s[r * HD + c * 16 + j2] = __uint_as_float(raw[j2]);
      }
    }
    if (S > 1 && mine) {
      ml_s[r * 2] = have_o ? m_run : -INFINITY;   // a CTA that gave up contributes nothing
      ml_s[r * 2 + 1] = have_o ? l_run : 0.0f;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
  if (S == 1) return;

  // --------------------------------------------- merge across the cluster
  cg::cluster_group cluster = cg::this_cluster();
  cluster.sync();
  const int rank = (int)cluster.block_rank();
  const int my_rows = (rows - rank + S - 1) / S;          // rows rank, rank + S, ...
  if ((int)threadIdx.x < my_rows) {
    const int ri = rank + (int)threadIdx.x * S;
    float mv[16], lv[16];
#pragma unroll
    for (int s2 = 0; s2 < 16; ++s2) {
      if (s2 < S) {
        const float* ml = cluster.map_shared_rank(ml_s, s2);
        mv[s2] = ml[ri * 2];
        lv[s2] = ml[ri * 2 + 1];
      }
    }
    float M = -INFINITY;
#pragma unroll
    for (int s2 = 0; s2 < 16; ++s2)
      if (s2 < S) M = fmaxf(M, mv[s2]);
    float den = 0.0f;
#pragma unroll
    for (int s2 = 0; s2 < 16; ++s2) {
      if (s2 < S) {
        mv[s2] = mv[s2] == -INFINITY ? 0.0f : exp2f(mv[s2] - M);
        den += mv[s2] * lv[s2];
      }
    }
    const float inv = den > 0.0f ? 1.0f / den : 0.0f;
#pragma unroll
    for (int s2 = 0; s2 < 16; ++s2)
      if (s2 < S) w_s[threadIdx.x * 16 + s2] = mv[s2] * inv;
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < my_rows * (HD / 2); idx += blockDim.x) {
    const int k = idx / (HD / 2), d = (idx % (HD / 2)) * 2;
    const int ri = rank + k * S;
    float2 pv[16];
#pragma unroll
    for (int s2 = 0; s2 < 16; ++s2)
      if (s2 < S) pv[s2] = *reinterpret_cast<const float2*>(cluster.map_shared_rank(part_s, s2) + ri * HD + d);
    float o0 = 0.0f, o1 = 0.0f;
#pragma unroll
    for (int s2 = 0; s2 < 16; ++s2) {
      if (s2 < S) {
        o0 += w_s[k * 16 + s2] * pv[s2].x;
        o1 += w_s[k * 16 + s2] * pv[s2].y;
      }
    }
    const int hh = ri / a.gamma, i = ri % a.gamma;
    *reinterpret_cast<__half2*>(a.out + (size_t)(b * a.gamma + i) * a.ld_out + (size_t)(g * group + hh) * HD + d) =
        __floats2half2_rn(o0, o1);
  }
  // no CTA may leave while another still reads its shared memory
  cluster.sync();
}

template <int HD>
int launch_tc(const CUtensorMap& tk, const CUtensorMap& tv, const AttnArgs& a, int B, cudaStream_t s) {
  constexpr size_t smem = 1024 + (size_t)TcLayout<HD>::kBytes;
  static_assert(96 * (HD + 2 + 16) * 4 <= TcLayout<HD>::oP, "merge state must fit the dead stage data");
  auto kern = attn_tc_kernel<HD>;
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return DFLASH_ERR_LAUNCH;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
      return DFLASH_ERR_LAUNCH;
    attr = true;
  }
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

int launch_attention_tc(const void* ring_k_layer, const void* ring_v_layer, const AttnArgs& a, int B,
                        cudaStream_t s) {
  if (a.n_q / a.n_kv * a.gamma > 96) return DFLASH_ERR_UNSUPPORTED;
  CUtensorMap tk, tv;
  const uint64_t rows = (uint64_t)a.ring_batch * a.n_kv * a.window;
  int rc = encode_2d(&tk, ring_k_layer, OPND_BF16, (uint64_t)a.hd, rows, 64, kKeysT);
  if (rc) return rc;
  rc = encode_2d(&tv, ring_v_layer, OPND_BF16, (uint64_t)a.hd, rows, 64, kKeysT);
  if (rc) return rc;
  if (a.hd == 128) return launch_tc<128>(tk, tv, a, B, s);
  return launch_tc<64>(tk, tv, a, B, s);
}

}  // namespace dfl
