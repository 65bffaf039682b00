// Block attention of the drafter on the 5th-generation tensor cores ("DFlash
// vs DFlash 2" blog, section "Conditioning on the target model": the gamma
// block queries of each head attend over [context window ; whole block],
// non-causally inside the block; model card "Beam-1.0-501B-A23B-DFlash2",
// section "Model": 4,096-token sliding window, 40 query / 8 KV heads), for
// head dims 64 and 128 and at most 128 query rows per KV head (query heads of
// the group x gamma).
//
// One CTA serves one (request, KV head, key split); the splits of a head form
// a thread-block cluster and merge their partial softmax states through
// distributed shared memory in split order.  Inside a CTA the query rows are
// the 128 rows of every MMA (zero-padded), so one K/V byte read from HBM
// serves every query head of the group:
//   warp 0       TMA producer: 64-key K/V tiles of the ring, 5 stages
//   warp 1       tensor-memory allocation; lane 0 issues the MMAs
//                  S_i = Q K_i^T     (fp16, A = Q and B = K_i in shared memory)
//                  O  += P_i V_i     (bf16 for ring tiles, fp16 for the block's
//                                     own keys; A = P_i in tensor memory, B =
//                                     V_i read MN-major from the TMA tile)
//                S_{i+2} is issued before P_i V_i, so the softmax of a tile
//                finds its scores ready and overlaps the MMAs of its
//                neighbours (S triple-, P double-buffered)
//   warps 2-3    widen each ring K tile from bf16 to fp16 in place (exact in
//                fp16's range), zero the rows of keys past the visible window
//   warps 4-7    softmax, one query row per thread (warp 4 + q owns tensor-
//                memory lanes 32q..32q+31): scale, mask, running max, P = 2^(s -
//                m) into tensor memory, running sum.  O lives in tensor memory
//                and is rescaled only when a row's maximum grows by more than
//                2^8 (P <= 256 meanwhile), which happens a few times per row.
//                A warp whose lanes hold only padding rows just keeps the
//                barriers' phases.
// Before the loop warps 2-7 load Q (and the block's own K/V) with
// asynchronous copies.  All waits are bounded (mbar_wait_bounded); a CTA that
// gives up still meets its cluster barriers and frees its tensor memory.
// Each CTA takes all 512 tensor-memory columns and at least 128 KiB of shared
// memory, so no other CTA holding tensor memory shares its SM.
#include <cooperative_groups.h>

#include "attention.h"
#include "attention_util.cuh"
#include "common.cuh"
#include "gemm.h"

namespace dfl {
namespace {

namespace cg = cooperative_groups;
using namespace attn;

constexpr int kKT = 64;             // keys per ring tile
constexpr int kST = 5;              // ring stages
constexpr int kMT = 128;            // MMA rows: query rows, zero-padded
constexpr int kBT = 16;             // the block's own keys (gamma <= 16), zero-padded
constexpr float kHeadroom = 8.0f;   // log2 growth of a row maximum before O is rescaled
constexpr int kThreads = 256;
constexpr int kLoaders = 192;       // warps 2-7 load Q and the block K/V

#ifndef DFLASH_ATTN_MAX_CLUSTER
#define DFLASH_ATTN_MAX_CLUSTER 8
#endif

template <int HD>
struct Tc {
  static constexpr int kTile = kKT * HD * 2;            // K or V of one ring tile
  static constexpr int kStage = 2 * kTile;
  static constexpr int kQ = kMT * HD * 2;
  static constexpr int kBlk = kBT * HD * 2;
  // at least 128 KiB, so that no other CTA with tensor memory shares the SM
  // (a CTA waiting in tcgen05.alloc beside one that waits for it would hang)
  static constexpr size_t kSmemUsed = 1024 + (size_t)kST * kStage + kQ + 2 * kBlk;
  static constexpr size_t kSmem = kSmemUsed < 128 * 1024 ? 128 * 1024 : kSmemUsed;
  static constexpr uint32_t kColO = 0;                  // O: HD columns
  static constexpr uint32_t kColS = HD;                 // S: three buffers of kKT columns
  static constexpr uint32_t kColP = HD + 3 * kKT;       // P: two buffers of kKT / 2 columns
  static constexpr uint32_t kCols = 512;
  static_assert(kColP + kKT <= kCols, "tensor memory columns");
  static_assert(kMT * HD * 4 + kMT * 2 * 4 + kMT * 16 * 4 <= kST * kStage,
                "merge partials must fit the stage buffers");
};

// Matrix descriptor of an MN-major operand stored as TMA writes it with the
// 128-byte swizzle: rows along K of 128 bytes (64 elements along M/N), 8-row
// atoms 1024 bytes apart, further blocks of 64 elements along M/N `mn_block`
// bytes apart.
__device__ __forceinline__ uint64_t smem_desc_sw128_mn(uint32_t smem_addr, uint32_t mn_block) {
  uint64_t d = 0;
  d |= (uint64_t)((smem_addr & 0x3FFFFu) >> 4);          // start address
  d |= (uint64_t)((mn_block >> 4) & 0x3FFFu) << 16;      // leading byte offset: next 64 along M/N
  d |= (uint64_t)(1024 >> 4) << 32;                      // stride byte offset: next 8 rows along K
  d |= (uint64_t)1 << 46;                                // descriptor version (sm_100 family)
  d |= (uint64_t)2 << 61;                                // 128-byte swizzle
  return d;
}

// Completions of an mbarrier used by every other tile: tile t's is number
// t / 2 (by every third tile: t / 3).
__device__ __forceinline__ uint32_t par2(int t) { return (uint32_t)(t >> 1) & 1u; }
__device__ __forceinline__ uint32_t par3(int t) { return (uint32_t)(t / 3) & 1u; }

template <int HD>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                   const AttnArgs a) {
  using Sh = Tc<HD>;
  pdl_enter();
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[kST], kready_bar[kST], empty_bar[kST];
  __shared__ __align__(8) uint64_t sfull_bar[3], sfree_bar[3], pfull_bar[2], pvdone_bar[2];
  __shared__ __align__(8) uint64_t q_bar, fin_bar;
  __shared__ uint32_t tmem_sh;
  __shared__ int abort_sh;

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* q_s = smem + kST * Sh::kStage;       // fp16 Q [128][HD], K-major halves [128][64]
  uint8_t* bk_s = q_s + Sh::kQ;                 // block K fp16 [16][HD], same layout
  uint8_t* bv_s = bk_s + Sh::kBlk;              // block V fp16 [16][HD]: MN-major for P.V
  float* part_s = reinterpret_cast<float*>(smem);   // after the loop: [128][HD] partial O
  float* ml_s = part_s + kMT * HD;                  // [128][2] (max (log2), sum)
  float* w_s = ml_s + kMT * 2;                      // [rows of this CTA][16] merge weights

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int S = gridDim.x;
  const int group = a.n_q / a.n_kv;
  const int rows = group * a.gamma;
  const long long L = a.ctx_len[b];
  const int n_valid = (int)(L < (long long)a.window ? (L < 0 ? 0 : L) : a.window);
  const int tiles = (n_valid + kKT - 1) / kKT;
  const int t0 = (int)((long long)split * tiles / S), t1 = (int)((long long)(split + 1) * tiles / S);
  const int nt = t1 - t0;
  const bool do_block = split == S - 1;
  const int nb = do_block ? 1 : 0;              // tile 0 is the block's own keys on the last split
  const int T = nb + nt;
  int slot_b = a.req_slot ? a.req_slot[b] : b;
  if (slot_b < 0 || slot_b >= a.ring_batch) {
    // reads then fall outside the ring and come back as zeros (TMA bounds check)
    if (threadIdx.x == 0 && split == 0) report_status(a.status, DFLASH_ERR_ARG);
    slot_b = a.ring_batch;
  }
  const int row_base = (slot_b * a.n_kv + g) * a.window;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kST; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&kready_bar[s], 2);
      mbar_init(&empty_bar[s], 1);
    }
    for (int i = 0; i < 3; ++i) {
      mbar_init(&sfull_bar[i], 1);
      mbar_init(&sfree_bar[i], 4);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&pfull_bar[i], 4);
      mbar_init(&pvdone_bar[i], 1);
    }
    mbar_init(&q_bar, 1);
    mbar_init(&fin_bar, 1);
    abort_sh = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_sh, Sh::kCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_sh;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && nt > 0) {
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      const uint64_t pol = policy_evict_first();
      int issued = 0;
      for (int j = 0; j < nt; ++j) {
        const int s = j % kST;
        if (!mbar_wait_bounded(&empty_bar[s], ((uint32_t)(j / kST) & 1u) ^ 1u, &abort_sh, a.status)) break;
        uint8_t* ks = smem + s * Sh::kStage;
        mbar_arrive_expect_tx(&full_bar[s], Sh::kStage);
        const int row = row_base + (t0 + j) * kKT;
#pragma unroll
        for (int h = 0; h < HD / 64; ++h) {
          tma_load_2d(ks + h * (kKT * 128), &tmK, &full_bar[s], h * 64, row, pol);
          tma_load_2d(ks + Sh::kTile + h * (kKT * 128), &tmV, &full_bar[s], h * 64, row, pol);
        }
        issued = j + 1;
      }
      if (abort_sh) {
        // a wait gave up: let the copies in flight land before the CTA leaves
        int dummy = 0;
        for (int j = (issued > kST ? issued - kST : 0); j < issued; ++j)
          (void)mbar_wait_bounded(&full_bar[j % kST], (uint32_t)(j / kST) & 1u, &dummy, nullptr, 100000000ull);
      }
    }
  } else if (warp == 1) {
    // --------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t id_qk_ring = idesc_f32acc(kMT, kKT, false);
      const uint32_t id_qk_blk = idesc_f32acc(kMT, kBT, false);
      const uint32_t id_pv_ring = idesc_f32acc(kMT, HD, true) | (1u << 16);   // B (V) MN-major
      const uint32_t id_pv_blk = idesc_f32acc(kMT, HD, false) | (1u << 16);
      const uint32_t q_addr = smem_u32(q_s);
      bool ok = mbar_wait_bounded(&q_bar, 0, &abort_sh, a.status);
      auto issue_qk = [&](int i) -> bool {
        const int bf = i % 3;
        if (i >= 3 && !mbar_wait_bounded(&sfree_bar[bf], par3(i - 3), &abort_sh, a.status)) return false;
        const bool blk = i < nb;
        uint32_t k_addr, k_half;
        if (blk) {
          k_addr = smem_u32(bk_s);
          k_half = kBT * 128;
        } else {
          const int j = i - nb, s = j % kST;
          if (!mbar_wait_bounded(&kready_bar[s], (uint32_t)(j / kST) & 1u, &abort_sh, a.status)) return false;
          k_addr = smem_u32(smem + s * Sh::kStage);
          k_half = kKT * 128;
        }
        tc_fence_after();
        const uint32_t d = tmem + Sh::kColS + (uint32_t)(bf * kKT);
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint32_t off = (uint32_t)(kk & 3) * 32;  // 16 dims of the 64-dim half
          tc_mma_f16(d, smem_desc_sw128(q_addr + (kk >> 2) * (kMT * 128) + off),
                     smem_desc_sw128(k_addr + (kk >> 2) * k_half + off), blk ? id_qk_blk : id_qk_ring,
                     kk > 0 ? 1u : 0u);
        }
        tc_commit(&sfull_bar[bf]);
        return true;
      };
      auto issue_pv = [&](int i) -> bool {
        const int bf = i & 1;
        if (!mbar_wait_bounded(&pfull_bar[bf], par2(i), &abort_sh, a.status)) return false;
        tc_fence_after();
        const bool blk = i < nb;
        const int nk = blk ? kBT : kKT;
        uint32_t v_addr, v_half;
        if (blk) {
          v_addr = smem_u32(bv_s);
          v_half = kBT * 128;
        } else {
          const int s = (i - nb) % kST;
          v_addr = smem_u32(smem + s * Sh::kStage + Sh::kTile);
          v_half = kKT * 128;
        }
        const uint32_t p = tmem + Sh::kColP + (uint32_t)(bf * (kKT / 2));
        for (int kk = 0; kk < nk / 16; ++kk)
          tc_mma_f16_ta(tmem + Sh::kColO, p + kk * 8, smem_desc_sw128_mn(v_addr + kk * 2048, v_half),
                        blk ? id_pv_blk : id_pv_ring, (i > 0 || kk > 0) ? 1u : 0u);
        tc_commit(&pvdone_bar[bf]);
        if (!blk) tc_commit(&empty_bar[(i - nb) % kST]);
        return true;
      };
      // scores two tiles ahead of P . V: the softmax of a tile never waits
      // for its scores behind the previous tile's P . V
      if (ok && T > 0) ok = issue_qk(0);
      if (ok && T > 1) ok = issue_qk(1);
      for (int i = 0; ok && i < T; ++i) {
        if (i + 2 < T && !issue_qk(i + 2)) break;
        if (!issue_pv(i)) break;
      }
      tc_commit(&fin_bar);  // every MMA this thread issued
    }
  } else {
    // Q (rows past `rows` zero) and, on the last split, the block's own K and
    // V (keys past gamma zero), by warps 2-7 with asynchronous copies
    const int lt = threadIdx.x - 64;
    for (int idx = lt; idx < kMT * (HD / 8); idx += kLoaders) {
      const int ri = idx / (HD / 8), ch = idx % (HD / 8);
      const bool ok = ri < rows;
      const int hh = ok ? ri / a.gamma : 0, i = ok ? ri % a.gamma : 0;
      const size_t src = (size_t)(b * a.gamma + i) * a.ld_qkv + (size_t)(g * group + hh) * HD + ch * 8;
      const int col = ch * 8;
      cp_async16(q_s + (col >> 6) * (kMT * 128) + swz(ri, col & 63), a.qkv + src, ok);
    }
    if (do_block) {
      const size_t kcol = (size_t)a.n_q * HD + (size_t)g * HD;
      const size_t vcol = (size_t)(a.n_q + a.n_kv) * HD + (size_t)g * HD;
      for (int idx = lt; idx < kBT * (HD / 8); idx += kLoaders) {
        const int r = idx / (HD / 8), ch = idx % (HD / 8);
        const bool ok = r < a.gamma;
        const __half* row = a.qkv + (size_t)(b * a.gamma + (ok ? r : 0)) * a.ld_qkv;
        const int col = ch * 8;
        const uint32_t off = (col >> 6) * (kBT * 128) + swz(r, col & 63);
        cp_async16(bk_s + off, row + kcol + ch * 8, ok);
        cp_async16(bv_s + off, row + vcol + ch * 8, ok);
      }
    }
    cp_async_wait_all();
    fence_proxy_async_smem();  // read next by the tensor cores (async proxy)
    named_sync(1, kLoaders);
    if (lt == 0) mbar_arrive(&q_bar);

    if (warp < 4) {
      // --------------------------------------------------------- converters
      const int ct = threadIdx.x - 64;  // 0..63
      for (int j = 0; j < nt; ++j) {
        const int s = j % kST;
        if (!warp_wait(&full_bar[s], (uint32_t)(j / kST) & 1u, &abort_sh, a.status)) break;
        uint8_t* ks = smem + s * Sh::kStage;
        uint4* k4 = reinterpret_cast<uint4*>(ks);
#pragma unroll 4
        for (int idx = ct; idx < Sh::kTile / 16; idx += 64) {
          uint4 u = k4[idx];
          u.x = bf16x2_to_f16x2(u.x);
          u.y = bf16x2_to_f16x2(u.y);
          u.z = bf16x2_to_f16x2(u.z);
          u.w = bf16x2_to_f16x2(u.w);
          k4[idx] = u;
        }
        // keys past the visible window: K and V rows zeroed (whatever those
        // ring slots hold cannot turn 0 * V into NaN)
        const int valid = n_valid - (t0 + j) * kKT;
        if (valid < kKT) {
          for (int idx = ct; idx < (kKT - valid) * (HD / 8) * 2; idx += 64) {
            const int half_rows = (kKT - valid) * 8;  // 16-byte pieces per half of K or V
            const int kv = idx / (half_rows * (HD / 64)), rem = idx % (half_rows * (HD / 64));
            const int h = rem / half_rows, r = valid + (rem % half_rows) / 8, c = rem % 8;
            reinterpret_cast<uint4*>(ks + kv * Sh::kTile + h * (kKT * 128) + r * 128)[c] =
                make_uint4(0u, 0u, 0u, 0u);
          }
        }
        fence_proxy_async_smem();  // generic writes, read next by the tensor cores
        __syncwarp();
        if (lane == 0) mbar_arrive(&kready_bar[s]);
      }
    } else {
      // ----------------------------------------------------------- softmax
      const int q = warp & 3;
      const int row = q * 32 + lane;
      const uint32_t lane_off = (uint32_t)(q * 32) << 16;
      float m_ref = -INFINITY, l_sum = 0.0f;
      bool ok = true;
      const bool live = q * 32 < rows;  // some of this warp's lanes are query rows
      for (int i = 0; i < T && ok; ++i) {
        const int bf = i & 1;
        const bool blk = i < nb;
        const int valid = blk ? a.gamma : n_valid - (t0 + i - nb) * kKT;  // visible keys of the tile
        const int sb = i % 3;  // S buffer
        if (!warp_wait(&sfull_bar[sb], par3(i), &abort_sh, a.status)) {
          ok = false;
          break;
        }
        if (!live) {
          // only padding rows in this warp's lanes: keep the barriers'
          // phases.  Its arrival for tile i must not count toward tile
          // i - 2's phase of the same P barrier (scores run two tiles ahead
          // of P . V): wait, like the live warps, for that tile's P . V.
          if (i >= 2 && !warp_wait(&pvdone_bar[bf], par2(i - 2), &abort_sh, a.status)) {
            ok = false;
            break;
          }
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&sfree_bar[sb]);
            mbar_arrive(&pfull_bar[bf]);
          }
          continue;
        }
        tc_fence_after();
        float sv[kKT];
        {
          uint32_t r0[16], r1[16], r2[16], r3[16];
          const uint32_t sa = tmem + lane_off + Sh::kColS + (uint32_t)(sb * kKT);
          tmem_ld_x16(sa, r0);
          if (!blk) {
            tmem_ld_x16(sa + 16, r1);
            tmem_ld_x16(sa + 32, r2);
            tmem_ld_x16(sa + 48, r3);
          }
          tc_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            sv[e] = __uint_as_float(r0[e]);
            sv[16 + e] = blk ? -INFINITY : __uint_as_float(r1[e]);
            sv[32 + e] = blk ? -INFINITY : __uint_as_float(r2[e]);
            sv[48 + e] = blk ? -INFINITY : __uint_as_float(r3[e]);
          }
        }
        // S buffer read: the MMA of tile i + 3 may overwrite it
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sfree_bar[sb]);
        if (valid < kKT) {
#pragma unroll
          for (int e = 0; e < kKT; ++e)
            if (e >= valid) sv[e] = -INFINITY;
        }
        // row maximum of the raw scores (the scale is positive), as a tree
        float mx[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          mx[k] = sv[k];
#pragma unroll
          for (int e = k + 8; e < kKT; e += 8) mx[k] = fmaxf(mx[k], sv[e]);
        }
        const float m_tile =
            fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])), fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) *
            a.scale_log2;
        const bool grow = m_tile > m_ref + kHeadroom || (m_ref == -INFINITY && m_tile > -INFINITY);
        if (__any_sync(0xffffffffu, grow)) {
          const float m_new = grow ? m_tile : m_ref;
          const float f = grow ? ex2_approx(m_ref - m_new) : 1.0f;  // 0 while nothing was seen
          if (i > 0) {
            // O holds tiles 0..i-1: wait for the last of their MMAs, rescale in place
            if (!warp_wait(&pvdone_bar[(i - 1) & 1], par2(i - 1), &abort_sh, a.status)) {
              ok = false;
              break;
            }
            tc_fence_after();
            uint32_t r[16];
#pragma unroll
            for (int c = 0; c < HD / 16; ++c) {
              const uint32_t oa = tmem + lane_off + Sh::kColO + c * 16;
              tmem_ld_x16(oa, r);
              tc_wait_ld();
#pragma unroll
              for (int e = 0; e < 16; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * f);
              tmem_st_x16(oa, r);
            }
            tc_wait_st();
          }
          l_sum *= f;
          m_ref = m_new;
        }
        // P = 2^(s * scale - m_ref), masked keys 0; partial sums as a tree
        const float nbase = m_ref == -INFINITY ? 0.0f : -m_ref;
        uint32_t pw0[16], pw1[16];  // keys 0-31 and 32-63 as 16-bit pairs
        float ls[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float p0 = ex2_approx(fmaf(sv[2 * e], a.scale_log2, nbase));
          const float p1 = ex2_approx(fmaf(sv[2 * e + 1], a.scale_log2, nbase));
          const float p2 = ex2_approx(fmaf(sv[32 + 2 * e], a.scale_log2, nbase));
          const float p3 = ex2_approx(fmaf(sv[32 + 2 * e + 1], a.scale_log2, nbase));
          ls[e & 3] += (p0 + p1) + (p2 + p3);
          pw0[e] = blk ? pack_f16(p0, p1) : pack_bf16(p0, p1);
          pw1[e] = blk ? pack_f16(p2, p3) : pack_bf16(p2, p3);
        }
        l_sum += (ls[0] + ls[1]) + (ls[2] + ls[3]);
        // P buffer `bf` was last read by the MMAs of tile i - 2
        if (i >= 2 && !warp_wait(&pvdone_bar[bf], par2(i - 2), &abort_sh, a.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t pa = tmem + lane_off + Sh::kColP + (uint32_t)(bf * (kKT / 2));
        tmem_st_x16(pa, pw0);
        tmem_st_x16(pa + 16, pw1);
        tc_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&pfull_bar[bf]);
      }
      // every MMA done (O final), then O / l out, or the unnormalised partial
      bool have = ok && T > 0 && warp_wait(&fin_bar, 0, &abort_sh, a.status);
      tc_fence_after();
      if (S == 1) {
        if (have) {
          const float inv = 1.0f / l_sum;
          const int hh = row / a.gamma, i = row % a.gamma;
          const size_t off = (size_t)(b * a.gamma + i) * a.ld_out + (size_t)(g * group + hh) * HD;
          uint32_t r[16];
#pragma unroll
          for (int c = 0; c < HD / 16; ++c) {
            tmem_ld_x16(tmem + lane_off + Sh::kColO + c * 16, r);
            tc_wait_ld();
            if (row < rows) {
#pragma unroll
              for (int e = 0; e < 16; e += 2)
                store_h2(a.out, off + c * 16 + e, __uint_as_float(r[e]) * inv, __uint_as_float(r[e + 1]) * inv);
            }
          }
        }
      } else {
        // the stage buffers are free: every tile has been consumed
        uint32_t r[16];
#pragma unroll
        for (int c = 0; c < HD / 16; ++c) {
          if (have) {
            tmem_ld_x16(tmem + lane_off + Sh::kColO + c * 16, r);
            tc_wait_ld();
          }
#pragma unroll
          for (int e = 0; e < 16; ++e) part_s[row * HD + c * 16 + e] = have ? __uint_as_float(r[e]) : 0.0f;
        }
        ml_s[row * 2 + 0] = have ? m_ref : -INFINITY;
        ml_s[row * 2 + 1] = have ? l_sum : 0.0f;
      }
    }
  }

  // tensor memory is no longer read: free it once every MMA has completed
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    int dummy = 0;
    if (lane == 0) (void)mbar_wait_bounded(&fin_bar, 0, &dummy, nullptr, 100000000ull);
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, Sh::kCols);
  }
  if (S == 1) return;

  // ------------------------------------------------ merge across the cluster
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

template <int HD>
int launch_tc_t(const CUtensorMap& tk, const CUtensorMap& tv, const AttnArgs& a, int B, cudaStream_t s) {
  auto kern = attn_tc_kernel<HD>;
  constexpr size_t smem = Tc<HD>::kSmem;
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return DFLASH_ERR_LAUNCH;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
      return DFLASH_ERR_LAUNCH;
    attr = true;
  }
  // largest power-of-two cluster the GPU can co-schedule for this kernel
  static int max_cluster = 0;
  if (max_cluster == 0) {
    max_cluster = 1;
    for (int c = DFLASH_ATTN_MAX_CLUSTER; c >= 2; c >>= 1) {
      cudaLaunchConfig_t q = {};
      q.gridDim = dim3(c, 1, 1);
      q.blockDim = dim3(kThreads);
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
  cfg.blockDim = dim3(kThreads);
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

bool attention_tc_supported(const AttnArgs& a) {
  return (a.hd == 64 || a.hd == 128) && a.n_kv > 0 && a.n_q % a.n_kv == 0 &&
         (a.n_q / a.n_kv) * a.gamma <= kMT && a.gamma >= 1 && a.gamma <= kBT;
}

int launch_attention_tc(const CUtensorMap& tk, const CUtensorMap& tv, const AttnArgs& a, int B,
                        cudaStream_t s) {
  if (a.hd == 128) return launch_tc_t<128>(tk, tv, a, B, s);
  if (a.hd == 64) return launch_tc_t<64>(tk, tv, a, B, s);
  return DFLASH_ERR_UNSUPPORTED;
}

}  // namespace dfl
