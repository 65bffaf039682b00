// Device code and launch templates of the tcgen05 GEMMs, shared by the
// translation units that instantiate them (gemm.cu, gemm_tiles_*.cu) so that
// the many token-tile widths compile in parallel.  See gemm.cu for the design.
#pragma once

#include <cooperative_groups.h>

#include <cmath>

#include "common.cuh"
#include "gemm.h"

namespace dfl {
namespace {

namespace cg = cooperative_groups;

constexpr int kBK = 64;                   // K elements per stage (128 bytes of 16-bit values)
constexpr int kABytes = 128 * kBK * 2;    // weight box per stage

__device__ __forceinline__ float silu(float x) { return x / (1.0f + __expf(-x)); }

// Rotate-half RoPE of dimension d (< hd) of one row: x pairs with the
// partner dimension d +- hd/2; (cos, sin) come from the token's table row.
__device__ __forceinline__ float rope_apply(float x, float partner, float2 cs, bool first_half) {
  return first_half ? fmaf(x, cs.x, -partner * cs.y) : fmaf(x, cs.x, partner * cs.y);
}

__device__ __forceinline__ void store_f16(const GemmEpi& e, size_t o, float y) {
  static_cast<__half*>(e.out)[o] = to_f16_checked(y, e.status);
}

// Floats of one exchange buffer: a chunk of 16 tokens x 128 rows.
constexpr int kXchg = 16 * 128;

// Epilogue of up to 16 tokens of this thread's row: v[j] is token
// tok_base + j * tok_step, the first `ntok` are real.  `xchg` holds the
// chunk as [16][128] floats so that partner rows can be read.  Every thread
// of one epilogue group (four warps, one per TMEM lane quarter, named
// barrier `bar`) calls it: it synchronises once, after writing `xchg`;
// callers alternate between two buffers per group so that a chunk's writes
// never meet the previous chunk's reads.
__device__ __forceinline__ void epi_sync(int bar) {
  // immediate barrier ids: a register id would reserve all sixteen
  if (bar == 1)
    asm volatile("bar.sync 1, 128;" ::: "memory");
  else
    asm volatile("bar.sync 2, 128;" ::: "memory");
}

// Output row of token tok for EPI_F32 (the MASK rows with out_gather), or -1.
__device__ __forceinline__ int f32_out_row(const GemmEpi& e, int tok) {
  if (e.out_gather <= 0) return tok;
  const int G = e.out_gather, jj = tok % G;
  return jj ? (tok / G) * (G - 1) + jj - 1 : -1;
}

// Top-k partial of one 16-token chunk of an LM-head tile (xchg = the chunk's
// logits as [16 tokens][128 rows], rows beyond the vocabulary at -inf).  The
// eight threads r = 8 jt .. 8 jt + 7 of the group serve token jt: each keeps
// a sorted top-KT of 16 rows and their (max, sum of exp), the eight merge by
// shuffles, and the first writes the tile's partial for the token's row.
template <int KT>
__device__ __forceinline__ void tile_topk_partial(const GemmEpi& e, const float* xchg, int tok_base,
                                                  int tok_step, int ntok, int tile_n, int r) {
  const int jt = r >> 3, part = r & 7;
  unsigned long long top[KT];
#pragma unroll
  for (int j = 0; j < KT; ++j) top[j] = 0;
  float m = -INFINITY, s = 0.0f;
  const float* row = xchg + jt * 128 + part * 16;
  float x[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    x[i] = row[i];
    m = fmaxf(m, x[i]);
  }
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    if (x[i] != -INFINITY) {
      s += expf(x[i] - m);
      insert_key<KT>(top, vkey(x[i], tile_n * 128 + part * 16 + i));
    }
  }
  // merge the eight lists of the token (lanes differing in bits 0-2)
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) {
    unsigned long long other[KT];
#pragma unroll
    for (int j = 0; j < KT; ++j) other[j] = __shfl_xor_sync(0xffffffffu, top[j], o);
#pragma unroll
    for (int j = 0; j < KT; ++j) insert_key<KT>(top, other[j]);
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o), s2 = __shfl_xor_sync(0xffffffffu, s, o);
    lse_merge(m, s, m2, s2);
  }
  const int tok = tok_base + jt * tok_step;
  if (part == 0 && jt < ntok && tok < e.M) {
    const int orow = f32_out_row(e, tok);
    if (orow >= 0) {
      const size_t slot = (size_t)orow * e.tk_tiles + tile_n;
      unsigned long long* dst = e.tk_keys + slot * e.tk_slots;
#pragma unroll
      for (int j = 0; j < KT; ++j)
        if (j < e.tk_k) dst[j] = top[j];
      e.tk_ml[slot] = make_float2(m, s);
    }
  }
}

__device__ __forceinline__ void epilogue_chunk(const GemmEpi& e, const GemmAOpts& ao, const float (&v_in)[16],
                               int tok_base, int tok_step, int ntok, int tile_n, int r,
                               float* xchg, int bar, const float* rs = nullptr,
                               float wscale = 1.0f, const float* resid_pre = nullptr) {
  // resid_pre (EPI_RESID): the residual stream's values of the chunk already
  // in shared memory, [16 tokens][128 rows] of the tile, or nullptr
  const int kind = e.kind;
  // row scale of a folded RMSNorm: rs[j * tok_step] is token j's rstd; the
  // weight row's dequantization scale (E4M3 weights) multiplies every token
  float v[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) v[j] = (rs && j < ntok) ? v_in[j] * rs[j * tok_step] : v_in[j];
  if (wscale != 1.0f) {
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] *= wscale;
  }
  const bool topk = kind == EPI_F32 && e.tk_keys != nullptr;
  const bool needs_xchg = (kind == EPI_QKV || kind == EPI_SWIGLU || kind == EPI_KV_RING || topk);
  if (needs_xchg) {
    const bool live = !topk || tile_n * 128 + r < e.N;   // top-k: rows past the vocabulary lose
#pragma unroll
    for (int j = 0; j < 16; ++j) xchg[j * 128 + r] = live ? v[j] : -INFINITY;
    epi_sync(bar);
  }
  if (topk) {
    if (e.tk_slots == 16)
      tile_topk_partial<16>(e, xchg, tok_base, tok_step, ntok, tile_n, r);
    else
      tile_topk_partial<4>(e, xchg, tok_base, tok_step, ntok, tile_n, r);
  }
  // Every kind loads what it needs for its 16 tokens into registers first and
  // stores afterwards: loads placed after stores that might alias them would
  // each wait for a full memory round trip.
  if (kind == EPI_F32 || kind == EPI_F16 || kind == EPI_RESID || kind == EPI_NORM_IN) {
    const int n = tile_n * 128 + r;
    float nw[16];  // EPI_RESID: the updated stream, zero outside the tile
#pragma unroll
    for (int j = 0; j < 16; ++j) nw[j] = 0.0f;
    if (n < e.N) {
      if (kind == EPI_NORM_IN) {
        // the accumulator is the norm's input: its gained fp16 copy only
        const float gn = __ldg(e.xg_g + n);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int tok = tok_base + j * tok_step;
          nw[j] = (j < ntok && tok < e.M) ? v[j] : 0.0f;
          if (j < ntok && tok < e.M) e.xg[(size_t)tok * e.ld + n] = to_f16_checked(v[j] * gn, e.status);
        }
      } else if (kind == EPI_RESID) {
        float* out = static_cast<float*>(e.out);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int tok = tok_base + j * tok_step;
          nw[j] = (j < ntok && tok < e.M)
                      ? (resid_pre ? resid_pre[j * 128 + r] : __ldcg(out + (size_t)tok * e.ld + n)) + v[j]
                      : 0.0f;
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int tok = tok_base + j * tok_step;
          if (j < ntok && tok < e.M) out[(size_t)tok * e.ld + n] = nw[j];
        }
        if (e.xg) {
          const float gn = __ldg(e.xg_g + n);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int tok = tok_base + j * tok_step;
            if (j < ntok && tok < e.M) e.xg[(size_t)tok * e.ld + n] = to_f16_checked(nw[j] * gn, e.status);
          }
        }
      } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int tok = tok_base + j * tok_step;
          if (j < ntok && tok < e.M && e.out) {
            const int row = f32_out_row(e, tok);  // MASK rows only with out_gather
            if (row >= 0) {
              const size_t o = (size_t)row * e.ld + n;
              if (kind == EPI_F32)
                static_cast<float*>(e.out)[o] = v[j];
              else
                store_f16(e, o, v[j]);
            }
          }
        }
      }
    }
    if ((kind == EPI_RESID || kind == EPI_NORM_IN) && e.ssq) {
      // sum over this tile's 128 rows of each token's squared stream values
      // (warp butterflies, then the group's four warps in order): the next
      // GEMM's RMSNorm adds these per-tile sums
      const int q = r >> 5, lane = r & 31;
      float mine = 0.0f;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        float sq = nw[j] * nw[j];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
        if (lane == j) mine = sq;
      }
      if (lane < 16) xchg[q * 16 + lane] = mine;
      epi_sync(bar);
      if (q == 0 && lane < 16) {
        const int tok = tok_base + lane * tok_step;
        if (lane < ntok && tok < e.M)
          e.ssq[(size_t)tile_n * e.M + tok] =
              (xchg[lane] + xchg[16 + lane]) + (xchg[32 + lane] + xchg[48 + lane]);
      }
    }
  } else if (kind == EPI_QKV) {
    const int n = tile_n * 128 + r;
    if (n < e.N) {
      const bool rot = n < e.rope_rows;
      const int d = n % e.hd, half = e.hd >> 1;
      const float2* cs = e.rope_cs + d % half;
      const int pr = r ^ half;
      float y[16];
      if (rot) {
        float2 c[16];
        float partner[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int tok = tok_base + j * tok_step;
          const bool ok = j < ntok && tok < e.M;
          c[j] = ok ? __ldg(cs + (size_t)tok * half) : make_float2(1.0f, 0.0f);
          partner[j] = xchg[j * 128 + pr];
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) y[j] = rope_apply(v[j], partner[j], c[j], d < half);
      } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) y[j] = v[j];
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int tok = tok_base + j * tok_step;
        if (j < ntok && tok < e.M) store_f16(e, (size_t)tok * e.ld + n, y[j]);
      }
    }
  } else if (kind == EPI_SWIGLU) {
    const int f = tile_n * 64 + r;
    if (r < 64 && f < e.N) {
      float u[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) u[j] = xchg[j * 128 + r + 64];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int tok = tok_base + j * tok_step;
        if (j < ntok && tok < e.M) store_f16(e, (size_t)tok * e.ld + f, silu(v[j]) * u[j]);
      }
    }
  } else if (kind == EPI_KV_RING) {
    const int local = (tile_n % ao.tiles_per_map) * 128 + r;
    const int layer = e.layer0 + tile_n / ao.tiles_per_map;
    const int kv = local / e.kv_dim;            // 0 = K, 1 = V
    const int g = (local % e.kv_dim) / e.hd;
    const int d = local % e.hd, half = e.hd >> 1;
    const bool cs_table = e.rope_cs != nullptr;
    const float2* cs = e.rope_cs + d % half;
    const int pr = r ^ half;
    __nv_bfloat16* ring = static_cast<__nv_bfloat16*>(kv ? e.ring_v : e.ring_k);
    // gather: position, ring row and rotation of each token
    long long pos[16];
    int slot[16];
    float y[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int tok = tok_base + j * tok_step;
      pos[j] = -1;
      slot[j] = -1;
      y[j] = v[j];
      if (j < ntok && tok < e.M) {
        const int b = tok / e.n_max, jr = tok % e.n_max;
        if (jr < __ldg(e.n_new + b)) {
          pos[j] = __ldg(e.ctx_len + b) + jr;
          slot[j] = e.req_slot ? __ldg(e.req_slot + b) : b;
          if (kv == 0) {
            float2 c;
            if (cs_table) {
              c = __ldg(cs + (size_t)tok * half);
            } else {  // no table: the rotation of this position and frequency here
              rope_sincos((float)pos[j], e.rope_inv.f[d % half].x, e.rope_inv.f[d % half].y, &c.y, &c.x);
            }
            y[j] = rope_apply(v[j], xchg[j * 128 + pr], c, d < half);
          }
        }
      }
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int tok = tok_base + j * tok_step;
      if (j < ntok && tok < e.M && slot[j] != -1) {
        if (pos[j] < 0 || slot[j] < 0 || slot[j] >= e.ring_batch) {
          report_status(e.status, DFLASH_ERR_ARG);
          continue;
        }
        // the attention kernel reads ring entries as fp16
        if (!(fabsf(y[j]) <= kF16Max)) report_status(e.status, DFLASH_ERR_RANGE);
        const size_t o = ((((size_t)layer * e.ring_batch + slot[j]) * e.n_kv + g) * e.window +
                          (size_t)(pos[j] % e.window)) * e.hd + d;
        ring[o] = __float2bfloat16_rn(y[j]);
      }
    }
  }
}

// Epilogue of a one-tile GEMM CTA once its accumulator is complete (or its
// mainloop gave up: `aborted`): every thread of the CTA calls it.  Warps form
// groups of four (one warp per TMEM lane quarter) taking alternate 16-token
// chunks.  With split-K the tile's splits are reduced first: through global
// memory and a ticket, or inside the thread-block cluster the splits form.
// The stage buffers at `smem` are free by now and serve as scratch.  rs_tile:
// the folded RMSNorm's rstd per local token, or nullptr; wscale: this thread's
// weight-row dequantization scale (1 for fp16 weights).  free_bytes: the
// size of the free buffers at `smem`.
template <int BN, int kGroups>
__device__ __forceinline__ void one_tile_epilogue(uint8_t* smem, int free_bytes, uint32_t tmem, bool aborted,
                                                  const GemmAOpts& ao, const GemmArgs& args,
                                                  const GemmEpi& epi, int tile_n, int tile_m, int split,
                                                  const float* rs_tile, int* last_sh, float wscale) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q = warp & 3, grp = warp >> 2;  // TMEM lane quarter, epilogue group
  const int r = q * 32 + lane;
  const uint32_t t_row = tmem + ((uint32_t)(q * 32) << 16);
  float* xchg = reinterpret_cast<float*>(smem) + grp * 2 * kXchg;  // this group's two buffers
  const int bar = 1 + grp;

  constexpr int T = BN;  // tokens per tile
  constexpr int ntok = 16;
  constexpr int n_chunks = T / 16;
  auto load_chunk = [&](int c, float (&v)[16]) {
    uint32_t raw[16];
    tmem_ld_x16(t_row + c * 16, raw);
    tc_wait_ld();
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(raw[j]);
  };

  if (args.splits == 1) {
    if (!aborted) {
      for (int c = grp, it = 0; c < n_chunks; c += kGroups, ++it) {
        float v[16];
        load_chunk(c, v);
        epilogue_chunk(epi, ao, v, tile_m * T + c * 16, 1, ntok, tile_n, r, xchg + (it & 1) * kXchg, bar,
                       rs_tile ? rs_tile + c * 16 : nullptr, wscale);
      }
    }
  } else if (!args.cluster) {
    // Ticketed reduction: every split stores its fp32 partial [T][128] in
    // global memory; the last split of the tile to arrive (atomic ticket after
    // a fence) sums them in split order and runs the epilogue.  At batch 1 each
    // global round trip on this path costs the tile's last split about a
    // microsecond, so its reads are issued together as asynchronous copies
    // into the free stage buffers: the residual stream (EPI_RESID) before the
    // ticket, then the splits' partials (all at once when they fit).
    const int tile_lin = tile_m * gridDim.x + tile_n;
    const size_t per_split = (size_t)n_chunks * 16 * 128;
    const int per16 = (int)(per_split / 4);  // 16-byte pieces of one partial
    float* part = args.partial + (size_t)tile_lin * args.splits * per_split;
    float* mine = part + (size_t)split * per_split;
    float* land = reinterpret_cast<float*>(smem) + kGroups * 2 * kXchg;  // past the exchange buffers
    const long long land_cap = (long long)free_bytes / 4 - kGroups * 2 * kXchg;
    const float* xres = static_cast<const float*>(epi.out);
    const bool resid_s = epi.kind == EPI_RESID && !aborted && (epi.N & 3) == 0 && (epi.ld & 3) == 0 &&
                         (reinterpret_cast<uintptr_t>(xres) & 15) == 0 && land_cap >= 2 * (long long)per_split;
    float* land_p = land + (resid_s ? per_split : 0);
    const int batch = (int)((land_cap - (resid_s ? (long long)per_split : 0)) / (long long)per_split);
    if (resid_s) {
      // only this tile's last split writes these values, after every split
      // has taken its ticket; the other splits discard what they read
      for (int idx = threadIdx.x; idx < T * 32; idx += blockDim.x) {
        const int tl = idx >> 5, q4 = (idx & 31) * 4;
        const int tok = tile_m * T + tl, n = tile_n * 128 + q4;
        const bool ok = tok < epi.M && n < epi.N;
        cp_async16(land + tl * 128 + q4, ok ? xres + (size_t)tok * epi.ld + n : xres, ok);
      }
    }
    if (!aborted) {
      for (int c = grp; c < n_chunks; c += kGroups) {
        float v[16];
        load_chunk(c, v);
#pragma unroll
        for (int j = 0; j < 16; ++j) mine[(c * 16 + j) * 128 + r] = v[j];
      }
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) *last_sh = (atomicAdd(&args.counters[tile_lin], 1) == args.splits - 1);
    __syncthreads();
    if (*last_sh) {
      __threadfence();
      const int S = args.splits;
      if (!aborted && batch >= 1 && (S <= batch || n_chunks == 1)) {
        // rounds of up to `batch` partials (one round unless a single chunk
        // accumulates across several)
        const int nb = S < batch ? S : batch;
        float acc[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) acc[j] = 0.0f;
        for (int s0 = 0; s0 < S; s0 += nb) {
          const int cnt = S - s0 < nb ? S - s0 : nb;
          for (int idx = threadIdx.x; idx < cnt * per16; idx += blockDim.x) {
            const int sl = idx / per16, off = (idx - sl * per16) * 4;
            cp_async16(land_p + (size_t)sl * per_split + off, part + (size_t)(s0 + sl) * per_split + off, true);
          }
          cp_async_wait_all();
          __syncthreads();
          if (n_chunks == 1) {
            if (grp == 0)
              for (int k = 0; k < cnt; ++k) {
#pragma unroll
                for (int j = 0; j < 16; ++j) acc[j] += land_p[(size_t)k * per_split + j * 128 + r];  // split order
              }
            if (s0 + nb < S) __syncthreads();  // the next round overwrites the landing zone
          }
        }
        for (int c = grp, it = 0; c < n_chunks; c += kGroups, ++it) {
          float v[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] = acc[j];
          if (n_chunks > 1) {
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = 0.0f;
            for (int k = 0; k < S; ++k) {
#pragma unroll
              for (int j = 0; j < 16; ++j) v[j] += land_p[(size_t)k * per_split + (c * 16 + j) * 128 + r];
            }
          }
          epilogue_chunk(epi, ao, v, tile_m * T + c * 16, 1, ntok, tile_n, r, xchg + (it & 1) * kXchg,
                         bar, rs_tile ? rs_tile + c * 16 : nullptr, wscale,
                         resid_s ? land + (size_t)(c * 16) * 128 : nullptr);
        }
      } else if (!aborted) {
        cp_async_wait_all();  // the residual block
        __syncthreads();
        for (int c = grp, it = 0; c < n_chunks; c += kGroups, ++it) {
          float v[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] = 0.0f;
          for (int s = 0; s < S; ++s) {
            const float* ps = part + (size_t)s * per_split;
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] += __ldcg(ps + (c * 16 + j) * 128 + r);
          }
          epilogue_chunk(epi, ao, v, tile_m * T + c * 16, 1, ntok, tile_n, r, xchg + (it & 1) * kXchg,
                         bar, rs_tile ? rs_tile + c * 16 : nullptr, wscale,
                         resid_s ? land + (size_t)(c * 16) * 128 : nullptr);
        }
      }
      if (threadIdx.x == 0) atomicExch(&args.counters[tile_lin], 0);
    }
    cp_async_wait_all();  // no copy may land after the CTA has left
  } else {
    // The K splits of this tile form a thread-block cluster.  Each leaves its
    // fp32 partial [T tokens][128 rows] in its own shared memory (the stage
    // buffers are free: every stage has been consumed); after a cluster
    // barrier CTA `rank` sums, over distributed shared memory and in split
    // order, the tokens rank, rank + S, ... of the tile and runs the epilogue
    // on them.  A CTA whose wait gave up still takes part in both cluster
    // barriers (its siblings would otherwise wait for it) but writes nothing.
    float* part_s = reinterpret_cast<float*>(smem);
    float* xchg_s = part_s + (size_t)n_chunks * 16 * 128 + grp * 2 * kXchg;
    for (int c = grp; c < n_chunks; c += kGroups) {
      float v[16];
      if (!aborted) {
        load_chunk(c, v);
      } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = 0.0f;
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) part_s[(c * 16 + j) * 128 + r] = v[j];
    }
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();
    if (!aborted) {
      const int S = args.splits;
      const int rank = split;  // cluster dims (1, 1, S): rank = blockIdx.z
      const int mine = (T - rank + S - 1) / S;
      for (int g0 = grp * 16, it = 0; g0 < mine; g0 += 16 * kGroups, ++it) {
        float v[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = 0.0f;
        for (int s = 0; s < S; ++s) {
          const float* ps = cluster.map_shared_rank(part_s, s);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int t = rank + (g0 + j) * S;
            if (g0 + j < mine) v[j] += ps[t * 128 + r];
          }
        }
        const int cnt = mine - g0 < 16 ? mine - g0 : 16;
        epilogue_chunk(epi, ao, v, tile_m * T + rank + g0 * S, S, cnt, tile_n, r,
                       xchg_s + (it & 1) * kXchg, bar, rs_tile ? rs_tile + rank + g0 * S : nullptr,
                       wscale);
      }
    }
    // no CTA may leave while another still reads its shared memory
    cluster.sync();
  }
}

// Threads of gemm_tc_kernel: four warps, eight (two epilogue groups taking
// alternate chunks of 16 tokens) for tiles of 128 or more tokens, whose
// one-tile epilogue would otherwise run serially after the mainloop.
__host__ __device__ constexpr int gemm_threads(int BN) { return BN >= 128 ? 256 : 128; }

// TMEM allocations are powers of two of at least 32 columns.
__host__ __device__ constexpr uint32_t tmem_cols(int n) {
  return n <= 32 ? 32u : n <= 64 ? 64u : n <= 128 ? 128u : n <= 256 ? 256u : 512u;
}

template <int BN, int STAGES>
__global__ void __launch_bounds__(gemm_threads(BN), 1)
    gemm_tc_kernel(const __grid_constant__ GemmAMaps A, const __grid_constant__ CUtensorMap tmB,
                        const GemmAOpts ao, const GemmArgs args, const GemmEpi epi) {
  constexpr int kBBytes = BN * kBK * 2;
  constexpr int kStage = kABytes + kBBytes;
  constexpr uint32_t kTmemCols = tmem_cols(BN);
  constexpr int kGroups = gemm_threads(BN) / 128;
  static_assert(kStage % 1024 == 0, "stage buffers must keep 1024-byte alignment");
  static_assert((BN + 64) * 128 * 4 <= STAGES * kStage, "split partials must fit the stage buffers");

  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[STAGES];
  __shared__ __align__(8) uint64_t empty_bar[STAGES];
  __shared__ __align__(8) uint64_t acc_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  __shared__ int last_sh;
  __shared__ float rs_sh[BN <= 32 ? 32 : 1];  // row scale (RMSNorm rstd) of the tile's tokens

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile_n = blockIdx.x, tile_m = blockIdx.y, split = blockIdx.z;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int kb_total = (args.K + kBK - 1) / kBK;
  const int kb0 = (int)((long long)split * kb_total / args.splits);
  const int kb1 = (int)((long long)(split + 1) * kb_total / args.splits);
  const int nkb = kb1 - kb0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    mbar_init(&acc_bar, 1);
    abort_sh = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    for (int i = 0; i < ao.n_maps; ++i) tma_prefetch_desc(&A.map[i]);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  // the next kernel may be scheduled now; it waits for our completion before
  // reading what we write
  grid_dependents_launch();

  int issued = 0;
  if (warp == 0 && lane == 0) {
    // ---------------------------------------------------------- producer
    const uint64_t pol_w = policy_evict_first();
    const uint64_t pol_x = policy_evict_last();
    int map_i = 0, row0;
    if (ao.dual) {
      row0 = ao.row_offset + tile_n * 64;
    } else {
      map_i = tile_n / ao.tiles_per_map;
      row0 = ao.row_offset + (tile_n % ao.tiles_per_map) * 128;
    }
    const int tok0 = tile_m * BN;
    // weights do not depend on the previous kernel: start streaming them
    // before waiting for it (programmatic dependent launch)
    const int pre = nkb < STAGES ? nkb : STAGES;
    for (int i = 0; i < pre; ++i) {
      uint8_t* sa = smem + i * kStage;
      mbar_arrive_expect_tx(&full_bar[i], kStage);
      const int kc = (kb0 + i) * kBK;
      if (ao.dual) {
        tma_load_2d(sa, &A.map[0], &full_bar[i], kc, row0, pol_w);
        tma_load_2d(sa + 64 * 128, &A.map[1], &full_bar[i], kc, row0, pol_w);
      } else {
        tma_load_2d(sa, &A.map[map_i], &full_bar[i], kc, row0, pol_w);
      }
    }
    grid_dependency_wait();
    for (int i = 0; i < pre; ++i)
      tma_load_2d(smem + i * kStage + kABytes, &tmB, &full_bar[i], (kb0 + i) * kBK, tok0, pol_x);
    issued = pre;
    for (int i = pre; i < nkb; ++i) {
      const int s = i % STAGES;
      const uint32_t ph = (uint32_t)(i / STAGES) & 1u;
      if (!mbar_wait_bounded(&empty_bar[s], ph ^ 1u, &abort_sh, args.status)) break;
      uint8_t* sa = smem + s * kStage;
      mbar_arrive_expect_tx(&full_bar[s], kStage);
      const int kc = (kb0 + i) * kBK;
      if (ao.dual) {
        tma_load_2d(sa, &A.map[0], &full_bar[s], kc, row0, pol_w);
        tma_load_2d(sa + 64 * 128, &A.map[1], &full_bar[s], kc, row0, pol_w);
      } else {
        tma_load_2d(sa, &A.map[map_i], &full_bar[s], kc, row0, pol_w);
      }
      tma_load_2d(sa + kABytes, &tmB, &full_bar[s], kc, tok0, pol_x);
      issued = i + 1;
    }
  } else if (warp == 1 && lane == 0) {
    // --------------------------------------------------------- MMA issuer
    const uint32_t idesc = idesc_f32acc(128, BN, args.type == OPND_BF16);
    for (int i = 0; i < nkb; ++i) {
      const int s = i % STAGES;
      const uint32_t ph = (uint32_t)(i / STAGES) & 1u;
      if (!mbar_wait_bounded(&full_bar[s], ph, &abort_sh, args.status)) break;
      tc_fence_after();
      const uint32_t a_addr = smem_u32(smem + s * kStage);
      const uint32_t b_addr = a_addr + kABytes;
#pragma unroll
      for (int k = 0; k < kBK / 16; ++k)
        tc_mma_f16(tmem, smem_desc_sw128(a_addr + k * 32), smem_desc_sw128(b_addr + k * 32), idesc,
                   (i | k) ? 1u : 0u);
      tc_commit(&empty_bar[s]);
    }
    tc_commit(&acc_bar);
  }
  if constexpr (BN <= 32) {
    if (warp == 2 && args.rs_ssq) {
      // rstd of the tile's tokens for a folded RMSNorm, while the mainloop runs
      grid_dependency_wait();
      if (lane < BN) {
        const int m = tile_m * BN + lane;
        float rsv = 0.0f;
        if (m < epi.M) {
          float ss = 0.0f;
          for (int p = 0; p < args.rs_parts; ++p) ss += __ldcg(args.rs_ssq + (size_t)p * epi.M + m);
          rsv = rsqrtf(ss / (float)args.rs_n + args.rs_eps);
        }
        rs_sh[lane] = rsv;
      }
    }
  }
  __syncwarp();

  // ----------------------------------------------------------- epilogue
  const bool acc_ok = mbar_wait_bounded(&acc_bar, 0, &abort_sh, args.status);
  tc_fence_after();
  if (warp == 0 && lane == 0 && abort_sh) {
    // a wait gave up: let this CTA's copies in flight land before exiting
    int dummy = 0;
    for (int i = (issued > STAGES ? issued - STAGES : 0); i < issued; ++i)
      (void)mbar_wait_bounded(&full_bar[i % STAGES], (uint32_t)(i / STAGES) & 1u, &dummy, nullptr,
                              100000000ull);
  }
  __syncthreads();
  one_tile_epilogue<BN, kGroups>(smem, STAGES * kStage, tmem, abort_sh != 0 || !acc_ok, ao, args, epi, tile_n, tile_m,
                                 split, (BN <= 32 && args.rs_ssq) ? rs_sh : nullptr, &last_sh, 1.0f);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// Persistent, warp-specialised variant for many token columns (no split-K):
// one CTA per SM walks the tiles t = blockIdx.x, blockIdx.x + gridDim.x, ...
// (token tiles fastest, so CTAs running at the same time share weight tiles in
// L2).  Warp 0 lane 0 issues TMA, warp 1 lane 0 issues MMAs, warps 2-9 run
// the epilogue as two groups of four (one warp per TMEM lane quarter) taking
// alternate chunks of 16 tokens.  Two TMEM accumulators let the epilogue of
// one tile overlap the mainloop of the next.
template <int BN, int STAGES>
__global__ void __launch_bounds__(320, 1)
    gemm_tc_persistent_kernel(const __grid_constant__ GemmAMaps A,
                                   const __grid_constant__ CUtensorMap tmB, const GemmAOpts ao,
                                   const GemmArgs args, const GemmEpi epi, int n_tiles, int m_tiles) {
  constexpr int kBBytes = BN * kBK * 2;
  constexpr int kStage = kABytes + kBBytes;
  constexpr uint32_t kTmemCols = tmem_cols(2 * BN);  // two accumulators, at columns 0 and BN
  static_assert(kStage % 1024 == 0, "stage buffers must keep 1024-byte alignment");
  static_assert(2 * BN <= 512, "two accumulators must fit tensor memory");

  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[STAGES];
  __shared__ __align__(8) uint64_t empty_bar[STAGES];
  __shared__ __align__(8) uint64_t accf_bar[2];
  __shared__ __align__(8) uint64_t acce_bar[2];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* xchg = reinterpret_cast<float*>(smem + STAGES * kStage);
  constexpr int T = BN;
  const int kb_total = (args.K + kBK - 1) / kBK;
  const int total = n_tiles * m_tiles;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&accf_bar[b], 1);
      mbar_init(&acce_bar[b], 8);
    }
    abort_sh = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    for (int i = 0; i < ao.n_maps; ++i) tma_prefetch_desc(&A.map[i]);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  grid_dependents_launch();

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------- producer
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_x = policy_evict_last();
      bool waited = false;
      int it = 0;
      for (int t = blockIdx.x; t < total && !abort_sh; t += gridDim.x) {
        const int tile_m = t % m_tiles, tile_n = t / m_tiles;
        int map_i = 0, row0;
        if (ao.dual) {
          row0 = ao.row_offset + tile_n * 64;
        } else {
          map_i = tile_n / ao.tiles_per_map;
          row0 = ao.row_offset + (tile_n % ao.tiles_per_map) * 128;
        }
        const int tok0 = tile_m * T;
        for (int kb = 0; kb < kb_total; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (uint32_t)(it / STAGES) & 1u;
          if (!mbar_wait_bounded(&empty_bar[s], ph ^ 1u, &abort_sh, args.status)) break;
          uint8_t* sa = smem + s * kStage;
          mbar_arrive_expect_tx(&full_bar[s], kStage);
          const int kc = kb * kBK;
          if (ao.dual) {
            tma_load_2d(sa, &A.map[0], &full_bar[s], kc, row0, pol_w);
            tma_load_2d(sa + 64 * 128, &A.map[1], &full_bar[s], kc, row0, pol_w);
          } else {
            tma_load_2d(sa, &A.map[map_i], &full_bar[s], kc, row0, pol_w);
          }
          if (!waited) {  // activations come from the previous kernel
            grid_dependency_wait();
                    waited = true;
          }
          tma_load_2d(sa + kABytes, &tmB, &full_bar[s], kc, tok0, pol_x);
        }
      }
      if (abort_sh) {
        int dummy = 0;
        for (int i = (it > STAGES ? it - STAGES : 0); i < it; ++i)
          (void)mbar_wait_bounded(&full_bar[i % STAGES], (uint32_t)(i / STAGES) & 1u, &dummy, nullptr,
                                  100000000ull);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------- MMA issuer
      const uint32_t idesc = idesc_f32acc(128, BN, args.type == OPND_BF16);
      int it = 0, lt = 0;
      for (int t = blockIdx.x; t < total && !abort_sh; t += gridDim.x, ++lt) {
        const int buf = lt & 1;
        const uint32_t use = (uint32_t)(lt >> 1);
        if (!mbar_wait_bounded(&acce_bar[buf], (use & 1u) ^ 1u, &abort_sh, args.status)) break;
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(buf * BN);
        for (int kb = 0; kb < kb_total; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (uint32_t)(it / STAGES) & 1u;
          if (!mbar_wait_bounded(&full_bar[s], ph, &abort_sh, args.status)) break;
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + s * kStage);
          const uint32_t b_addr = a_addr + kABytes;
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)
            tc_mma_f16(d, smem_desc_sw128(a_addr + k * 32), smem_desc_sw128(b_addr + k * 32), idesc,
                       (kb | k) ? 1u : 0u);
          tc_commit(&empty_bar[s]);
        }
        tc_commit(&accf_bar[buf]);
      }
    }
  } else {
    // --------------------------------------------------------- epilogue
    const int r = 32 * (warp & 3) + lane;  // TMEM lane quarter of this warp
    const uint32_t t_row = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    const int grp = (warp - 2) >> 2, bar = 1 + grp;
    float* gx = xchg + grp * 2 * kXchg;   // this group's two exchange buffers
    constexpr int ntok = 16;
    constexpr int n_chunks = T / 16;
    int lt = 0;
    unsigned xc = 0;  // exchange buffer of the next chunk, alternating across tiles
    for (int t = blockIdx.x; t < total; t += gridDim.x, ++lt) {
      const int tile_m = t % m_tiles, tile_n = t / m_tiles;
      const int buf = lt & 1;
      const uint32_t use = (uint32_t)(lt >> 1);
      const bool ok = mbar_wait_bounded(&accf_bar[buf], use & 1u, &abort_sh, args.status);
      // the four warps of the group agree before acting on the outcome
      epi_sync(bar);
      if (!ok || abort_sh) break;
      tc_fence_after();
      const uint32_t base = t_row + (uint32_t)(buf * BN);
      for (int c = grp; c < n_chunks; c += 2) {
        float v[16];
        uint32_t raw[16];
        tmem_ld_x16(base + c * 16, raw);
        tc_wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(raw[j]);
        if (c + 2 >= n_chunks) {
          // every column of this accumulator is in registers: hand it back
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acce_bar[buf]);
        }
        epilogue_chunk(epi, ao, v, tile_m * T + c * 16, 1, ntok, tile_n, r, gx + (xc++ & 1) * kXchg,
                       bar);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// Persistent kernel over CTA pairs (cta_group::2).  A cluster of two CTAs
// owns a unit of two adjacent weight tiles (256 rows) x one token tile: each
// CTA loads its own 128 weight rows and half of the token tile, and one
// thread of the even CTA issues M = 256 MMAs that read both CTAs' shared
// memory and accumulate each CTA's 128 rows in its own tensor memory.  Per
// k-block a CTA then moves 16 KiB of weights + BN * 64 bytes of activations
// through shared memory instead of 16 KiB + BN * 128, which is what bounds
// the single-CTA kernel's mainloop (TMA fills and MMA operand reads share the
// SM's shared-memory bandwidth).
//   Barriers: the even CTA's full[s] takes one expect-tx arrival (its
// producer's, for both CTAs' bytes) and both CTAs' TMA bytes; the even CTA's MMA commits arrive on empty[s] and
// accf[b] of both CTAs; the even CTA's acce[b] counts the epilogue warps of
// both CTAs.  Both CTAs meet at cluster barriers after setup and before exit,
// so neither leaves while the other may still touch its memory.
template <int BN, int STAGES>
__global__ void __launch_bounds__(320, 1)
    gemm_tc_pair_kernel(const __grid_constant__ GemmAMaps A, const __grid_constant__ CUtensorMap tmB,
                        const GemmAOpts ao, const GemmArgs args, const GemmEpi epi, int n_tiles,
                        int m_tiles) {
  constexpr int kBHalf = BN / 2;                  // token rows of B held by each CTA
  constexpr int kBBytes = kBHalf * kBK * 2;
  constexpr int kStage = kABytes + kBBytes;
  constexpr uint32_t kTmemCols = tmem_cols(2 * BN);  // two accumulators, at columns 0 and BN
  static_assert(kStage % 1024 == 0, "stage buffers must keep 1024-byte alignment");
  static_assert(kBHalf % 8 == 0, "half token tiles must hold whole 8-row swizzle atoms");
  static_assert(2 * BN <= 512, "two accumulators must fit tensor memory");

  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[STAGES];
  __shared__ __align__(8) uint64_t empty_bar[STAGES];
  __shared__ __align__(8) uint64_t accf_bar[2];
  __shared__ __align__(8) uint64_t acce_bar[2];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* xchg = reinterpret_cast<float*>(smem + STAGES * kStage);
  constexpr int T = BN;
  const int kb_total = (args.K + kBK - 1) / kBK;
  const int n_pairs_n = (n_tiles + 1) / 2;
  const int total = n_pairs_n * m_tiles;
  const int unit0 = (int)(blockIdx.x >> 1), unit_step = (int)(gridDim.x >> 1);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&accf_bar[b], 1);
      mbar_init(&acce_bar[b], 16);
    }
    abort_sh = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    for (int i = 0; i < ao.n_maps; ++i) tma_prefetch_desc(&A.map[i]);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc_pair(&tmem_base_sh, kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  // the peer's barriers are initialised and its tensor memory allocated
  cluster_arrive();
  cluster_wait();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  if (threadIdx.x == 0) {
    // the pair's MMAs address both CTAs' accumulators by one column address
    uint32_t peer;
    asm volatile("ld.shared::cluster.u32 %0, [%1];"
                 : "=r"(peer)
                 : "r"(mapa_shared(smem_u32(&tmem_base_sh), rank ^ 1u))
                 : "memory");
    if (peer != tmem) {
      abort_sh = 1;
      report_status(args.status, DFLASH_ERR_UNSUPPORTED);
    }
  }
  __syncthreads();
  grid_dependents_launch();

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------- producer
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_x = policy_evict_last();
      bool waited = false;
      int it = 0;
      for (int t = unit0; t < total && !abort_sh; t += unit_step) {
        const int tile_m = t % m_tiles;
        int tile_n = (t / m_tiles) * 2 + (int)rank;
        // an odd tile count leaves the last unit one tile: the other CTA loads
        // the live tile's rows again (its results are not stored)
        if (tile_n >= n_tiles) tile_n = n_tiles - 1;
        int map_i = 0, row0;
        if (ao.dual) {
          row0 = ao.row_offset + tile_n * 64;
        } else {
          map_i = tile_n / ao.tiles_per_map;
          row0 = ao.row_offset + (tile_n % ao.tiles_per_map) * 128;
        }
        const int tok0 = tile_m * T + (int)rank * kBHalf;
        for (int kb = 0; kb < kb_total; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (uint32_t)(it / STAGES) & 1u;
          if (!mbar_wait_bounded(&empty_bar[s], ph ^ 1u, &abort_sh, args.status)) break;
          uint8_t* sa = smem + s * kStage;
          const uint32_t fb = mapa_shared(smem_u32(&full_bar[s]), 0);
          // the even CTA announces both CTAs' bytes; the odd CTA's copies may
          // land before that (the transaction count runs negative meanwhile)
          if (rank == 0) mbar_arrive_expect_tx(&full_bar[s], 2 * kStage);
          const int kc = kb * kBK;
          if (ao.dual) {
            tma_load_2d_pair(sa, &A.map[0], fb, kc, row0, pol_w);
            tma_load_2d_pair(sa + 64 * 128, &A.map[1], fb, kc, row0, pol_w);
          } else {
            tma_load_2d_pair(sa, &A.map[map_i], fb, kc, row0, pol_w);
          }
          if (!waited) {  // activations come from the previous kernel
            grid_dependency_wait();
                    waited = true;
          }
          tma_load_2d_pair(sa + kABytes, &tmB, fb, kc, tok0, pol_x);
        }
      }
      if (abort_sh) {
        // let this CTA's copies in flight land: wait for the stages it filled
        // to be consumed or give up after a short bound
        int dummy = 0;
        for (int i = (it > STAGES ? it - STAGES : 0); i < it; ++i)
          (void)mbar_wait_bounded(&empty_bar[i % STAGES], (uint32_t)(i / STAGES) & 1u, &dummy, nullptr,
                                  100000000ull);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ------------------------------------------------------- MMA issuer
      const uint32_t idesc = idesc_f32acc(256, BN, args.type == OPND_BF16);
      int it = 0, lt = 0;
      for (int t = unit0; t < total && !abort_sh; t += unit_step, ++lt) {
        const int buf = lt & 1;
        const uint32_t use = (uint32_t)(lt >> 1);
        if (!mbar_wait_bounded(&acce_bar[buf], (use & 1u) ^ 1u, &abort_sh, args.status)) break;
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(buf * BN);
        for (int kb = 0; kb < kb_total; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (uint32_t)(it / STAGES) & 1u;
          if (!mbar_wait_bounded(&full_bar[s], ph, &abort_sh, args.status)) break;
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + s * kStage);
          const uint32_t b_addr = a_addr + kABytes;
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)
            tc_mma_f16_pair(d, smem_desc_sw128(a_addr + k * 32), smem_desc_sw128(b_addr + k * 32), idesc,
                            (kb | k) ? 1u : 0u);
          tc_commit_pair(&empty_bar[s], (uint16_t)3);
        }
        tc_commit_pair(&accf_bar[buf], (uint16_t)3);
      }
    }
  } else {
    // --------------------------------------------------------- epilogue
    const int r = 32 * (warp & 3) + lane;  // TMEM lane quarter of this warp
    const uint32_t t_row = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    const int grp = (warp - 2) >> 2, bar = 1 + grp;
    float* gx = xchg + grp * 2 * kXchg;   // this group's two exchange buffers
    constexpr int ntok = 16;
    constexpr int n_chunks = T / 16;
    int lt = 0;
    unsigned xc = 0;
    for (int t = unit0; t < total; t += unit_step, ++lt) {
      const int tile_m = t % m_tiles, tile_n = (t / m_tiles) * 2 + (int)rank;
      const int buf = lt & 1;
      const uint32_t use = (uint32_t)(lt >> 1);
      const bool ok = mbar_wait_bounded(&accf_bar[buf], use & 1u, &abort_sh, args.status);
      epi_sync(bar);
      if (!ok || abort_sh) break;
      tc_fence_after();
      const uint32_t base = t_row + (uint32_t)(buf * BN);
      const bool live = tile_n < n_tiles;  // the last unit may hold one weight tile
      for (int c = grp; c < n_chunks; c += 2) {
        float v[16];
        uint32_t raw[16];
        tmem_ld_x16(base + c * 16, raw);
        tc_wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(raw[j]);
        if (c + 2 >= n_chunks) {
          // every column of this accumulator is in registers: hand it back
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&acce_bar[buf]), 0));
        }
        if (live)
          epilogue_chunk(epi, ao, v, tile_m * T + c * 16, 1, ntok, tile_n, r, gx + (xc++ & 1) * kXchg,
                         bar);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  // the peer may still read this CTA's stages (MMA) or arrive on its barriers
  cluster_arrive();
  cluster_wait();
  if (warp == 1) tmem_dealloc_pair(tmem, kTmemCols);
}

// ------------------------------------------------------------------ launch


template <int BN, int STAGES>
constexpr size_t smem_bytes() {
  return (size_t)STAGES * (kABytes + BN * kBK * 2) + 1024;
}

template <int BN, int STAGES>
int launch_one(const GemmAMaps& A, const CUtensorMap& tmB, const GemmAOpts& ao, const GemmArgs& args,
               const GemmEpi& epi, dim3 grid, cudaStream_t s, bool pdl) {
  auto kern = gemm_tc_kernel<BN, STAGES>;
  constexpr size_t smem = smem_bytes<BN, STAGES>();
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
      return DFLASH_ERR_LAUNCH;
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(gemm_threads(BN));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  if (args.splits > 1 && args.cluster) {  // the K splits of a tile run as one cluster
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = 1;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = args.splits;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  if (cudaLaunchKernelEx(&cfg, kern, A, tmB, ao, args, epi) != cudaSuccess) return DFLASH_ERR_LAUNCH;
  return DFLASH_OK;
}



template <int BN, int STAGES>
int launch_persistent(const GemmAMaps& A, const CUtensorMap& tmB, const GemmAOpts& ao,
                      const GemmArgs& args, const GemmEpi& epi, int n_tiles, int m_tiles,
                      int num_sms, cudaStream_t s, bool pdl) {
  auto kern = gemm_tc_persistent_kernel<BN, STAGES>;
  constexpr size_t smem = (size_t)STAGES * (kABytes + BN * kBK * 2) + 4 * kXchg * 4 + 1024;
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
      return DFLASH_ERR_LAUNCH;
    attr_set = true;
  }
  const int total = n_tiles * m_tiles;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(total < num_sms ? total : num_sms);
  cfg.blockDim = dim3(320);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  if (cudaLaunchKernelEx(&cfg, kern, A, tmB, ao, args, epi, n_tiles, m_tiles) != cudaSuccess)
    return DFLASH_ERR_LAUNCH;
  return DFLASH_OK;
}

template <int BN, int STAGES>
int launch_pair(const GemmAMaps& A, const CUtensorMap& tmB, const GemmAOpts& ao, const GemmArgs& args,
                const GemmEpi& epi, int n_tiles, int m_tiles, int num_sms, cudaStream_t s, bool pdl) {
  auto kern = gemm_tc_pair_kernel<BN, STAGES>;
  constexpr size_t smem = (size_t)STAGES * (kABytes + BN / 2 * kBK * 2) + 4 * kXchg * 4 + 1024;
  static int max_pairs = -1;
  if (max_pairs < 0) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
      return DFLASH_ERR_LAUNCH;
    // how many pairs fit at once: a persistent grid must not exceed it
    cudaLaunchConfig_t q = {};
    q.gridDim = dim3(2 * (num_sms / 2));
    q.blockDim = dim3(320);
    q.dynamicSmemBytes = smem;
    cudaLaunchAttribute qa[1];
    qa[0].id = cudaLaunchAttributeClusterDimension;
    qa[0].val.clusterDim.x = 2;
    qa[0].val.clusterDim.y = 1;
    qa[0].val.clusterDim.z = 1;
    q.attrs = qa;
    q.numAttrs = 1;
    int nc = 0;
    if (cudaOccupancyMaxActiveClusters(&nc, kern, &q) != cudaSuccess || nc < 1) {
      (void)cudaGetLastError();
      return DFLASH_ERR_LAUNCH;
    }
    max_pairs = nc;
  }
  const int units = ((n_tiles + 1) / 2) * m_tiles;
  const int pairs = units < max_pairs ? units : max_pairs;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs);
  cfg.blockDim = dim3(320);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  if (cudaLaunchKernelEx(&cfg, kern, A, tmB, ao, args, epi, n_tiles, m_tiles) != cudaSuccess)
    return DFLASH_ERR_LAUNCH;
  return DFLASH_OK;
}

}  // namespace

// Launch of one token-tile width: the non-persistent kernel on `grid`, or the
// persistent one; defined by the translation unit that instantiates it.
#define DFL_TILE_CASES_ONE(X) X(16, 6) X(32, 5) X(64, 4)
// pair kernel: stages of 16 KiB + BN * 64 bytes within about 192 KiB
#define DFL_PAIR_CASES(X)                                                                    \
  X(80, 8) X(96, 8) X(112, 8) X(128, 8) X(144, 7) X(160, 7) X(176, 7) X(192, 6) X(208, 6) \
  X(224, 6) X(240, 6) X(256, 6)

// Token tiles of 80 to 256 (two widths per translation unit, gemm_tiles_*.cu).
#define DFL_TILE_UNIT_DECL(name)                                                                 \
  int name(int BN, bool persistent, const GemmAMaps& A, const CUtensorMap& tmB, const GemmAOpts& ao, \
           const GemmArgs& args, const GemmEpi& epi, dim3 grid, int n_tiles, int m_tiles, int num_sms, \
           cudaStream_t s, bool pdl);
DFL_TILE_UNIT_DECL(launch_tile_080)
DFL_TILE_UNIT_DECL(launch_tile_112)
DFL_TILE_UNIT_DECL(launch_tile_144)
DFL_TILE_UNIT_DECL(launch_tile_176)
DFL_TILE_UNIT_DECL(launch_tile_208)
DFL_TILE_UNIT_DECL(launch_tile_240)
#undef DFL_TILE_UNIT_DECL
// The pair kernel of one token-tile width; tmB_half describes boxes of BN / 2
// token rows.
int launch_tile_pair(int BN, const GemmAMaps& A, const CUtensorMap& tmB_half, const GemmAOpts& ao,
                     const GemmArgs& args, const GemmEpi& epi, int n_tiles, int m_tiles, int num_sms,
                     cudaStream_t s, bool pdl);

}  // namespace dfl
