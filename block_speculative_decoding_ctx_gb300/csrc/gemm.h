// Internal interface of the tcgen05 GEMM (gemm.cu).
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "dflash.h"

namespace dfl {

constexpr int kMaxAMaps = 8;

enum EpiKind : int {
  EPI_F32 = 0,     // out fp32 [M, ld] = acc
  EPI_F16 = 1,     // out fp16 [M, ld] = acc
  EPI_QKV = 2,     // out fp16 [M, ld]; rows < rope_rows rotated (table row m)
  EPI_RESID = 3,   // out fp32 [M, ld] += acc
  EPI_SWIGLU = 4,  // A tile = 64 gate rows + 64 up rows; out fp16 [M, ld] = silu(g) * u
  EPI_KV_RING = 5,  // scatter K (rotated) / V rows into the bf16 context ring
  EPI_NORM_IN = 6   // a folded RMSNorm's input: xg = fp16(acc * xg_g) and per-tile sums of
                    // squares ssq (GemmEpi); nothing else is written
};

// Element type of both MMA operands (tcgen05 kind::f16 takes A and B of one
// type).  OPND_E4M3: E4M3 weights (one float32 scale per row, GemmAOpts::
// scale) widened to fp16 in shared memory, fp16 tokens (gemm_f8.cu).
enum OperandType : int { OPND_F16 = 0, OPND_BF16 = 1, OPND_E4M3 = 2 };

// TMA descriptors of the weight operand (rows = output features, K inner).
struct GemmAMaps {
  CUtensorMap map[kMaxAMaps];
};

struct GemmAOpts {
  int n_maps;         // descriptors in use
  int tiles_per_map;  // 128-row tiles served by each descriptor (multi-map mode)
  int row_offset;     // first weight row inside each descriptor
  int dual;           // SwiGLU: map[0] gate rows, map[1] up rows, 64-row boxes
  // E4M3 weights: float32 scale of every row of each descriptor's matrix
  // (indexed like its rows, row_offset included); nullptr for fp16 weights
  const float* scale[kMaxAMaps];
};

struct GemmArgs {
  int K;
  int type;         // OperandType of weights and tokens
  int splits;       // K splits per tile
  int cluster;      // 1: the splits of a tile form a cluster and reduce through
                    //    distributed shared memory (splits <= 8)
                    // 0: each split stores an fp32 partial in global memory and the
                    //    last split of the tile (atomic ticket) reduces them
  float* partial;   // [tiles][splits][T][128] when cluster == 0
  int* counters;    // [tiles] when cluster == 0, zero between launches
  int* status;
  // Row scale (see GemmRowScale); rs_ssq == nullptr: none.
  const float* rs_ssq;
  int rs_parts;
  int rs_n;
  float rs_eps;
};

// RMSNorm folded into the GEMM that consumes it.  The residual-add epilogue of
// the GEMM that last updated the fp32 stream x wrote X = fp16(x * g) (the
// norm's gains, GemmEpi::xg) and, per 128-row tile p, the sums over its rows
// of x^2 (GemmEpi::ssq: ssq[p][token]).  The consuming GEMM multiplies every
// accumulator value of token m by rstd(m) = 1 / sqrt(sum_p ssq[p][m] / n +
// eps), which makes its input RMSNorm(x) * g up to rounding.  Used for token
// tiles of at most 32, where a separate RMSNorm launch would cost more than
// the pass's arithmetic.
struct GemmRowScale {
  const float* ssq;  // [parts][M]
  int parts;
  int n;             // row length of the stream (the norm's mean divides by it)
  float eps;
};

struct GemmEpi {
  int kind;
  int M;            // valid token rows
  int N;            // valid output features (SwiGLU: F)
  void* out;
  long long ld;
  // rotary positions
  const int64_t* ctx_len;
  int gamma;
  const float2* rope_cs;  // [M][hd/2] (cos, sin) of token m's position x inv_freq_j; for
                          // EPI_KV_RING nullptr means: computed here from rope_inv
  RopeInv rope_inv;
  int rope_rows;
  int hd;
  // context ring scatter
  void* ring_k;
  void* ring_v;
  int ring_batch;
  int window;
  int n_kv;
  int kv_dim;
  int n_max;
  const int32_t* n_new;
  const int32_t* req_slot;
  int layer0;
  // EPI_RESID (and EPI_NORM_IN, where the "stream" is the accumulator): per
  // weight tile, the sums over its rows of the updated stream's squares,
  // ssq[tile][token], and xg = fp16(stream * xg_g) [M][ld]: the input of the
  // next GEMM, which applies the RMSNorm's rstd (GemmRowScale); or nullptr
  float* ssq;
  __half* xg;
  const float* xg_g;
  // EPI_F32: with out_gather = G > 0 only the MASK rows are written, token t
  // to row (t / G) * (G - 1) + t % G - 1 (t % G == 0 skipped); out may be
  // nullptr when only the top-k partials below are wanted
  int out_gather;
  // EPI_F32 (the LM head): per weight tile and output row, the tile's top
  // tk_k keys (ordered logit << 32 | ~id, descending, 0 = none) at
  // tk_keys[(row * tk_tiles + tile) * tk_slots] and the tile's (max, sum of
  // exp(logit - max)) at tk_ml[row * tk_tiles + tile]; or tk_keys nullptr
  unsigned long long* tk_keys;
  float2* tk_ml;
  int tk_slots;  // 4 or 16
  int tk_k;
  int tk_tiles;
  int* status;      // device status word: argument errors found on the device, and fp16
                    // outputs (or ring entries) beyond the fp16 range (DFLASH_ERR_RANGE)
};

struct GemmScratch {
  float* partial;   // split-K partial tiles of the ticketed reduction
  size_t partial_cap_floats;
  int* counters;    // tickets, zero between launches
  int counters_cap;
  int* status;      // device status word
  int num_sms;      // persistent kernels launch one CTA per SM
};

// Largest K-split count reduced through a cluster; above it the ticketed
// reduction through global memory is used.
#ifndef DFLASH_SPLITK_CLUSTER_MAX
#define DFLASH_SPLITK_CLUSTER_MAX 8
#endif

// TMA descriptor of a row-major matrix of 16-bit elements (OperandType)
// [outer, inner] with a (box_outer x box_inner) box and the 128-byte swizzle.
int encode_2d(CUtensorMap* map, const void* ptr, int type, uint64_t inner, uint64_t outer,
              uint32_t box_inner, uint32_t box_outer);
// The same for a matrix of bytes (E4M3 codes): box_inner bytes (<= 128).
int encode_2d_u8(CUtensorMap* map, const void* ptr, uint64_t inner, uint64_t outer, uint32_t box_inner,
                 uint32_t box_outer);

int gemm_token_tile(int M);
// The token tile launch_gemm takes for n_tiles weight tiles on num_sms SMs.
int gemm_token_tile_for(int M, int n_tiles, int num_sms);
int gemm_plan_splits(int tiles, int K, int target_ctas);

// Y = X W^T through the epilogue.  n_tiles = number of 128-row weight tiles
// (SwiGLU: F / 64).  x: [M, K] row-major, of the same OperandType `type` as
// the weights behind A.
// With rs, every output of token m is scaled by the RMSNorm rstd rs
// describes (token tiles of at most 32 only).
// type OPND_E4M3: the weights behind A are E4M3 codes with ao.scale set, x
// is fp16; the split count is planned by launch_gemm_f8 (`splits` ignored).
int launch_gemm(const GemmAMaps& A, const GemmAOpts& ao, int n_tiles, const void* x, int type,
                int M, int K, const GemmEpi& epi, const GemmScratch& scratch, int splits,
                cudaStream_t s, bool pdl, const GemmRowScale* rs = nullptr);
// E4M3 weights x fp16 tokens (gemm_f8.cu); token tiles of 16, 32, 64 or 128.
int launch_gemm_f8(const GemmAMaps& A, const GemmAOpts& ao, int n_tiles, const void* x, int M, int K,
                   const GemmEpi& epi, const GemmScratch& scratch, cudaStream_t s, bool pdl,
                   const GemmRowScale* rs);
int f8_token_tile(int M);

}  // namespace dfl
