// Internal interface of the tcgen05 GEMM (gemm.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dflash.h"

namespace dfl {

constexpr int kMaxAMaps = 8;

enum EpiKind : int {
  EPI_F32 = 0,     // out fp32 [M, ld] = acc
  EPI_BF16 = 1,    // out bf16 [M, ld] = acc
  EPI_QKV = 2,     // out bf16 [M, ld]; rows < rope_rows rotated at pos = ctx_len[m/gamma] + m%gamma
  EPI_RESID = 3,   // out fp32 [M, ld] += acc
  EPI_SWIGLU = 4,  // A tile = 64 gate rows + 64 up rows; out bf16 [M, ld] = silu(g) * u
  EPI_KV_RING = 5  // scatter K (rotated) / V rows into the context ring
};

// TMA descriptors of the weight operand (rows = output features, K inner).
struct GemmAMaps {
  CUtensorMap map[kMaxAMaps];
};

struct GemmAOpts {
  int n_maps;         // descriptors in use
  int tiles_per_map;  // 128-row tiles served by each descriptor (multi-map mode)
  int row_offset;     // first weight row inside each descriptor
  int dual;           // SwiGLU: map[0] gate rows, map[1] up rows, 64-row boxes
  int split;          // token operand is [2M, K]: rows [0, M) bf16 hi parts, rows [M, 2M) the
                      // bf16 remainders (x - hi); a tile of BN columns holds BN/2 tokens as
                      // (hi, lo) column pairs and the epilogue adds them
};

struct GemmArgs {
  int K;
  int splits;       // K splits per tile
  int cluster;      // 1: the splits of a tile form a cluster and reduce through
                    //    distributed shared memory (splits <= 8)
                    // 0: each split stores an fp32 partial in global memory and the
                    //    last split of the tile (atomic ticket) reduces them
  float* partial;   // [tiles][splits][T][128] when cluster == 0
  int* counters;    // [tiles] when cluster == 0, zero between launches
  int* status;
};

struct GemmEpi {
  int kind;
  int M;            // valid token rows
  int N;            // valid output features (SwiGLU: F)
  void* out;
  long long ld;
  void* out_lo;     // EPI_BF16 / EPI_QKV / EPI_SWIGLU: bf16 remainder x - bf16(x) is written
                    // here too ([M, ld_lo]; EPI_QKV: only the rope_rows_lo first columns)
  long long ld_lo;
  int lo_cols;      // EPI_QKV: columns [0, lo_cols) get a remainder
  // rotary positions
  const int64_t* ctx_len;
  int gamma;
  float2 rope_inv[64];  // inv_freq_j = theta^(-2j/hd) as a float pair (hi, lo), j < hd/2
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
  int* status;      // device status word for argument errors found on the device
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

// TMA descriptor of a row-major bf16 matrix [outer, inner] with a
// (box_outer x box_inner) box and the 128-byte swizzle.
int encode_bf16_2d(CUtensorMap* map, const void* ptr, uint64_t inner, uint64_t outer,
                   uint32_t box_inner, uint32_t box_outer);

int gemm_token_tile(int M);
int gemm_plan_splits(int tiles, int K, int target_ctas);

// Y = X W^T through the epilogue.  n_tiles = number of 128-row weight tiles
// (SwiGLU: F / 64).  x: bf16 [M, K] row-major, or [2M, K] (hi rows then
// remainder rows) when ao.split.
int launch_gemm(const GemmAMaps& A, const GemmAOpts& ao, int n_tiles, const void* x, int M, int K,
                const GemmEpi& epi, const GemmScratch& scratch, int splits, cudaStream_t s,
                bool pdl);

}  // namespace dfl
