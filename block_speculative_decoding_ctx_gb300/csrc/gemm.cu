// Dense contractions of the drafter on the 5th-generation tensor cores.
//
// Every linear layer of the pass (QKV, O, gate/up, down, LM head, W_c and the
// per-layer context K/V projections) is Y[tokens, rows] = X[tokens, K] W[rows,
// K]^T with few tokens (8 at batch 1) and many weight rows.  The kernel is
// therefore "swap-AB": the weight tile is the 128-row A operand of
// tcgen05.mma, the tokens are the N side (16..256 columns), and the fp32
// accumulator lives in tensor memory as 128 lanes (weight rows) x BN columns
// (tokens).  Operands are fp16 (the drafter's matrices re-encoded exactly,
// activations rounded to 11 significant bits) or bf16 (W_c with the target's
// bf16 features); kind::f16 takes both, A and B of one type.
//
// Pipeline (one CTA = 4 warps, 8 for token tiles of 128 or more):
//   warp 0 lane 0   TMA producer: 128x64 weight box + BNx64 token box per
//                   stage, 128-byte swizzle, weights marked evict-first;
//   warp 1          allocates TMEM; lane 0 issues 4 MMAs (K = 16 each) per
//                   stage and commits the stage back to the producer;
//   warp 2          with a folded RMSNorm, the rstd of the tile's tokens
//                   while the mainloop runs;
//   all warps       epilogue, in groups of 4 (one warp per TMEM lane quarter)
//                   taking alternate 16-token chunks: tcgen05.ld, then the
//                   fused epilogue of the layer (RoPE, residual add with the
//                   next norm's input, SwiGLU, fp32 logits, or scatter into
//                   the context ring).
// Split-K: the grid's z dimension partitions K.  The splits of one tile
// either run as a thread-block cluster (each keeps its fp32 partial tile in
// shared memory and, after a cluster barrier, every CTA of the cluster sums a
// disjoint subset of the tile's tokens over distributed shared memory, in
// split order — deterministic) or store their partials in global memory, the
// last to arrive summing them in split order.
// Many token columns and no split-K: a persistent kernel walks the output
// tiles (gemm_tc_persistent_kernel), by default over CTA pairs
// (gemm_tc_pair_kernel: cta_group::2 MMAs of 256 weight rows, the token tile
// split between the pair's shared memories).
// All waits are bounded (see mbar_wait_bounded).
#include <cudaTypedefs.h>

#include <mutex>

#include "gemm_kernels.cuh"

// Persistent GEMMs over CTA pairs (cta_group::2) instead of single CTAs.
#ifndef DFLASH_GEMM_PAIR
#define DFLASH_GEMM_PAIR 1
#endif

namespace dfl {
namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
}  // namespace

int encode_2d(CUtensorMap* map, const void* ptr, int type, uint64_t inner, uint64_t outer,
              uint32_t box_inner, uint32_t box_outer) {
  std::call_once(g_encode_once, [] {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!g_encode) return DFLASH_ERR_CUDA;
  if ((reinterpret_cast<uintptr_t>(ptr) & 15) || (inner * 2) % 16) return DFLASH_ERR_ALIGN;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType dt =
      type == OPND_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUresult r = g_encode(map, dt, 2, const_cast<void*>(ptr), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DFLASH_OK : DFLASH_ERR_CUDA;
}

int encode_2d_u8(CUtensorMap* map, const void* ptr, uint64_t inner, uint64_t outer, uint32_t box_inner,
                 uint32_t box_outer) {
  std::call_once(g_encode_once, [] {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!g_encode) return DFLASH_ERR_CUDA;
  if ((reinterpret_cast<uintptr_t>(ptr) & 15) || inner % 16) return DFLASH_ERR_ALIGN;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box,
                        estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DFLASH_OK : DFLASH_ERR_CUDA;
}

int gemm_token_tile(int M) {
  if (M <= 16) return 16;
  if (M <= 32) return 32;
  if (M <= 64) return 64;
  // the tokens cut into equal tiles of at most 256, rounded up to 16 (an MMA
  // N): no tile is mostly padding (224 tokens take one 224-wide tile, not 256)
  const int m_tiles = (M + 255) / 256;
  const int per = (M + m_tiles - 1) / m_tiles;
  return (per + 15) / 16 * 16;
}

// A GEMM with fewer weight tiles than SMs whose wide token tile would take
// exactly two K splits takes two token tiles per weight tile instead: the same
// CTA count, no partials to reduce.
#ifndef DFLASH_TOKEN_SPLIT
#define DFLASH_TOKEN_SPLIT 1
#endif
int gemm_token_tile_for(int M, int n_tiles, int num_sms) {
  const int T0 = gemm_token_tile(M);
  if (!DFLASH_TOKEN_SPLIT || T0 <= 128 || n_tiles < 1) return T0;
  const int m0 = (M + T0 - 1) / T0;
  if (num_sms / (n_tiles * m0) != 2) return T0;
  const int per = (M + 2 * m0 - 1) / (2 * m0);
  return (per + 15) / 16 * 16;
}

int gemm_plan_splits(int tiles, int K, int target_ctas) {
  const int kb = (K + kBK - 1) / kBK;
  // as many splits as fit in one wave of CTA slots: a second, mostly empty
  // wave would cost a whole extra CTA lifetime
  int s = target_ctas / tiles;
  const int max_s = kb / 4 > 0 ? kb / 4 : 1;  // at least 4 k-blocks per split
  if (s > max_s) s = max_s;
  if (s < 1) s = 1;
  return s;
}

int launch_gemm(const GemmAMaps& A, const GemmAOpts& ao, int n_tiles, const void* x, int type,
                int M, int K, const GemmEpi& epi, const GemmScratch& scratch, int splits,
                cudaStream_t s, bool pdl, const GemmRowScale* rs) {
  if (type == OPND_E4M3) return launch_gemm_f8(A, ao, n_tiles, x, M, K, epi, scratch, s, pdl, rs);
  const int BN = gemm_token_tile_for(M, n_tiles, scratch.num_sms);
  const int T = BN;
  if (rs && (T > 32 || !rs->ssq || rs->parts < 1 || rs->n < 1)) return DFLASH_ERR_UNSUPPORTED;
  CUtensorMap tmB;
  int rc = encode_2d(&tmB, x, type, (uint64_t)K, (uint64_t)M, kBK, (uint32_t)T);
  if (rc) return rc;
  const int m_tiles = (M + T - 1) / T;
  const int kb = (K + kBK - 1) / kBK;
  if (splits < 1) splits = 1;
  if (splits > kb) splits = kb;
  const size_t tiles = (size_t)n_tiles * m_tiles;
  const size_t per_split = (size_t)T * 128;
  // Measured on GB300: with small token tiles (8-16 tokens, partials of
  // 4-8 KiB) the ticketed reduction wins — non-last splits leave at once;
  // with 32+ token tiles the partials are large and the cluster reduction
  // through distributed shared memory wins.
  const bool cluster = splits > 1 && splits <= DFLASH_SPLITK_CLUSTER_MAX && T >= 32;
  if (splits > 1 && !cluster) {
    if (tiles > (size_t)scratch.counters_cap || !scratch.partial) splits = 1;
    while (splits > 1 && tiles * splits * per_split > scratch.partial_cap_floats) --splits;
  }
  GemmArgs args;
  args.K = K;
  args.type = type;
  args.splits = splits;
  args.cluster = cluster ? 1 : 0;
  args.partial = scratch.partial;
  args.counters = scratch.counters;
  args.status = scratch.status;
  args.rs_ssq = rs ? rs->ssq : nullptr;
  args.rs_parts = rs ? rs->parts : 0;
  args.rs_n = rs ? rs->n : 0;
  args.rs_eps = rs ? rs->eps : 0.0f;
  // many token columns and no split-K: the persistent kernel
  const bool persistent = !rs && splits == 1 && T >= 64 && (size_t)n_tiles * m_tiles >= (size_t)scratch.num_sms;
  dim3 grid(n_tiles, m_tiles, splits);
  if (persistent && DFLASH_GEMM_PAIR && BN >= 80) {
    CUtensorMap tmBh;
    rc = encode_2d(&tmBh, x, type, (uint64_t)K, (uint64_t)M, kBK, (uint32_t)(T / 2));
    if (rc) return rc;
    return launch_tile_pair(BN, A, tmBh, ao, args, epi, n_tiles, m_tiles, scratch.num_sms, s, pdl);
  }
  if (BN >= 80) {
    auto unit = BN >= 240   ? launch_tile_240
                : BN >= 208 ? launch_tile_208
                : BN >= 176 ? launch_tile_176
                : BN >= 144 ? launch_tile_144
                : BN >= 112 ? launch_tile_112
                            : launch_tile_080;
    return unit(BN, persistent, A, tmB, ao, args, epi, grid, n_tiles, m_tiles, scratch.num_sms, s, pdl);
  }
  switch (BN) {
#define DFL_ONE(bn, st) \
  case bn: return launch_one<bn, st>(A, tmB, ao, args, epi, grid, s, pdl);
    DFL_TILE_CASES_ONE(DFL_ONE)
#undef DFL_ONE
    default: return DFLASH_ERR_UNSUPPORTED;
  }
}

}  // namespace dfl
