// Weight-streaming GEMM over E4M3 (FP8) drafter weights with fp16 activations.
//
// Y[tokens, rows] = X W^T with W stored as E4M3 codes and one float32 scale
// per weight row (see dflash_quantize_e4m3).  At small batch the draft pass
// is bound by the bytes of its weights; E4M3 halves them.  The activations
// stay fp16 (an E4M3 activation would keep 4 significant bits), so the
// tensor cores still run kind::f16: converter warps widen each weight stage
// to fp16 into tensor memory (every E4M3 value is exactly an fp16 value; one
// weight row per TMEM lane), the MMAs take their A operand from there, and
// the epilogue multiplies each accumulator row by its weight row's scale.
// Keeping the widened weights out of shared memory leaves it to the E4M3
// stages in flight from HBM.
//
// One CTA = 8 warps per (weight tile, token tile, K split):
//   warp 0 lane 0   TMA producer: a 128-row x 128-byte E4M3 box (128 K
//                   elements) and the matching two 64-deep token boxes per
//                   stage, 128-byte swizzle, weights marked evict-first;
//   warp 1          allocates TMEM; lane 0 issues 4 MMAs (K = 16 each) per
//                   64-deep fp16 slot and commits slots and stages back;
//   warp 2          with a folded RMSNorm, the rstd of the tile's tokens;
//   warps 4-7       converters: thread t widens weight row t of each stage,
//                   16 codes per 16-byte load, into a ring of 64-deep fp16
//                   slots in tensor memory (lane t, 32 columns per slot);
//   all warps       epilogue in two groups (one_tile_epilogue), with split-K
//                   reduced by ticket or inside a cluster as in gemm.cu.
// Every wait is bounded (mbar_wait_bounded).
#include <cuda_fp8.h>

#include "gemm_kernels.cuh"

namespace dfl {
namespace {

constexpr int kBK8 = 128;                 // K elements (bytes) of one E4M3 weight row per stage
constexpr int kA8Bytes = 128 * kBK8;      // E4M3 weight box per stage (16 KiB)
constexpr int kSlotCols = kBK / 2;        // TMEM columns of one 64-deep fp16 slot (2 per column)

// Shape per token-tile width: two CTAs share an SM up to 32 tokens.  The
// widened fp16 slots live in tensor memory, so shared memory holds only the
// E4M3 stages in flight (and their token boxes).  Measured at batch 1 (full
// dimensions) with the slots in shared memory instead: two CTAs per SM with
// three stages and two slots streamed the pass's E4M3 weights at 2.8 TB/s,
// one CTA per SM with nine stages and two slots at 1.8 TB/s — the converters
// waited on the slots' round trip through the tensor cores.
template <int BN>
struct F8Shape {
  static constexpr bool kTwo = BN <= 32;      // two CTAs per SM
  static constexpr int kBBytes = BN * kBK * 2;
  static constexpr int kStage = kA8Bytes + 2 * kBBytes;
  static constexpr int S = kTwo ? 100 * 1024 / kStage : 192 * 1024 / kStage;  // E4M3 stages
  static constexpr int NC = 6;                // fp16 slots in tensor memory
  static constexpr int kAccCols = BN < 32 ? 32 : BN;
  static constexpr uint32_t kTmemCols = tmem_cols(kAccCols + NC * kSlotCols);
  static constexpr size_t smem = (size_t)S * kStage + 1024;
  static_assert(!kTwo || kTmemCols <= 256, "two CTAs per SM share the 512 TMEM columns");
};

// Dequantization scale of this thread's weight row (row r of tile tile_n),
// 0 for rows beyond the matrix.
__device__ __forceinline__ float weight_row_scale(const GemmAOpts& ao, const GemmEpi& epi, int tile_n,
                                                  int r) {
  if (ao.dual) {
    const int f = tile_n * 64 + (r & 63);
    return f < epi.N ? __ldg(ao.scale[r >> 6] + ao.row_offset + f) : 0.0f;
  }
  const int map = tile_n / ao.tiles_per_map;
  const int local = (tile_n % ao.tiles_per_map) * 128 + r;
  if (ao.n_maps == 1 && local >= epi.N) return 0.0f;
  return __ldg(ao.scale[map] + ao.row_offset + local);
}

// 16 E4M3 codes -> 16 fp16 values (two 16-byte chunks).
__device__ __forceinline__ void widen16(const uint4 c, uint4& lo, uint4& hi) {
  auto two = [](uint32_t w) -> uint32_t {
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w & 0xFFFFu), __NV_E4M3);
    return (uint32_t)h.x | ((uint32_t)h.y << 16);
  };
  lo = make_uint4(two(c.x), two(c.x >> 16), two(c.y), two(c.y >> 16));
  hi = make_uint4(two(c.z), two(c.z >> 16), two(c.w), two(c.w >> 16));
}

// Up to 32 tokens two CTAs share an SM: 128 registers per thread at most.
template <int BN>
__global__ void __launch_bounds__(256, BN <= 32 ? 2 : 1)
    gemm_f8_kernel(const __grid_constant__ GemmAMaps A, const __grid_constant__ CUtensorMap tmB,
                   const GemmAOpts ao, const GemmArgs args, const GemmEpi epi) {
  using Sh = F8Shape<BN>;
  constexpr int S = Sh::S, NC = Sh::NC;
  constexpr int kBBytes = Sh::kBBytes, kStage = Sh::kStage;
  constexpr uint32_t kTmemCols = Sh::kTmemCols;
  static_assert(kStage % 1024 == 0, "stage buffers must keep 1024-byte alignment");
  static_assert((BN + 64) * 128 * 4 <= S * kStage,
                "split partials and exchange buffers must fit the stage buffers");

  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[S];
  __shared__ __align__(8) uint64_t empty_bar[S];
  __shared__ __align__(8) uint64_t cfull_bar[NC];   // fp16 slot written to tensor memory
  __shared__ __align__(8) uint64_t cempty_bar[NC];  // fp16 slot consumed by the MMAs
  __shared__ __align__(8) uint64_t acc_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  __shared__ int last_sh;
  __shared__ float rs_sh[BN <= 32 ? 32 : 1];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile_n = blockIdx.x, tile_m = blockIdx.y, split = blockIdx.z;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int kb_total = (args.K + kBK8 - 1) / kBK8;
  const int kb0 = (int)((long long)split * kb_total / args.splits);
  const int kb1 = (int)((long long)(split + 1) * kb_total / args.splits);
  const int nkb = kb1 - kb0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int c = 0; c < NC; ++c) {
      mbar_init(&cfull_bar[c], 4);
      mbar_init(&cempty_bar[c], 1);
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
  const uint32_t tmem = tmem_base_sh;           // accumulator at columns 0 .. BN - 1
  const uint32_t tslot = tmem + Sh::kAccCols;    // fp16 slot c at tslot + c * kSlotCols
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
    auto load_a = [&](int i, int s) {
      uint8_t* sa = smem + s * kStage;
      const int kc = (kb0 + i) * kBK8;
      if (ao.dual) {
        tma_load_2d(sa, &A.map[0], &full_bar[s], kc, row0, pol_w);
        tma_load_2d(sa + 64 * 128, &A.map[1], &full_bar[s], kc, row0, pol_w);
      } else {
        tma_load_2d(sa, &A.map[map_i], &full_bar[s], kc, row0, pol_w);
      }
    };
    auto load_b = [&](int i, int s) {
      uint8_t* sb = smem + s * kStage + kA8Bytes;
      const int kc = (kb0 + i) * kBK8;
      tma_load_2d(sb, &tmB, &full_bar[s], kc, tok0, pol_x);
      tma_load_2d(sb + kBBytes, &tmB, &full_bar[s], kc + kBK, tok0, pol_x);
    };
    // weights do not depend on the previous kernel: stream them first
    const int pre = nkb < S ? nkb : S;
    for (int i = 0; i < pre; ++i) {
      mbar_arrive_expect_tx(&full_bar[i], kStage);
      load_a(i, i);
    }
    grid_dependency_wait();
    for (int i = 0; i < pre; ++i) load_b(i, i);
    issued = pre;
    for (int i = pre; i < nkb; ++i) {
      const int s = i % S;
      const uint32_t ph = (uint32_t)(i / S) & 1u;
      if (!mbar_wait_bounded(&empty_bar[s], ph ^ 1u, &abort_sh, args.status)) break;
      mbar_arrive_expect_tx(&full_bar[s], kStage);
      load_a(i, s);
      load_b(i, s);
      issued = i + 1;
    }
  } else if (warp == 1 && lane == 0) {
    // --------------------------------------------------------- MMA issuer
    const uint32_t idesc = idesc_f32acc(128, BN, false);
    for (int i = 0; i < nkb && !abort_sh; ++i) {
      const int s = i % S;
      if (!mbar_wait_bounded(&full_bar[s], (uint32_t)(i / S) & 1u, &abort_sh, args.status)) break;
      bool ok = true;
      for (int h = 0; h < 2; ++h) {
        const int n = 2 * i + h, c = n % NC;
        if (!mbar_wait_bounded(&cfull_bar[c], (uint32_t)(n / NC) & 1u, &abort_sh, args.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a_col = tslot + (uint32_t)(c * kSlotCols);
        const uint32_t b_addr = smem_u32(smem + s * kStage + kA8Bytes + h * kBBytes);
#pragma unroll
        for (int k = 0; k < kBK / 16; ++k)
          tc_mma_f16_ta(tmem, a_col + k * 8, smem_desc_sw128(b_addr + k * 32), idesc, (i | h | k) ? 1u : 0u);
        tc_commit(&cempty_bar[c]);
      }
      if (!ok) break;
      tc_commit(&empty_bar[s]);
    }
    tc_commit(&acc_bar);
  } else if (warp >= 4) {
    // ---------------------------------------------------------- converters
    // thread t owns weight row t (TMEM lane t: warp w reaches lanes
    // 32 (w % 4) .. + 31): its E4M3 row (128 bytes, 16-byte chunk j stored at
    // chunk j ^ (t % 8) of the row) becomes, per 64-deep half, 32 columns of
    // fp16 pairs in K order
    const int t = threadIdx.x - 128;
    const uint32_t sw = (uint32_t)(t & 7);
    const uint32_t row_off = (uint32_t)(t >> 3) * 1024u + sw * 128u;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    for (int i = 0; i < nkb; ++i) {
      const int s = i % S;
      if (!mbar_wait_bounded(&full_bar[s], (uint32_t)(i / S) & 1u, &abort_sh, args.status)) break;
      const uint8_t* a8 = smem + s * kStage + row_off;
      bool ok = true;
      for (int h = 0; h < 2; ++h) {
        const int n = 2 * i + h, c = n % NC;
        if (!mbar_wait_bounded(&cempty_bar[c], ((uint32_t)(n / NC) & 1u) ^ 1u, &abort_sh, args.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // the half's four 16-code chunks, loaded together, widened into two
        // 16-column stores (register arrays indexed by constants only)
        const uint32_t j0 = (uint32_t)(h * 4);
        const uint4 r0 = *reinterpret_cast<const uint4*>(a8 + (((j0 + 0u) ^ sw) << 4));
        const uint4 r1 = *reinterpret_cast<const uint4*>(a8 + (((j0 + 1u) ^ sw) << 4));
        const uint4 r2 = *reinterpret_cast<const uint4*>(a8 + (((j0 + 2u) ^ sw) << 4));
        const uint4 r3 = *reinterpret_cast<const uint4*>(a8 + (((j0 + 3u) ^ sw) << 4));
        uint4 l0, h0, l1, h1, l2, h2, l3, h3;
        widen16(r0, l0, h0);
        widen16(r1, l1, h1);
        widen16(r2, l2, h2);
        widen16(r3, l3, h3);
        const uint32_t w0[16] = {l0.x, l0.y, l0.z, l0.w, h0.x, h0.y, h0.z, h0.w,
                                 l1.x, l1.y, l1.z, l1.w, h1.x, h1.y, h1.z, h1.w};
        const uint32_t w1[16] = {l2.x, l2.y, l2.z, l2.w, h2.x, h2.y, h2.z, h2.w,
                                 l3.x, l3.y, l3.z, l3.w, h3.x, h3.y, h3.z, h3.w};
        const uint32_t dst = tslot + lane_base + (uint32_t)(c * kSlotCols);
        tmem_st_x16(dst, w0);
        tmem_st_x16(dst + 16, w1);
        tc_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&cfull_bar[c]);
      }
      if (!ok) break;
    }
  } else if (BN <= 32 && warp == 2 && args.rs_ssq) {
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
  __syncwarp();

  // ----------------------------------------------------------- epilogue
  const bool acc_ok = mbar_wait_bounded(&acc_bar, 0, &abort_sh, args.status);
  tc_fence_after();
  if (warp == 0 && lane == 0 && abort_sh) {
    // a wait gave up: let this CTA's copies in flight land before exiting
    int dummy = 0;
    for (int i = (issued > S ? issued - S : 0); i < issued; ++i)
      (void)mbar_wait_bounded(&full_bar[i % S], (uint32_t)(i / S) & 1u, &dummy, nullptr, 100000000ull);
  }
  __syncthreads();
  const float wscale = weight_row_scale(ao, epi, tile_n, (warp & 3) * 32 + lane);
  one_tile_epilogue<BN, 2>(smem, S * kStage, tmem, abort_sh != 0 || !acc_ok, ao, args, epi, tile_n, tile_m, split,
                           (BN <= 32 && args.rs_ssq) ? rs_sh : nullptr, &last_sh, wscale);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

template <int BN>
int launch_f8(const GemmAMaps& A, const CUtensorMap& tmB, const GemmAOpts& ao, const GemmArgs& args,
              const GemmEpi& epi, dim3 grid, cudaStream_t s, bool pdl) {
  auto kern = gemm_f8_kernel<BN>;
  constexpr size_t smem = F8Shape<BN>::smem;
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return DFLASH_ERR_LAUNCH;
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  if (args.splits > 1 && args.cluster) {
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

}  // namespace

int f8_token_tile(int M) {
  if (M <= 16) return 16;
  if (M <= 32) return 32;
  if (M <= 64) return 64;
  return 128;
}

int launch_gemm_f8(const GemmAMaps& A, const GemmAOpts& ao, int n_tiles, const void* x, int M, int K,
                   const GemmEpi& epi, const GemmScratch& scratch, cudaStream_t s, bool pdl,
                   const GemmRowScale* rs) {
  const int BN = f8_token_tile(M);
  if (rs && (BN > 32 || !rs->ssq || rs->parts < 1 || rs->n < 1)) return DFLASH_ERR_UNSUPPORTED;
  if (!ao.scale[0] || (ao.dual && !ao.scale[1])) return DFLASH_ERR_ARG;
  CUtensorMap tmB;
  int rc = encode_2d(&tmB, x, OPND_F16, (uint64_t)K, (uint64_t)M, kBK, (uint32_t)BN);
  if (rc) return rc;
  const int m_tiles = (M + BN - 1) / BN;
  const int kb = (K + kBK8 - 1) / kBK8;
  const size_t tiles = (size_t)n_tiles * m_tiles;
  // one wave of CTA slots (two CTAs per SM up to 32 tokens), at least two
  // 128-deep k-blocks per split
  const int per_sm = BN <= 32 ? 2 : 1;
  int splits = (int)((size_t)scratch.num_sms * per_sm / tiles);
  const int max_s = kb / 2 > 0 ? kb / 2 : 1;
  if (splits > max_s) splits = max_s;
  if (splits < 1) splits = 1;
  const bool cluster = splits > 1 && splits <= DFLASH_SPLITK_CLUSTER_MAX && BN >= 32;
  const size_t per_split = (size_t)BN * 128;
  if (splits > 1 && !cluster) {
    if (tiles > (size_t)scratch.counters_cap || !scratch.partial) splits = 1;
    while (splits > 1 && tiles * splits * per_split > scratch.partial_cap_floats) --splits;
  }
  GemmArgs args;
  args.K = K;
  args.type = OPND_F16;
  args.splits = splits;
  args.cluster = (splits > 1 && cluster) ? 1 : 0;
  args.partial = scratch.partial;
  args.counters = scratch.counters;
  args.status = scratch.status;
  args.rs_ssq = rs ? rs->ssq : nullptr;
  args.rs_parts = rs ? rs->parts : 0;
  args.rs_n = rs ? rs->n : 0;
  args.rs_eps = rs ? rs->eps : 0.0f;
  const dim3 grid(n_tiles, m_tiles, splits);
  switch (BN) {
    case 16: return launch_f8<16>(A, tmB, ao, args, epi, grid, s, pdl);
    case 32: return launch_f8<32>(A, tmB, ao, args, epi, grid, s, pdl);
    case 64: return launch_f8<64>(A, tmB, ao, args, epi, grid, s, pdl);
    case 128: return launch_f8<128>(A, tmB, ao, args, epi, grid, s, pdl);
    default: return DFLASH_ERR_UNSUPPORTED;
  }
}

}  // namespace dfl
