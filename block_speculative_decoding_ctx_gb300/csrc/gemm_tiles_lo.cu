// Instantiations of the tcgen05 GEMMs for the middle token-tile widths
// (see gemm.cu); a translation unit of their own so that they compile in
// parallel with the rest.
#include "gemm_kernels.cuh"

namespace dfl {

int launch_tile_lo(int BN, bool persistent, const GemmAMaps& A, const CUtensorMap& tmB,
                   const GemmAOpts& ao, const GemmArgs& args, const GemmEpi& epi, dim3 grid,
                   int n_tiles, int m_tiles, int num_sms, cudaStream_t s, bool pdl) {
  if (persistent) {
    switch (BN) {
#define DFL_P(bn, st) \
  case bn: return launch_persistent<bn, st>(A, tmB, ao, args, epi, n_tiles, m_tiles, num_sms, s, pdl);
      DFL_TILE_CASES_LO(DFL_P)
#undef DFL_P
      default: break;
    }
  }
  switch (BN) {
#define DFL_O(bn, st) \
  case bn: return launch_one<bn, st>(A, tmB, ao, args, epi, grid, s, pdl);
    DFL_TILE_CASES_LO(DFL_O)
#undef DFL_O
    default: return DFLASH_ERR_UNSUPPORTED;
  }
}

}  // namespace dfl
