// Body of one translation unit of tcgen05 GEMM instantiations: the unit
// defines DFL_UNIT_NAME (the launcher's name) and DFL_UNIT_CASES(X) (its
// token-tile widths and stage counts) and includes this file.  Each unit
// holds two widths so that the widths compile in parallel.
#include "gemm_kernels.cuh"

namespace dfl {

int DFL_UNIT_NAME(int BN, bool persistent, const GemmAMaps& A, const CUtensorMap& tmB,
                  const GemmAOpts& ao, const GemmArgs& args, const GemmEpi& epi, dim3 grid,
                  int n_tiles, int m_tiles, int num_sms, cudaStream_t s, bool pdl) {
  if (persistent) {
    switch (BN) {
#define DFL_P(bn, st) \
  case bn: return launch_persistent<bn, st>(A, tmB, ao, args, epi, n_tiles, m_tiles, num_sms, s, pdl);
      DFL_UNIT_CASES(DFL_P)
#undef DFL_P
      default: break;
    }
  }
  switch (BN) {
#define DFL_O(bn, st) \
  case bn: return launch_one<bn, st>(A, tmB, ao, args, epi, grid, s, pdl);
    DFL_UNIT_CASES(DFL_O)
#undef DFL_O
    default: return DFLASH_ERR_UNSUPPORTED;
  }
}

}  // namespace dfl
