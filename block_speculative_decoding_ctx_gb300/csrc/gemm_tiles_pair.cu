// Instantiations of the CTA-pair (cta_group::2) persistent GEMM for the wider
// token-tile widths (see gemm.cu); a translation unit of their own so that
// they compile in parallel with the rest.
#include "gemm_kernels.cuh"

namespace dfl {

int launch_tile_pair(int BN, const GemmAMaps& A, const CUtensorMap& tmB_half, const GemmAOpts& ao,
                     const GemmArgs& args, const GemmEpi& epi, int n_tiles, int m_tiles, int num_sms,
                     cudaStream_t s, bool pdl) {
  switch (BN) {
#define DFL_Q(bn, st) \
  case bn: return launch_pair<bn, st>(A, tmB_half, ao, args, epi, n_tiles, m_tiles, num_sms, s, pdl);
    DFL_PAIR_CASES(DFL_Q)
#undef DFL_Q
    default: return DFLASH_ERR_UNSUPPORTED;
  }
}

}  // namespace dfl
