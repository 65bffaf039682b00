// tcgen05 GEMM instantiations for token tiles of 144 and 160.
#define DFL_UNIT_NAME launch_tile_144
#define DFL_UNIT_CASES(X) X(144, 5) X(160, 5)
#include "gemm_tiles_unit.cuh"
