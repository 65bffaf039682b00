// tcgen05 GEMM instantiations for token tiles of 112 and 128.
#define DFL_UNIT_NAME launch_tile_112
#define DFL_UNIT_CASES(X) X(112, 6) X(128, 6)
#include "gemm_tiles_unit.cuh"
