// tcgen05 GEMM instantiations for token tiles of 80 and 96.
#define DFL_UNIT_NAME launch_tile_080
#define DFL_UNIT_CASES(X) X(80, 6) X(96, 6)
#include "gemm_tiles_unit.cuh"
