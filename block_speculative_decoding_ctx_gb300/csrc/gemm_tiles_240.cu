// tcgen05 GEMM instantiations for token tiles of 240 and 256.
#define DFL_UNIT_NAME launch_tile_240
#define DFL_UNIT_CASES(X) X(240, 4) X(256, 4)
#include "gemm_tiles_unit.cuh"
