// tcgen05 GEMM instantiations for token tiles of 208 and 224.
#define DFL_UNIT_NAME launch_tile_208
#define DFL_UNIT_CASES(X) X(208, 4) X(224, 4)
#include "gemm_tiles_unit.cuh"
