// tcgen05 GEMM instantiations for token tiles of 176 and 192.
#define DFL_UNIT_NAME launch_tile_176
#define DFL_UNIT_CASES(X) X(176, 5) X(192, 4)
#include "gemm_tiles_unit.cuh"
