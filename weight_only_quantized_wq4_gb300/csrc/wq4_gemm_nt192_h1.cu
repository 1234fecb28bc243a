// GEMM instantiations for a token tile of 192 with 1 scale set per 128-K record.
#include "wq4_gemm_unit.cuh"

WQ4_GEMM_UNIT(192, 1)
