// GEMM instantiations for a token tile of 16.
#include "wq4_gemm.cuh"
#include "wq4_launch.h"

namespace wq4 {

template <bool GROUPED, bool BF16, bool ZP, bool ATMEM>
static cudaError_t go(const void* p, int grid, bool pdl, cudaStream_t st) {
    constexpr int MAXP = GROUPED ? kMaxGroupedProblems : 1;
    return launch_gemm<16, BF16, ZP, MAXP, ATMEM>(*static_cast<const GemmParams<MAXP>*>(p), grid, pdl, st);
}

template <bool GROUPED, bool BF16, bool ZP>
static cudaError_t pick_a(const void* p, bool a_tmem, int grid, bool pdl, cudaStream_t st) {
    return a_tmem ? go<GROUPED, BF16, ZP, true>(p, grid, pdl, st) : go<GROUPED, BF16, ZP, false>(p, grid, pdl, st);
}

template <bool GROUPED>
static cudaError_t pick_types(const void* p, bool bf16, bool zp, bool a_tmem, int grid, bool pdl, cudaStream_t st) {
    if (bf16) return zp ? pick_a<GROUPED, true, true>(p, a_tmem, grid, pdl, st) : pick_a<GROUPED, true, false>(p, a_tmem, grid, pdl, st);
    return zp ? pick_a<GROUPED, false, true>(p, a_tmem, grid, pdl, st) : pick_a<GROUPED, false, false>(p, a_tmem, grid, pdl, st);
}

cudaError_t launch_gemm_nt16(const void* params, bool grouped, bool bf16, bool zp, bool a_tmem, int grid,
                             bool pdl, cudaStream_t st) {
    return grouped ? pick_types<true>(params, bf16, zp, a_tmem, grid, pdl, st)
                   : pick_types<false>(params, bf16, zp, a_tmem, grid, pdl, st);
}

}  // namespace wq4
