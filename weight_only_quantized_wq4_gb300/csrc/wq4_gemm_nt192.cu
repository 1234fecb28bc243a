// GEMM instantiations for a token tile of 192.
#include "wq4_gemm.cuh"
#include "wq4_launch.h"

namespace wq4 {

template <bool GROUPED, bool BF16, int QT, bool ATMEM, int H>
static cudaError_t go(const void* p, int grid, bool pdl, cudaStream_t st) {
    constexpr int MAXP = GROUPED ? kMaxGroupedProblems : 1;
    return launch_gemm<192, BF16, QT, MAXP, ATMEM, H>(*static_cast<const GemmParams<MAXP>*>(p), grid, pdl, st);
}

template <bool GROUPED, bool BF16, int QT, int H>
static cudaError_t pick_a(const void* p, bool a_tmem, int grid, bool pdl, cudaStream_t st) {
    return a_tmem ? go<GROUPED, BF16, QT, true, H>(p, grid, pdl, st) : go<GROUPED, BF16, QT, false, H>(p, grid, pdl, st);
}

template <bool GROUPED, bool BF16, int H>
static cudaError_t pick_q(const void* p, int qt, bool a_tmem, int grid, bool pdl, cudaStream_t st) {
    switch (qt) {
        case kQtU4B8: return pick_a<GROUPED, BF16, kQtU4B8, H>(p, a_tmem, grid, pdl, st);
        case kQtU4Zp: return pick_a<GROUPED, BF16, kQtU4Zp, H>(p, a_tmem, grid, pdl, st);
        default:   // float zeros: single-problem calls only (the activation sums are per call)
            if constexpr (GROUPED) return cudaErrorInvalidValue;
            else return pick_a<GROUPED, BF16, kQtU4FZp, H>(p, a_tmem, grid, pdl, st);
    }
}

template <int H>
static cudaError_t pick_h(const void* params, bool grouped, bool bf16, int qt, bool a_tmem, int grid, bool pdl,
                          cudaStream_t st) {
    if (grouped) return bf16 ? pick_q<true, true, H>(params, qt, a_tmem, grid, pdl, st) : pick_q<true, false, H>(params, qt, a_tmem, grid, pdl, st);
    return bf16 ? pick_q<false, true, H>(params, qt, a_tmem, grid, pdl, st) : pick_q<false, false, H>(params, qt, a_tmem, grid, pdl, st);
}

// scale_sets: 2 for a group size of 64 (not at this token tile: its partials would not fit in tensor memory)
cudaError_t launch_gemm_nt192(const void* params, bool grouped, bool bf16, int qt, bool a_tmem, int scale_sets,
                             int grid, bool pdl, cudaStream_t st) {
    if (scale_sets != 1) return cudaErrorInvalidValue;
    return pick_h<1>(params, grouped, bf16, qt, a_tmem, grid, pdl, st);
}

}  // namespace wq4
