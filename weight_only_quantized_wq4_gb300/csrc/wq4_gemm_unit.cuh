// One GEMM translation unit: the instantiations of a token tile NT and a scale-set count H, and
// their launcher launch_gemm_unit<NT, H> (every activation type, weight format, operand source
// and problem-table size). Each wq4_gemm_nt*_h*.cu file includes this and instantiates one pair,
// so that the pairs compile in parallel.
#pragma once

#include "wq4_gemm.cuh"
#include "wq4_launch.h"

namespace wq4 {

template <int NT, int H, bool GROUPED, bool BF16, int QT, bool ATMEM>
cudaError_t unit_go(const void* p, int grid, bool pdl, cudaStream_t st) {
    constexpr int MAXP = GROUPED ? kMaxGroupedProblems : 1;
    return launch_gemm<NT, BF16, QT, MAXP, ATMEM, H>(*static_cast<const GemmParams<MAXP>*>(p), grid, pdl, st);
}

template <int NT, int H, bool GROUPED, bool BF16, int QT>
cudaError_t unit_pick_a(const void* p, bool a_tmem, int grid, bool pdl, cudaStream_t st) {
    return a_tmem ? unit_go<NT, H, GROUPED, BF16, QT, true>(p, grid, pdl, st)
                  : unit_go<NT, H, GROUPED, BF16, QT, false>(p, grid, pdl, st);
}

template <int NT, int H, bool GROUPED, bool BF16>
cudaError_t unit_pick_q(const void* p, int qt, bool a_tmem, int grid, bool pdl, cudaStream_t st) {
    switch (qt) {
        case kQtU4B8: return unit_pick_a<NT, H, GROUPED, BF16, kQtU4B8>(p, a_tmem, grid, pdl, st);
        case kQtU4Zp: return unit_pick_a<NT, H, GROUPED, BF16, kQtU4Zp>(p, a_tmem, grid, pdl, st);
        default: return unit_pick_a<NT, H, GROUPED, BF16, kQtU4FZp>(p, a_tmem, grid, pdl, st);
    }
}

template <int NT, int H>
cudaError_t launch_gemm_unit(const void* params, bool grouped, bool bf16, int qt, bool a_tmem, int grid, bool pdl,
                             cudaStream_t st) {
    if (grouped)
        return bf16 ? unit_pick_q<NT, H, true, true>(params, qt, a_tmem, grid, pdl, st)
                    : unit_pick_q<NT, H, true, false>(params, qt, a_tmem, grid, pdl, st);
    return bf16 ? unit_pick_q<NT, H, false, true>(params, qt, a_tmem, grid, pdl, st)
                : unit_pick_q<NT, H, false, false>(params, qt, a_tmem, grid, pdl, st);
}

}  // namespace wq4

// The exported launcher of one (token tile, scale sets) pair, declared in wq4_launch.h.
#define WQ4_GEMM_UNIT(NT, H)                                                                               \
    namespace wq4 {                                                                                        \
    cudaError_t launch_gemm_nt##NT##_h##H(const void* params, bool grouped, bool bf16, int qt, bool a_tmem, \
                                          int grid, bool pdl, cudaStream_t st) {                          \
        return launch_gemm_unit<NT, H>(params, grouped, bf16, qt, a_tmem, grid, pdl, st);                  \
    }                                                                                                      \
    }
