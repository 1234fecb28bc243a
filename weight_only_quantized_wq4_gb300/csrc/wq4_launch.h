// Launchers of the GEMM instantiations and of prepack.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace wq4 {

// Epilogue of wq4_mm_ex: Y = alpha acc + beta C + bias (C read only when beta != 0).
struct EpilogueArgs {
    float alpha, beta;
    const void* c;
    const void* bias;
};

// `params` points to a GemmParams<1> (grouped == false) or GemmParams<kMaxGroupedProblems>. One
// launcher per token tile (16, 64, 128, 160, 192) and scale-set count (h1: one scale per 128-K
// record, h2: two, group size 64), each in its own translation unit (wq4_gemm_nt*_h*.cu).
#define WQ4_DECLARE_GEMM_UNIT(NT, H)                                                                  \
    cudaError_t launch_gemm_nt##NT##_h##H(const void* params, bool grouped, bool bf16, int qt, bool a_tmem, \
                                          int grid, bool pdl, cudaStream_t st);
WQ4_DECLARE_GEMM_UNIT(16, 1)
WQ4_DECLARE_GEMM_UNIT(16, 2)
WQ4_DECLARE_GEMM_UNIT(64, 1)
WQ4_DECLARE_GEMM_UNIT(64, 2)
WQ4_DECLARE_GEMM_UNIT(128, 1)
WQ4_DECLARE_GEMM_UNIT(128, 2)
WQ4_DECLARE_GEMM_UNIT(160, 1)
WQ4_DECLARE_GEMM_UNIT(160, 2)
WQ4_DECLARE_GEMM_UNIT(192, 1)
WQ4_DECLARE_GEMM_UNIT(192, 2)
#undef WQ4_DECLARE_GEMM_UNIT

// Decode-sized M (<= 32 tokens): warp-level MMA kernel, no workspace.
struct DecodeLaunch {
    int sm_count;
    unsigned int* status;       // device status word
    long long timeout_cycles;   // bound of every pipeline wait
    void* encode_fn;            // cuTensorMapEncodeTiled
    bool pdl;                   // programmatic dependent launch
    int test_stall;             // (tests) one wait per CTA that nothing ends
    int const_weights;          // 1: the blob is read before the kernel ahead on the stream completes
    int trigger_late;           // 1: the next kernel is let in once the activations landed
    int depth;                  // weight ring slots; 0 = automatic
    int hdr_trusted;            // 1: the blob was prepacked here for these arguments: stream before the check
};
bool decode_fits(int M, int K);
cudaError_t launch_decode(const DecodeLaunch& L, const void* X, const void* Wp, void* Y, int M, int N, int K,
                          int group_size, int dtype, int qtype, const EpilogueArgs* epi, int* grid_out,
                          int* depth_out, cudaStream_t st);
// P decode-sized problems (every M[p] > 0, decode_fits at the largest M and K) in one launch.
cudaError_t launch_decode_grouped(const DecodeLaunch& L, int P, const void* const* X, const void* const* Wp,
                                  void* const* Y, const int* M, const int* N, const int* K, int group_size, int dtype,
                                  int qtype, int* grid_out, int* depth_out, cudaStream_t st);

cudaError_t launch_prepack(const uint32_t* wq, const void* scales, const void* zeros, int N, int K, int G,
                           int dtype, int qtype, void* blob, cudaStream_t st);
cudaError_t launch_unprepack(const void* blob, int N, int K, int G, int qtype, uint32_t* wq, void* scales,
                             void* zeros, cudaStream_t st);

}  // namespace wq4
