// Launchers of the GEMM instantiations (one translation unit per token tile) and of prepack.
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

// `params` points to a GemmParams<1> (grouped == false) or GemmParams<kMaxGroupedProblems>.
cudaError_t launch_gemm_nt16(const void* params, bool grouped, bool bf16, int qt, bool a_tmem, int scale_sets, int grid,
                             bool pdl, cudaStream_t st);
cudaError_t launch_gemm_nt64(const void* params, bool grouped, bool bf16, int qt, bool a_tmem, int scale_sets, int grid,
                             bool pdl, cudaStream_t st);
cudaError_t launch_gemm_nt128(const void* params, bool grouped, bool bf16, int qt, bool a_tmem, int scale_sets, int grid,
                              bool pdl, cudaStream_t st);
cudaError_t launch_gemm_nt160(const void* params, bool grouped, bool bf16, int qt, bool a_tmem, int scale_sets, int grid,
                              bool pdl, cudaStream_t st);
cudaError_t launch_gemm_nt192(const void* params, bool grouped, bool bf16, int qt, bool a_tmem, int scale_sets, int grid,
                              bool pdl, cudaStream_t st);

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

cudaError_t launch_prepack(const uint32_t* wq, const void* scales, const void* zeros, int N, int K, int G,
                           int dtype, int qtype, void* blob, cudaStream_t st);
cudaError_t launch_unprepack(const void* blob, int N, int K, int G, int qtype, uint32_t* wq, void* scales,
                             void* zeros, cudaStream_t st);

}  // namespace wq4
