// Prepack and its inverse: reorder packed 4-bit weights, scales and zero points into the tile
// records the GEMM streams (the offline weight reordering of "machete_mainloop.cuh", header
// comment, with a layout made for this kernel).
//
// Blob: a 256-byte header of little-endian uint32 (magic "WQ4P", version 1, N, K, group size,
// dtype code, qtype code, record bytes, N/128, K/128, then zeros), then one record per
// (n_tile, group) in n_tile-major order. A record holds
//   * 8192 B of codes: 16-byte chunk (j * 128 + r) = row 128 n_tile + r, K elements
//     128 g + 32 j + [0, 32); its word w holds elements 8w + e (e = 0..7) of that run with element
//     e in nibble e/2 + 4 (e % 2), so that (word >> 4i) & 0x000F000F holds elements 2i, 2i+1.
//     A dequant thread then reads its row's 32-element runs with one 128-bit load, and the 32
//     threads of a warp read 512 consecutive bytes;
//   * 256 B of scales, row r at byte 2r (the scale of the quantisation group the record lies in:
//     with a group size G that is a multiple of 128, record g carries group 128 g / G; without
//     scales every slot holds 1.0);
//   * (zero-point mode) 64 B of zero points, row r in nibble r % 8 of word r / 8; then zero
//     padding to 8576 B.
#include <cuda_runtime.h>

#include <cstdint>

#include "wq4_params.h"

namespace wq4 {

constexpr uint32_t kBlobMagic = 0x50345157u;

__device__ __forceinline__ uint32_t interleave_codes(uint32_t in) {
    uint32_t out = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) out |= ((in >> (4 * e)) & 0xFu) << (4 * ((e >> 1) + 4 * (e & 1)));
    return out;
}

__device__ __forceinline__ uint32_t deinterleave_codes(uint32_t in) {
    uint32_t out = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) out |= ((in >> (4 * ((e >> 1) + 4 * (e & 1)))) & 0xFu) << (4 * e);
    return out;
}

// Byte offset (from the first record) of the code word holding elements [8 kw, 8 kw + 8) of row n.
__device__ __forceinline__ size_t code_word_offset(int n, int kw, int k_groups, int rec) {
    const int g = kw >> 4, j = (kw >> 2) & 3, w = kw & 3;
    const int nt = n >> 7, r = n & 127;
    return (static_cast<size_t>(nt) * k_groups + g) * rec + static_cast<size_t>((j * 128 + r) * 16 + 4 * w);
}

__global__ void prepack_codes_kernel(const uint32_t* __restrict__ wq, uint8_t* __restrict__ recs, int N,
                                     int K, int rec) {
    const int kwords = K / 8;
    const long long total = static_cast<long long>(N) * kwords;
    for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int n = static_cast<int>(idx / kwords), kw = static_cast<int>(idx % kwords);
        *reinterpret_cast<uint32_t*>(recs + code_word_offset(n, kw, K / 128, rec)) = interleave_codes(wq[idx]);
    }
}

__global__ void unprepack_codes_kernel(const uint8_t* __restrict__ recs, uint32_t* __restrict__ wq, int N,
                                       int K, int rec) {
    const int kwords = K / 8;
    const long long total = static_cast<long long>(N) * kwords;
    for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int n = static_cast<int>(idx / kwords), kw = static_cast<int>(idx % kwords);
        wq[idx] = deinterleave_codes(*reinterpret_cast<const uint32_t*>(recs + code_word_offset(n, kw, K / 128, rec)));
    }
}

// Scales (one thread per (group, row)), zero-point words (one per (group, 8 rows)), record
// padding and the header.
__global__ void prepack_side_kernel(const uint16_t* __restrict__ scales, const uint32_t* __restrict__ zeros,
                                    uint8_t* __restrict__ blob, int N, int K, int G, int dtype, int qtype, int rec) {
    const uint16_t one = dtype == 0 ? 0x3F80u : 0x3C00u;     // 1.0 in bf16 / fp16
    const int ng = K / 128, nT = N / 128;
    uint8_t* recs = blob + kBlobHeader;
    const long long n_scale = static_cast<long long>(ng) * N;
    const long long n_zero = zeros ? static_cast<long long>(ng) * (N / 8) : 0;
    const int pad_words = (rec - (8192 + 256 + (zeros ? 64 : 0))) / 4;
    const long long n_pad = static_cast<long long>(ng) * nT * pad_words;
    const long long total = n_scale + n_zero + n_pad + 64;
    for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<long long>(gridDim.x) * blockDim.x) {
        if (idx < n_scale) {
            const int g = static_cast<int>(idx / N), n = static_cast<int>(idx % N);
            const int src = (g * 128) / G;                           // quantisation group of record g
            uint8_t* r = recs + (static_cast<size_t>(n >> 7) * ng + g) * rec;
            reinterpret_cast<uint16_t*>(r + 8192)[n & 127] = scales ? scales[static_cast<size_t>(src) * N + n] : one;
        } else if (idx < n_scale + n_zero) {
            const long long z = idx - n_scale;
            const int g = static_cast<int>(z / (N / 8)), wz = static_cast<int>(z % (N / 8));
            const int src = (g * 128) / G;
            uint8_t* r = recs + (static_cast<size_t>(wz >> 4) * ng + g) * rec;
            reinterpret_cast<uint32_t*>(r + 8448)[wz & 15] = zeros[static_cast<size_t>(src) * (N / 8) + wz];
        } else if (idx < n_scale + n_zero + n_pad) {
            const long long z = idx - n_scale - n_zero;
            const long long rr = z / pad_words;
            const int w = static_cast<int>(z % pad_words);
            uint8_t* r = recs + rr * rec;
            reinterpret_cast<uint32_t*>(r + (rec - 4 * pad_words))[w] = 0u;
        } else {
            const int w = static_cast<int>(idx - n_scale - n_zero - n_pad);
            uint32_t v = 0;
            switch (w) {
                case 0: v = kBlobMagic; break;
                case 1: v = 1u; break;
                case 2: v = static_cast<uint32_t>(N); break;
                case 3: v = static_cast<uint32_t>(K); break;
                case 4: v = static_cast<uint32_t>(G); break;
                case 5: v = static_cast<uint32_t>(dtype); break;
                case 6: v = static_cast<uint32_t>(qtype); break;
                case 7: v = static_cast<uint32_t>(rec); break;
                case 8: v = static_cast<uint32_t>(nT); break;
                case 9: v = static_cast<uint32_t>(ng); break;
                default: v = 0u;
            }
            reinterpret_cast<uint32_t*>(blob)[w] = v;
        }
    }
}

// Output row j (quantisation group j) is read from its first record, 128-K record j G / 128.
__global__ void unprepack_side_kernel(const uint8_t* __restrict__ blob, uint16_t* __restrict__ scales,
                                      uint32_t* __restrict__ zeros, int N, int K, int G, int rec) {
    const int ng = K / 128, nq = K / G;
    const uint8_t* recs = blob + kBlobHeader;
    const long long n_scale = scales ? static_cast<long long>(nq) * N : 0;
    const long long n_zero = zeros ? static_cast<long long>(nq) * (N / 8) : 0;
    for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < n_scale + n_zero;
         idx += static_cast<long long>(gridDim.x) * blockDim.x) {
        if (idx < n_scale) {
            const int j = static_cast<int>(idx / N), n = static_cast<int>(idx % N);
            const int g = (j * G) / 128;
            const uint8_t* r = recs + (static_cast<size_t>(n >> 7) * ng + g) * rec;
            scales[idx] = reinterpret_cast<const uint16_t*>(r + 8192)[n & 127];
        } else {
            const long long z = idx - n_scale;
            const int j = static_cast<int>(z / (N / 8)), wz = static_cast<int>(z % (N / 8));
            const int g = (j * G) / 128;
            const uint8_t* r = recs + (static_cast<size_t>(wz >> 4) * ng + g) * rec;
            zeros[z] = reinterpret_cast<const uint32_t*>(r + 8448)[wz & 15];
        }
    }
}

static int grid_for(long long work, int threads) {
    long long b = (work + threads - 1) / threads;
    if (b < 1) b = 1;
    if (b > 16384) b = 16384;
    return static_cast<int>(b);
}

cudaError_t launch_prepack(const uint32_t* wq, const void* scales, const uint32_t* zeros, int N, int K, int G,
                           int dtype, int qtype, void* blob, cudaStream_t st) {
    const int rec = tile_record_bytes(qtype == 1);
    uint8_t* b = static_cast<uint8_t*>(blob);
    const long long words = static_cast<long long>(N) * (K / 8);
    prepack_codes_kernel<<<grid_for(words, 256), 256, 0, st>>>(wq, b + kBlobHeader, N, K, rec);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const long long side = static_cast<long long>(K / 128) * N * 2;
    prepack_side_kernel<<<grid_for(side, 256), 256, 0, st>>>(static_cast<const uint16_t*>(scales), zeros, b, N, K, G,
                                                            dtype, qtype, rec);
    return cudaGetLastError();
}

cudaError_t launch_unprepack(const void* blob, int N, int K, int G, int qtype, uint32_t* wq, void* scales,
                             uint32_t* zeros, cudaStream_t st) {
    const int rec = tile_record_bytes(qtype == 1);
    const uint8_t* b = static_cast<const uint8_t*>(blob);
    const long long words = static_cast<long long>(N) * (K / 8);
    unprepack_codes_kernel<<<grid_for(words, 256), 256, 0, st>>>(b + kBlobHeader, wq, N, K, rec);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const long long side = static_cast<long long>(K / 128) * N * 2;
    unprepack_side_kernel<<<grid_for(side, 256), 256, 0, st>>>(b, static_cast<uint16_t*>(scales), zeros, N, K, G,
                                                              rec);
    return cudaGetLastError();
}

}  // namespace wq4
