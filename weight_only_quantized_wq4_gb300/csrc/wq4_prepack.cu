// Prepack and its inverse: reorder packed 4-bit weights, scales and zero points into the tile
// records the GEMM streams (the offline weight reordering of "machete_mainloop.cuh", header
// comment, with a layout made for this hardware).
//
// Blob (version 2): a 256-byte header of little-endian uint32 (magic "WQ4P", version 2, N, K,
// group size, dtype code, qtype code, record bytes, N/128, K/128, then zeros), then one record
// per (n_tile, group) in n_tile-major order. A record is eight blocks of 16 weight rows
// (wq4_params.h); block b of record (nt, g) holds, for rows n = 128 nt + 16 b + rr:
//   * 1024 B of codes: 16-byte chunk (16 j + rr) = row rr's K elements 128 g + 32 j + [0, 32); its
//     word w holds elements 8w + e (e = 0..7) of that run with element e in nibble e/2 + 4 (e % 2),
//     so that (word >> 4i) & 0x000F000F holds elements 2i, 2i+1. A thread that owns a row reads a
//     32-element run with one 128-bit load; a warp's 8-row 16-byte pieces are 128 contiguous bytes;
//   * 32 B of scales per scale set, row rr at byte 4 (rr % 8) + 2 (rr / 8) of the set (one set with
//     a group size G that is a multiple of 128, record g carrying group 128 g / G; two with G = 64,
//     set h carrying group 2 g + h; without scales every slot holds 1.0);
//   * (zero-point mode) 8 B of zero points, row rr in byte rr % 8 (high nibble for rr >= 8), then
//     zero padding to 1072 B; (float-zero mode) 32 B of float zeros placed like the scales (1088 B).
#include <cuda_runtime.h>

#include <cstdint>

#include "wq4_params.h"

namespace wq4 {

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
__device__ __forceinline__ size_t code_word_offset(int n, int kw, int k_groups, int zp, int H) {
    const int g = kw >> 4, j = (kw >> 2) & 3, w = kw & 3;
    const int nt = n >> 7, r = n & 127;
    return (static_cast<size_t>(nt) * k_groups + g) * tile_record_bytes(zp, H) +
           static_cast<size_t>(rec_code_off(zp, r, j, H) + 4 * w);
}

__global__ void prepack_codes_kernel(const uint32_t* __restrict__ wq, uint8_t* __restrict__ recs, int N,
                                     int K, int zp, int H) {
    const int kwords = K / 8;
    const long long total = static_cast<long long>(N) * kwords;
    for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int n = static_cast<int>(idx / kwords), kw = static_cast<int>(idx % kwords);
        *reinterpret_cast<uint32_t*>(recs + code_word_offset(n, kw, K / 128, zp, H)) = interleave_codes(wq[idx]);
    }
}

__global__ void unprepack_codes_kernel(const uint8_t* __restrict__ recs, uint32_t* __restrict__ wq, int N,
                                       int K, int zp, int H) {
    const int kwords = K / 8;
    const long long total = static_cast<long long>(N) * kwords;
    for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int n = static_cast<int>(idx / kwords), kw = static_cast<int>(idx % kwords);
        wq[idx] = deinterleave_codes(*reinterpret_cast<const uint32_t*>(recs + code_word_offset(n, kw, K / 128, zp, H)));
    }
}

// Scales and float zeros (one thread per (record, row), every scale set), zero points and padding
// (one thread per (record, 16-row block): the eight zero-point bytes of a block combine two of the
// API's words), and the header. Set h of record g carries quantisation group (128 g + 64 h) / G.
__global__ void prepack_side_kernel(const uint16_t* __restrict__ scales, const void* __restrict__ zeros_in,
                                    uint8_t* __restrict__ blob, int N, int K, int G, int dtype, int qtype) {
    const int zp = qtype;                                            // record layout of this format
    const int H = scale_sets(G);
    const uint32_t* zeros = static_cast<const uint32_t*>(zeros_in);  // 4-bit zero points (zero-point mode)
    const uint16_t* fzeros = static_cast<const uint16_t*>(zeros_in); // float zeros (float-zero mode)
    const int rec = tile_record_bytes(zp, H);
    const uint16_t one = dtype == 0 ? 0x3F80u : 0x3C00u;     // 1.0 in bf16 / fp16
    const int ng = K / 128, nT = N / 128;
    uint8_t* recs = blob + kBlobHeader;
    const long long n_scale = static_cast<long long>(ng) * N;
    const long long n_block = qtype == kQtU4Zp ? static_cast<long long>(ng) * (N / kBlockRows) : 0;
    const long long total = n_scale + n_block + 64;
    for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<long long>(gridDim.x) * blockDim.x) {
        if (idx < n_scale) {
            const int g = static_cast<int>(idx / N), n = static_cast<int>(idx % N);
            uint8_t* r = recs + (static_cast<size_t>(n >> 7) * ng + g) * rec;
            for (int h = 0; h < H; ++h) {
                const int src = (g * 128 + 64 * h) / G;              // quantisation group of set h
                *reinterpret_cast<uint16_t*>(r + rec_scale_off(zp, n & 127, H, h)) =
                    scales ? scales[static_cast<size_t>(src) * N + n] : one;
                if (qtype == kQtU4FZp)
                    *reinterpret_cast<uint16_t*>(r + rec_fzero_off(zp, n & 127, H, h)) =
                        fzeros[static_cast<size_t>(src) * N + n];
            }
        } else if (idx < n_scale + n_block) {
            const long long z = idx - n_scale;
            const int g = static_cast<int>(z / (N / kBlockRows)), blk = static_cast<int>(z % (N / kBlockRows));
            uint8_t* r = recs + (static_cast<size_t>(blk >> 3) * ng + g) * rec + (blk & 7) * block_bytes(kQtU4Zp, H);
            uint32_t* zw = reinterpret_cast<uint32_t*>(r + block_zero_off(H));
            for (int h = 0; h < H; ++h) {
                const int src = (g * 128 + 64 * h) / G;
                const uint32_t lo = zeros[static_cast<size_t>(src) * (N / 8) + 2 * blk];       // rows 16 blk + 0..7
                const uint32_t hi = zeros[static_cast<size_t>(src) * (N / 8) + 2 * blk + 1];   // rows 16 blk + 8..15
                uint32_t w[2] = {0u, 0u};
#pragma unroll
                for (int p = 0; p < 8; ++p) {
                    const uint32_t byte = ((lo >> (4 * p)) & 0xFu) | (((hi >> (4 * p)) & 0xFu) << 4);
                    w[p >> 2] |= byte << (8 * (p & 3));
                }
                zw[2 * h] = w[0];
                zw[2 * h + 1] = w[1];
            }
            // zero padding up to the block's end (8 B with one set, none with two)
            for (int i = 2 * H; i < (block_bytes(kQtU4Zp, H) - block_zero_off(H)) / 4; ++i) zw[i] = 0u;
        } else {
            const int w = static_cast<int>(idx - n_scale - n_block);
            uint32_t v = 0;
            switch (w) {
                case 0: v = kBlobMagic; break;
                case 1: v = kBlobVersion; break;
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

// Output row j (quantisation group j) is read from the first record and scale set holding it:
// record j G / 128, set (j G % 128) / 64.
__global__ void unprepack_side_kernel(const uint8_t* __restrict__ blob, uint16_t* __restrict__ scales,
                                      void* __restrict__ zeros_out, int N, int K, int G, int zp) {
    const int H = scale_sets(G);
    const int rec = tile_record_bytes(zp, H);
    const int ng = K / 128, nq = K / G;
    const uint8_t* recs = blob + kBlobHeader;
    uint32_t* zeros = static_cast<uint32_t*>(zeros_out);
    uint16_t* fzeros = static_cast<uint16_t*>(zeros_out);
    const long long n_scale = scales ? static_cast<long long>(nq) * N : 0;
    const long long n_zero = zeros_out ? static_cast<long long>(nq) * (zp == kQtU4FZp ? N : N / 8) : 0;
    for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < n_scale + n_zero;
         idx += static_cast<long long>(gridDim.x) * blockDim.x) {
        if (idx < n_scale) {
            const int j = static_cast<int>(idx / N), n = static_cast<int>(idx % N);
            const int g = (j * G) / 128, h = ((j * G) % 128) / 64;
            const uint8_t* r = recs + (static_cast<size_t>(n >> 7) * ng + g) * rec;
            scales[idx] = *reinterpret_cast<const uint16_t*>(r + rec_scale_off(zp, n & 127, H, h));
        } else if (zp == kQtU4FZp) {
            const long long z = idx - n_scale;
            const int j = static_cast<int>(z / N), n = static_cast<int>(z % N);
            const int g = (j * G) / 128, h = ((j * G) % 128) / 64;
            const uint8_t* r = recs + (static_cast<size_t>(n >> 7) * ng + g) * rec;
            fzeros[z] = *reinterpret_cast<const uint16_t*>(r + rec_fzero_off(zp, n & 127, H, h));
        } else {
            // API word wz: rows 8 wz .. 8 wz + 7, the low (wz even) or high (wz odd) nibbles of a block
            const long long z = idx - n_scale;
            const int j = static_cast<int>(z / (N / 8)), wz = static_cast<int>(z % (N / 8));
            const int g = (j * G) / 128, h = ((j * G) % 128) / 64;
            const int n0 = 8 * wz;
            const uint8_t* r = recs + (static_cast<size_t>(n0 >> 7) * ng + g) * rec;
            uint32_t out = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int rr = (n0 + i) & 127;
                const uint32_t byte = r[rec_zero_off(kQtU4Zp, rr, H, h)];
                out |= ((byte >> (4 * ((rr >> 3) & 1))) & 0xFu) << (4 * i);
            }
            zeros[z] = out;
        }
    }
}

static int grid_for(long long work, int threads) {
    long long b = (work + threads - 1) / threads;
    if (b < 1) b = 1;
    if (b > 16384) b = 16384;
    return static_cast<int>(b);
}

cudaError_t launch_prepack(const uint32_t* wq, const void* scales, const void* zeros, int N, int K, int G,
                           int dtype, int qtype, void* blob, cudaStream_t st) {
    const int zp = qtype;
    uint8_t* b = static_cast<uint8_t*>(blob);
    const long long words = static_cast<long long>(N) * (K / 8);
    prepack_codes_kernel<<<grid_for(words, 256), 256, 0, st>>>(wq, b + kBlobHeader, N, K, zp, scale_sets(G));
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const long long side = static_cast<long long>(K / 128) * N * 2;
    prepack_side_kernel<<<grid_for(side, 256), 256, 0, st>>>(static_cast<const uint16_t*>(scales), zeros, b, N, K, G,
                                                            dtype, qtype);
    return cudaGetLastError();
}

cudaError_t launch_unprepack(const void* blob, int N, int K, int G, int qtype, uint32_t* wq, void* scales,
                             void* zeros, cudaStream_t st) {
    const int zp = qtype;
    const uint8_t* b = static_cast<const uint8_t*>(blob);
    const long long words = static_cast<long long>(N) * (K / 8);
    unprepack_codes_kernel<<<grid_for(words, 256), 256, 0, st>>>(b + kBlobHeader, wq, N, K, zp, scale_sets(G));
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const long long side = static_cast<long long>(K / 128) * N * 2;
    unprepack_side_kernel<<<grid_for(side, 256), 256, 0, st>>>(b, static_cast<uint16_t*>(scales), zeros, N, K, G,
                                                              zp);
    return cudaGetLastError();
}

}  // namespace wq4
