// Kernel parameter blocks shared by the host planner and the GEMM kernels.
#pragma once

#include <cstdint>
#include <cuda.h>

namespace wq4 {

constexpr int kTileN = 128;          // weight rows per tile (the MMA's M side after the transpose)
constexpr int kTileK = 128;          // K elements per tile = one quantisation group
constexpr int kBlobHeader = 256;     // bytes before the first tile record of a prepacked blob
constexpr int kMaxGroupedProblems = 64;
constexpr uint32_t kBlobMagic = 0x50345157u;   // "WQ4P"
constexpr uint32_t kBlobVersion = 2;

// Bits of the device status word: a bounded pipeline wait ran out; a blob header did not match
// the call's arguments; a bounds check of the debug build failed.
enum : uint32_t { kStatusTimeout = 1u, kStatusBadBlob = 2u, kStatusBounds = 4u };

// Weight formats (the blob header's qtype code): uint4b8 (value = (q - 8) s), uint4 with a 4-bit
// zero point per (group, row) (value = (q - z) s), uint4 with a float zero per (group, row), added
// after the scale (value = q s + zf: the scale-with-zero conversion of "machete_mainloop.cuh",
// transform_A_kblock).
enum : int { kQtU4B8 = 0, kQtU4Zp = 1, kQtU4FZp = 2 };

// A (128-row, 128-K) record of the prepacked blob is eight blocks of 16 weight rows. Block b
// holds, for its rows rr = 0..15: 1024 B of codes (16-byte chunk 16 j + rr = the row's K elements
// 32 j + [0, 32)), then H scale sets (H = 2 for a group size of 64, set h covering the record's K
// elements from 64 h; else H = 1) of 32 B each (row rr at byte 4 (rr % 8) + 2 (rr / 8) of the
// set), then per set the zeros: in zero-point mode 8 B (row rr in byte rr % 8, high nibble for
// rr >= 8), in float-zero mode 32 B placed like the scales; padded to 16 B. A block is one
// contiguous run, so a kernel that owns a few 16-row blocks stages exactly those with one tensor
// copy per run of groups, and a kernel that owns whole tiles copies the record at once.
constexpr int kBlockRows = 16;
constexpr int kBlockCodes = 1024;
constexpr int kBlockScaleOff = 1024;
__host__ __device__ constexpr int scale_sets(int group_size) { return group_size == 64 ? 2 : 1; }
__host__ __device__ constexpr int block_zero_off(int H) { return kBlockScaleOff + 32 * H; }
__host__ __device__ constexpr int block_bytes(int qt, int H = 1) {
    return (block_zero_off(H) + H * (qt == kQtU4Zp ? 8 : qt == kQtU4FZp ? 32 : 0) + 15) / 16 * 16;
}
__host__ __device__ constexpr int tile_record_bytes(int qt, int H = 1) { return 8 * block_bytes(qt, H); }
// Byte offsets, inside a record, of row r's (0..127) 16-byte code chunk j, its scale of set h, the
// byte holding its zero point of set h (nibble (r / 8) & 1) and its float zero of set h.
__host__ __device__ constexpr int rec_code_off(int qt, int r, int j, int H = 1) {
    return (r >> 4) * block_bytes(qt, H) + (16 * j + (r & 15)) * 16;
}
__host__ __device__ constexpr int rec_scale_off(int qt, int r, int H = 1, int h = 0) {
    return (r >> 4) * block_bytes(qt, H) + kBlockScaleOff + 32 * h + 4 * (r & 7) + 2 * ((r >> 3) & 1);
}
__host__ __device__ constexpr int rec_zero_off(int qt, int r, int H = 1, int h = 0) {
    return (r >> 4) * block_bytes(qt, H) + block_zero_off(H) + 8 * h + (r & 7);
}
__host__ __device__ constexpr int rec_fzero_off(int qt, int r, int H = 1, int h = 0) {
    return (r >> 4) * block_bytes(qt, H) + block_zero_off(H) + 32 * h + 4 * (r & 7) + 2 * ((r >> 3) & 1);
}

struct ProblemDesc {
    const uint8_t* wp;       // first tile record (blob + kBlobHeader)
    void* y;                 // [M][N] row-major
    const void* c;           // epilogue source [M][N] (read when beta != 0), or null
    const void* bias;        // epilogue bias [N], or null
    int M, N, K;
    int n_tiles;             // N / 128
    int m_tiles;             // ceil(M / token tile), 0 for an empty problem
    int k_groups;            // K / 128
    int tile_begin;          // global index of the problem's first tile
    int unit_begin;          // global index of the problem's first (tile, group) unit
    int valid;               // 0: its pointers failed the device-side check (its tiles are skipped)
    int pad;
};

// Per-problem pointers in device memory (wq4_grouped_mm_dev_ptrs): a set-up kernel on the stream
// writes each problem's descriptor and activation tensor map into the workspace (any number of
// problems up to kMaxDevPtrProblems); the GEMM reads them from there instead of its parameters.
constexpr int kMaxDevPtrProblems = 4096;
constexpr int kPtrSetupChunk = 128;       // problems per set-up launch (its parameters hold their maps)
constexpr int kPtrSetupSmall = 16;        // a call with at most this many problems: a small parameter block
template <int C>
struct PtrSetup {
    // Problem i's activation map, encoded on the host for its rows and K with a stand-in address;
    // the set-up kernel replaces only the global address. (The encoder also derives a flag from the
    // tensor's total size, which replacing the row count on the device would leave stale.)
    CUtensorMap tmpl[C];
    int p0, count;                        // problems [p0, p0 + count) of this launch
    int group_size, dtype, qtype;         // what every blob header must say
    int M[C], N[C], K[C];
    int m_tiles[C], tile_begin[C], unit_begin[C];
};
static_assert(sizeof(PtrSetup<kPtrSetupChunk>) <= 32000, "kernel parameter space");

// Problem sizes known only on the device (tokens routed to experts by a kernel): a set-up kernel
// writes this table from the device array of token counts; the GEMM then reads M, the tile counts
// and the first tile of each problem from here instead of its parameters (whole tiles only).
struct DynTable {
    int total_tiles;
    int pad[3];
    int M[kMaxGroupedProblems];
    int tile_begin[kMaxGroupedProblems];
};

// A tile is (problem, m_tile, n_tile); inside a problem tiles run m-major (consecutive tiles
// share the same activation rows and walk the weight tiles), so the CTAs working at one time
// share operands in L2. Tiles [0, dp_tiles) are processed whole, tile t by CTA t % num_ctas.
// The units (tile, group) of tiles [dp_tiles, total_tiles) are split evenly and contiguously
// over the CTAs (CTA c takes units [floor(c U / C), floor((c+1) U / C)) counted from
// sk_unit_begin); a tile split between CTAs is summed in the workspace in CTA order.
// Cluster mode (few tiles, e.g. decode-sized M): the grid is tiles x S CTAs in clusters of S;
// cluster t computes tile t, its CTA of rank q the groups [q kg / S, (q+1) kg / S), and the S
// partial sums are added in rank order through distributed shared memory (no workspace).
// The constants of the code-to-16-bit conversion (a code pair sits in bits [0,4) and [16,20) of a
// word): the mask that keeps it and the magic bits OR-ed around it (128.0 in bf16, 1024.0 in
// fp16). Kernels take them as arguments, not as literals: held in registers, they let one
// three-input logic instruction form each pair, where two literals cost two instructions (one
// instruction encodes one literal). Measured on the decode kernel's 16 x 128 unit: 94 integer-pipe
// warp instructions per unit with literals, 61 with registers.
struct NibbleConsts {
    uint32_t mask;
    uint32_t magic;
};
inline NibbleConsts nibble_consts(bool bf16) { return NibbleConsts{0x000F000Fu, bf16 ? 0x43004300u : 0x64006400u}; }

template <int MAXP>
struct GemmParams {
    CUtensorMap xmap[MAXP];  // activations of each problem: 2-D (K, M), box (64, token tile), 128B swizzle
    ProblemDesc prob[MAXP];
    int num_problems;
    int total_tiles;
    int dp_tiles;
    int num_ctas;
    int sk_unit_begin;
    int sk_units;            // the host keeps sk_units * num_ctas < 2^31 (32-bit index math)
    int cluster_split;       // S > 0: cluster mode (below); 0: the data-parallel / K-split plan above
    float* partials;         // [2 * num_ctas][token tile * 128] fp32
    int* counters;           // [total_tiles - dp_tiles], zero between calls
    unsigned int* status;    // device status word (timeouts)
    long long timeout_cycles;
    int test_stall;          // 1: one wait per CTA on a barrier nothing arrives on (tests)
    int has_epi;             // 1: Y = alpha acc + beta C + bias (else Y = acc)
    float alpha, beta;
    const DynTable* dyn;     // device-resident problem sizes (see DynTable), or null
    int group_size, dtype, qtype;   // what every problem's blob header must say
    int early;               // 1: the caller's constant-weights promise: the weight records (and blob
                             // headers) may be read before the kernel ahead on the stream completes
    int hdr_trusted;         // 1: every blob was prepacked here for these arguments (records may be read
                             // while the headers are being checked); 0: check before the first read
    NibbleConsts nib;        // nibble_consts(dtype == bf16)
    // float-zero mode: each problem's activation sums per (token, zero group), split into high and
    // low 16-bit parts: [rows][2 zpad], high in columns [0, zpad), low in [zpad, 2 zpad), zpad =
    // (K / zero-group span) rounded up to 64; box (64, token tile), 128B swizzle
    CUtensorMap sxmap[MAXP];
    // the fused epilogue's C ([M][N] 16-bit; box (128, token tile), rows past M zero): single-problem
    // calls with beta != 0, copied into shared memory per whole tile where the kernel has room
    CUtensorMap cmap;
    const ProblemDesc* prob_tab;    // device-resident problem table (num_problems entries), or null
    const CUtensorMap* xmap_tab;    // their activation tensor maps (patched on the device), or null
};

}  // namespace wq4
