// Host side of the C ABI declared in include/wq4.h: argument checks, the tile/work plan, the
// activation tensor maps and the launches.
//
// Argument rules follow "machete_mainloop.cuh", can_implement: 128-bit alignment of every
// operand for TMA; group_size == K or a multiple of the K tile, and non-zero; the scale pointer
// present in the scaled modes; the zero pointer present exactly in the zero-point mode. This
// build supports group sizes that are multiples of 128 dividing K (group_size == K included;
// "machete_mainloop.cuh", load: the scale row of a k-tile is k_tile / (group_size / tile_k)),
// the no-scale mode for uint4b8 (get_conversion_mode: direct conversion) and N, K multiples of 128.
//
// The work plan mirrors the grouped persistent kernel of
// "sm90_gemm_array_tma_warpspecialized_cooperative.hpp" (grid sized from the SM count, a
// problem-shape array walked by one scheduler, work tiles past the last real one ending the CTA)
// with a data-parallel / K-split hybrid: whole waves of tiles go one per CTA, the remaining
// tiles' (tile, group) units are divided evenly over the CTAs and K-split tiles are summed in a
// fixed order (deterministic).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <memory>
#include <mutex>
#include <unordered_map>
#include <vector>

#include "wq4.h"
#include "wq4_device.cuh"
#include "wq4_launch.h"
#include "wq4_params.h"

namespace wq4 {
namespace {

// device-side error word (bounded-wait timeouts, bad blobs, bounds checks), then the first
// bounds violation of the debug build (site and three values)
__device__ unsigned int g_status[1 + check::kRecordWords];

constexpr int kMaxDevices = 64;
constexpr long long kDefaultTimeoutCycles = 4000000000LL;   // ~2 s at 2 GHz
constexpr long long kFixupSteps = 10;   // cost of a K-split tile's fixup, in (tile, group) steps

struct Options {
    int token_tile = 0;
    int grid = 0;
    int split_all = 0;
    long long timeout_cycles = 0;
    int trace = -1;
    int a_in_smem = 0;
    int cluster = 0;          // 0 automatic, -1 never, S >= 2 force clusters of S
    int decode = 0;           // 0 automatic, -1 never, 1 always when the shape allows it
    int pdl = 0;              // 0 programmatic dependent launch on, -1 off
    int test_stall = 0;       // 1: kernels wait once on a barrier nothing arrives on (tests)
    int const_weights = 0;    // 1: blobs are not written by pending work; weights are read early
    int decode_depth = 0;     // decode weight ring slots, 0 = automatic
    int decode_trigger = 0;   // 0: the next kernel is let in once the activations landed, 1: at once
    int verify_dev_ptrs = 0;  // 1: the device-pointer grouped call stops after its set-up and checks its maps
};
Options g_opt;

struct DeviceInfo {
    bool init = false;
    int sm_count = 0;
    unsigned int* status = nullptr;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_mu;
int g_violation[1 + check::kRecordWords];   // the last violation read back (count, site, three values)

bool trace_on() {
    if (g_opt.trace < 0) {
        const char* e = std::getenv("WQ4_TRACE");
        g_opt.trace = (e && e[0] == '1') ? 1 : 0;
    }
    return g_opt.trace == 1;
}

int device_info(DeviceInfo** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return WQ4_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceInfo& d = g_dev[dev];
    if (!d.init) {
        if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return WQ4_ERR_CUDA;
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return WQ4_ERR_CUDA;
        d.status = static_cast<unsigned int*>(p);
        d.init = true;
    }
    *out = &d;
    return WQ4_OK;
}

// Bound of every pipeline wait: the option if set, else WQ4_TIMEOUT_CYCLES from the environment,
// else about two seconds.
long long timeout_cycles() {
    if (g_opt.timeout_cycles > 0) return g_opt.timeout_cycles;
    static long long env = -1;
    if (env < 0) {
        const char* e = std::getenv("WQ4_TIMEOUT_CYCLES");
        env = e ? std::atoll(e) : 0;
    }
    return env > 0 ? env : kDefaultTimeoutCycles;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Blobs this process wrote with wq4_prepack, with the arguments they were written for. A GEMM call
// whose arguments match its blob's entry lets the kernels stream weight records at once, checking
// the blob header alongside; a call on any other blob (made by other means, or passed with other
// arguments) waits for the device-side header check before the first record is read, so that a
// blob smaller than the call expects is never read past its end.
struct BlobKey {
    int N, K, G, dtype, qtype;
    bool operator==(const BlobKey& o) const {
        return N == o.N && K == o.K && G == o.G && dtype == o.dtype && qtype == o.qtype;
    }
};
std::mutex g_blob_mu;
std::unordered_map<uintptr_t, BlobKey> g_blobs;
constexpr size_t kMaxBlobEntries = 1 << 16;

void blob_register(const void* wp, const BlobKey& k) {
    std::lock_guard<std::mutex> lk(g_blob_mu);
    if (g_blobs.size() >= kMaxBlobEntries) g_blobs.clear();
    g_blobs[reinterpret_cast<uintptr_t>(wp)] = k;
}

bool blob_trusted(const void* wp, const BlobKey& k) {
    std::lock_guard<std::mutex> lk(g_blob_mu);
    const auto it = g_blobs.find(reinterpret_cast<uintptr_t>(wp));
    return it != g_blobs.end() && it->second == k;
}

int check_types(int group_size, int dtype, int qtype) {
    if (dtype != WQ4_BF16 && dtype != WQ4_FP16) return WQ4_ERR_INVALID;
    if (qtype != WQ4_U4B8 && qtype != WQ4_U4_ZP && qtype != WQ4_U4_FZP) return WQ4_ERR_INVALID;
    if (group_size <= 0) return WQ4_ERR_INVALID;
    return WQ4_OK;
}

// Group sizes of this build: multiples of the 128-element K tile that divide K (group_size == K is
// the channel-wise case), every 128-K record of the blob then carrying its group's scale; and 64,
// each record then carrying two scale sets (one per 64-K half).
int check_group(int group_size, int K) {
    if ((group_size % kTileK && group_size != 64) || K % group_size) return WQ4_ERR_UNSUPPORTED;
    return WQ4_OK;
}

// Rows per decode-kernel launch when wq4_mm takes that kernel (no workspace) for this M, N, K
// under the current options, else 0. Up to 32 tokens in one launch when their activations fit
// in shared memory; beyond that (17..32 tokens at large K) two launches of at most 16 tokens each
// for weights up to 12 Mi elements, which read the weights twice and still beat the
// tensor-core kernel there (measured, 32 tokens, K = 4096: N = 2048 8.8 vs 11.3 us; at N = 4096
// the two are even, beyond it the tensor-core kernel wins).
int decode_rows_per_launch(int M, int N, int K) {
    const bool auto_decode = g_opt.decode == 0 && !g_opt.token_tile && !g_opt.grid && !g_opt.split_all &&
                             !g_opt.cluster && !g_opt.a_in_smem;
    if (!(g_opt.decode == 1 || auto_decode)) return 0;
    if (decode_fits(M, K)) return M;
    if (M > 16 && M <= 32 && decode_fits(16, K) && static_cast<long long>(N) * K <= 12LL * 1024 * 1024) return 16;
    return 0;
}

bool uses_decode_kernel(int M, int N, int K) { return decode_rows_per_launch(M, N, K) > 0; }

// A grouped call whose non-empty problems all have at most 32 tokens takes the decode kernel, in
// one launch (under the same options as a single problem does).
bool grouped_uses_decode(int P, const int* M, const int* K) {
    const bool auto_decode = g_opt.decode == 0 && !g_opt.token_tile && !g_opt.grid && !g_opt.split_all &&
                             !g_opt.cluster && !g_opt.a_in_smem;
    if (!(g_opt.decode == 1 || auto_decode)) return false;
    int Mmax = 0, Kmax = 0;
    for (int p = 0; p < P; ++p) {
        if (M[p] <= 0) continue;
        Mmax = std::max(Mmax, M[p]);
        Kmax = std::max(Kmax, K[p]);
    }
    return Mmax > 0 && decode_fits(Mmax, Kmax);
}

int check_nk(int N, int K) {
    if (N <= 0 || K <= 0) return WQ4_ERR_INVALID;
    if (N % kTileN || K % kTileK) return WQ4_ERR_UNSUPPORTED;
    return WQ4_OK;
}

// ---------------------------------------------------------------------------- planning
struct Shape {
    int M, N, K;
};

struct Plan {
    int nt = 0;              // token tile
    int grid = 0;
    int total_tiles = 0;
    int dp_tiles = 0;
    int sk_unit_begin = 0;
    int sk_units = 0;
    int cluster = 0;
    size_t counters_bytes = 0;
    size_t partials_bytes = 0;
    int m_tiles[kMaxDevPtrProblems] = {};
    int tile_begin[kMaxDevPtrProblems] = {};
    int unit_begin[kMaxDevPtrProblems] = {};
    size_t workspace() const { return counters_bytes + partials_bytes; }
};

// Token tile for a launch (one tile size serves every problem of a grouped call). Up to 64 tokens
// the narrow tiles; beyond, the tile of 128, 160 or 192 tokens that minimises the padded work
// sum_p ceil(M_p / NT) * t(NT), t = the measured time of one (tile, group) step of the GEMM
// kernel on GB300 at M = 4096 (584, 633 and 693 ns: a wider tile costs more per step but less
// per token, and a narrower one holds more operand buffers in tensor memory).
int token_tile_for(const int* M, int P) {
    if (g_opt.token_tile) return g_opt.token_tile;
    int maxM = 0;
    for (int p = 0; p < P; ++p) maxM = std::max(maxM, M[p]);
    if (maxM <= 16) return 16;
    if (maxM <= 64) return 64;
    static const int kTiles[3] = {128, 160, 192};
    static const long long kStepNs[3] = {584, 633, 693};
    int best = 192;
    long long best_cost = -1;
    for (int t = 0; t < 3; ++t) {
        long long cost = 0;
        for (int p = 0; p < P; ++p) cost += static_cast<long long>((M[p] + kTiles[t] - 1) / kTiles[t]) * kStepNs[t];
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = kTiles[t];
        }
    }
    return best;
}

// The token tile for these problems (any group size).
int pick_token_tile(const Shape* shapes, int P, int /*group_size*/) {
    int Ms[kMaxDevPtrProblems];
    for (int p = 0; p < P; ++p) Ms[p] = shapes[p].M;
    return token_tile_for(Ms, P);
}

// Splitting the last partial wave of tiles over all CTAs pays only if it saves more (tile, group)
// steps than the fixup of the split tiles costs (the last CTA of a tile reads and adds the
// others' fp32 partials: about kFixupSteps steps, measured). Otherwise every tile stays whole and
// the last wave is partly idle.
bool keep_tiles_whole(long long tiles, long long units, int C) {
    if (g_opt.split_all || g_opt.grid) return false;
    const long long kg_avg = (units + tiles - 1) / tiles;
    const long long whole = (tiles + C - 1) / C * kg_avg;
    const long long split = (tiles / C) * kg_avg + ((tiles % C) * kg_avg + C - 1) / C + kFixupSteps;
    return whole <= split;
}

// The launch plan for P problems (P <= kMaxGroupedProblems). ws_cap bounds the workspace the plan
// may ask for: a K-split plan that would need more keeps every tile whole instead (no workspace;
// the same sums in another order), unless an option forces the split (then the caller's size
// check fails).
int make_plan(const Shape* shapes, int P, int sm_count, size_t ws_cap, int group_size, Plan* pl) {
    pl->nt = pick_token_tile(shapes, P, group_size);
    long long tiles = 0, units = 0;
    for (int p = 0; p < P; ++p) {
        const Shape& s = shapes[p];
        const int mt = s.M > 0 ? (s.M + pl->nt - 1) / pl->nt : 0;
        pl->m_tiles[p] = mt;
        pl->tile_begin[p] = static_cast<int>(tiles);
        pl->unit_begin[p] = static_cast<int>(units);
        const long long t = static_cast<long long>(mt) * (s.N / kTileN);
        tiles += t;
        units += t * (s.K / kTileK);
        if (units >= (1LL << 30) || tiles >= (1LL << 30)) return WQ4_ERR_UNSUPPORTED;
    }
    pl->total_tiles = static_cast<int>(tiles);
    if (tiles == 0) return WQ4_OK;

    // Few tiles (e.g. decode-sized M): clusters of S CTAs split each tile's K range and add their
    // partial sums through distributed shared memory (no global workspace, no atomics).
    int min_kg = 1 << 30;
    for (int p = 0; p < P; ++p)
        if (pl->m_tiles[p] > 0) min_kg = std::min(min_kg, shapes[p].K / kTileK);
    int S = 0;
    if (g_opt.cluster >= 2) {
        S = g_opt.cluster;
    } else if (g_opt.cluster == 0 && !g_opt.split_all && !g_opt.grid && tiles * 2 <= sm_count) {
        // clusters of 8 only for at most 8 tiles: 16 clusters of 8 did not fit in one wave
        // (N = 2048, 16 tiles: 19.7 us with 8, 11.3 us with 4)
        S = static_cast<int>(std::min<long long>(tiles <= 8 ? 8 : 4, sm_count / tiles));
    }
    S = std::min(S, min_kg);
    if (S >= 2) {
        if (tiles * S >= (1LL << 31)) return WQ4_ERR_UNSUPPORTED;
        pl->cluster = S;
        pl->grid = static_cast<int>(tiles * S);
        pl->dp_tiles = 0;
        pl->sk_unit_begin = static_cast<int>(units);
        pl->sk_units = 0;
        return WQ4_OK;
    }

    int C = g_opt.grid ? g_opt.grid : sm_count;
    auto all_whole = [&] {
        pl->grid = static_cast<int>(std::min<long long>(C, tiles));
        pl->dp_tiles = static_cast<int>(tiles);
        pl->sk_unit_begin = static_cast<int>(units);
        pl->sk_units = 0;
        return WQ4_OK;
    };
    // whole waves of tiles are processed data-parallel; the rest is K-split over all CTAs
    int dp = g_opt.split_all ? 0 : static_cast<int>((tiles / C) * C);
    if (dp < tiles && keep_tiles_whole(tiles, units, C)) dp = static_cast<int>(tiles);
    if (dp == tiles && !g_opt.split_all) return all_whole();
    // units of the K-split region
    auto units_before = [&](int tile) {
        int p = 0;
        while (p + 1 < P && pl->tile_begin[p + 1] <= tile) ++p;
        return pl->unit_begin[p] + static_cast<long long>(tile - pl->tile_begin[p]) * (shapes[p].K / kTileK);
    };
    long long sk_begin = units_before(dp);
    // a thin remainder (under two units per CTA) takes one more wave into the split region
    if (dp >= C && units - sk_begin < 2LL * C) {
        dp -= C;
        sk_begin = units_before(dp);
    }
    const long long sk_units = units - sk_begin;
    // a K-split CTA should get at least a few groups; with little work use fewer CTAs
    if (dp == 0 && !g_opt.grid) {
        const long long want = std::max<long long>(1, sk_units / 4);
        C = static_cast<int>(std::min<long long>(C, want));
    }
    if (sk_units * static_cast<long long>(C) >= (1LL << 31)) return WQ4_ERR_UNSUPPORTED;
    const size_t counters = ((static_cast<size_t>(tiles - dp) * 4) + 255) / 256 * 256;
    const size_t partials = static_cast<size_t>(2) * C * pl->nt * kTileN * 4;
    if (counters + partials > ws_cap && !g_opt.split_all && !g_opt.grid) {
        C = g_opt.grid ? g_opt.grid : sm_count;
        return all_whole();
    }
    pl->grid = C;
    pl->dp_tiles = dp;
    pl->sk_unit_begin = static_cast<int>(sk_begin);
    pl->sk_units = static_cast<int>(sk_units);
    pl->counters_bytes = counters;
    pl->partials_bytes = partials;
    return WQ4_OK;
}

// ---------------------------------------------------------------------------- tensor maps
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// X [M][K] 16-bit row-major; box = 64 K elements (128 B) x nt rows, 128-byte swizzle; rows past M
// read as zero.
int encode_x_map(CUtensorMap* map, const void* X, int M, int K, int dtype, int nt) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return WQ4_ERR_CUDA;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
    const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(nt)};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(map, dtype == WQ4_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                          2, const_cast<void*>(X), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? WQ4_OK : WQ4_ERR_CUDA;
}

cudaError_t dispatch(const void* params, bool grouped, int nt, int dtype, int qtype, int group_size, int grid,
                     cudaStream_t st) {
    const bool two = scale_sets(group_size) == 2;
    const bool bf16 = dtype == WQ4_BF16, a_tmem = !g_opt.a_in_smem;
    const int qt = qtype;                                       // record layout of the format
    const bool pdl = g_opt.pdl == 0;
#define WQ4_GO(NT) (two ? launch_gemm_nt##NT##_h2 : launch_gemm_nt##NT##_h1)(params, grouped, bf16, qt, a_tmem, grid, pdl, st)
    switch (nt) {
        case 16: return WQ4_GO(16);
        case 64: return WQ4_GO(64);
        case 128: return WQ4_GO(128);
        case 160: return WQ4_GO(160);
        default: return WQ4_GO(192);
    }
#undef WQ4_GO
}

// Float-zero mode: the activation sums of every (token m, zero group z) for the GEMM's zero steps,
// xs = the sum of X[m][span z .. span z + span - 1] in fp32 (span = 128, or 64 with two scale sets
// per record), split into hi = xs rounded to the 16-bit type and lo = xs - hi rounded likewise
// (hi + lo carries 16 (bf16) or 22 (fp16) significant bits). One table per problem, [ld][2 zpad]
// 16-bit values: hi at column z, lo at column zpad + z; zero for rows m >= M (up to ld) and for
// z >= K / span (up to zpad, a multiple of 64), so that a zero step's copies never read past it and
// the masked-off zeros never meet a NaN. One thread per (problem, m, z), consecutive threads on
// consecutive z of a row: 16-byte loads of its span, added in K order (the same order every run).
// Launched with programmatic dependent launch: the GEMM behind it may set up at once, and X is
// read only once the kernel ahead (which may write it) has completed.
struct XsumJob {
    const uint16_t* X;
    uint16_t* out;
    int M, K, ld, zpad;
    long long begin;             // first thread of this problem
};
struct XsumBatch {
    int P, span;
    long long total;             // threads over all problems
    unsigned int* status;        // device status word (the debug build's checks)
    XsumJob job[kMaxGroupedProblems];
};

template <bool BF16>
__global__ void xsum_kernel(const __grid_constant__ XsumBatch b) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    for (long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; t < b.total;
         t += static_cast<long long>(gridDim.x) * blockDim.x) {
        int p = 0;
        while (p + 1 < b.P && b.job[p + 1].begin <= t) ++p;
        const XsumJob& J = b.job[p];
        const long long u = t - J.begin;
        const int m = static_cast<int>(u / J.zpad), z = static_cast<int>(u % J.zpad);
        float v = 0.f;
        if (m < J.M && z < J.K / b.span) {
            const uint4* xp =
                reinterpret_cast<const uint4*>(J.X + static_cast<size_t>(m) * J.K + static_cast<size_t>(b.span) * z);
            for (int c = 0; c < b.span / 8; ++c) {
                const uint4 q = __ldg(xp + c);
                const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if constexpr (BF16) {
                        v += __uint_as_float(w[e] << 16);
                        v += __uint_as_float(w[e] & 0xFFFF0000u);
                    } else {
                        v += __half2float(__ushort_as_half(static_cast<unsigned short>(w[e] & 0xFFFFu)));
                        v += __half2float(__ushort_as_half(static_cast<unsigned short>(w[e] >> 16)));
                    }
                }
            }
        }
        uint16_t hi, lo;
        if constexpr (BF16) {
            const __nv_bfloat16 h = __float2bfloat16_rn(v);
            hi = __bfloat16_as_ushort(h);
            lo = __bfloat16_as_ushort(__float2bfloat16_rn(v - __bfloat162float(h)));
        } else {
            const __half h = __float2half_rn(v);
            hi = __half_as_ushort(h);
            lo = __half_as_ushort(__float2half_rn(v - __half2float(h)));
        }
        if (!WQ4_CHECK(m < J.ld && z < J.zpad, b.status, nullptr, check::kSiteXSums, m, z, J.ld)) continue;
        uint16_t* row = J.out + static_cast<size_t>(m) * 2 * J.zpad;
        row[z] = hi;
        row[J.zpad + z] = lo;
    }
}

// Zero groups of a problem (K / span) rounded up to a whole zero step (64).
int zero_groups_padded(int K, int group_size) {
    const int nz = K / (kTileK / scale_sets(group_size));
    return (nz + 63) / 64 * 64;
}

// Bytes of the float-zero sums table for one problem at token tile nt (0 otherwise).
size_t xsum_table_bytes(int qtype, const Shape& s, int nt, int group_size) {
    if (qtype != WQ4_U4_FZP || s.M <= 0) return 0;
    const size_t ld = static_cast<size_t>((s.M + nt - 1) / nt) * nt;
    return ld * 2 * zero_groups_padded(s.K, group_size) * 2;
}

// The tables of all P problems, each 256-byte aligned: total bytes (offsets relative to the first).
size_t xsum_tables_bytes(int qtype, const Shape* shapes, int P, int nt, int group_size, size_t* offs = nullptr) {
    size_t total = 0;
    for (int p = 0; p < P; ++p) {
        if (offs) offs[p] = total;
        total += (xsum_table_bytes(qtype, shapes[p], nt, group_size) + 255) / 256 * 256;
    }
    return total;
}

// Plans and launches the GEMM kernel for P problems. With fixed_scratch the workspace is the
// library's own array (kept between calls): the plan is bounded by its size and the counters it
// uses are cleared on `st` first; otherwise it is the caller's (counters already zero).
template <int MAXP>
int run_gemm(const Shape* shapes, int P, const void* const* X, const void* const* Wp, void* const* Y,
             int group_size, int dtype, int qtype, void* workspace, size_t workspace_bytes, bool fixed_scratch,
             cudaStream_t st, const EpilogueArgs* epi = nullptr) {
    DeviceInfo* dev = nullptr;
    int rc = device_info(&dev);
    if (rc) return rc;
    // float zeros: the activation-sum tables follow the plan's part of the workspace
    size_t xsum_rel[MAXP];
    const size_t xsum_bytes = xsum_tables_bytes(qtype, shapes, P, pick_token_tile(shapes, P, group_size), group_size,
                                                xsum_rel);
    if (fixed_scratch && xsum_bytes + 256 > workspace_bytes) return WQ4_ERR_WORKSPACE;
    Plan pl;
    rc = make_plan(shapes, P, dev->sm_count, fixed_scratch ? workspace_bytes - xsum_bytes - 256 : SIZE_MAX, group_size,
                   &pl);
    if (rc) return rc;
    if (pl.total_tiles == 0) return WQ4_OK;
    const size_t xsum_off = xsum_bytes ? (pl.workspace() + 255) / 256 * 256 : 0;
    const size_t need = xsum_bytes ? xsum_off + xsum_bytes : pl.workspace();
    if (need > 0 && (workspace == nullptr || workspace_bytes < need)) {
        if (trace_on())
            std::fprintf(stderr, "[wq4] the plan needs %zu bytes of workspace, %zu given\n", need,
                         workspace == nullptr ? static_cast<size_t>(0) : workspace_bytes);
        return WQ4_ERR_WORKSPACE;
    }
    if (need > 0 && !aligned16(workspace)) return WQ4_ERR_ALIGN;

    GemmParams<MAXP> params;
    GemmParams<MAXP>* prm = &params;
    std::memset(static_cast<void*>(prm), 0, sizeof(GemmParams<MAXP>));
    for (int p = 0; p < P; ++p) {
        ProblemDesc& d = prm->prob[p];
        d.wp = static_cast<const uint8_t*>(Wp[p]) + kBlobHeader;
        d.y = Y[p];
        d.M = shapes[p].M;
        d.N = shapes[p].N;
        d.K = shapes[p].K;
        d.n_tiles = shapes[p].N / kTileN;
        d.m_tiles = pl.m_tiles[p];
        d.k_groups = shapes[p].K / kTileK;
        d.tile_begin = pl.tile_begin[p];
        d.unit_begin = pl.unit_begin[p];
        d.valid = 1;
        if (d.M > 0) {
            rc = encode_x_map(&prm->xmap[p], X[p], d.M, d.K, dtype, pl.nt);
            if (rc) return rc;
        }
    }
    prm->num_problems = P;
    prm->hdr_trusted = 1;
    for (int p = 0; p < P; ++p)
        if (shapes[p].M > 0 && !blob_trusted(Wp[p], BlobKey{shapes[p].N, shapes[p].K, group_size, dtype, qtype}))
            prm->hdr_trusted = 0;
    prm->group_size = group_size;
    prm->dtype = dtype;
    prm->qtype = qtype;
    prm->early = g_opt.const_weights;
    prm->nib = nibble_consts(dtype == WQ4_BF16);
    prm->total_tiles = pl.total_tiles;
    prm->dp_tiles = pl.dp_tiles;
    prm->num_ctas = pl.grid;
    prm->sk_unit_begin = pl.sk_unit_begin;
    prm->sk_units = pl.sk_units;
    prm->cluster_split = pl.cluster;
    prm->counters = pl.counters_bytes ? static_cast<int*>(workspace) : nullptr;
    prm->partials = pl.partials_bytes ? reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + pl.counters_bytes)
                                      : nullptr;
    prm->status = dev->status;
    prm->timeout_cycles = timeout_cycles();
    prm->test_stall = g_opt.test_stall;
    if (epi) {   // single-problem calls only (wq4_mm_ex)
        prm->has_epi = 1;
        prm->alpha = epi->alpha;
        prm->beta = epi->beta;
        prm->prob[0].c = epi->c;
        prm->prob[0].bias = epi->bias;
        if (epi->beta != 0.f && epi->c) {
            EncodeTiledFn fn = encode_fn();
            if (!fn) return WQ4_ERR_CUDA;
            const cuuint64_t dims[2] = {static_cast<cuuint64_t>(shapes[0].N), static_cast<cuuint64_t>(shapes[0].M)};
            const cuuint64_t strides[1] = {static_cast<cuuint64_t>(shapes[0].N) * 2};
            // (half the token tile: the kernel copies a C tile as two halves)
            const cuuint32_t box[2] = {static_cast<cuuint32_t>(kTileN), static_cast<cuuint32_t>(pl.nt / 2)};
            const cuuint32_t estr[2] = {1, 1};
            if (fn(&prm->cmap, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(epi->c), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
                return WQ4_ERR_CUDA;
        }
    }

    // the fixed array keeps the previous call's contents: the arrival counters must start at zero
    if (fixed_scratch && pl.counters_bytes && cudaMemsetAsync(workspace, 0, pl.counters_bytes, st) != cudaSuccess)
        return WQ4_ERR_CUDA;
    if (xsum_bytes) {                                           // the pre-pass, in stream order before the GEMM
        EncodeTiledFn fn = encode_fn();
        if (!fn) return WQ4_ERR_CUDA;
        XsumBatch xb;
        std::memset(static_cast<void*>(&xb), 0, sizeof(xb));
        xb.span = kTileK / scale_sets(group_size);
        xb.status = prm->status;
        for (int p = 0; p < P; ++p) {
            if (shapes[p].M <= 0) continue;
            uint16_t* xs = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(workspace) + xsum_off + xsum_rel[p]);
            const int ld = pl.m_tiles[p] * pl.nt;
            const int zpad = zero_groups_padded(shapes[p].K, group_size);
            const cuuint64_t dims[2] = {static_cast<cuuint64_t>(2 * zpad), static_cast<cuuint64_t>(ld)};
            const cuuint64_t strides[1] = {static_cast<cuuint64_t>(2 * zpad) * 2};
            const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(pl.nt)};
            const cuuint32_t estr[2] = {1, 1};
            if (fn(&prm->sxmap[p], dtype == WQ4_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                   2, xs, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
                return WQ4_ERR_CUDA;
            XsumJob& J = xb.job[xb.P++];
            J.X = static_cast<const uint16_t*>(X[p]);
            J.out = xs;
            J.M = shapes[p].M;
            J.K = shapes[p].K;
            J.ld = ld;
            J.zpad = zpad;
            J.begin = xb.total;
            xb.total += static_cast<long long>(ld) * zpad;
        }
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(std::min<long long>((xb.total + 255) / 256, 65535)), 1, 1);
        cfg.blockDim = dim3(256, 1, 1);
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = g_opt.pdl == 0 ? 1 : 0;
        const cudaError_t e = dtype == WQ4_BF16 ? cudaLaunchKernelEx(&cfg, xsum_kernel<true>, xb)
                                                : cudaLaunchKernelEx(&cfg, xsum_kernel<false>, xb);
        if (e != cudaSuccess || cudaGetLastError() != cudaSuccess) return WQ4_ERR_CUDA;
    }
    if (trace_on()) {
        std::fprintf(stderr,
                     "[wq4] problems=%d token_tile=%d grid=%d cluster=%d tiles=%d dp_tiles=%d sk_units=%d a_src=%s "
                     "ws=%zu%s\n",
                     P, pl.nt, pl.grid, pl.cluster, pl.total_tiles, pl.dp_tiles, pl.sk_units,
                     g_opt.a_in_smem ? "smem" : "tmem", pl.workspace(), fixed_scratch ? " (fixed array)" : "");
    }
    const cudaError_t e = dispatch(prm, MAXP > 1, pl.nt, dtype, qtype, group_size, pl.grid, st);
    return e == cudaSuccess ? WQ4_OK : WQ4_ERR_CUDA;
}

// ---------------------------------------------------------------------------- fixed scratch
// For callers that may not allocate device memory: wq4_mm_static_scratch below runs wq4_mm's
// kernels with the K-split workspace taken from this array. It is zero when the module loads;
// every GPU that loads the library holds it until the process exits.
constexpr size_t kStaticScratchBytes = static_cast<size_t>(24) << 20;
__device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];
uint8_t* g_static_scratch_addr[kMaxDevices];   // device address of the array, per device
std::mutex g_static_mu;

// Device address of g_static_scratch on the current device, looked up once per device.
int static_scratch(uint8_t** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return WQ4_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_static_mu);
    if (!g_static_scratch_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr) return WQ4_ERR_CUDA;
        g_static_scratch_addr[dev] = static_cast<uint8_t*>(p);
    }
    *out = g_static_scratch_addr[dev];
    return WQ4_OK;
}

}  // namespace
}  // namespace wq4

using namespace wq4;

extern "C" {

int wq4_version(void) { return 100; }

const char* wq4_status_string(int status) {
    switch (status) {
        case WQ4_OK: return "ok";
        case WQ4_ERR_INVALID: return "invalid argument";
        case WQ4_ERR_ALIGN: return "pointer not 16-byte aligned";
        case WQ4_ERR_UNSUPPORTED: return "unsupported shape or group size";
        case WQ4_ERR_WORKSPACE: return "workspace missing or too small";
        case WQ4_ERR_CUDA: return "CUDA error";
        case WQ4_ERR_TIMEOUT: return "device pipeline wait timed out";
        case WQ4_ERR_BOUNDS: return "bounds check failed (debug build)";
        default: return "unknown status";
    }
}

size_t wq4_prepacked_bytes(int N, int K, int group_size, int qtype) {
    if (check_types(group_size, WQ4_BF16, qtype) || check_nk(N, K) || check_group(group_size, K)) return 0;
    return kBlobHeader + static_cast<size_t>(N / kTileN) * (K / kTileK) * tile_record_bytes(qtype, scale_sets(group_size));
}

int wq4_prepack(const uint32_t* Wq, const void* scales, const void* zeros, int N, int K, int group_size,
                int dtype, int qtype, void* Wp_out, wq4_stream_t stream) {
    int rc = check_types(group_size, dtype, qtype);
    if (rc) return rc;
    if ((rc = check_nk(N, K))) return rc;
    if ((rc = check_group(group_size, K))) return rc;
    if (!Wq || !Wp_out) return WQ4_ERR_INVALID;
    if (!scales && qtype != WQ4_U4B8) return WQ4_ERR_INVALID;    // zero points need scales
    if ((qtype != WQ4_U4B8) != (zeros != nullptr)) return WQ4_ERR_INVALID;
    if (!aligned16(Wq) || (scales && !aligned16(scales)) || !aligned16(Wp_out) || (zeros && !aligned16(zeros)))
        return WQ4_ERR_ALIGN;
    const cudaError_t e = launch_prepack(Wq, scales, zeros, N, K, group_size, dtype, qtype, Wp_out, stream);
    if (e != cudaSuccess) return WQ4_ERR_CUDA;
    blob_register(Wp_out, BlobKey{N, K, group_size, dtype, qtype});
    return WQ4_OK;
}

int wq4_unprepack(const void* Wp, int N, int K, int group_size, int dtype, int qtype, uint32_t* Wq_out,
                  void* scales_out, void* zeros_out, wq4_stream_t stream) {
    int rc = check_types(group_size, dtype, qtype);
    if (rc) return rc;
    if ((rc = check_nk(N, K))) return rc;
    if ((rc = check_group(group_size, K))) return rc;
    if (!Wp || !Wq_out) return WQ4_ERR_INVALID;
    if ((qtype != WQ4_U4B8) != (zeros_out != nullptr)) return WQ4_ERR_INVALID;
    if (!aligned16(Wp) || !aligned16(Wq_out) || (scales_out && !aligned16(scales_out)) ||
        (zeros_out && !aligned16(zeros_out)))
        return WQ4_ERR_ALIGN;
    const cudaError_t e = launch_unprepack(Wp, N, K, group_size, qtype, Wq_out, scales_out, zeros_out, stream);
    return e == cudaSuccess ? WQ4_OK : WQ4_ERR_CUDA;
}

int wq4_grouped_workspace_bytes(int P, const int* M, const int* N, const int* K, int group_size, size_t* bytes) {
    if (!bytes || P <= 0 || P > kMaxGroupedProblems || !M || !N || !K) return WQ4_ERR_INVALID;
    int rc = check_types(group_size, WQ4_BF16, WQ4_U4B8);
    if (rc) return rc;
    Shape shapes[kMaxGroupedProblems];
    for (int p = 0; p < P; ++p) {
        if (M[p] < 0) return WQ4_ERR_INVALID;
        if ((rc = check_nk(N[p], K[p]))) return rc;
        if ((rc = check_group(group_size, K[p]))) return rc;
        shapes[p] = Shape{M[p], N[p], K[p]};
    }
    DeviceInfo* dev = nullptr;
    if ((rc = device_info(&dev))) return rc;
    if (grouped_uses_decode(P, M, K)) {                        // the decode kernel needs none
        *bytes = 0;
        return WQ4_OK;
    }
    Plan pl;
    if ((rc = make_plan(shapes, P, dev->sm_count, SIZE_MAX, group_size, &pl))) return rc;
    *bytes = pl.workspace();
    return WQ4_OK;
}

int wq4_workspace_bytes_ex(int M, int N, int K, int group_size, int qtype, size_t* bytes) {
    int rc = check_types(group_size, WQ4_BF16, qtype);
    if (rc) return rc;
    if ((rc = wq4_workspace_bytes(M, N, K, group_size, bytes))) return rc;
    DeviceInfo* dev = nullptr;
    if ((rc = device_info(&dev))) return rc;
    if (M > 0 && !uses_decode_kernel(M, N, K)) {
        const Shape sh{M, N, K};
        const size_t xs = xsum_table_bytes(qtype, sh, pick_token_tile(&sh, 1, group_size), group_size);
        if (xs) *bytes = (*bytes + 255) / 256 * 256 + xs;
    }
    return WQ4_OK;
}

int wq4_grouped_workspace_bytes_ex(int P, const int* M, const int* N, const int* K, int group_size, int qtype,
                                   size_t* bytes) {
    int rc = check_types(group_size, WQ4_BF16, qtype);
    if (rc) return rc;
    if ((rc = wq4_grouped_workspace_bytes(P, M, N, K, group_size, bytes))) return rc;
    if (qtype != WQ4_U4_FZP || grouped_uses_decode(P, M, K)) return WQ4_OK;
    Shape shapes[kMaxGroupedProblems];
    for (int p = 0; p < P; ++p) shapes[p] = Shape{M[p], N[p], K[p]};
    const size_t xs = xsum_tables_bytes(qtype, shapes, P, pick_token_tile(shapes, P, group_size), group_size);
    if (xs) *bytes = (*bytes + 255) / 256 * 256 + xs;
    return WQ4_OK;
}

int wq4_workspace_bytes(int M, int N, int K, int group_size, size_t* bytes) {
    const int rc = wq4_grouped_workspace_bytes(1, &M, &N, &K, group_size, bytes);
    if (rc == WQ4_OK && M > 0 && uses_decode_kernel(M, N, K)) *bytes = 0;   // that kernel needs none
    return rc;
}

// The decode kernel's launch settings from the options.
static DecodeLaunch decode_launch(DeviceInfo* dev, EncodeTiledFn fn, bool hdr_trusted) {
    DecodeLaunch L;
    L.sm_count = dev->sm_count;
    L.status = dev->status;
    L.timeout_cycles = timeout_cycles();
    L.encode_fn = reinterpret_cast<void*>(fn);
    L.pdl = g_opt.pdl == 0;
    L.test_stall = g_opt.test_stall;
    L.const_weights = g_opt.const_weights;
    L.trigger_late = g_opt.decode_trigger == 0 ? 1 : 0;
    L.depth = g_opt.decode_depth;
    L.hdr_trusted = hdr_trusted ? 1 : 0;
    return L;
}

static int mm_impl(const void* X, const void* Wp, void* Y, int M, int N, int K, int group_size, int dtype,
                   int qtype, const EpilogueArgs* epi, void* workspace, size_t workspace_bytes, bool fixed_scratch,
                   wq4_stream_t stream) {
    int rc = check_types(group_size, dtype, qtype);
    if (rc) return rc;
    if (M < 0) return WQ4_ERR_INVALID;
    if ((rc = check_nk(N, K))) return rc;
    if ((rc = check_group(group_size, K))) return rc;
    if (M == 0) return WQ4_OK;
    if (!X || !Wp || !Y) return WQ4_ERR_INVALID;
    if (!aligned16(X) || !aligned16(Wp) || !aligned16(Y)) return WQ4_ERR_ALIGN;
    // decode-sized M: the warp-level MMA kernel (whole row blocks per CTA, no workspace)
    if (const int rows = decode_rows_per_launch(M, N, K)) {
        DeviceInfo* dev = nullptr;
        if ((rc = device_info(&dev))) return rc;
        EncodeTiledFn fn = encode_fn();
        if (!fn) return WQ4_ERR_CUDA;
        for (int m0 = 0; m0 < M; m0 += rows) {   // one launch, or two of at most 16 rows
            const int mr = M - m0 < rows ? M - m0 : rows;
            const uint8_t* x = static_cast<const uint8_t*>(X) + static_cast<size_t>(m0) * K * 2;
            uint8_t* y = static_cast<uint8_t*>(Y) + static_cast<size_t>(m0) * N * 2;
            EpilogueArgs e_part;
            if (epi) {
                e_part = *epi;
                if (e_part.c) e_part.c = static_cast<const uint8_t*>(e_part.c) + static_cast<size_t>(m0) * N * 2;
            }
            const DecodeLaunch L =
                decode_launch(dev, fn, blob_trusted(Wp, BlobKey{N, K, group_size, dtype, qtype}));
            int grid = 0, depth = 0;
            const cudaError_t e = launch_decode(L, x, Wp, y, mr, N, K, group_size, dtype, qtype, epi ? &e_part : nullptr,
                                                &grid, &depth, stream);
            if (trace_on())
                std::fprintf(stderr, "[wq4] decode kernel: M=%d (rows %d..%d) N=%d K=%d grid=%d ring=%d const_weights=%d "
                             "header_alongside=%d (%s)\n", M, m0, m0 + mr, N, K, grid, depth, g_opt.const_weights,
                             L.hdr_trusted, e == cudaSuccess ? "ok" : cudaGetErrorString(e));
            if (e != cudaSuccess) return WQ4_ERR_CUDA;
        }
        return WQ4_OK;
    }
    const Shape shape{M, N, K};
    const void* xs[1] = {X};
    const void* ws[1] = {Wp};
    void* ys[1] = {Y};
    return run_gemm<1>(&shape, 1, xs, ws, ys, group_size, dtype, qtype, workspace, workspace_bytes, fixed_scratch,
                       stream, epi);
}

int wq4_mm(const void* X, const void* Wp, void* Y, int M, int N, int K, int group_size, int dtype, int qtype,
           void* workspace, size_t workspace_bytes, wq4_stream_t stream) {
    return mm_impl(X, Wp, Y, M, N, K, group_size, dtype, qtype, nullptr, workspace, workspace_bytes, false, stream);
}

int wq4_mm_ex(const void* X, const void* Wp, void* Y, int M, int N, int K, int group_size, int dtype, int qtype,
              float alpha, const void* C, float beta, const void* bias, void* workspace, size_t workspace_bytes,
              wq4_stream_t stream) {
    if (beta != 0.f && !C) return WQ4_ERR_INVALID;
    if ((C && !aligned16(C)) || (bias && !aligned16(bias))) return WQ4_ERR_ALIGN;
    const EpilogueArgs epi{alpha, beta, beta != 0.f ? C : nullptr, bias};
    return mm_impl(X, Wp, Y, M, N, K, group_size, dtype, qtype, &epi, workspace, workspace_bytes, false, stream);
}

int wq4_grouped_mm(int P, const int* M, const int* N, const int* K, const void* const* X, const void* const* Wp,
                   void* const* Y, int group_size, int dtype, int qtype, void* workspace, size_t workspace_bytes,
                   wq4_stream_t stream) {
    int rc = check_types(group_size, dtype, qtype);
    if (rc) return rc;
    if (P <= 0 || !M || !N || !K || !X || !Wp || !Y) return WQ4_ERR_INVALID;
    if (P > kMaxGroupedProblems) return WQ4_ERR_UNSUPPORTED;
    Shape shapes[kMaxGroupedProblems];
    for (int p = 0; p < P; ++p) {
        if (M[p] < 0) return WQ4_ERR_INVALID;
        if ((rc = check_nk(N[p], K[p]))) return rc;
        if ((rc = check_group(group_size, K[p]))) return rc;
        if (M[p] > 0) {
            if (!X[p] || !Wp[p] || !Y[p]) return WQ4_ERR_INVALID;
            if (!aligned16(X[p]) || !aligned16(Wp[p]) || !aligned16(Y[p])) return WQ4_ERR_ALIGN;
        }
        shapes[p] = Shape{M[p], N[p], K[p]};
    }
    if (grouped_uses_decode(P, M, K)) {
        // decode-sized: the non-empty problems in one launch of the decode kernel (no workspace)
        DeviceInfo* dev = nullptr;
        if ((rc = device_info(&dev))) return rc;
        EncodeTiledFn fn = encode_fn();
        if (!fn) return WQ4_ERR_CUDA;
        const void* xs[kMaxGroupedProblems];
        const void* wps[kMaxGroupedProblems];
        void* ys[kMaxGroupedProblems];
        int ms[kMaxGroupedProblems], ns[kMaxGroupedProblems], ks[kMaxGroupedProblems];
        int n = 0;
        bool trusted = true;
        for (int p = 0; p < P; ++p) {
            if (M[p] == 0) continue;
            xs[n] = X[p];
            wps[n] = Wp[p];
            ys[n] = Y[p];
            ms[n] = M[p];
            ns[n] = N[p];
            ks[n] = K[p];
            trusted = trusted && blob_trusted(Wp[p], BlobKey{N[p], K[p], group_size, dtype, qtype});
            ++n;
        }
        int grid = 0, depth = 0;
        const cudaError_t e = launch_decode_grouped(decode_launch(dev, fn, trusted), n, xs, wps, ys, ms, ns, ks, group_size,
                                                    dtype, qtype, &grid, &depth, stream);
        if (trace_on())
            std::fprintf(stderr, "[wq4] grouped decode kernel: problems=%d grid=%d ring=%d (%s)\n", n, grid, depth,
                         e == cudaSuccess ? "ok" : cudaGetErrorString(e));
        return e == cudaSuccess ? WQ4_OK : WQ4_ERR_CUDA;
    }
    return run_gemm<kMaxGroupedProblems>(shapes, P, X, Wp, Y, group_size, dtype, qtype, workspace, workspace_bytes,
                                         false, stream);
}

// ------------------------------------------------------------------ device-resident shapes
namespace wq4 {
struct DynSetup {
    int P, nt;
    int cap[kMaxGroupedProblems];
    int n_tiles[kMaxGroupedProblems];
};

// Turns the device array of token counts into the GEMM's tile table: counts clamped to
// [0, capacity], tiles per problem, first tile of each problem, total (one thread; P <= 64).
__global__ void dyn_table_kernel(const int* __restrict__ M_dev, const __grid_constant__ DynSetup su, DynTable* t) {
    if (threadIdx.x != 0) return;
    int acc = 0;
    for (int p = 0; p < su.P; ++p) {
        int m = M_dev[p];
        m = m < 0 ? 0 : (m > su.cap[p] ? su.cap[p] : m);
        t->M[p] = m;
        t->tile_begin[p] = acc;
        acc += (m + su.nt - 1) / su.nt * su.n_tiles[p];
    }
    t->total_tiles = acc;
}
}  // namespace wq4

extern "C++" {
namespace wq4 {
// Device-resident per-problem pointers: one thread per problem of this launch's chunk writes the
// problem's descriptor (pointers read from the device arrays, shape and tile ranges from the
// launch parameters) and, for a non-empty problem, its activation tensor map: the map the host
// encoded for its shape copied into the table, then its global address replaced in place
// (tensormap.replace) and released to the tensor-map proxy. A null or misaligned pointer,
// or a blob whose header does not match the call, marks the problem invalid (the GEMM skips its
// tiles) and sets the status word's bad-argument bit.
template <int C>
__global__ void ptr_setup_kernel(const __grid_constant__ PtrSetup<C> su, const void* const* __restrict__ X,
                                 const void* const* __restrict__ W, void* const* __restrict__ Y,
                                 ProblemDesc* __restrict__ tab, CUtensorMap* __restrict__ maps,
                                 unsigned int* status) {
    // Launched with programmatic dependent launch: the GEMM behind it may start its set-up at once
    // (it reads the tables only after this grid has completed); the pointer arrays and the tables
    // are touched only after the kernel ahead (which may write the former or read the latter) has.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= su.count) return;
    const int p = su.p0 + i;
    ProblemDesc d;
    memset(&d, 0, sizeof(d));
    d.M = su.M[i];
    d.N = su.N[i];
    d.K = su.K[i];
    d.n_tiles = su.N[i] / kTileN;
    d.m_tiles = su.m_tiles[i];
    d.k_groups = su.K[i] / kTileK;
    d.tile_begin = su.tile_begin[i];
    d.unit_begin = su.unit_begin[i];
    d.valid = 1;
    if (d.M > 0) {
        const void* x = X[p];
        const void* w = W[p];
        void* y = Y[p];
        // the host-encoded map goes to the table while the pointers load (an invalid problem's map
        // is never used)
        const uint4* src = reinterpret_cast<const uint4*>(&su.tmpl[i]);
        uint4* dst = reinterpret_cast<uint4*>(&maps[p]);
#pragma unroll
        for (int k = 0; k < 8; ++k) dst[k] = src[k];
        const bool ok = x && w && y &&
                        ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(w) |
                          reinterpret_cast<uintptr_t>(y)) & 15u) == 0 &&
                        blob_header_ok(static_cast<const uint32_t*>(w), d.N, d.K, su.group_size, su.dtype, su.qtype);
        if (ok) {
            d.wp = static_cast<const uint8_t*>(w) + kBlobHeader;
            d.y = y;
            asm volatile("tensormap.replace.tile.global_address.global.b1024.b64 [%0], %1;" ::"l"(dst),
                         "l"(reinterpret_cast<uint64_t>(x))
                         : "memory");
            asm volatile("fence.proxy.tensormap::generic.release.gpu;" ::: "memory");
        } else {
            d.valid = 0;
            atomicOr(status, kStatusBadBlob);
        }
    }
    tab[p] = d;
}
}  // namespace wq4
}  // extern "C++"

int wq4_grouped_device_m_workspace_bytes(int P, size_t* bytes) {
    if (!bytes || P <= 0) return WQ4_ERR_INVALID;
    if (P > kMaxGroupedProblems) return WQ4_ERR_UNSUPPORTED;
    *bytes = (sizeof(DynTable) + 255) / 256 * 256;
    return WQ4_OK;
}

int wq4_grouped_mm_device_m(int P, const int* M_dev, const int* M_cap, const int* N, const int* K,
                            const void* const* X, const void* const* Wp, void* const* Y, int group_size, int dtype,
                            int qtype, void* workspace, size_t workspace_bytes, wq4_stream_t stream) {
    int rc = check_types(group_size, dtype, qtype);
    if (rc) return rc;
    if (qtype == WQ4_U4_FZP) return WQ4_ERR_UNSUPPORTED;        // float zeros: host-known shapes only
    if (P <= 0 || !M_dev || !M_cap || !N || !K || !X || !Wp || !Y) return WQ4_ERR_INVALID;
    if (P > kMaxGroupedProblems) return WQ4_ERR_UNSUPPORTED;
    if (reinterpret_cast<uintptr_t>(M_dev) & 3) return WQ4_ERR_ALIGN;
    if (!workspace || workspace_bytes < (sizeof(DynTable) + 255) / 256 * 256) return WQ4_ERR_WORKSPACE;
    if (!aligned16(workspace)) return WQ4_ERR_ALIGN;
    for (int p = 0; p < P; ++p) {
        if (M_cap[p] < 0) return WQ4_ERR_INVALID;
        if ((rc = check_nk(N[p], K[p]))) return rc;
        if ((rc = check_group(group_size, K[p]))) return rc;
        if (M_cap[p] > 0) {
            if (!X[p] || !Wp[p] || !Y[p]) return WQ4_ERR_INVALID;
            if (!aligned16(X[p]) || !aligned16(Wp[p]) || !aligned16(Y[p])) return WQ4_ERR_ALIGN;
        }
    }
    DeviceInfo* dev = nullptr;
    if ((rc = device_info(&dev))) return rc;
    // Plan for the capacities: the token tile and the grid; every tile whole (the tile count is
    // known only on the device).
    const int nt = token_tile_for(M_cap, P);
    long long max_tiles = 0;
    auto* prm = new (std::nothrow) GemmParams<kMaxGroupedProblems>();
    if (!prm) return WQ4_ERR_CUDA;
    std::memset(static_cast<void*>(prm), 0, sizeof(*prm));
    DynSetup su;
    std::memset(static_cast<void*>(&su), 0, sizeof(su));
    su.P = P;
    su.nt = nt;
    for (int p = 0; p < P; ++p) {
        ProblemDesc& d = prm->prob[p];
        d.wp = static_cast<const uint8_t*>(Wp[p]) + kBlobHeader;
        d.y = Y[p];
        d.M = M_cap[p];
        d.N = N[p];
        d.K = K[p];
        d.n_tiles = N[p] / kTileN;
        d.m_tiles = (M_cap[p] + nt - 1) / nt;
        d.k_groups = K[p] / kTileK;
        d.tile_begin = static_cast<int>(max_tiles);
        d.valid = 1;
        max_tiles += static_cast<long long>(d.m_tiles) * d.n_tiles;
        su.cap[p] = M_cap[p];
        su.n_tiles[p] = d.n_tiles;
        if (M_cap[p] > 0) {
            rc = encode_x_map(&prm->xmap[p], X[p], M_cap[p], K[p], dtype, nt);
            if (rc) {
                delete prm;
                return rc;
            }
        }
    }
    if (max_tiles >= (1LL << 30)) {
        delete prm;
        return WQ4_ERR_UNSUPPORTED;
    }
    const int grid = static_cast<int>(std::max<long long>(1, std::min<long long>(dev->sm_count, max_tiles)));
    prm->num_problems = P;
    prm->group_size = group_size;
    prm->dtype = dtype;
    prm->qtype = qtype;
    prm->nib = nibble_consts(dtype == WQ4_BF16);
    prm->total_tiles = static_cast<int>(max_tiles);
    prm->dp_tiles = static_cast<int>(max_tiles);
    prm->num_ctas = grid;
    prm->status = dev->status;
    prm->timeout_cycles = timeout_cycles();
    prm->test_stall = g_opt.test_stall;
    prm->dyn = static_cast<const DynTable*>(workspace);
    dyn_table_kernel<<<1, 32, 0, stream>>>(M_dev, su, static_cast<DynTable*>(workspace));
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) e = dispatch(prm, true, nt, dtype, qtype, group_size, grid, stream);
    if (trace_on())
        std::fprintf(stderr, "[wq4] device-resident shapes: problems=%d token_tile=%d grid=%d max_tiles=%lld (%s)\n", P,
                     nt, grid, max_tiles, e == cudaSuccess ? "ok" : cudaGetErrorString(e));
    delete prm;
    return e == cudaSuccess ? WQ4_OK : WQ4_ERR_CUDA;
}

// ------------------------------------------------------------------ device-resident pointers
extern "C++" {
namespace wq4 {
namespace {
// Workspace of the device-pointer grouped call: the plan's K-split part (counters first, zero
// between calls), then the problem table, then one 128-byte activation map per problem.
struct PtrLayout {
    size_t tab_off, map_off, total;
};
PtrLayout ptr_layout(const Plan& pl, int P) {
    PtrLayout L;
    L.tab_off = (pl.workspace() + 255) / 256 * 256;
    L.map_off = (L.tab_off + static_cast<size_t>(P) * sizeof(ProblemDesc) + 127) / 128 * 128;
    L.total = L.map_off + static_cast<size_t>(P) * sizeof(CUtensorMap);
    return L;
}

int ptr_shapes(int P, const int* M, const int* N, const int* K, int group_size, Shape* shapes) {
    int rc = WQ4_OK;
    for (int p = 0; p < P; ++p) {
        if (M[p] < 0) return WQ4_ERR_INVALID;
        if ((rc = check_nk(N[p], K[p]))) return rc;
        if ((rc = check_group(group_size, K[p]))) return rc;
        shapes[p] = Shape{M[p], N[p], K[p]};
    }
    return WQ4_OK;
}

// Reads back the maps the set-up kernels wrote and compares each with the host encoder's map for
// the same address and row count (the test aid of WQ4_OPT_VERIFY_DEV_PTRS).
int verify_ptr_maps(int P, const Shape* shapes, const void* const* X_dev, const uint8_t* maps_dev, int dtype, int nt,
                    cudaStream_t st) {
    if (cudaStreamSynchronize(st) != cudaSuccess) return WQ4_ERR_CUDA;
    std::vector<const void*> xs(P);
    std::vector<uint8_t> got(static_cast<size_t>(P) * sizeof(CUtensorMap));
    if (cudaMemcpy(xs.data(), X_dev, sizeof(void*) * P, cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemcpy(got.data(), maps_dev, got.size(), cudaMemcpyDeviceToHost) != cudaSuccess)
        return WQ4_ERR_CUDA;
    int bad = 0;
    for (int p = 0; p < P; ++p) {
        if (shapes[p].M == 0 || !xs[p] || !aligned16(xs[p])) continue;
        CUtensorMap want;
        const int rc = encode_x_map(&want, xs[p], shapes[p].M, shapes[p].K, dtype, nt);
        if (rc) return rc;
        const uint8_t* g = got.data() + static_cast<size_t>(p) * sizeof(CUtensorMap);
        const uint8_t* w = reinterpret_cast<const uint8_t*>(&want);
        const int bad_before = bad;
        for (size_t b = 0; b < sizeof(CUtensorMap); ++b) bad += g[b] != w[b];
        if (trace_on() && bad != bad_before)
            std::fprintf(stderr, "[wq4] map %d differs: X=%p M=%d K=%d\n", p, xs[p], shapes[p].M, shapes[p].K);
        if (trace_on() && bad != bad_before && bad_before == 0) {   // the first mismatching map in full
            std::fprintf(stderr, "[wq4] problem %d (M=%d K=%d, X=%p): map bytes differ\n", p, shapes[p].M, shapes[p].K,
                         xs[p]);
            for (int row = 0; row < 8; ++row) {
                std::fprintf(stderr, "[wq4]  %3d device", row * 16);
                for (int b = 0; b < 16; ++b) std::fprintf(stderr, " %02x", g[row * 16 + b]);
                std::fprintf(stderr, "\n[wq4]      host  ");
                for (int b = 0; b < 16; ++b) std::fprintf(stderr, " %02x", w[row * 16 + b]);
                std::fprintf(stderr, "\n");
            }
        }
    }
    if (trace_on() && bad) std::fprintf(stderr, "[wq4] %d map bytes differ in all\n", bad);
    return bad ? WQ4_ERR_UNSUPPORTED : WQ4_OK;
}
// Launches the set-up kernel over P problems, C per launch (their maps in its parameters).
template <int C>
int ptr_setup(int P, const int* M, const int* N, const int* K, const Plan& pl, const void* const* X_dev,
              const void* const* Wp_dev, void* const* Y_dev, int group_size, int dtype, int qtype, void* stand_in,
              ProblemDesc* tab, CUtensorMap* maps, unsigned int* status, cudaStream_t stream) {
    auto su = std::make_unique<PtrSetup<C>>();
    std::memset(static_cast<void*>(su.get()), 0, sizeof(PtrSetup<C>));
    su->group_size = group_size;
    su->dtype = dtype;
    su->qtype = qtype;
    for (int p0 = 0; p0 < P; p0 += C) {
        const int cnt = std::min(C, P - p0);
        su->p0 = p0;
        su->count = cnt;
        for (int i = 0; i < cnt; ++i) {
            const int p = p0 + i;
            su->M[i] = M[p];
            su->N[i] = N[p];
            su->K[i] = K[p];
            su->m_tiles[i] = pl.m_tiles[p];
            su->tile_begin[i] = pl.tile_begin[p];
            su->unit_begin[i] = pl.unit_begin[p];
            // the stand-in address (the workspace: any 16-byte aligned one) is replaced on the device
            if (M[p] > 0) {
                const int rc = encode_x_map(&su->tmpl[i], stand_in, M[p], K[p], dtype, pl.nt);
                if (rc) return rc;
            }
        }
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((cnt + 127) / 128, 1, 1);
        cfg.blockDim = dim3(C < 128 ? C : 128, 1, 1);
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = g_opt.pdl == 0 ? 1 : 0;
        if (cudaLaunchKernelEx(&cfg, ptr_setup_kernel<C>, static_cast<const PtrSetup<C>&>(*su), X_dev, Wp_dev, Y_dev,
                               tab, maps, status) != cudaSuccess ||
            cudaGetLastError() != cudaSuccess)
            return WQ4_ERR_CUDA;
    }
    return WQ4_OK;
}
}  // namespace
}  // namespace wq4
}  // extern "C++"

int wq4_grouped_dev_ptrs_workspace_bytes(int P, const int* M, const int* N, const int* K, int group_size,
                                         size_t* bytes) {
    if (!bytes || P <= 0 || !M || !N || !K) return WQ4_ERR_INVALID;
    if (P > kMaxDevPtrProblems) return WQ4_ERR_UNSUPPORTED;
    int rc = check_types(group_size, WQ4_BF16, WQ4_U4B8);
    if (rc) return rc;
    std::vector<Shape> shapes(P);
    if ((rc = ptr_shapes(P, M, N, K, group_size, shapes.data()))) return rc;
    DeviceInfo* dev = nullptr;
    if ((rc = device_info(&dev))) return rc;
    auto pl = std::make_unique<Plan>();
    if ((rc = make_plan(shapes.data(), P, dev->sm_count, SIZE_MAX, group_size, pl.get()))) return rc;
    *bytes = ptr_layout(*pl, P).total;
    return WQ4_OK;
}

int wq4_grouped_mm_dev_ptrs(int P, const int* M, const int* N, const int* K, const void* const* X_dev,
                            const void* const* Wp_dev, void* const* Y_dev, int group_size, int dtype, int qtype,
                            void* workspace, size_t workspace_bytes, wq4_stream_t stream) {
    int rc = check_types(group_size, dtype, qtype);
    if (rc) return rc;
    if (P <= 0 || !M || !N || !K || !X_dev || !Wp_dev || !Y_dev) return WQ4_ERR_INVALID;
    if (P > kMaxDevPtrProblems || qtype == WQ4_U4_FZP) return WQ4_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(X_dev) | reinterpret_cast<uintptr_t>(Wp_dev) |
         reinterpret_cast<uintptr_t>(Y_dev)) & 7u)
        return WQ4_ERR_ALIGN;
    std::vector<Shape> shapes(P);
    if ((rc = ptr_shapes(P, M, N, K, group_size, shapes.data()))) return rc;
    DeviceInfo* dev = nullptr;
    if ((rc = device_info(&dev))) return rc;
    auto pl = std::make_unique<Plan>();
    if ((rc = make_plan(shapes.data(), P, dev->sm_count, SIZE_MAX, group_size, pl.get()))) return rc;
    if (pl->total_tiles == 0) return WQ4_OK;
    const PtrLayout L = ptr_layout(*pl, P);
    if (!workspace || workspace_bytes < L.total) return WQ4_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) & 127u) return WQ4_ERR_ALIGN;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    auto* tab = reinterpret_cast<ProblemDesc*>(ws + L.tab_off);
    auto* maps = reinterpret_cast<CUtensorMap*>(ws + L.map_off);

    rc = P <= kPtrSetupSmall ? ptr_setup<kPtrSetupSmall>(P, M, N, K, *pl, X_dev, Wp_dev, Y_dev, group_size, dtype, qtype,
                                                         workspace, tab, maps, dev->status, stream)
                             : ptr_setup<kPtrSetupChunk>(P, M, N, K, *pl, X_dev, Wp_dev, Y_dev, group_size, dtype, qtype,
                                                         workspace, tab, maps, dev->status, stream);
    if (rc) return rc;
    if (g_opt.verify_dev_ptrs)
        return verify_ptr_maps(P, shapes.data(), X_dev, ws + L.map_off, dtype, pl->nt, stream);

    GemmParams<1> prm;
    std::memset(static_cast<void*>(&prm), 0, sizeof(prm));
    prm.prob_tab = tab;
    prm.xmap_tab = maps;
    prm.num_problems = P;
    prm.group_size = group_size;
    prm.dtype = dtype;
    prm.qtype = qtype;
    prm.nib = nibble_consts(dtype == WQ4_BF16);
    prm.total_tiles = pl->total_tiles;
    prm.dp_tiles = pl->dp_tiles;
    prm.num_ctas = pl->grid;
    prm.sk_unit_begin = pl->sk_unit_begin;
    prm.sk_units = pl->sk_units;
    prm.cluster_split = pl->cluster;
    prm.counters = pl->counters_bytes ? reinterpret_cast<int*>(ws) : nullptr;
    prm.partials = pl->partials_bytes ? reinterpret_cast<float*>(ws + pl->counters_bytes) : nullptr;
    prm.status = dev->status;
    prm.timeout_cycles = timeout_cycles();
    prm.test_stall = g_opt.test_stall;
    const cudaError_t e = dispatch(&prm, false, pl->nt, dtype, qtype, group_size, pl->grid, stream);
    if (trace_on())
        std::fprintf(stderr,
                     "[wq4] device pointers: problems=%d token_tile=%d grid=%d cluster=%d tiles=%d "
                     "dp_tiles=%d sk_units=%d ws=%zu (%s)\n",
                     P, pl->nt, pl->grid, pl->cluster, pl->total_tiles, pl->dp_tiles, pl->sk_units, L.total,
                     e == cudaSuccess ? "ok" : cudaGetErrorString(e));
    return e == cudaSuccess ? WQ4_OK : WQ4_ERR_CUDA;
}

int wq4_get_last_error(wq4_stream_t stream) {
    const cudaError_t se = cudaStreamSynchronize(stream);
    DeviceInfo* dev = nullptr;
    int rc = device_info(&dev);
    if (rc) return rc;
    unsigned int w[1 + check::kRecordWords] = {};
    if (cudaMemcpy(w, dev->status, sizeof(w), cudaMemcpyDeviceToHost) != cudaSuccess) return WQ4_ERR_CUDA;
    const unsigned int st = w[0];
    if (st) {
        const unsigned int zero[1 + check::kRecordWords] = {};
        cudaMemcpy(dev->status, zero, sizeof(zero), cudaMemcpyHostToDevice);
        if (st & kStatusBounds) {
            std::lock_guard<std::mutex> lk(g_mu);
            g_violation[0] = 1;
            for (int i = 0; i < check::kRecordWords; ++i) g_violation[1 + i] = static_cast<int>(w[1 + i]);
            return WQ4_ERR_BOUNDS;
        }
        return (st & kStatusBadBlob) ? WQ4_ERR_INVALID : WQ4_ERR_TIMEOUT;
    }
    if (se != cudaSuccess || cudaGetLastError() != cudaSuccess) return WQ4_ERR_CUDA;
    return WQ4_OK;
}

int wq4_debug_checks(void) { return kDebugChecks ? 1 : 0; }

int wq4_last_violation(int* record) {
    if (!record) return WQ4_ERR_INVALID;
    std::lock_guard<std::mutex> lk(g_mu);
    const int seen = g_violation[0];
    for (int i = 0; i < check::kRecordWords; ++i) record[i] = seen ? g_violation[1 + i] : 0;
    g_violation[0] = 0;
    return seen;
}

int wq4_set_option(int key, long long value) {
    switch (key) {
        case WQ4_OPT_TOKEN_TILE:
            if (value != 0 && value != 16 && value != 64 && value != 128 && value != 160 && value != 192)
                return WQ4_ERR_INVALID;
            g_opt.token_tile = static_cast<int>(value);
            return WQ4_OK;
        case WQ4_OPT_GRID:
            if (value < 0 || value > 4096) return WQ4_ERR_INVALID;
            g_opt.grid = static_cast<int>(value);
            return WQ4_OK;
        case WQ4_OPT_SPLIT_ALL:
            g_opt.split_all = value ? 1 : 0;
            return WQ4_OK;
        case WQ4_OPT_TIMEOUT_CYCLES:
            if (value < 0) return WQ4_ERR_INVALID;
            g_opt.timeout_cycles = value;
            return WQ4_OK;
        case WQ4_OPT_TRACE:
            g_opt.trace = value ? 1 : 0;
            return WQ4_OK;
        case WQ4_OPT_A_IN_SMEM:
            g_opt.a_in_smem = value ? 1 : 0;
            return WQ4_OK;
        case WQ4_OPT_CLUSTER:
            if (value < -1 || value == 1 || value > 8) return WQ4_ERR_INVALID;
            g_opt.cluster = static_cast<int>(value);
            return WQ4_OK;
        case WQ4_OPT_DECODE:
            if (value < -1 || value > 1) return WQ4_ERR_INVALID;
            g_opt.decode = static_cast<int>(value);
            return WQ4_OK;
        case WQ4_OPT_PDL:
            if (value < -1 || value > 0) return WQ4_ERR_INVALID;
            g_opt.pdl = static_cast<int>(value);
            return WQ4_OK;
        case WQ4_OPT_TEST_STALL:
            if (value < 0 || value > 1) return WQ4_ERR_INVALID;
            g_opt.test_stall = static_cast<int>(value);
            return WQ4_OK;
        case WQ4_OPT_CONST_WEIGHTS:
            if (value < 0 || value > 1) return WQ4_ERR_INVALID;
            g_opt.const_weights = static_cast<int>(value);
            return WQ4_OK;
        case WQ4_OPT_DECODE_DEPTH:
            if (value != 0 && (value < 2 || value > 16)) return WQ4_ERR_INVALID;
            g_opt.decode_depth = static_cast<int>(value);
            return WQ4_OK;
        case WQ4_OPT_DECODE_TRIGGER:
            if (value < 0 || value > 1) return WQ4_ERR_INVALID;
            g_opt.decode_trigger = static_cast<int>(value);
            return WQ4_OK;
        case WQ4_OPT_VERIFY_DEV_PTRS:
            if (value < 0 || value > 1) return WQ4_ERR_INVALID;
            g_opt.verify_dev_ptrs = static_cast<int>(value);
            return WQ4_OK;
        default: return WQ4_ERR_INVALID;
    }
}

long long wq4_get_option(int key) {
    switch (key) {
        case WQ4_OPT_TOKEN_TILE: return g_opt.token_tile;
        case WQ4_OPT_GRID: return g_opt.grid;
        case WQ4_OPT_SPLIT_ALL: return g_opt.split_all;
        case WQ4_OPT_TIMEOUT_CYCLES: return g_opt.timeout_cycles;
        case WQ4_OPT_TRACE: return trace_on() ? 1 : 0;
        case WQ4_OPT_A_IN_SMEM: return g_opt.a_in_smem;
        case WQ4_OPT_CLUSTER: return g_opt.cluster;
        case WQ4_OPT_DECODE: return g_opt.decode;
        case WQ4_OPT_PDL: return g_opt.pdl;
        case WQ4_OPT_TEST_STALL: return g_opt.test_stall;
        case WQ4_OPT_CONST_WEIGHTS: return g_opt.const_weights;
        case WQ4_OPT_DECODE_DEPTH: return g_opt.decode_depth;
        case WQ4_OPT_DECODE_TRIGGER: return g_opt.decode_trigger;
        case WQ4_OPT_VERIFY_DEV_PTRS: return g_opt.verify_dev_ptrs;
        default: return -1;
    }
}

int wq4_mm_static_scratch(const void* X, const void* Wp, void* Y, int M, int N, int K, int group_size, int dtype,
                          int qtype, wq4_stream_t stream) {
    int rc = check_types(group_size, dtype, qtype);
    if (rc) return rc;
    // resolved before the shape is looked at, so that a device's first call always does the
    // lookup, even one that needs no scratch (M == 0, or a decode-sized M)
    uint8_t* scratch = nullptr;
    if ((rc = static_scratch(&scratch))) return rc;
    return mm_impl(X, Wp, Y, M, N, K, group_size, dtype, qtype, nullptr, scratch, kStaticScratchBytes, true, stream);
}

}  // extern "C"
