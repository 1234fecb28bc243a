// Bounds checks of the debug build (compiled with -DWQ4_DEBUG=1 into libwq4_debug.so; the release
// library compiles every check away, its condition unevaluated).
//
// In place of a memory checker, each kernel checks the coordinates it derives before it uses them:
// every tiled tensor copy's innermost coordinate (16-byte multiple, box inside the extent), every
// weight record's address range inside its blob, every scheduled tile against its problem's M, N
// and K groups, the K-split workspace slots and counters, and every output column against N: the
// conditions the host establishes for each call ("machete_mainloop.cuh", can_implement), checked
// again where the device relies on them.
//
// A failed check skips the access and never faults or waits: a skipped copy is replaced by a
// plain arrival on its barrier (the stage's phase completes, its data undefined), the first
// violation (site and three values) is recorded after the status word, the status word's bounds
// bit is set and the CTA's abort flag raised; the call then reports WQ4_ERR_BOUNDS and its outputs
// are undefined. The predicates are plain functions, host-callable, so that they are tested on
// the CPU as well.
#pragma once

#include <cstdint>

#if defined(__CUDACC__)
#include "wq4_params.h"
#define WQ4_HD __host__ __device__
#else
#define WQ4_HD
#endif

namespace wq4 {
namespace check {

// The check sites (the first word of a violation record) and the three values recorded with each.
enum Site : int {
    kSiteTile = 1,        // scheduled tile outside its problem: m-tile, n-tile, end of its group range
    kSiteXTile = 2,       // activation tile copy: K coordinate, token row, K
    kSiteXSums = 3,       // activation-sum panel copy: zero-group coordinate, token row, padded width;
                          // or the sums kernel's store: token row, zero group, rows of the table
    kSiteWRecord = 4,     // weight record copy: byte offset in the blob, n-tile, group
    kSiteCTile = 5,       // epilogue C tile copy: column coordinate, token row, N
    kSitePartial = 6,     // K-split partial slot: slot, tile, slots in the workspace
    kSiteCounter = 7,     // K-split tile counter: counter index, tile, counters in the workspace
    kSiteYStore = 8,      // output column: column, token row, N
    kSiteDecW = 9,        // decode weight stage copy: 16-row block, first group, blocks
    kSiteDecX = 10,       // decode activation piece copy: first 64-wide K panel, piece, K
    kSiteProblem = 11,    // problem index of a scheduled tile: index, problems, 0
};

// The words after the status word that hold the first violation: site, then three values.
constexpr int kRecordWords = 4;

// A tiled tensor copy's innermost coordinate x: x times the element size a multiple of 16 bytes
// (the TMA rule) and the box [x, x + box) inside [0, extent).
WQ4_HD inline bool tma_x_ok(long long x, int elem_bytes, int box, long long extent) {
    return x >= 0 && (x * elem_bytes) % 16 == 0 && x + box <= extent;
}

// [begin, begin + len) inside [lo, hi).
WQ4_HD inline bool span_ok(long long begin, long long len, long long lo, long long hi) {
    return len >= 0 && begin >= lo && begin + len <= hi;
}

WQ4_HD inline bool aligned16(unsigned long long addr) { return (addr & 15ull) == 0; }

// A tile of a problem with `rows` tokens, N weight rows and k_groups groups: m-tile mt of
// token_tile tokens holds at least one token, n-tile nt's 128 weight rows are inside N and the
// group range [g0, g1) is non-empty and inside [0, k_groups).
WQ4_HD inline bool tile_ok(int mt, int token_tile, int rows, int nt, int N, int g0, int g1, int k_groups) {
    return mt >= 0 && static_cast<long long>(mt) * token_tile < rows && nt >= 0 &&
           (static_cast<long long>(nt) + 1) * 128 <= N && g0 >= 0 && g0 < g1 && g1 <= k_groups;
}

}  // namespace check

#if defined(__CUDACC__)
// Records the first violation after the status word (site, a, b, limit), sets the bounds bit and
// raises the CTA's abort flag (when there is one to raise).
__device__ __noinline__ inline void bounds_fail(unsigned int* status, volatile int* abort_flag, int site, long long a,
                                               long long b, long long limit) {
    if (atomicCAS(status + 1, 0u, static_cast<unsigned int>(site)) == 0u) {
        status[2] = static_cast<unsigned int>(a);
        status[3] = static_cast<unsigned int>(b);
        status[4] = static_cast<unsigned int>(limit);
        __threadfence();
    }
    atomicOr(status, kStatusBounds);
    if (abort_flag) *abort_flag = 1;
}
#endif

}  // namespace wq4

// WQ4_CHECK(cond, status, abort_flag, site, a, b, limit): true when cond holds; otherwise records
// the violation and yields false. Without WQ4_DEBUG it is the constant true and cond is not
// evaluated.
#if defined(WQ4_DEBUG) && WQ4_DEBUG
#define WQ4_CHECK(cond, status, abort_flag, site, a, b, limit)                                                  \
    ((cond) ? true                                                                                              \
            : (::wq4::bounds_fail((status), (abort_flag), (site), static_cast<long long>(a),                    \
                                  static_cast<long long>(b), static_cast<long long>(limit)),                    \
               false))
namespace wq4 { constexpr bool kDebugChecks = true; }
#else
#define WQ4_CHECK(cond, status, abort_flag, site, a, b, limit) true
namespace wq4 { constexpr bool kDebugChecks = false; }
#endif
