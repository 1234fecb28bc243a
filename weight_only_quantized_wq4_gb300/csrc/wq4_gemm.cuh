// The W4A16 GEMM kernel for sm_103a.
//
// Problem (after "machete_mainloop.cuh", header comment): Y = X W^T is computed transposed,
// Y^T = W X^T, so that the 4-bit weight is the MMA's A operand: 128 weight rows form the MMA's
// M = 128 side (one row per TMEM lane) and a tile of NT tokens the N side.
//
// Dequantisation (after "machete_mainloop.cuh", transform_A_kblock and get_conversion_mode):
// the value of a weight is (code - zero) * scale with zero = 8 (uint4b8) or the stored per-group
// zero point. The pages round each scaled weight to the 16-bit type before the MMA; that
// rounding, summed over K = 4096..14336, exceeds the required |dY| <= 1e-2 + 1e-2 |Y|. Here the
// MMA operand is the exact integer (code - zero) (|v| <= 15 is exact in bf16 and fp16), every
// 128-K group's product P_g = (q - z) . X^T lands in its own TMEM buffer, and the group's scale
// is applied in fp32: acc += s[n, g] * P_g[n, :], one scalar per TMEM lane.
//
// Warp roles in one CTA (one CTA per SM, persistent):
//   warp 0        TMA producer: per group, one bulk copy of the prepacked weight record (codes,
//                 scales, zero points) and two 2-D tensor copies of the activation tile (two
//                 64-element K panels, 128-byte swizzle) into a ring of shared-memory stages.
//                 (After "machete_mainloop.cuh", load: A, B, scale and zero per stage.)
//   warps 1, 3    MMA issuers (warp 1 even groups, warp 3 odd groups): one thread each issues
//                 8 tcgen05.mma (K = 16 each) per group into P[b], b = group parity, then
//                 commits to the fold, dequant and stage barriers.
//                 (After "sm100_implicit_gemm_umma_warpspecialized.hpp", mma.)
//   dequant warps turn the 4-bit codes of a stage into the 16-bit integer operand (q - z) with
//                 bit logic and one packed subtraction per pair, written to tensor memory (or to
//                 a swizzled shared-memory tile), double buffered.
//   fold warps    read P[b] from TMEM (lane = weight row), acc = s * P + acc in registers, and at
//                 the end of a tile round to bf16/fp16 and store Y, or (for a tile split over
//                 CTAs) write fp32 partials to the workspace, the last CTA to arrive summing them
//                 in CTA order (after the split-K fixup in
//                 "sm90_gemm_array_tma_warpspecialized_cooperative.hpp", TileScheduler::fixup).
//
// Every wait is bounded (see mbar_wait); a timed-out wait records WQ4_ERR_TIMEOUT in the status
// word, the CTA stops issuing work, drains its copies and MMAs, frees its TMEM and returns.
#pragma once

#include "wq4_device.cuh"
#include "wq4_params.h"

namespace wq4 {

// Weight-ring stages that leave `want` activation stages in `avail` bytes of shared memory: the
// deepest ring of 2..8 stages that does, else 8 (the activation ring then gets what is left).
constexpr int wring_for_x(int avail, int wstage_bytes, int xstage_bytes, int want) {
    for (int w = 8; w >= 2; --w)
        if (((avail - (w * wstage_bytes + 1023) / 1024 * 1024) / xstage_bytes & ~1) >= want) return w;
    return 8;
}

template <int NT, int QT, bool ATMEM, int H>
struct GemmCfg {
    static_assert(NT == 16 || NT == 64 || NT == 128 || NT == 160 || NT == 192, "token tile");
    // H scale sets per 128-K record (2 for a group size of 64): the MMAs of each 64-K half of a
    // group accumulate into a partial of their own, folded with the half's scale.
    static_assert(H == 1 || H == 2, "scale sets");
    // Four warpgroups: WG0 = the two TMA producer warps (0, 2) and the two MMA warps (1, 3);
    // then the dequant warps; then the fold warps. Any four consecutive warps cover the four TMEM lane quarters (warp % 4).
    static constexpr int kDQW = NT <= 64 ? 8 : 4;            // dequant warps
    static constexpr int kFW = NT <= 64 ? 4 : 8;             // fold / epilogue warps
    static constexpr int kWarps = 4 + kDQW + kFW;
    // With wide token tiles the fold warps hold 64..96 fp32 accumulators each: registers move
    // to them from the other warpgroups (setmaxnreg). Launched with 128 per thread, the split
    // (128 x 56 + 128 x 104 + 256 x 176 = 65536 for NT >= 128; 128 x 56 + 256 x 96 + 128 x 200 =
    // 57344 for NT = 64) stays within the 512 x 128 = 65536 launched. The dequant warps hold one
    // group's operand (64 words at NT >= 128) while the previous group's stores complete.
    static constexpr bool kRegSplit = NT >= 64;
    static constexpr int kRegWg0 = 56, kRegDequant = NT >= 128 ? 104 : 96, kRegFold = NT == 64 ? 200 : 176;
    static_assert(!kRegSplit || (128 * kRegWg0 + 32 * kDQW * kRegDequant + 32 * kFW * kRegFold <= kWarps * 32 * 128),
                  "register split exceeds the launched registers");
    static constexpr int kThreads = kWarps * 32;
    static constexpr int kKParts = kDQW / 4;                 // dequant warps per TMEM lane quarter
    static constexpr int kChunks = 4 / kKParts;              // 32-element K chunks per dequant thread
    static constexpr int kColParts = kFW / 4;                // fold warps per TMEM lane quarter
    static constexpr int kNC = NT / kColParts;               // accumulator columns per fold thread
    // epilogue: C values loaded together per thread (16 at NT = 192 spill the bf16 fold warps)
    static constexpr int kEpiBatch = 8;
    static constexpr int kRec = tile_record_bytes(QT, H);
    static constexpr int kXPanel = NT * 128;                 // one 64-K panel of NT token rows
    // Two rings: activation tiles (two panels per group; consumed by the MMA, released by its
    // commit) and weight records (codes + scales + zeros; released once the dequant warps and
    // the fold warps are done with them). The weight ring is deep so that dequantisation can run
    // ahead of the MMA; the activation ring only has to cover the copy latency.
    static constexpr int kXStageBytes = 2 * kXPanel;
    static constexpr int kWStageBytes = (kRec + 127) / 128 * 128;
    static constexpr int kABuf = 128 * 128 * 2;              // one 128 x 128 16-bit operand tile
    // Dequantised operand buffers: as many as tensor memory holds beside the two P buffers
    // (64 columns each). With two, the dequantisation of group g waits for the MMAs of group
    // g - 2 and that chain, not the tensor pipe, sets the pace; a third or fourth buffer lets it
    // run further ahead. In shared memory (the comparison path) two.
    // P buffers (partials), NT columns each. One scale set: two, one per MMA warp (the warps take
    // alternate groups); at NT = 128 three P buffers with two operand buffers were measured slower
    // than two P buffers with four operand buffers (the dequantisation chain binds before the fold
    // chain does). Two scale sets: MMA warp h issues half h of every group into buffers of its
    // own, two each where tensor memory leaves two operand buffers beside them, else one; so
    // every buffer is walked in consecutive phases by a single issuer.
    static constexpr int kPBufs = H == 1 ? 2 : (4 * NT + 2 * 64 <= 512 ? 4 : 2);
    static constexpr int kPPerHalf = kPBufs / H;             // P buffers of one issuer
    static constexpr int kPCols = NT;                        // tensor-memory columns of one P buffer
    // the P buffer of group i's partial h, and the round (phase parity) of its use
    __device__ static int pbuf(int i, int h) { return h + H * (i % kPPerHalf); }
    __device__ static uint32_t pround(int i) { return static_cast<uint32_t>(i / kPPerHalf) & 1u; }
    // (an even count: at NT = 160 two buffers, one per MMA warp, measured 1 % faster than three
    // shared by both on the grouped workload)
    static constexpr int kABufs = !ATMEM ? 2 : (512 - kPBufs * kPCols) / 64 >= 4 ? 4 : ((512 - kPBufs * kPCols) / 64) & ~1;
    static constexpr int kABytes = ATMEM ? 0 : 2 * kABuf;
    // Float zeros: the zero term sum over groups of zf[n][g] * (sum of X[m] over group g) runs on
    // the tensor core as one extra step (a "zero step") after every kZRec records of a segment and
    // after its last: A = the rows' float zeros of those records' kZRec * H zero groups (64 at
    // most), B = the activation sums split into a high and a low 16-bit part (a pre-pass table
    // copied like an activation tile, high part in K 0..63 and low part in K 64..127, each against
    // the same zeros). The dequant warps stage each row's zeros in shared memory as they pass
    // (row stride 132 B: the 32 lanes of a warp write different banks), one copy per dequant warp
    // of a lane quarter.
    static constexpr bool kZ = QT == kQtU4FZp;
    static constexpr int kZRec = 64 / H;                     // records per zero step
    static constexpr int kZRow = 132;                        // staging bytes per row
    static constexpr int kZBytes = kZ ? ((NT <= 64 ? 2 : 1) * 128 * kZRow + 1023) / 1024 * 1024 : 0;
    __device__ static bool zstep_after(int g, int g1) { return kZ && ((g + 1) % kZRec == 0 || g + 1 == g1); }
    static constexpr int kBarBytes = 1024;
    static constexpr int kMaxDynSmem = 232448;
    // Weight ring: 8 stages; with activation tiles of 160 and 192 tokens, as many as leave four
    // activation stages (measured at prefill, NT = 192: 2 activation + 8 weight stages 421.6 us,
    // 4 + 4 364.0 us: the activation copies, not the weight records, are the ones that wait).
    static constexpr int kWStages =
        NT <= 16 ? (kZ && !ATMEM ? 8 : 16)
                 : (ATMEM ? (NT >= 160 ? wring_for_x(kMaxDynSmem - 1024 - kBarBytes - kABytes - kZBytes,
                                                     kWStageBytes, kXStageBytes, 4)
                                       : 8)
                          : (kZ ? 4 : 6));
    // the ring is padded to 1024 B so that the operand tiles after it keep their swizzle atoms aligned
    static constexpr int kWRingBytes = (kWStages * kWStageBytes + 1023) / 1024 * 1024;
    static constexpr int kXStagesFit = (kMaxDynSmem - 1024 - kBarBytes - kABytes - kZBytes - kWRingBytes) / kXStageBytes;
    // An even count: the two MMA warps take alternate groups, so each then owns every other slot
    // and waits on consecutive phases of it (a parity wait is unambiguous one phase ahead only; with
    // an odd count a warp would skip the other warp's phase of a slot).
    static constexpr int kXStages = (kXStagesFit > 16 ? 16 : kXStagesFit) & ~1;
    // The fused epilogue's C tile ([NT][128] 16-bit, copied by TMA while the tile's groups run) where
    // shared memory has room for it. Otherwise a whole tile's C goes through the activation ring: a
    // "C step" after the tile's last step takes two consecutive activation stages, half the tile's
    // token rows in each (two stages keep every stage with the MMA warp of its parity; each fold
    // warp's columns lie in one half).
    static constexpr int kCTile = NT * 128 * 2;
    static constexpr int kCBytes =
        kMaxDynSmem - (1024 + kXStages * kXStageBytes + kWRingBytes + kABytes + kZBytes + kBarBytes) >= kCTile ? kCTile : 0;
    static constexpr int kSmemBytes = 1024 + kXStages * kXStageBytes + kWRingBytes + kABytes + kZBytes + kCBytes + kBarBytes;
    static constexpr int kColA = kPBufs * kPCols;            // TMEM column of A buffer 0
    static constexpr int kTmemNeed = kPBufs * kPCols + (ATMEM ? 64 * kABufs : 0);
    static constexpr int kTmemCols = kTmemNeed <= 32 ? 32 : kTmemNeed <= 64 ? 64 : kTmemNeed <= 128 ? 128
                                     : kTmemNeed <= 256 ? 256 : 512;
    static_assert(kXStages >= 2 && kWStages <= 16, "shared memory");
    static_assert(kXStageBytes % 1024 == 0 && kWRingBytes % 1024 == 0, "1024-byte aligned operand tiles");
    static_assert(kXStages * kXStageBytes >= NT * 128 * 4, "cluster reduction buffer");
    static_assert(kSmemBytes <= kMaxDynSmem, "shared memory");
    static_assert(kTmemNeed <= 512 && kABufs >= 2 && kABufs <= 4, "tensor memory");
};

// slot: -1 whole tile, >= 0 workspace slot of a K-split part, kSlotCluster a cluster part.
struct Seg {
    int prob, tile, nt, mt, g0, g1, slot;
};
constexpr int kSlotCluster = -2;

// Problem p's descriptor and activation map: from the kernel parameters, or from the tables a
// set-up kernel wrote into the workspace (device-resident per-problem pointers).
template <int MAXP>
__device__ __forceinline__ const ProblemDesc& prob_at(const GemmParams<MAXP>& prm, int p) {
    return prm.prob_tab ? prm.prob_tab[p] : prm.prob[p];
}
template <int MAXP>
__device__ __forceinline__ const CUtensorMap* xmap_at(const GemmParams<MAXP>& prm, int p) {
    return prm.xmap_tab ? &prm.xmap_tab[p] : &prm.xmap[p];
}

template <int MAXP>
struct Sched {
    const GemmParams<MAXP>& prm;
    int cta;
    int dp_t;
    int u, u_end;
    bool first_sk;
    bool cluster_done = false;

    __device__ Sched(const GemmParams<MAXP>& p, int c) : prm(p), cta(c), dp_t(c), first_sk(true) {
        u = p.sk_unit_begin + (p.sk_units * c) / p.num_ctas;
        u_end = p.sk_unit_begin + (p.sk_units * (c + 1)) / p.num_ctas;
    }

    // first tile of problem p: from the parameters, or from the device table
    __device__ int tile_begin(int p) const { return prm.dyn ? prm.dyn->tile_begin[p] : prob_at(prm, p).tile_begin; }

    // the last problem whose first tile (unit) is <= t (v): a binary search (begins are non-decreasing)
    __device__ int problem_of_tile(int t) const {
        int lo = 0, hi = prm.num_problems - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (tile_begin(mid) <= t) lo = mid; else hi = mid - 1;
        }
        return lo;
    }

    __device__ int problem_of_unit(int v) const {
        int lo = 0, hi = prm.num_problems - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (prob_at(prm, mid).unit_begin <= v) lo = mid; else hi = mid - 1;
        }
        return lo;
    }

    __device__ bool next(Seg& s) {
        if (prm.cluster_split > 0) {
            if (cluster_done) return false;
            cluster_done = true;
            const int S = prm.cluster_split;
            const int t = cta / S, q = cta % S;
            const int p = problem_of_tile(t);
            const ProblemDesc& P = prob_at(prm, p);
            if (!P.valid) return false;
            const int local = t - P.tile_begin;
            s.prob = p;
            s.tile = t;
            s.mt = local / P.n_tiles;
            s.nt = local % P.n_tiles;
            s.g0 = (q * P.k_groups) / S;
            s.g1 = ((q + 1) * P.k_groups) / S;
            s.slot = kSlotCluster;
            return true;
        }
        while (dp_t < (prm.dyn ? prm.dyn->total_tiles : prm.dp_tiles)) {
            const int t = dp_t;
            dp_t += prm.num_ctas;
            const int p = problem_of_tile(t);
            const ProblemDesc& P = prob_at(prm, p);
            if (!P.valid) continue;                      // every role skips the same tiles
            const int local = t - tile_begin(p);
            s.prob = p;
            s.tile = t;
            s.mt = local / P.n_tiles;
            s.nt = local % P.n_tiles;
            s.g0 = 0;
            s.g1 = P.k_groups;
            s.slot = -1;
            return true;
        }
        while (u < u_end) {
            const int p = problem_of_unit(u);
            const ProblemDesc& P = prob_at(prm, p);
            const int local = u - P.unit_begin;
            const int tl = local / P.k_groups;
            const int g = local - tl * P.k_groups;
            const int left = u_end - u;
            const int take = left < (P.k_groups - g) ? left : (P.k_groups - g);
            if (!P.valid) {
                u += take;
                continue;
            }
            s.prob = p;
            s.tile = P.tile_begin + tl;
            s.mt = tl / P.n_tiles;
            s.nt = tl % P.n_tiles;
            s.g0 = g;
            s.g1 = g + take;
            const bool whole = (g == 0 && take == P.k_groups);
            s.slot = whole ? -1 : 2 * cta + (first_sk ? 0 : 1);
            first_sk = false;
            u += take;
            return true;
        }
        return false;
    }
};

// Rows (tokens) of problem p: from the parameters, or from the device table.
template <int MAXP>
__device__ __forceinline__ int problem_rows(const GemmParams<MAXP>& prm, int p) {
    return prm.dyn ? prm.dyn->M[p] : prob_at(prm, p).M;
}

// CTA whose K-split range holds split-relative unit v (ranges [floor(c U / C), floor((c+1) U / C))).
__device__ __forceinline__ int sk_cta_of(int v, int U, int C) {
    return ((v + 1) * C - 1) / U;
}

template <bool BF16>
__device__ __forceinline__ uint32_t sub2(uint32_t a, uint32_t b) {
    // packed 16-bit subtraction on the raw 32-bit registers (no pair-struct round trip)
    uint32_t d;
    if constexpr (BF16) {
        asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    } else {
        asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    }
    return d;
}

// Two codes (in bits [0,4) and [16,20) of `w`) to two exact 16-bit integers code - zero.
// OR-ing a code into the low mantissa bits of 128.0 (bf16 0x4300) or 1024.0 (fp16 0x6400), whose
// unit in the last place is 1, gives 128 + q (1024 + q) exactly; subtracting 128 + z (1024 + z),
// also exact, leaves q - z.
template <bool BF16>
__device__ __forceinline__ uint32_t codes_to_pair(uint32_t w, uint32_t sub, const NibbleConsts& nc) {
    return sub2<BF16>(and_or(w, nc.mask, nc.magic), sub);
}

template <bool BF16>
__device__ __forceinline__ float scale_to_float(uint16_t bits) {
    if constexpr (BF16) {
        return __uint_as_float(static_cast<uint32_t>(bits) << 16);
    } else {
        return __half2float(__ushort_as_half(bits));
    }
}

template <bool BF16>
__device__ __forceinline__ uint16_t float_to_out(float v) {
    if constexpr (BF16) {
        return __bfloat16_as_ushort(__float2bfloat16_rn(v));
    } else {
        return __half_as_ushort(__float2half_rn(v));
    }
}

// Writes Y[m0 + j][n] = v[j0 + j] for j < nc (at most B) and m0 + j < Mrows, with the epilogue
// when the call has one: alpha * v + bias[n] + beta * C[m][n] in fp32 (after the C load and alpha /
// beta of the epilogue in "sm90_gemm_array_tma_warpspecialized_cooperative.hpp", plus a bias per
// weight row), rounded once. The epilogue rewrites the B values in registers without branches and
// the stores are the plain path's; the C values of the B columns are loaded together (from the
// tile's copy in shared memory when c_s != 0: this thread's element of the tile's first column),
// and C may be Y itself, each element being read and then written by the same thread. `bias` is the
// row's bias as float (0 without one).
template <bool BF16, int B, int MAXP, int NV>
__device__ __forceinline__ void store_cols(const GemmParams<MAXP>& prm, const ProblemDesc& P, float (&v)[NV],
                                           int j0, int nc, int m0, int n, int Mrows, float bias, uint32_t c_s = 0) {
    if (!WQ4_CHECK(n >= 0 && n < P.N, prm.status, nullptr, check::kSiteYStore, n, m0, P.N)) return;
    uint16_t* y = reinterpret_cast<uint16_t*>(P.y);
    float* r = v + j0;                                   // (rewritten in place: the values are final here)
    if (prm.has_epi) {
        const float alpha = prm.alpha, beta = prm.beta;
#pragma unroll
        for (int j = 0; j < B; ++j) r[j] = fmaf(alpha, r[j], bias);
        if (beta != 0.f) {
            uint32_t cv[B];
            if (c_s) {
#pragma unroll
                for (int j = 0; j < B; ++j) {
                    cv[j] = 0;
                    if (j < nc) asm volatile("ld.shared.u16 %0, [%1];" : "=r"(cv[j]) : "r"(c_s + (j0 + j) * 256));
                }
            } else {
                const uint16_t* c = static_cast<const uint16_t*>(P.c);
#pragma unroll
                for (int j = 0; j < B; ++j) cv[j] = (j < nc && m0 + j < Mrows) ? c[static_cast<size_t>(m0 + j) * P.N + n] : 0u;
            }
#pragma unroll
            for (int j = 0; j < B; ++j) r[j] = fmaf(beta, scale_to_float<BF16>(static_cast<uint16_t>(cv[j])), r[j]);
        }
    }
#pragma unroll
    for (int j = 0; j < B; ++j)
        if (j < nc && m0 + j < Mrows) y[static_cast<size_t>(m0 + j) * P.N + n] = float_to_out<BF16>(r[j]);
}

// The row's bias as float, 0 without one (or without the epilogue).
template <bool BF16, int MAXP>
__device__ __forceinline__ float row_bias(const GemmParams<MAXP>& prm, const ProblemDesc& P, int n) {
    return (prm.has_epi && P.bias) ? scale_to_float<BF16>(static_cast<const uint16_t*>(P.bias)[n]) : 0.f;
}

// (d0, d1) += a * (b0, b1) with one packed fp32 FMA (fma.rn.f32x2).
__device__ __forceinline__ void fma2(float& d0, float& d1, float a, uint32_t b0, uint32_t b1) {
    uint64_t d, bb, cc, aa;
    asm("mov.b64 %0, {%1, %2};" : "=l"(bb) : "r"(b0), "r"(b1));
    asm("mov.b64 %0, {%1, %2};" : "=l"(cc) : "f"(d0), "f"(d1));
    asm("mov.b64 %0, {%1, %1};" : "=l"(aa) : "f"(a));
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(aa), "l"(bb), "l"(cc));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(d0), "=f"(d1) : "l"(d));
}

template <int NT, bool BF16, int QT, int MAXP, bool ATMEM, int H>
__global__ void __launch_bounds__(GemmCfg<NT, QT, ATMEM, H>::kThreads, 1)
wq4_gemm_kernel(const __grid_constant__ GemmParams<MAXP> prm) {
    using C = GemmCfg<NT, QT, ATMEM, H>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t sbase = (raw_s + 1023u) & ~1023u;
    uint8_t* const gbase = smem_raw + (sbase - raw_s);

    const uint32_t s_x0 = sbase;                                         // activation ring
    const uint32_t s_w0 = s_x0 + C::kXStages * C::kXStageBytes;           // weight-record ring
    const uint32_t s_A = s_w0 + C::kWRingBytes;
    const uint32_t s_Z = s_A + C::kABytes;                                // float-zero staging
    const uint32_t s_C = s_Z + C::kZBytes;                                // epilogue C tile
    const uint32_t s_bar = s_C + C::kCBytes;
    auto xfull_bar = [&](int s) { return s_bar + 8u * s; };
    auto xempty_bar = [&](int s) { return s_bar + 8u * (16 + s); };
    auto wfull_bar = [&](int s) { return s_bar + 8u * (32 + s); };
    auto wempty_bar = [&](int s) { return s_bar + 8u * (48 + s); };
    auto afull_bar = [&](int a) { return s_bar + 8u * (64 + a); };
    auto aempty_bar = [&](int a) { return s_bar + 8u * (68 + a); };
    auto pfull_bar = [&](int b) { return s_bar + 8u * (72 + b); };
    auto pempty_bar = [&](int b) { return s_bar + 8u * (76 + b); };
    const uint32_t drain_bar = s_bar + 8u * 80;
    const uint32_t fsync_bar = s_bar + 8u * 81;   // fold warps meet here in the split epilogue
    const uint32_t stall_bar = s_bar + 8u * 82;   // never arrived on (test of the timeout path)
    const uint32_t cfull_bar = s_bar + 8u * 83;   // the epilogue's C tile landed
    const uint32_t cempty_bar = s_bar + 8u * 84;  // ... and was read by the fold warps
    // C through shared memory: whole tiles of a fused epilogue that reads C, where it fits
    const bool c_smem = C::kCBytes > 0 && prm.has_epi && prm.beta != 0.f;
    // ... or, without room, the CTA's last whole tile through the activation stage after its last step
    // (where the fold warps split the token columns in two halves, as the C step's stages do)
    const bool c_xstage = C::kCBytes == 0 && C::kColParts == 2 && prm.has_epi && prm.beta != 0.f &&
                          prm.cluster_split == 0;
    uint8_t* const gmisc = gbase + (s_bar - sbase) + 8 * 88;
    uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(gmisc);
    volatile int* const abort_flag = reinterpret_cast<volatile int*>(gmisc + 4);
    volatile int* const fin_flag = reinterpret_cast<volatile int*>(gmisc + 8);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        // a stage or operand buffer is released by the commit of each MMA warp that read it: the
        // one that issued the group, or both with two scale sets (one half each)
        for (int s = 0; s < C::kXStages; ++s) {
            mbar_init(xfull_bar(s), 1);
            mbar_init(xempty_bar(s), H);
        }
        for (int s = 0; s < C::kWStages; ++s) {
            mbar_init(wfull_bar(s), 1);
            mbar_init(wempty_bar(s), C::kDQW + C::kFW);
        }
        for (int a = 0; a < C::kABufs; ++a) {
            mbar_init(afull_bar(a), C::kDQW);
            mbar_init(aempty_bar(a), H);
        }
        for (int b = 0; b < C::kPBufs; ++b) {
            mbar_init(pfull_bar(b), 1);
            mbar_init(pempty_bar(b), C::kFW);
        }
        mbar_init(drain_bar, 2);                 // one commit from each MMA warp
        mbar_init(fsync_bar, C::kFW);
        mbar_init(stall_bar, 1);
        mbar_init(cfull_bar, 1);
        mbar_init(cempty_bar, C::kFW);
        *abort_flag = 0;
        *fin_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0 && !prm.prob_tab) {      // (device tables: written by the kernel ahead)
        for (int p = 0; p < prm.num_problems; ++p) {
            if (prm.prob[p].m_tiles > 0) prefetch_tensormap(&prm.xmap[p]);   // empty problems have no map
        }
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // Programmatic dependent launch: the set-up above (barriers, tensor maps, tensor memory)
    // overlaps the tail of the kernel ahead on the stream; every global access below (copies,
    // split counters and partials, Y) waits for it to complete. Both are no-ops when the launch
    // carries no programmatic dependency.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // Under the constant-weights promise (problems in the parameters only) the weight producer
    // copies its first ring of records, and the header checks read the blobs, before the kernel
    // ahead completes; the MMA and dequant warps touch only shared and tensor memory and never
    // wait; the activation producer and the fold warps wait here as every warp does otherwise.
    const bool w_early = prm.early != 0 && !prm.prob_tab && !prm.dyn;
    if (!w_early || warp == 0 || warp >= 4 + C::kDQW) asm volatile("griddepcontrol.wait;" ::: "memory");
    const WaitCtl ctl{abort_flag, prm.status, prm.timeout_cycles};

    if (warp < 4) {
        if constexpr (C::kRegSplit) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::kRegWg0));
    }
    int issued = 0;                                      // copies a producer thread has issued
    // Every problem's blob header against the call: by the weight producer's warp before its first
    // record copy, or (blobs prepacked here for these arguments) by lanes 1..31 of MMA warp 1 while
    // the copies already stream; a mismatch stops the CTA and is reported as WQ4_ERR_INVALID.
    // (Device tables: the set-up kernel checked every header and marked mismatches invalid.)
    bool hdr_ok = true;
    const bool hdr_alongside = prm.hdr_trusted != 0;
    if (!prm.prob_tab && ((warp == 2 && !hdr_alongside) || (warp == 1 && hdr_alongside && lane > 0))) {
        const unsigned int mask = hdr_alongside ? 0xfffffffeu : 0xffffffffu;
        const int l0 = hdr_alongside ? 1 : 0, nl = hdr_alongside ? 31 : 32;
        bool mine = true;
        for (int p = lane - l0; p < prm.num_problems; p += nl) {
            const ProblemDesc& P = prob_at(prm, p);
            if (P.m_tiles > 0 && P.valid)
                mine = blob_header_ok(reinterpret_cast<const uint32_t*>(P.wp - kBlobHeader), P.N, P.K, prm.group_size,
                                      prm.dtype, prm.qtype) && mine;
        }
        hdr_ok = __all_sync(mask, mine ? 1 : 0) != 0;
        if (!hdr_ok && lane == l0) {
            atomicOr(prm.status, kStatusBadBlob);
            *abort_flag = 1;
        }
        if (warp == 1) hdr_ok = true;                    // the MMA issuer (lane 0) is unaffected here
    }
    if (warp == 0 || warp == 2) {
        // ------------------------------------------------------------------ producers
        // warp 0: activation tiles (two 2-D tensor copies per group); warp 2: weight records (one
        // bulk copy per group, up to kWStages groups ahead)
        if (lane == 0) {
            const bool is_x = warp == 0;
            const uint64_t pol_stream = policy_evict_first();
            const uint64_t pol_keep = policy_evict_last();
            const int depth = is_x ? C::kXStages : C::kWStages;
            Sched<MAXP> sch(prm, blockIdx.x);
            Seg seg;
            int i = 0;
            int last_prob = -1;
            bool ok = hdr_ok;
            bool dep_done = is_x || !w_early;            // (the early weight producer waits after a ring)
            while (ok && sch.next(seg)) {
                if (!WQ4_CHECK(seg.prob >= 0 && seg.prob < prm.num_problems, prm.status, abort_flag,
                               check::kSiteProblem, seg.prob, prm.num_problems, 0)) break;
                const ProblemDesc& P = prob_at(prm, seg.prob);
                if (!WQ4_CHECK(check::tile_ok(seg.mt, NT, problem_rows(prm, seg.prob), seg.nt, P.N, seg.g0, seg.g1,
                                              P.k_groups),
                               prm.status, abort_flag, check::kSiteTile, seg.mt, seg.nt, seg.g1)) break;
                const uint64_t pol_w = P.m_tiles == 1 ? pol_stream : pol_keep;
                const uint8_t* wrec = P.wp + (static_cast<size_t>(seg.nt) * P.k_groups + seg.g0) * C::kRec;
                const CUtensorMap* xmap = xmap_at(prm, seg.prob);
                if (is_x && prm.xmap_tab && seg.prob != last_prob) {
                    // a map patched in global memory by the set-up kernel: acquire it for the
                    // tensor-map proxy before the first copy that uses it
                    asm volatile("fence.proxy.tensormap::generic.acquire.gpu [%0], 128;" ::"l"(reinterpret_cast<uint64_t>(xmap))
                                 : "memory");
                    last_prob = seg.prob;
                }
                for (int g = seg.g0; g < seg.g1; ++g, wrec += C::kRec) {
                    if (is_x) {
                        // the group's activation tile, then (float zeros) a zero step's sums
                        const int nstep = C::zstep_after(g, seg.g1) ? 2 : 1;
                        for (int t = 0; t < nstep; ++t, ++i) {
                            const int s = i % depth;
                            if (!mbar_wait(xempty_bar(s), ((i / depth) & 1) ^ 1, ctl)) { ok = false; break; }
                            const uint32_t stage = s_x0 + s * C::kXStageBytes;
                            mbar_arrive_expect_tx(xfull_bar(s), 2 * C::kXPanel);
                            if (t == 0) {
                                int kx = g * kTileK;     // (a failed check reads the tensor's origin instead)
                                if (!WQ4_CHECK(check::tma_x_ok(kx, 2, kTileK, P.K), prm.status, abort_flag,
                                               check::kSiteXTile, kx, seg.mt * NT, P.K)) kx = 0;
                                tma_load_2d(stage, xmap, xfull_bar(s), kx, seg.mt * NT, pol_keep);
                                tma_load_2d(stage + C::kXPanel, xmap, xfull_bar(s), kx + 64, seg.mt * NT, pol_keep);
                            } else {                     // zero groups [64 zc, 64 zc + 64): high, then low part
                                int zc = (g * H) / 64;
                                const int zpad = (P.K / (kTileK / H) + 63) / 64 * 64;
                                if (!WQ4_CHECK(check::tma_x_ok(64 * zc, 2, 64, zpad), prm.status, abort_flag,
                                               check::kSiteXSums, 64 * zc, seg.mt * NT, zpad)) zc = 0;
                                const CUtensorMap* sxm = &prm.sxmap[seg.prob];
                                tma_load_2d(stage, sxm, xfull_bar(s), 64 * zc, seg.mt * NT, pol_stream);
                                tma_load_2d(stage + C::kXPanel, sxm, xfull_bar(s), zpad + 64 * zc, seg.mt * NT, pol_stream);
                            }
                        }
                        if (!ok) break;
                    } else {
                        if (!dep_done && i == depth) {
                            asm volatile("griddepcontrol.wait;" ::: "memory");
                            dep_done = true;
                        }
                        const int s = i % depth;
                        if (!mbar_wait(wempty_bar(s), ((i / depth) & 1) ^ 1, ctl)) { ok = false; break; }
                        mbar_arrive_expect_tx(wfull_bar(s), C::kRec);
                        const uint8_t* src = wrec;   // (a failed check reads the blob's first record instead)
                        if (!WQ4_CHECK(check::span_ok(wrec - P.wp, C::kRec, 0,
                                                      static_cast<long long>(P.N / kTileN) * P.k_groups * C::kRec) &&
                                           check::aligned16(reinterpret_cast<uintptr_t>(wrec)),
                                       prm.status, abort_flag, check::kSiteWRecord, wrec - P.wp, seg.nt, g)) src = P.wp;
                        bulk_load(s_w0 + s * C::kWStageBytes, src, C::kRec, wfull_bar(s), pol_w);
                        ++i;
                    }
                }
                if (is_x && ok && c_xstage && seg.slot == -1) {
                    // the C step: the tile's C in two halves of NT / 2 token rows, one stage each
                    for (int hf = 0; hf < 2; ++hf, ++i) {
                        const int s = i % depth;
                        if (!mbar_wait(xempty_bar(s), ((i / depth) & 1) ^ 1, ctl)) { ok = false; break; }
                        mbar_arrive_expect_tx(xfull_bar(s), C::kCTile / 2);
                        int cn = seg.nt * kTileN;
                        if (!WQ4_CHECK(check::tma_x_ok(cn, 2, kTileN, P.N), prm.status, abort_flag, check::kSiteCTile,
                                       cn, seg.mt * NT, P.N)) cn = 0;
                        tma_load_2d(s_x0 + s * C::kXStageBytes, &prm.cmap, xfull_bar(s), cn,
                                    seg.mt * NT + hf * (NT / 2), pol_stream);
                    }
                }
            }
            if (!dep_done) asm volatile("griddepcontrol.wait;" ::: "memory");
            issued = i;                                  // drained at the end if the CTA gives up
        }
        __syncwarp();
    } else if (warp == 1 || warp == 3) {
        // ------------------------------------------------------------------ MMA issuers
        // Two issuing threads: warp 1 takes the even groups, warp 3 the odd ones (the P and A
        // buffers alternate with the group's parity, the X stages are distinct). One thread
        // alone leaves the tensor pipe idle between groups while it checks the next group's
        // three barriers and runs its loop (measured ~0.3 us of a ~0.85 us group at 192
        // tokens); with two, one thread's checks overlap the other's MMAs. Each thread's
        // tcgen05.commit tracks only the MMAs that thread issued.
        const int mine = warp == 1 ? 0 : 1;
        if (lane == 0) {
            Sched<MAXP> sch(prm, blockIdx.x);
            Seg seg;
            int i = 0;                                   // compute steps (groups and zero steps)
            int cx = 0;                                  // activation stages taken by C steps (2 each)
            // (tests) a wait that nothing ends: it runs out, records the timeout, stops the CTA
            bool ok = !(prm.test_stall && mine == 0) || mbar_wait(stall_bar, 0, ctl);
            while (ok && sch.next(seg)) {
                const ProblemDesc& P = prob_at(prm, seg.prob);
                const int rows = problem_rows(prm, seg.prob) - seg.mt * NT;
                const int n_valid = rows < NT ? rows : NT;
                const uint32_t idesc = make_idesc(BF16, 128, static_cast<uint32_t>((n_valid + 15) & ~15));
                for (int g = seg.g0; g < seg.g1 && ok; ++g)
                for (int t = 0, nstep = C::zstep_after(g, seg.g1) ? 2 : 1; t < nstep; ++t, ++i) {
                    // step i: group g, or (t = 1) the zero step after it; both alike here
                    if (H == 1 && (i & 1) != mine) continue;    // one scale set: alternate steps
                    const int xi = i + cx;                      // its activation stage (same parity as i)
                    const int s = xi % C::kXStages;
                    const int b = C::pbuf(i, H == 1 ? 0 : mine);   // P buffer (two sets: half `mine`)
                    const uint32_t u = C::pround(i);
                    const int a = i % C::kABufs;                // A buffer
                    if (!mbar_wait(xfull_bar(s), (xi / C::kXStages) & 1, ctl)) { ok = false; break; }
                    if (!mbar_wait(afull_bar(a), (i / C::kABufs) & 1, ctl)) { ok = false; break; }
                    if (!mbar_wait(pempty_bar(b), u ^ 1u, ctl)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t xs = s_x0 + s * C::kXStageBytes;
                    const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(b * C::kPCols);
#pragma unroll
                    for (int k = 0; k < 8 / H; ++k) {
                        const int kk = (H == 2 ? 4 * mine : 0) + k;    // K step (panel kk / 4)
                        const bool accum = k > 0;
                        const uint64_t bdesc = make_sdesc_sw128(xs + (kk >> 2) * C::kXPanel + (kk & 3) * 32);
                        if constexpr (ATMEM) {
                            mma_ts(d_tmem, tmem_base + C::kColA + a * 64 + kk * 8, bdesc, idesc, accum);
                        } else {
                            const uint64_t adesc = make_sdesc_sw128(s_A + a * C::kABuf + (kk >> 2) * (C::kABuf / 2) + (kk & 3) * 32);
                            mma_ss(d_tmem, adesc, bdesc, idesc, accum);
                        }
                    }
                    mma_commit(pfull_bar(b));
                    mma_commit(aempty_bar(a));
                    mma_commit(xempty_bar(s));
                }
                if (ok && c_xstage && seg.slot == -1) {
                    // the C step: no MMA, but the warp that owns a stage waits for its copy, so that
                    // it walks every phase of its stages in order (the fold warps release them)
                    for (int hf = 0; hf < 2; ++hf) {
                        const int xi = i + cx + hf;
                        if ((H == 1 && (xi & 1) != mine) || !ok) continue;
                        ok = mbar_wait(xfull_bar(xi % C::kXStages), (xi / C::kXStages) & 1, ctl);
                    }
                    cx += 2;
                }
            }
            // Every MMA issued so far completes before the CTA frees its tensor memory.
            mma_commit(drain_bar);
            mbar_wait_plain(drain_bar, 0, drain_limit(prm.timeout_cycles));
        }
        __syncwarp();
    } else if (warp < 4 + C::kDQW) {
        // ------------------------------------------------------------------ dequant
        if constexpr (C::kRegSplit) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::kRegDequant));
        const int q4 = warp & 3;
        const int part = (warp - 4) >> 2;
        const int r = 32 * q4 + lane;
        const NibbleConsts nib = prm.nib;
        // this thread's float-zero staging row (one copy per dequant warp of a lane quarter)
        const uint32_t zrow = s_Z + static_cast<uint32_t>((part * 128 + r) * C::kZRow);
        // stores one 32-K chunk (16 pairs) of the operand in buffer a
        auto put_chunk = [&](int a, int j, const uint32_t (&out)[16]) {
            if constexpr (ATMEM) {
                tmem_st16(tmem_base + (static_cast<uint32_t>(32 * q4) << 16) + C::kColA + a * 64 + 16 * j, out);
            } else {
                const uint32_t pbase = s_A + a * C::kABuf + (j >> 1) * (C::kABuf / 2) + r * 128;
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    const uint32_t chunk = static_cast<uint32_t>((4 * (j & 1) + w) ^ (r & 7));
                    sts128(pbase + chunk * 16, out[4 * w], out[4 * w + 1], out[4 * w + 2], out[4 * w + 3]);
                }
            }
        };
        auto operand_done = [&](int a) {                 // buffer a written: hand it to the MMA warps
            if constexpr (ATMEM) {
                tmem_st_wait();
                tc_fence_before();
            } else {
                fence_proxy_async_smem();
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(afull_bar(a));
        };
        // Software-pipelined: a step's operand is computed into registers first, then the previous
        // step's stores are waited for and that buffer handed to the MMA warps, then this step's
        // stores are issued, so the store latency overlaps the next step's bit work.
        int pend_a = -1;                                 // buffer whose stores are in flight
        auto handover = [&]() {
            if (pend_a >= 0) operand_done(pend_a);
            pend_a = -1;
        };
        Sched<MAXP> sch(prm, blockIdx.x);
        Seg seg;
        int i = 0;                                       // steps (groups and zero steps)
        int wi = 0;                                      // weight records
        bool ok = true;
        while (ok && sch.next(seg)) {
            for (int g = seg.g0; g < seg.g1; ++g, ++i, ++wi) {
                const int s = wi % C::kWStages;
                const int a = i % C::kABufs;
                if (!mbar_wait(wfull_bar(s), (wi / C::kWStages) & 1, ctl)) { ok = false; break; }
                const uint32_t rec = s_w0 + s * C::kWStageBytes;
                uint32_t subs[H];                             // per scale set
#pragma unroll
                for (int h = 0; h < H; ++h) {
                    if constexpr (QT == kQtU4Zp) {
                        uint32_t zb;
                        asm volatile("ld.shared.u8 %0, [%1];" : "=r"(zb) : "r"(rec + rec_zero_off(QT, r, H, h)));
                        const uint32_t z = (zb >> (((r >> 3) & 1) * 4)) & 0xFu;
                        subs[h] = ((BF16 ? 0x4300u : 0x6400u) | z) * 0x10001u;
                    } else if constexpr (QT == kQtU4FZp) {
                        subs[h] = BF16 ? 0x43004300u : 0x64006400u;   // the code itself; its zero goes to a zero step
                        uint32_t zfb;
                        asm volatile("ld.shared.u16 %0, [%1];" : "=r"(zfb) : "r"(rec + rec_fzero_off(QT, r, H, h)));
                        asm volatile("st.shared.u16 [%0], %1;" ::"r"(zrow + 2 * ((g * H + h) % 64)), "r"(zfb) : "memory");
                    } else {
                        subs[h] = BF16 ? 0x43084308u : 0x64086408u;   // 128 + 8 (bf16), 1024 + 8 (fp16)
                    }
                }
                uint32_t out[C::kChunks][16];
#pragma unroll
                for (int jj = 0; jj < C::kChunks; ++jj) {
                    const int j = part * C::kChunks + jj;
                    const uint32_t sub = subs[H == 2 ? (j >> 1) : 0];   // 32-K chunk j lies in set j / 2
                    const uint4 v = lds128(rec + rec_code_off(QT, r, j, H));
                    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
#pragma unroll
                        for (int e = 0; e < 4; ++e) out[jj][4 * w + e] = codes_to_pair<BF16>(wv[w] >> (4 * e), sub, nib);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(wempty_bar(s));      // (the record is read)
                handover();
                if (!mbar_wait(aempty_bar(a), ((i / C::kABufs) & 1) ^ 1u, ctl)) { ok = false; break; }
#pragma unroll
                for (int jj = 0; jj < C::kChunks; ++jj) put_chunk(a, part * C::kChunks + jj, out[jj]);
                pend_a = a;
                if (C::zstep_after(g, seg.g1)) {
                    // zero step: the staged zeros of this chunk's zero groups that lie in the segment
                    // (K 0..63 and again K 64..127, against the high and the low part of the sums);
                    // the rest of the 64 are zero
                    ++i;
                    const int a2 = i % C::kABufs;
                    const int zc = (g * H) / 64;
                    const int zlo = max(seg.g0 * H - 64 * zc, 0), zhi = (g + 1) * H - 64 * zc;
                    handover();
                    if (!mbar_wait(aempty_bar(a2), ((i / C::kABufs) & 1) ^ 1u, ctl)) { ok = false; break; }
#pragma unroll 1
                    for (int jj = 0; jj < C::kChunks; ++jj) {
                        const int j = part * C::kChunks + jj;
                        const int z0 = 32 * (j & 1);
                        uint32_t zo[16];
#pragma unroll
                        for (int q = 0; q < 16; ++q) {
                            const int z = z0 + 2 * q;
                            uint32_t wv;
                            asm volatile("ld.shared.u32 %0, [%1];" : "=r"(wv) : "r"(zrow + 2 * z));
                            const uint32_t lo_ok = (z >= zlo && z < zhi) ? 0x0000FFFFu : 0u;
                            const uint32_t hi_ok = (z + 1 >= zlo && z + 1 < zhi) ? 0xFFFF0000u : 0u;
                            zo[q] = wv & (lo_ok | hi_ok);
                        }
                        put_chunk(a2, j, zo);
                    }
                    pend_a = a2;
                }
            }
        }
        if (pend_a >= 0) {                               // the last step's operand
            if (ok) {
                handover();
            } else if constexpr (ATMEM) {
                tmem_st_wait();                          // no store in flight when the tensor memory is freed
            }
        }
    } else {
        // ------------------------------------------------------------------ fold + epilogue
        if constexpr (C::kRegSplit) asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(C::kRegFold));
        const int f = warp - 4 - C::kDQW;
        const int q4 = warp & 3;
        const int col0 = (f >> 2) * C::kNC;
        const int r = 32 * q4 + lane;
        const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(32 * q4) << 16);
        float acc[C::kNC];
        uint32_t fs_phase = 0;
        // Bounded rendezvous of the fold warps (an mbarrier, so that an abort cannot strand them).
        auto fold_sync = [&]() -> bool {
            __syncwarp();
            if (lane == 0) mbar_arrive(fsync_bar);
            const bool r_ok = mbar_wait(fsync_bar, fs_phase, ctl);
            fs_phase ^= 1u;
            return r_ok;
        };
        Sched<MAXP> sch(prm, blockIdx.x);
        Seg seg;
        seg.prob = -1;                                   // stays -1 if the CTA gets no tile
        // acc += sc * (partial b, this thread's columns); then the partial goes back to the MMAs
        auto fold_partial = [&](int b, uint32_t round, float sc) -> bool {
            if (!mbar_wait(pfull_bar(b), round, ctl)) return false;
            tc_fence_after();
            // P in batches of up to 64 columns per wait (the loads of a batch overlap)
            // (the last batch may be shorter: 80 columns = 48 + 32)
            constexpr int kBatchCols = C::kNC <= 64 ? C::kNC : 48;
            const uint32_t t_p = t_lane + b * C::kPCols + col0;
#pragma unroll
            for (int c = 0; c < C::kNC; c += kBatchCols) {
                constexpr int kLeft = C::kNC;
                const int nbc = kLeft - c < kBatchCols ? kLeft - c : kBatchCols;
                uint32_t v[kBatchCols];
#pragma unroll
                for (int q = 0; q < kBatchCols; q += 16)
                    if (q < nbc) tmem_ld16(t_p + c + q, *reinterpret_cast<uint32_t(*)[16]>(&v[q]));
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < kBatchCols; j += 4) {
                    // (columns come in multiples of 16: j < nbc covers j + 3 too)
                    if (j < nbc) {
                        fma2(acc[c + j], acc[c + j + 1], sc, v[j], v[j + 1]);
                        fma2(acc[c + j + 2], acc[c + j + 3], sc, v[j + 2], v[j + 3]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(pempty_bar(b));
            return true;
        };
        int ct = 0;                                      // whole tiles whose C came through shared memory
        int c_issued = 0;                                // C copies issued (fold warp 0, lane 0)
        int cx = 0;                                      // activation stages taken by C steps (2 each)
        int i = 0;                                       // steps (groups and zero steps)
        int wi = 0;                                      // weight records
        bool ok = true;
        while (ok && sch.next(seg)) {
            for (int g = seg.g0; g < seg.g1; ++g, ++i, ++wi) {
                const int s = wi % C::kWStages;
                if (!mbar_wait(wfull_bar(s), (wi / C::kWStages) & 1, ctl)) { ok = false; break; }
                const uint32_t rec = s_w0 + s * C::kWStageBytes;
                if (g == seg.g0) {
#pragma unroll
                    for (int j = 0; j < C::kNC; ++j) acc[j] = 0.f;
                    // The epilogue's C load ("sm90_gemm_array_tma_warpspecialized_cooperative.hpp",
                    // the epilogue load), issued by one fold thread as a whole tile starts, once every
                    // fold warp has read the previous tile's C: it lands while the tile's groups run.
                    // (a wait that runs out issues nothing: the epilogue's wait for the copy then runs out)
                    if (c_smem && seg.slot == -1 && f == 0 && lane == 0 &&
                        mbar_wait(cempty_bar, static_cast<uint32_t>(ct & 1) ^ 1u, ctl)) {
                        mbar_arrive_expect_tx(cfull_bar, C::kCTile);
                        int cn = seg.nt * kTileN;
                        if (!WQ4_CHECK(check::tma_x_ok(cn, 2, kTileN, prob_at(prm, seg.prob).N), prm.status, abort_flag,
                                       check::kSiteCTile, cn, seg.mt * NT, prob_at(prm, seg.prob).N)) cn = 0;
                        for (int hf = 0; hf < 2; ++hf)        // (the map's box is half the token rows)
                            tma_load_2d(s_C + hf * (C::kCTile / 2), &prm.cmap, cfull_bar, cn,
                                        seg.mt * NT + hf * (NT / 2), policy_evict_first());
                        c_issued = ct + 1;
                    }
                }
                float sc[H];                                    // the record's scale per set
#pragma unroll
                for (int h = 0; h < H; ++h) {
                    uint32_t sbits;
                    asm volatile("ld.shared.u16 %0, [%1];" : "=r"(sbits) : "r"(rec + rec_scale_off(QT, r, H, h)));
                    sc[h] = scale_to_float<BF16>(static_cast<uint16_t>(sbits));
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(wempty_bar(s));      // (the scales are read: the record may go)
#pragma unroll 1
                for (int h = 0; h < H; ++h)                     // scale set h: its partial with its scale
                    if (!fold_partial(C::pbuf(i, h), C::pround(i), h == 0 ? sc[0] : sc[H - 1])) { ok = false; break; }
                if (!ok) break;
                if (C::zstep_after(g, seg.g1)) {                // float zeros: the zero step, scale 1
                    ++i;
#pragma unroll 1
                    for (int h = 0; h < H; ++h)
                        if (!fold_partial(C::pbuf(i, h), C::pround(i), 1.0f)) { ok = false; break; }
                    if (!ok) break;
                }
            }
            if (!ok) break;

            // ---------------------------------------------------------- tile epilogue
            const ProblemDesc& P = prob_at(prm, seg.prob);
            const int Mrows = problem_rows(prm, seg.prob);
            const int n = seg.nt * kTileN + r;
            const int m0 = seg.mt * NT + col0;
            if (seg.slot == kSlotCluster) {
                // partial sum to this CTA's shared memory (the stages are idle now); after the
                // cluster barrier below every rank adds the S partials of its slice of columns
#pragma unroll
                for (int j = 0; j < C::kNC; ++j)
                    asm volatile("st.shared.f32 [%0], %1;" ::"r"(s_x0 + ((col0 + j) * 128 + r) * 4), "f"(acc[j])
                                 : "memory");
                continue;
            }
            if (seg.slot >= 0) {
                float* mine = prm.partials + static_cast<size_t>(seg.slot) * (NT * 128);
                if (WQ4_CHECK(seg.slot < 2 * prm.num_ctas, prm.status, abort_flag, check::kSitePartial, seg.slot,
                              seg.tile, 2 * prm.num_ctas)) {
#pragma unroll
                    for (int j = 0; j < C::kNC; ++j) mine[(col0 + j) * 128 + r] = acc[j];
                }
                if (!fold_sync()) break;
                // the units of this tile, relative to the start of the K-split region
                const int U = prm.sk_units;
                const int t_u0 = P.unit_begin + (seg.tile - P.tile_begin) * P.k_groups - prm.sk_unit_begin;
                const int c_first = sk_cta_of(t_u0, U, prm.num_ctas);
                const int c_last = sk_cta_of(t_u0 + P.k_groups - 1, U, prm.num_ctas);
                if (f == 0 && lane == 0) {
                    // CTAs whose range is empty (fewer units than CTAs) hold no part of the tile
                    int nseg = 0;
                    for (int cc = c_first; cc <= c_last; ++cc)
                        nseg += ((cc * U) / prm.num_ctas < ((cc + 1) * U) / prm.num_ctas) ? 1 : 0;
                    // release this CTA's partial (written by all fold threads before the rendezvous
                    // above) and, for the last arrival, acquire everyone else's
                    const int ci = seg.tile - prm.dp_tiles;
                    if (WQ4_CHECK(ci >= 0 && ci < prm.total_tiles - prm.dp_tiles, prm.status, abort_flag,
                                  check::kSiteCounter, ci, seg.tile, prm.total_tiles - prm.dp_tiles)) {
                        int* cnt = prm.counters + ci;
                        const int old = atomic_add_acq_rel_gpu(cnt, 1);
                        const int last = (old == nseg - 1) ? 1 : 0;
                        if (last) st_relaxed_gpu(cnt, 0);
                        *fin_flag = last;
                    } else {
                        *fin_flag = 0;
                    }
                }
                if (!fold_sync()) break;
                if (!*fin_flag) continue;
                // sum the parts in CTA order, loading kBatch parts at a time
                constexpr int kBatch = C::kNC <= 64 ? 4 : 2;   // parts of a 16-column batch loaded together
#pragma unroll
                for (int c = 0; c < C::kNC; c += 16) {
                    bool firstv = true;
                    for (int cc = c_first; cc <= c_last; cc += kBatch) {
                        float v[kBatch][16];
                        bool use[kBatch];
#pragma unroll
                        for (int b = 0; b < kBatch; ++b) {
                            const int c2 = cc + b;
                            const int start = (c2 * U) / prm.num_ctas;
                            use[b] = c2 <= c_last && start < ((c2 + 1) * U) / prm.num_ctas;
                            if (use[b]) {
                                int sl = 2 * c2 + ((c2 == c_first && start < t_u0) ? 1 : 0);
                                if (!WQ4_CHECK(sl >= 0 && sl < 2 * prm.num_ctas, prm.status, abort_flag,
                                               check::kSitePartial, sl, seg.tile, 2 * prm.num_ctas)) sl = 0;
                                const float* src = prm.partials + static_cast<size_t>(sl) * (NT * 128) + r;
#pragma unroll
                                for (int j = 0; j < 16; ++j) v[b][j] = __ldcg(src + (col0 + c + j) * 128);
                            }
                        }
#pragma unroll
                        for (int b = 0; b < kBatch; ++b) {
                            if (use[b]) {
#pragma unroll
                                for (int j = 0; j < 16; ++j) acc[c + j] = firstv ? v[b][j] : acc[c + j] + v[b][j];
                                firstv = false;
                            }
                        }
                    }
                }
            }
            const float bias = row_bias<BF16>(prm, P, n);
            constexpr int kB = C::kEpiBatch;
            // a whole tile reads its C from shared memory (copied while its groups ran)
            const bool cs = c_smem && seg.slot == -1;
            if (cs && !mbar_wait(cfull_bar, static_cast<uint32_t>(ct & 1), ctl)) { ok = false; break; }
            uint32_t c_s = cs ? s_C + static_cast<uint32_t>((col0 * 128 + r) * 2) : 0u;
            const bool cstep = c_xstage && seg.slot == -1;
            if (cstep) {
                // the C step's stage holding this thread's half of the token rows (col0 is 0 or NT / 2)
                const int xh = i + cx + col0 / (NT / 2);
                if (!mbar_wait(xfull_bar(xh % C::kXStages), static_cast<uint32_t>(xh / C::kXStages) & 1u, ctl)) {
                    ok = false;
                    break;
                }
                c_s = s_x0 + static_cast<uint32_t>((xh % C::kXStages) * C::kXStageBytes + r * 2);
            }
#pragma unroll
            for (int j0 = 0; j0 < C::kNC; j0 += kB)
                store_cols<BF16, kB>(prm, P, acc, j0, C::kNC - j0 < kB ? C::kNC - j0 : kB, m0 + j0, n, Mrows, bias,
                                     c_s);
            if (cs) {
                __syncwarp();
                if (lane == 0) mbar_arrive(cempty_bar);
                ++ct;
            }
            if (cstep) {
                // every fold warp has read its half: the two stages go back to the activation ring
                // (standing in for the MMA warps' commits)
                if (!fold_sync()) { ok = false; break; }
                if (f == 0 && lane == 0) {
                    mbar_arrive_cnt(xempty_bar((i + cx) % C::kXStages), H);
                    mbar_arrive_cnt(xempty_bar((i + cx + 1) % C::kXStages), H);
                }
                cx += 2;
            }
        }
        if (prm.cluster_split > 0) {
            cluster_sync();   // every rank's partial is in its shared memory
            if (seg.prob >= 0) {   // (the whole cluster skips a tile of a problem marked invalid)
                // Each rank of the cluster adds the S partials (in rank order) for its own slice of
                // the token columns, [rank NT / S, (rank + 1) NT / S), and writes that slice of Y:
                // the reads through distributed shared memory are spread over the cluster.
                const ProblemDesc& P = prob_at(prm, seg.prob);
                const int Mrows = P.M;
                const int S = prm.cluster_split;
                const int q = static_cast<int>(cluster_rank());
                const int n = seg.nt * kTileN + r;
                const int cb = max((q * NT) / S, col0), ce = min(((q + 1) * NT) / S, col0 + C::kNC);
                constexpr int kBatch = C::kNC <= 64 ? 4 : 2;   // parts of a 16-column batch loaded together
                const float bias = row_bias<BF16>(prm, P, n);
                for (int c = cb; c < ce; c += 16) {
                    const int nc = ce - c < 16 ? ce - c : 16;
                    float sum[16];
                    for (int q0 = 0; q0 < S; q0 += kBatch) {
                        float v[kBatch][16];
#pragma unroll
                        for (int b = 0; b < kBatch; ++b) {
                            if (q0 + b < S) {
                                const uint32_t base = map_to_rank(s_x0, static_cast<uint32_t>(q0 + b));
#pragma unroll
                                for (int j = 0; j < 16; ++j)
                                    if (j < nc) v[b][j] = ld_cluster_f32(base + ((c + j) * 128 + r) * 4);
                            }
                        }
#pragma unroll
                        for (int b = 0; b < kBatch; ++b) {
                            if (q0 + b < S) {
#pragma unroll
                                for (int j = 0; j < 16; ++j) sum[j] = (q0 + b == 0) ? v[b][j] : sum[j] + v[b][j];
                            }
                        }
                    }
                    constexpr int kB = C::kEpiBatch;
#pragma unroll
                    for (int h = 0; h < 16; h += kB)
                        store_cols<BF16, kB>(prm, P, sum, h, nc - h < 0 ? 0 : (nc - h < kB ? nc - h : kB),
                                             seg.mt * NT + c + h, n, Mrows, bias);
                }
            }
            cluster_sync();   // no CTA leaves while another still reads its shared memory
        }
        // the last C copy lands before the CTA can leave (whether or not the epilogue read it)
        if (f == 0 && lane == 0 && c_issued > 0)
            mbar_wait_plain(cfull_bar, static_cast<uint32_t>(c_issued - 1) & 1u, drain_limit(prm.timeout_cycles));
    }
    if (prm.cluster_split > 0 && warp < 4 + C::kDQW) {
        cluster_sync();
        cluster_sync();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::kTmemCols);
    }
    // A CTA that gave up (any role's wait ran out; the flag is final after the barrier above) lets
    // every copy its producers issued land before it exits: the last ring's worth of each.
    if ((warp == 0 || warp == 2) && lane == 0 && *abort_flag) {
        const bool is_x = warp == 0;
        const int depth = is_x ? C::kXStages : C::kWStages;
        for (int j = issued > depth ? issued - depth : 0; j < issued; ++j)
            mbar_wait_plain(is_x ? xfull_bar(j % depth) : wfull_bar(j % depth), (j / depth) & 1,
                            drain_limit(prm.timeout_cycles));
    }
}

// Host-side launcher for one instantiation (cluster = S CTAs per cluster in cluster mode, else 1).
template <int NT, bool BF16, int QT, int MAXP, bool ATMEM, int H>
cudaError_t launch_gemm(const GemmParams<MAXP>& p, int grid, bool pdl, cudaStream_t stream) {
    using C = GemmCfg<NT, QT, ATMEM, H>;
    auto kern = wq4_gemm_kernel<NT, BF16, QT, MAXP, ATMEM, H>;
    if constexpr (C::kRegSplit) {
        // The register split assumes 128 registers per thread at launch; a build that launched
        // with fewer would leave the fold warps' setmaxnreg.inc waiting forever. Refuse it.
        static int launch_regs = -1;
        if (launch_regs < 0) {
            cudaFuncAttributes fa;
            if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) return cudaErrorInvalidDeviceFunction;
            launch_regs = fa.numRegs;
        }
        if (launch_regs != 128) return cudaErrorInvalidConfiguration;
    }
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(C::kThreads, 1, 1);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = p.cluster_split > 0 ? p.cluster_split : 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
    e = cudaLaunchKernelEx(&cfg, kern, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace wq4
