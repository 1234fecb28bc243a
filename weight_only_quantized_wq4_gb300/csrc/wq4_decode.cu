// W4A16 GEMM for decode-sized M (at most 32 tokens), sm_103a.
//
// At a few tokens the tensor core's per-instruction floor decides: a tcgen05.mma with M = 128
// costs the same ~78 cycles for any N up to 128, so 8 tokens (padded to N = 16) use a few percent
// of it, while mma.sync m16n8k16 takes exactly 8 tokens as its N. This kernel therefore keeps the
// pages' register-sourced design ("machete_mainloop.cuh", header comment and transform_A_kblock:
// the narrow weight is the MMA's A operand, up-converted in registers right before the MMA) on the
// warp-level MMA, and spends its effort on moving the weight bytes at the rate of HBM:
//
//   * every SM gets a CTA; CTA c owns a contiguous run of 16-row weight blocks over all of K, so no
//     partial sum leaves the CTA (a CTA's weight share differs by at most one block);
//   * a producer warp stages the CTA's blocks with 4-D tensor copies of the prepacked blob (one
//     copy = one block's records for 8 groups: its codes, scales and zero points are one contiguous
//     run per record), into a ring of stages under mbarriers with transaction counts (after
//     "machete_mainloop.cuh", load); the activations arrive as one tensor copy per 8 groups;
//   * 16 consumer warps: block b of the CTA has KS = 16 / blocks warps, warp ks takes the groups
//     g = ks (mod KS); per group, two ldmatrix.x4 give a lane its 8 code words (word c of rows g,
//     g + 8 of each 32-element chunk), bit logic turns them into the exact integers (q - z) as the
//     A fragments, and mma.sync accumulates P = sum (q - z) x in fp32; then acc += s[row] P (the
//     group's scale in fp32, as in the tcgen05 path); the KS partials of a block are added through
//     shared memory in slice order (deterministic);
//   * the blob header is compared with the call's arguments before any record is read; a
//     mismatch sets the status word (WQ4_ERR_INVALID) and the CTA stops;
//   * programmatic dependent launch: nothing that a kernel ahead on the stream may write (the
//     activations, the outputs, and by default the blob) is read before griddepcontrol.wait. With
//     constant weights (the caller's promise that no pending kernel writes the blob) the header
//     check and the first ring of weight copies are issued before that wait, so the weight stream
//     overlaps the tail of the kernel ahead. The next kernel is let in once this CTA's
//     activations have landed (its own early weight copies then do not queue ahead of them).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstring>
#include <memory>

#include "wq4_device.cuh"
#include "wq4_launch.h"
#include "wq4_params.h"

namespace wq4 {

constexpr int kDecWarps = 16;                           // consumer warps; warp 16 is the producer
constexpr int kDecThreads = (kDecWarps + 1) * 32;
constexpr int kDecStageGroups = 8;                      // groups per weight stage and per activation piece
constexpr int kDecMaxPieces = 64;                       // activation pieces: K up to 65536
constexpr int kDecMaxDepth = 16;
constexpr int kDecMaxSmem = 232448;
constexpr int kDecCoResident = 115712;                  // two CTAs of at most this much fit on one SM

// One problem of a launch: its operands, sizes and first CTA (a grouped launch gives each problem
// a contiguous range of CTAs; each CTA works on row blocks of its own problem only).
struct DecodeProblem {
    CUtensorMap xmap;        // X: 3-D (64, M, K/64) 16-bit, box (64, Mpad, 16), 128-byte swizzle
    CUtensorMap wmap;        // blob blocks: 4-D (block_bytes / 8, 8, K/128, N/128) u64, box (.., 1, 8, 1)
    const uint32_t* hdr;     // blob header
    void* y;                 // [M][N]
    const void* c;           // epilogue C [M][N], read when beta != 0 (may be Y itself); single problems
    const void* bias;        // epilogue bias [N] or null; single problems
    int M, N, K;
    int k_groups;
    int n_blocks;            // N / 16
    int n_stages;            // ceil(k_groups / 8): weight stages per block = activation pieces
    int cta_begin;           // first CTA of this problem
};

template <int MAXP>
struct DecodeParams {
    DecodeProblem prob[MAXP];
    int num_problems;
    int group_size, dtype, qtype;
    int depth;               // ring slots
    unsigned int* status;
    long long timeout_cycles;
    int test_stall;          // 1: one consumer thread per CTA waits on a barrier nothing arrives on (tests)
    int early;               // 1: header check and the first ring of weight copies before griddepcontrol.wait
    int trigger_late;        // 1: let the next kernel in once the activations landed (else at once)
    int hdr_trusted;         // 1: the blob was prepacked in this process for these arguments: records are
                             // copied while the header is checked (else only after the check passed)
    int has_epi;             // 1: Y = alpha acc + beta C + bias (else Y = acc)
    float alpha, beta;
    NibbleConsts nib;        // nibble_consts(dtype == bf16)
};

template <int NB>
struct DecCfg {
    static constexpr int kMpad = 8 * NB;
    static constexpr int kPieceBytes = kDecStageGroups * 2 * kMpad * 128;   // activations of 8 groups
    static constexpr int kRedBytes = kDecWarps * NB * 32 * 16;              // per-warp partials
};

__host__ __device__ constexpr int dec_stage_bytes(int qt, int H = 1) { return kDecStageGroups * block_bytes(qt, H); }

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z)
        : "memory");
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y, int z,
                                            int w, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4, %5, %6}], [%2], %7;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z), "r"(w), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& d0, uint32_t& d1, uint32_t& d2, uint32_t& d3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(d0), "=r"(d1), "=r"(d2), "=r"(d3)
                 : "r"(addr));
}

template <bool BF16>
__device__ __forceinline__ float dec_to_float(uint32_t b16) {
    if constexpr (BF16) {
        return __uint_as_float(b16 << 16);
    } else {
        return __half2float(__ushort_as_half(static_cast<uint16_t>(b16)));
    }
}

template <bool BF16>
__device__ __forceinline__ uint32_t dec_sub2(uint32_t a, uint32_t b) {
    // packed 16-bit subtraction on the raw 32-bit registers (no pair-struct round trip)
    uint32_t d;
    if constexpr (BF16) {
        asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    } else {
        asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    }
    return d;
}

// d = a . b (accumulator starts at zero: no register moves to clear it)
template <bool BF16>
__device__ __forceinline__ void mma16816_z(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    if constexpr (BF16) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%10,%10,%10,%10};"
            : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.f));
    } else {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%10,%10,%10,%10};"
            : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.f));
    }
}

template <bool BF16>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    if constexpr (BF16) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    } else {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
}

template <int NB, bool BF16, int QT, int H, int MAXP>
__global__ void __launch_bounds__(kDecThreads, NB == 1 ? 2 : 1)
    wq4_decode_kernel(const __grid_constant__ DecodeParams<MAXP> prm) {
    using C = DecCfg<NB>;
    // this CTA's problem (the last whose first CTA is <= blockIdx.x), its index and CTA count there
    int pidx = 0;
    if constexpr (MAXP > 1) {
        int lo = 0, hi = prm.num_problems - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (prm.prob[mid].cta_begin <= static_cast<int>(blockIdx.x)) lo = mid; else hi = mid - 1;
        }
        pidx = lo;
    }
    const DecodeProblem& Q = prm.prob[pidx];
    const int cta = static_cast<int>(blockIdx.x) - Q.cta_begin;
    const int ncta = (pidx + 1 < prm.num_problems ? prm.prob[pidx + 1].cta_begin : static_cast<int>(gridDim.x)) - Q.cta_begin;
    constexpr int kBB = block_bytes(QT, H);
    constexpr int kStage = dec_stage_bytes(QT, H);
    constexpr int kZ = block_zero_off(H);
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t sbase = (raw_s + 1023u) & ~1023u;
    const int depth = prm.depth;
    const int n_st = Q.n_stages;
    const uint32_t x_bytes = static_cast<uint32_t>(n_st) * C::kPieceBytes;
    const uint32_t x_region = x_bytes > static_cast<uint32_t>(C::kRedBytes) ? x_bytes : C::kRedBytes;
    const uint32_t s_x = sbase;                                        // activations, later the partials
    const uint32_t s_w = sbase + ((x_region + 127u) & ~127u);          // weight ring
    const uint32_t s_bar = s_w + depth * kStage;
    auto full_bar = [&](int i) { return s_bar + 8u * i; };
    auto empty_bar = [&](int i) { return s_bar + 8u * (kDecMaxDepth + i); };
    auto xfull_bar = [&](int p) { return s_bar + 8u * (2 * kDecMaxDepth + p); };
    const uint32_t stall_bar = s_bar + 8u * (2 * kDecMaxDepth + kDecMaxPieces);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem_raw + (stall_bar + 8 - raw_s));
    const uint8_t* const sm = smem_raw + (sbase - raw_s);              // generic view of the aligned base

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // this CTA's blocks [bb0, bb0 + nbc) and the K slices per block
    const int bb0 = static_cast<int>((static_cast<long long>(cta) * Q.n_blocks) / ncta);
    const int nbc = static_cast<int>((static_cast<long long>(cta + 1) * Q.n_blocks) / ncta) - bb0;
    const int KS = kDecWarps / nbc;
    const int n_items = nbc * n_st;                                    // weight stages of this CTA
    // Ring slots per block: block b uses slots [b Db, (b + 1) Db), stage s of it slot b Db + s % Db
    // at phase s / Db. Every waiter then walks consecutive phases of its slots (a parity wait is
    // only unambiguous one phase ahead; blocks sharing a slot would skip each other's phases).
    const int Db = depth / nbc;

    // with constant weights the producer fetches the blob header first thing (its latency then
    // overlaps the set-up below); otherwise only after the kernel ahead has completed
    BlobHeader hdr{};
    if (warp == kDecWarps && lane == 0 && prm.early) hdr = load_blob_header(Q.hdr);
    if (threadIdx.x == 0) {
        for (int i = 0; i < depth; ++i) {
            mbar_init(full_bar(i), 1);
            mbar_init(empty_bar(i), KS);
        }
        for (int p = 0; p < n_st; ++p) mbar_init(xfull_bar(p), 1);
        mbar_init(stall_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (!prm.trigger_late) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    const WaitCtl ctl{abort_flag, prm.status, prm.timeout_cycles};
    int issued = 0;                                                    // weight stages copied (producer)
    if (warp == kDecWarps) {
        // ------------------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tensormap(&Q.xmap);
            prefetch_tensormap(&Q.wmap);
            const uint64_t pol = policy_evict_first();
            // item `issued` = (stage is, block ib); its slot and the stage's position in the block's slots
            int is = 0, ib = 0, isd = 0;
            uint32_t iph = 0;
            auto issue_next = [&]() {
                const int slot = ib * Db + isd;
                mbar_arrive_expect_tx(full_bar(slot), kStage);
                int b = bb0 + ib, gz = is * kDecStageGroups;   // (a failed check reads the blob's origin)
                if (!WQ4_CHECK(b >= 0 && b < Q.n_blocks && gz >= 0 && gz < Q.k_groups, prm.status, abort_flag,
                               check::kSiteDecW, b, gz, Q.n_blocks)) b = gz = 0;
                tma_load_4d(s_w + slot * kStage, &Q.wmap, full_bar(slot), 0, b & 7, gz, b >> 3, pol);
                ++issued;
                if (++ib == nbc) {
                    ib = 0;
                    ++is;
                    if (++isd == Db) {
                        isd = 0;
                        iph ^= 1u;
                    }
                }
            };
            bool ok = true;
            // items in the first Db stages fill every slot once: no wait for a free slot
            const int first = n_items < Db * nbc ? n_items : Db * nbc;
            const bool trusted = prm.hdr_trusted != 0;
            if (prm.early) {
                if (trusted) {
                    while (issued < first) issue_next();
                    ok = blob_header_matches(hdr, Q.N, Q.K, prm.group_size, prm.dtype, prm.qtype);
                } else {
                    ok = blob_header_matches(hdr, Q.N, Q.K, prm.group_size, prm.dtype, prm.qtype);
                    while (ok && issued < first) issue_next();
                }
            }
            asm volatile("griddepcontrol.wait;" ::: "memory");
            // activations: one copy per 8 groups (rows past M and K past the end read as zero)
            for (int p = 0; p < n_st; ++p) {
                mbar_arrive_expect_tx(xfull_bar(p), C::kPieceBytes);
                int pz = 2 * kDecStageGroups * p;              // first 64-wide K panel of the piece
                if (!WQ4_CHECK(pz >= 0 && 64 * pz < Q.K, prm.status, abort_flag, check::kSiteDecX, pz, p, Q.K)) pz = 0;
                tma_load_3d(s_x + p * C::kPieceBytes, &Q.xmap, xfull_bar(p), 0, 0, pz);
            }
            if (!prm.early) {
                if (trusted) {
                    while (issued < first) issue_next();
                    ok = blob_header_ok(Q.hdr, Q.N, Q.K, prm.group_size, prm.dtype, prm.qtype);
                } else {
                    ok = blob_header_ok(Q.hdr, Q.N, Q.K, prm.group_size, prm.dtype, prm.qtype);
                    while (ok && issued < first) issue_next();
                }
            }
            if (!ok) {
                atomicOr(prm.status, kStatusBadBlob);
                *abort_flag = 1;
            }
            if (prm.trigger_late) {
                for (int p = 0; ok && p < n_st; ++p) ok = mbar_wait(xfull_bar(p), 0, ctl);
                asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
            }
            while (ok && issued < n_items) {
                if (!mbar_wait(empty_bar(ib * Db + isd), iph ^ 1u, ctl)) break;
                issue_next();
            }
        }
        __syncwarp();
    } else {
        asm volatile("griddepcontrol.wait;" ::: "memory");
    }

    // ---------------------------------------------------------------------- consumers
    float acc[NB][4];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[nb][i] = 0.f;
    const int bl = warp / KS, ks = warp % KS;                           // block and K slice of this warp
    const bool active = warp < kDecWarps && bl < nbc;
    const int g = lane >> 2, c = lane & 3;
    // activations: token 8 nb + g at 128-byte row (panel * Mpad + token), swizzle key g
    const uint32_t xo_even = g * 128 + ((c ^ g) << 4);
    const uint32_t xo_odd = g * 128 + (((4 + c) ^ g) << 4);
    bool ok = true;
    if (warp < kDecWarps) {
        // (tests) a wait that nothing ends: it runs out, records the timeout and stops the CTA
        ok = !(prm.test_stall && warp == 0 && lane == 0) || mbar_wait(stall_bar, 0, ctl);
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    }
    if (active && ok) {
        const uint32_t ld_off = 256u * (lane >> 4) + 16u * ((lane & 7) + 8 * ((lane >> 3) & 1));
        const NibbleConsts nib = prm.nib;
        int next_g = ks;                                                // next group of this slice
        int sd = 0;                                                     // stage's slot within the block's Db
        uint32_t ph = 0;
        for (int s = 0; s < n_st && ok; ++s) {
            const int slot = bl * Db + sd;
            ok = mbar_wait(full_bar(slot), ph, ctl);
            if (!ok) break;
            const int g_lo = s * kDecStageGroups;
            const int g_hi = min(g_lo + kDecStageGroups, Q.k_groups);
            const uint32_t st = s_w + slot * kStage;
            if (next_g < g_hi) {                                        // this stage's activation piece
                ok = mbar_wait(xfull_bar(s), 0, ctl);
                if (!ok) break;
            }
            for (; next_g < g_hi; next_g += KS) {
                const int gg = next_g;
                const uint32_t ua = st + (gg - g_lo) * kBB;             // this block's record of group gg
                const uint8_t* const up = sm + (ua - sbase);
                // per scale set q (one per 64-K half with a group size of 64, else one for both
                // halves): the scale word, the packed subtrahend base + z, the float zeros of rows g, g + 8
                uint32_t sw[H], sub_lo[H], sub_hi[H];
                float zf_lo[H], zf_hi[H];
#pragma unroll
                for (int q = 0; q < H; ++q) {
                    sw[q] = *reinterpret_cast<const uint32_t*>(up + kBlockScaleOff + 32 * q + 4 * g);
                    zf_lo[q] = zf_hi[q] = 0.f;
                    if constexpr (QT == kQtU4Zp) {
                        const uint32_t zb = up[kZ + 8 * q + g];
                        sub_lo[q] = ((BF16 ? 0x4300u : 0x6400u) | (zb & 0xFu)) * 0x10001u;
                        sub_hi[q] = ((BF16 ? 0x4300u : 0x6400u) | (zb >> 4)) * 0x10001u;
                    } else if constexpr (QT == kQtU4FZp) {
                        sub_lo[q] = sub_hi[q] = BF16 ? 0x43004300u : 0x64006400u;   // the code itself
                        const uint32_t zw = *reinterpret_cast<const uint32_t*>(up + kZ + 32 * q + 4 * g);
                        zf_lo[q] = dec_to_float<BF16>(zw & 0xFFFFu);
                        zf_hi[q] = dec_to_float<BF16>(zw >> 16);
                    } else {
                        sub_lo[q] = sub_hi[q] = BF16 ? 0x43084308u : 0x64086408u;
                    }
                }
                const uint32_t xg = s_x + static_cast<uint32_t>(gg) * (2 * C::kMpad * 128);
                const uint8_t* const xe = sm + (xg - sbase) + xo_even;
                const uint8_t* const xd = sm + (xg - sbase) + xo_odd;
                // two independent MMA chains, one per 64-element half of the group (half the
                // dependent latency of one chain over the group), added (or scaled apart) at the fold
                float pr[2][NB][4];
                // float zeros: the activation sum per token of each scale set's K range, from an
                // MMA with an all-ones A (the tensor pipe has room; the integer pipe does not)
                float ps[H][NB][4];
                constexpr uint32_t kOnes = BF16 ? 0x3F803F80u : 0x3C003C00u;
                const uint32_t ones[4] = {kOnes, kOnes, kOnes, kOnes};
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    constexpr int kOne = 0;
                    const int qs = H == 2 ? q : kOne;                  // this half's scale set
                    uint32_t w[4];                                      // (2q, g) (2q, g+8) (2q+1, g) (2q+1, g+8)
                    ldsm_x4(ua + 512u * q + ld_off, w[0], w[1], w[2], w[3]);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int j = 2 * q + h;
                        const uint32_t wlo = w[2 * h], whi = w[2 * h + 1];
                        uint32_t lo[4], hi[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            // bit logic on the integer pipe, the exact subtraction on the fp16/bf16 one
                            lo[e] = dec_sub2<BF16>(and_or(wlo >> (4 * e), nib.mask, nib.magic), sub_lo[qs]);
                            hi[e] = dec_sub2<BF16>(and_or(whi >> (4 * e), nib.mask, nib.magic), sub_hi[qs]);
                        }
                        const uint32_t a0[4] = {lo[0], hi[0], lo[1], hi[1]};
                        const uint32_t a1[4] = {lo[2], hi[2], lo[3], hi[3]};
#pragma unroll
                        for (int nb = 0; nb < NB; ++nb) {
                            const uint4 xb = *reinterpret_cast<const uint4*>(((j & 1) ? xd : xe) +
                                                                             (j >> 1) * C::kMpad * 128 + nb * 8 * 128);
                            if (h == 0) {
                                mma16816_z<BF16>(pr[q][nb], a0, xb.x, xb.y);
                            } else {
                                mma16816<BF16>(pr[q][nb], a0, xb.x, xb.y);
                            }
                            mma16816<BF16>(pr[q][nb], a1, xb.z, xb.w);
                            if constexpr (QT == kQtU4FZp) {
                                if (h == 0 && (q == 0 || H == 2)) {
                                    mma16816_z<BF16>(ps[qs][nb], ones, xb.x, xb.y);
                                } else {
                                    mma16816<BF16>(ps[qs][nb], ones, xb.x, xb.y);
                                }
                                mma16816<BF16>(ps[qs][nb], ones, xb.z, xb.w);
                            }
                        }
                    }
                }
                // group scales of rows g and g + 8 (one 32-bit word per set), in fp32
#pragma unroll
                for (int nb = 0; nb < NB; ++nb) {
                    if constexpr (H == 1) {
                        const float s_lo = dec_to_float<BF16>(sw[0] & 0xFFFFu);
                        const float s_hi = dec_to_float<BF16>(sw[0] >> 16);
                        acc[nb][0] = fmaf(s_lo, pr[0][nb][0] + pr[1][nb][0], acc[nb][0]);
                        acc[nb][1] = fmaf(s_lo, pr[0][nb][1] + pr[1][nb][1], acc[nb][1]);
                        acc[nb][2] = fmaf(s_hi, pr[0][nb][2] + pr[1][nb][2], acc[nb][2]);
                        acc[nb][3] = fmaf(s_hi, pr[0][nb][3] + pr[1][nb][3], acc[nb][3]);
                    } else {
#pragma unroll
                        for (int q = 0; q < 2; ++q) {
                            const float s_lo = dec_to_float<BF16>(sw[q] & 0xFFFFu);
                            const float s_hi = dec_to_float<BF16>(sw[q] >> 16);
                            acc[nb][0] = fmaf(s_lo, pr[q][nb][0], acc[nb][0]);
                            acc[nb][1] = fmaf(s_lo, pr[q][nb][1], acc[nb][1]);
                            acc[nb][2] = fmaf(s_hi, pr[q][nb][2], acc[nb][2]);
                            acc[nb][3] = fmaf(s_hi, pr[q][nb][3], acc[nb][3]);
                        }
                    }
                    if constexpr (QT == kQtU4FZp) {
#pragma unroll
                        for (int q = 0; q < H; ++q) {
                            acc[nb][0] = fmaf(zf_lo[q], ps[q][nb][0], acc[nb][0]);
                            acc[nb][1] = fmaf(zf_lo[q], ps[q][nb][1], acc[nb][1]);
                            acc[nb][2] = fmaf(zf_hi[q], ps[q][nb][2], acc[nb][2]);
                            acc[nb][3] = fmaf(zf_hi[q], ps[q][nb][3], acc[nb][3]);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty_bar(slot));
            if (++sd == Db) {
                sd = 0;
                ph ^= 1u;
            }
        }
    }

    __syncthreads();                                                   // every consumer is done with X
    // A CTA that gave up (the flag is final after the barrier above) lets every copy it issued land
    // before it exits: all activation pieces and the newest copy into each weight slot.
    if (*abort_flag) {
        if (warp == kDecWarps && lane == 0) {
            const long long lim = drain_limit(prm.timeout_cycles);
            for (int p = 0; p < n_st; ++p) mbar_wait_plain(xfull_bar(p), 0, lim);
            uint32_t seen = 0;
            for (int j = issued - 1; j >= 0 && j >= issued - Db * nbc; --j) {
                const int sj = j / nbc, slot = (j % nbc) * Db + sj % Db;
                if (seen & (1u << slot)) continue;
                seen |= 1u << slot;
                mbar_wait_plain(full_bar(slot), static_cast<uint32_t>(sj / Db) & 1u, lim);
            }
        }
        return;
    }
    // slice partials -> shared memory (over the activations), then every output element is the
    // sum of its block's KS slice partials in slice order (deterministic)
    if (active) {
#pragma unroll
        for (int nb = 0; nb < NB; ++nb)
            sts128(s_x + ((warp * NB + nb) * 32 + lane) * 16, __float_as_uint(acc[nb][0]), __float_as_uint(acc[nb][1]),
                   __float_as_uint(acc[nb][2]), __float_as_uint(acc[nb][3]));
    }
    __syncthreads();
    // (consumer threads only: they have all waited for the kernel ahead before touching C or Y)
    const int n_out = nbc * NB * 128;
    uint16_t* y = reinterpret_cast<uint16_t*>(Q.y);
    for (int t = threadIdx.x; warp < kDecWarps && t < n_out; t += kDecWarps * 32) {
        const int ob = t / (NB * 128), orem = t % (NB * 128);
        const int onb = orem / 128, olane = (orem % 128) >> 2, ot = orem & 3;
        const int om = onb * 8 + 2 * (olane & 3) + (ot & 1);
        const int on = (bb0 + ob) * 16 + (olane >> 2) + (ot >> 1) * 8;
        if (om >= Q.M) continue;
        if (!WQ4_CHECK(on >= 0 && on < Q.N, prm.status, nullptr, check::kSiteYStore, on, om, Q.N)) continue;
        float v = 0.f;
        for (int sl = 0; sl < KS; ++sl)
            v += *reinterpret_cast<const float*>(sm + (((ob * KS + sl) * NB + onb) * 32 + olane) * 16 + 4 * ot);
        if (prm.has_epi) {                                              // alpha acc + beta C + bias, rounded once
            v *= prm.alpha;
            if (prm.beta != 0.f)
                v = fmaf(prm.beta, dec_to_float<BF16>(static_cast<const uint16_t*>(Q.c)[static_cast<size_t>(om) * Q.N + on]), v);
            if (Q.bias) v += dec_to_float<BF16>(static_cast<const uint16_t*>(Q.bias)[on]);
        }
        uint16_t o;
        if constexpr (BF16) {
            o = __bfloat16_as_ushort(__float2bfloat16_rn(v));
        } else {
            o = __half_as_ushort(__float2half_rn(v));
        }
        y[static_cast<size_t>(om) * Q.N + on] = o;
    }
}

// ------------------------------------------------------------------------------------ host
static int dec_nb(int M) {
    const int nb = (M + 7) / 8;
    return nb == 3 ? 4 : nb;
}

static int dec_x_region(int nb, int K) {
    const int n_st = (K / kTileK + kDecStageGroups - 1) / kDecStageGroups;
    const int x = n_st * kDecStageGroups * 2 * 8 * nb * 128;
    const int red = kDecWarps * nb * 32 * 16;
    return ((x > red ? x : red) + 127) & ~127;
}

static int decode_smem_bytes(int nb, int K, int depth, int zp, int H) {
    return 1024 + dec_x_region(nb, K) + depth * dec_stage_bytes(zp, H) + 8 * (2 * kDecMaxDepth + kDecMaxPieces + 1) + 16;
}

// Ring depth: the deepest that fits, capped by the items a CTA has and, while the activations are
// small enough, by the size at which a CTA of the next launch still fits beside this one - unless
// that size leaves a block a single slot (no double buffering: each stage then waits a full HBM
// round trip) where the full size gives it two (measured, 8 tokens, N = 14336, K = 4096, constant
// weights: 6 blocks per CTA, 10.5 us with two CTAs per SM and one slot per block, 8.9 us with one
// CTA per SM and two slots per block).
static int decode_depth(int nb, int K, int zp, int H, int items_max, int nbc, int forced) {
    const int d_min = nbc > 2 ? nbc : 2;
    int d = forced > 0 ? forced : kDecMaxDepth;
    if (d > items_max) d = items_max;
    if (d < d_min) d = d_min;
    const bool small_x = dec_x_region(nb, K) <= 64 * 1024;
    while (d > d_min && decode_smem_bytes(nb, K, d, zp, H) > kDecMaxSmem) --d;
    if (forced <= 0 && small_x) {
        int dc = d;
        while (dc > d_min && decode_smem_bytes(nb, K, dc, zp, H) > kDecCoResident) --dc;
        const bool co_double = dc >= items_max || dc >= 2 * nbc;
        const bool full_double = d >= items_max || d >= 2 * nbc;
        if (co_double || !full_double) d = dc;
    }
    return d;
}

bool decode_fits(int M, int K) {
    if (M < 1 || M > 32) return false;
    const int n_st = (K / kTileK + kDecStageGroups - 1) / kDecStageGroups;
    if (n_st > kDecMaxPieces) return false;
    return decode_smem_bytes(dec_nb(M), K, 2, kQtU4FZp, 2) <= kDecMaxSmem;   // the largest records
}

template <int NB, bool BF16, int QT, int H, int MAXP>
static cudaError_t go_decode(const DecodeParams<MAXP>& p, int smem, int grid, bool pdl, cudaStream_t st) {
    auto kern = wq4_decode_kernel<NB, BF16, QT, H, MAXP>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(kDecThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    e = cudaLaunchKernelEx(&cfg, kern, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <int NB, int H, int MAXP>
static cudaError_t pick_decode_q(const DecodeParams<MAXP>& p, bool bf16, int qt, int smem, int grid, bool pdl,
                                 cudaStream_t st) {
    switch (qt) {
        case kQtU4B8:
            return bf16 ? go_decode<NB, true, kQtU4B8, H>(p, smem, grid, pdl, st)
                        : go_decode<NB, false, kQtU4B8, H>(p, smem, grid, pdl, st);
        case kQtU4Zp:
            return bf16 ? go_decode<NB, true, kQtU4Zp, H>(p, smem, grid, pdl, st)
                        : go_decode<NB, false, kQtU4Zp, H>(p, smem, grid, pdl, st);
        default:
            return bf16 ? go_decode<NB, true, kQtU4FZp, H>(p, smem, grid, pdl, st)
                        : go_decode<NB, false, kQtU4FZp, H>(p, smem, grid, pdl, st);
    }
}

template <int MAXP>
static cudaError_t pick_decode(const DecodeParams<MAXP>& p, int nb, bool bf16, int qt, int H, int smem, int grid,
                               bool pdl, cudaStream_t st) {
    switch (nb) {
        case 1:
            return H == 2 ? pick_decode_q<1, 2>(p, bf16, qt, smem, grid, pdl, st) : pick_decode_q<1, 1>(p, bf16, qt, smem, grid, pdl, st);
        case 2:
            return H == 2 ? pick_decode_q<2, 2>(p, bf16, qt, smem, grid, pdl, st) : pick_decode_q<2, 1>(p, bf16, qt, smem, grid, pdl, st);
        default:
            return H == 2 ? pick_decode_q<4, 2>(p, bf16, qt, smem, grid, pdl, st) : pick_decode_q<4, 1>(p, bf16, qt, smem, grid, pdl, st);
    }
}

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// A problem's record: its activation and weight-block maps (rows of X padded to 8 nb), pointers
// and sizes. False if a map could not be encoded.
static bool fill_problem(DecodeProblem& q, EncodeFn enc, const void* X, const void* Wp, void* Y, int M, int N, int K,
                         int nb, int dtype, int zp, int H) {
    {
        const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(M), static_cast<cuuint64_t>(K / 64)};
        const cuuint64_t strides[2] = {static_cast<cuuint64_t>(K) * 2, 128};
        const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(8 * nb), static_cast<cuuint32_t>(2 * kDecStageGroups)};
        const cuuint32_t estr[3] = {1, 1, 1};
        if (enc(&q.xmap, dtype == 0 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                const_cast<void*>(X), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return false;
    }
    {
        // the blob's records as 16-row blocks: (u64 words of a block, block, group, n-tile)
        const int bb = block_bytes(zp, H);
        const cuuint64_t dims[4] = {static_cast<cuuint64_t>(bb / 8), 8, static_cast<cuuint64_t>(K / kTileK),
                                    static_cast<cuuint64_t>(N / kTileN)};
        const cuuint64_t strides[3] = {static_cast<cuuint64_t>(bb), static_cast<cuuint64_t>(tile_record_bytes(zp, H)),
                                       static_cast<cuuint64_t>(tile_record_bytes(zp, H)) * (K / kTileK)};
        const cuuint32_t box[4] = {static_cast<cuuint32_t>(bb / 8), 1, kDecStageGroups, 1};
        const cuuint32_t estr[4] = {1, 1, 1, 1};
        if (enc(&q.wmap, CU_TENSOR_MAP_DATA_TYPE_UINT64, 4,
                const_cast<uint8_t*>(static_cast<const uint8_t*>(Wp) + kBlobHeader), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return false;
    }
    q.hdr = static_cast<const uint32_t*>(Wp);
    q.y = Y;
    q.M = M;
    q.N = N;
    q.K = K;
    q.k_groups = K / kTileK;
    q.n_blocks = N / kBlockRows;
    q.n_stages = (q.k_groups + kDecStageGroups - 1) / kDecStageGroups;
    return true;
}

// The parts of a launch that every problem shares, and the launch itself: the grid is the sum of
// the problems' CTA counts (cta_begin already set); the ring depth and shared memory are sized for
// the largest K and per-CTA block count.
template <int MAXP>
static cudaError_t launch_params(DecodeParams<MAXP>& p, const DecodeLaunch& L, int nb, int Kmax, int nbc_max,
                                 int items_max, int grid, int group_size, int dtype, int qtype, int* grid_out,
                                 int* depth_out, cudaStream_t st) {
    const int zp = qtype;                                       // record layout of the format
    const int H = scale_sets(group_size);
    p.group_size = group_size;
    p.dtype = dtype;
    p.qtype = qtype;
    p.nib = nibble_consts(dtype == 0);
    p.depth = decode_depth(nb, Kmax, zp, H, items_max, nbc_max, L.depth);
    const int smem = decode_smem_bytes(nb, Kmax, p.depth, zp, H);
    if (smem > kDecMaxSmem) return cudaErrorInvalidConfiguration;
    p.status = L.status;
    p.timeout_cycles = L.timeout_cycles;
    p.test_stall = L.test_stall;
    // (early copies only pay for a blob of some size: at 92 KB, 16 CTAs, they made the call slower)
    long long wbytes = 0;
    for (int i = 0; i < p.num_problems; ++i) wbytes += static_cast<long long>(p.prob[i].N) * p.prob[i].K / 2;
    p.early = L.const_weights && wbytes >= (1LL << 20);
    p.trigger_late = L.trigger_late;
    p.hdr_trusted = L.hdr_trusted;
    *grid_out = grid;
    *depth_out = p.depth;
    return pick_decode<MAXP>(p, nb, dtype == 0, zp, H, smem, grid, L.pdl, st);
}

// Blocks a CTA may own: ring slots (one per block at least, within shared memory) and warps (16).
static int decode_cap(int nb, int Kmax, int zp, int H) {
    const int cap = (kDecMaxSmem - decode_smem_bytes(nb, Kmax, 0, zp, H)) / dec_stage_bytes(zp, H);
    return cap > kDecWarps ? kDecWarps : cap;
}

// Host entry used by wq4_mm: X [M][K], blob, Y [M][N]; the caller has checked decode_fits().
cudaError_t launch_decode(const DecodeLaunch& L, const void* X, const void* Wp, void* Y, int M, int N, int K,
                          int group_size, int dtype, int qtype, const EpilogueArgs* epi, int* grid_out,
                          int* depth_out, cudaStream_t st) {
    const int nb = dec_nb(M);
    const int zp = qtype;
    const int H = scale_sets(group_size);
    DecodeParams<1> p;
    std::memset(static_cast<void*>(&p), 0, sizeof(p));
    DecodeProblem& q = p.prob[0];
    if (!fill_problem(q, reinterpret_cast<EncodeFn>(L.encode_fn), X, Wp, Y, M, N, K, nb, dtype, zp, H))
        return cudaErrorInvalidValue;
    p.num_problems = 1;
    // one CTA per SM; a CTA owns at most `cap` blocks: beyond that, more CTAs than SMs
    int grid = L.sm_count < q.n_blocks ? L.sm_count : q.n_blocks;
    const int cap = decode_cap(nb, K, zp, H);
    if (cap < 1) return cudaErrorInvalidConfiguration;
    if (q.n_blocks > cap * grid) grid = (q.n_blocks + cap - 1) / cap;
    const int nbc_max = (q.n_blocks + grid - 1) / grid;
    if (epi) {
        p.has_epi = 1;
        p.alpha = epi->alpha;
        p.beta = epi->beta;
        q.c = epi->c;
        q.bias = epi->bias;
    }
    return launch_params(p, L, nb, K, nbc_max, nbc_max * q.n_stages, grid, group_size, dtype, qtype, grid_out,
                         depth_out, st);
}

// Host entry used by wq4_grouped_mm when every problem is decode-sized: P problems with M[p] > 0,
// one launch. Each problem gets CTAs in proportion to its row blocks (at least one, and enough that
// no CTA owns more than `cap` blocks); a CTA works on blocks of its own problem only.
cudaError_t launch_decode_grouped(const DecodeLaunch& L, int P, const void* const* X, const void* const* Wp,
                                  void* const* Y, const int* M, const int* N, const int* K, int group_size, int dtype,
                                  int qtype, int* grid_out, int* depth_out, cudaStream_t st) {
    if (P < 1 || P > kMaxGroupedProblems) return cudaErrorInvalidValue;
    const int zp = qtype;
    const int H = scale_sets(group_size);
    int Mmax = 0, Kmax = 0;
    long long blocks = 0;
    for (int i = 0; i < P; ++i) {
        Mmax = M[i] > Mmax ? M[i] : Mmax;
        Kmax = K[i] > Kmax ? K[i] : Kmax;
        blocks += N[i] / kBlockRows;
    }
    const int nb = dec_nb(Mmax);
    const int cap = decode_cap(nb, Kmax, zp, H);
    if (cap < 1) return cudaErrorInvalidConfiguration;
    auto pp = std::make_unique<DecodeParams<kMaxGroupedProblems>>();
    DecodeParams<kMaxGroupedProblems>& p = *pp;
    std::memset(static_cast<void*>(&p), 0, sizeof(p));
    const EncodeFn enc = reinterpret_cast<EncodeFn>(L.encode_fn);
    int grid = 0, nbc_max = 0, items_max = 0;
    for (int i = 0; i < P; ++i) {
        DecodeProblem& q = p.prob[i];
        if (!fill_problem(q, enc, X[i], Wp[i], Y[i], M[i], N[i], K[i], nb, dtype, zp, H)) return cudaErrorInvalidValue;
        long long g = (static_cast<long long>(q.n_blocks) * L.sm_count + blocks / 2) / blocks;
        if (g < 1) g = 1;
        if (g < (q.n_blocks + cap - 1) / cap) g = (q.n_blocks + cap - 1) / cap;
        if (g > q.n_blocks) g = q.n_blocks;
        q.cta_begin = grid;
        grid += static_cast<int>(g);
        const int nbc = static_cast<int>((q.n_blocks + g - 1) / g);
        nbc_max = nbc > nbc_max ? nbc : nbc_max;
        items_max = nbc * q.n_stages > items_max ? nbc * q.n_stages : items_max;
    }
    p.num_problems = P;
    return launch_params(p, L, nb, Kmax, nbc_max, items_max, grid, group_size, dtype, qtype, grid_out, depth_out, st);
}

}  // namespace wq4
