// W4A16 GEMM for decode-sized M (at most 32 tokens), sm_103a.
//
// At a few tokens the tensor core's per-instruction floor decides: a tcgen05.mma with M = 128
// costs the same ~78 cycles for any N up to 128, so 8 tokens (padded to N = 16) use a few percent
// of it, while mma.sync m16n8k16 takes exactly 8 tokens as its N and sustains ~1000 FMA/clk/SM.
// This kernel therefore keeps the pages' register-sourced design ("machete_mainloop.cuh",
// header comment and transform_A_kblock: the narrow weight is the MMA's A operand, up-converted
// in registers right before the MMA) on the warp-level MMA:
//
//   * each CTA owns RB blocks of 16 weight rows over all of K, so no partial sum leaves the CTA;
//     its warps split K into KS = warps / RB slices (slice ks takes groups ks, ks + KS, ...; any
//     warps beyond RB x KS idle) and add their parts through shared memory in slice order
//     (deterministic);
//   * every warp streams its own weight pieces (16-byte cp.async from the prepacked records) into
//     a private ring of 2 or 4 group stages; the activations arrive through 4 to 8 3-D tensor copies
//     per CTA (each a run of the K/64 panels x Mpad token rows x 128 B, 128-byte swizzle, rows past
//     M zero), each on its own barrier, so the first groups start before all of X is in;
//   * programmatic dependent launch: the prologue (barriers, tensor-map prefetch) overlaps the
//     previous kernel's tail; every global access waits for griddepcontrol.wait;
//   * lane (g, c) of a warp reads word c of each 32-element chunk of rows g and g + 8; the k order
//     inside a chunk is permuted identically for A and B (slot 2c + t and 2c + 8 + t of k-step h
//     hold elements 8c + 4h + t and 8c + 4h + 2 + t), so a lane's B fragments for the chunk's two
//     k-steps are one 16-byte shared load;
//   * per group: P = sum over the group's 128 K of (q - z) x (exact integer operands, fp32
//     accumulate), then acc += s[row, group] * P in fp32 (the group scale, as in the tcgen05 path).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstring>

#include "wq4_device.cuh"
#include "wq4_launch.h"
#include "wq4_params.h"

namespace wq4 {

struct DecodeParams {
    CUtensorMap xmap;        // 3-D (64, M, K/64), strides (2K, 128) bytes, box (64, Mpad, 2 x_gp)
    const uint8_t* wp;       // first tile record
    void* y;                 // [M][N]
    int M, N, K;
    int k_groups;
    int n_blocks;            // N / 16
    int rb;                  // row blocks per CTA
    int depth;               // group stages per warp ring (2 or 4)
    int x_gp;                // groups per activation piece
    int x_pieces;            // activation pieces (at most kDecXPieces)
    unsigned int* status;
    long long timeout_cycles;
    int test_stall;          // 1: thread 0 of each CTA waits on a barrier nothing arrives on (tests)
    int has_epi;             // 1: Y = alpha acc + beta C + bias (else Y = acc)
    float alpha, beta;
    const void* c;           // [M][N], read when beta != 0 (may be Y itself)
    const void* bias;        // [N] or null
};

constexpr int kDecStage = 1024 + 32 + 16;                     // codes, scales, zero points
constexpr int kDecMaxX = 140 * 1024;                          // activation bytes held per CTA
constexpr int kDecXPieces = 8;                                // most activation copies per CTA

// warps per CTA: 16 at every token-block count (at one block 32 warps with half the groups each
// were measured ~1 % slower: the group loop is issue-bound, and fewer warps run more groups per
// loop setup)
__host__ __device__ constexpr int dec_warps(int) { return 16; }

template <int NB>
struct DecCfg {
    static constexpr int kMpad = 8 * NB;
    static constexpr int kWarps = dec_warps(NB);
    static constexpr int kRedBytes = kWarps * NB * 32 * 16;     // per-warp partials for the final sum
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async8(uint32_t dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z)
        : "memory");
}

template <bool BF16>
__device__ __forceinline__ float dec_to_float(uint16_t b) {
    if constexpr (BF16) {
        return __uint_as_float(static_cast<uint32_t>(b) << 16);
    } else {
        return __half2float(__ushort_as_half(b));
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

template <int NB, bool BF16, bool ZP>
__global__ void __launch_bounds__(dec_warps(NB) * 32, 1) wq4_decode_kernel(const __grid_constant__ DecodeParams prm) {
    using C = DecCfg<NB>;
    constexpr int kRec = tile_record_bytes(ZP);
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t sbase = (raw_s + 1023u) & ~1023u;
    const int depth = prm.depth;
    const uint32_t x_piece_bytes = static_cast<uint32_t>(C::kMpad * prm.x_gp * 256);
    const uint32_t x_bytes = x_piece_bytes * prm.x_pieces;
    const uint32_t s_x = sbase;                                       // activations (swizzled panels)
    const uint32_t s_w = sbase + ((x_bytes + 1023) & ~1023u);          // per-warp stage rings
    const uint32_t s_red = s_w + C::kWarps * depth * kDecStage;       // slice partials
    const uint32_t s_bar = s_red + C::kRedBytes;                      // one barrier per activation piece
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem_raw + (s_bar + 8 * kDecXPieces - raw_s));
    const uint8_t* const sm = smem_raw + (sbase - raw_s);              // generic view of the aligned base

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    const int KS = C::kWarps / prm.rb;                                // K slices
    const int bl = warp % prm.rb, ks = warp / prm.rb;
    const int block = blockIdx.x * prm.rb + bl;                       // 16-row block of this warp
    const bool active = (ks < KS) && block < prm.n_blocks;

    const uint32_t stall_bar = s_bar + 8 * kDecXPieces + 8;            // after the abort flag
    if (threadIdx.x == 0) {
        for (int q = 0; q < prm.x_pieces; ++q) mbar_init(s_bar + 8 * q, 1);
        mbar_init(stall_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    // Programmatic dependent launch: the next kernel on the stream may begin its own prologue and
    // weight prefetch now; this one waits for its predecessor before touching activations or
    // outputs (griddepcontrol is a no-op when the launch carries no programmatic dependency).
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (threadIdx.x == 0) prefetch_tensormap(&prm.xmap);
    // Nothing else happens before griddepcontrol.wait: the weights may be written by the kernel
    // ahead of this one on the stream (a prepack), whose writes are only guaranteed visible after
    // the wait. (An L2 prefetch of the weights ahead of the wait was measured slower: it queues
    // the activation copy behind weight traffic.)

    float acc[NB][4];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[nb][i] = 0.f;

    // this warp's groups: ks, ks + KS, ...
    const int n_my = active ? (prm.k_groups - ks + KS - 1) / KS : 0;
    const int nt = block >> 3, rblk = (block & 7) * 16;               // n-tile and first row inside it
    const uint32_t my_ring = s_w + warp * (depth * kDecStage);
    // per-lane constants of the copy pattern: this lane moves code pieces lane and lane + 32
    // (piece = chunk j * 16 + row), lanes 0..1 the two 16-byte halves of the scales, lane 2 the
    // eight bytes of zero points; a group's record advances by KS records per step
    const size_t rec_step = static_cast<size_t>(KS) * kRec;
    const uint8_t* rec_next = prm.wp + (static_cast<size_t>(nt) * prm.k_groups + ks) * kRec;
    const uint32_t goff0 = ((lane >> 4) * 128 + rblk + (lane & 15)) * 16;
    const uint32_t goff1 = (((lane + 32) >> 4) * 128 + rblk + (lane & 15)) * 16;
    const uint32_t soff_side = lane < 2 ? 1024 + lane * 16 : 1056;
    const uint32_t goff_side = lane < 2 ? 8192 + 2 * rblk + lane * 16 : 8448 + rblk / 2;
    auto issue = [&](int slot) {
        const uint32_t st = my_ring + slot * kDecStage;
        cp_async16(st + lane * 16, rec_next + goff0);
        cp_async16(st + lane * 16 + 512, rec_next + goff1);
        if (lane < 2) cp_async16(st + soff_side, rec_next + goff_side);
        if constexpr (ZP) {
            if (lane == 2) cp_async8(st + soff_side, rec_next + goff_side);
        }
        rec_next += rec_step;
    };
    const int pre = n_my < depth ? n_my : depth;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (threadIdx.x == 0) {
        // the activations in pieces of x_gp groups, so that the first groups start early
        for (int q = 0; q < prm.x_pieces; ++q) {
            mbar_arrive_expect_tx(s_bar + 8 * q, x_piece_bytes);
            tma_load_3d(s_x + q * x_piece_bytes, &prm.xmap, s_bar + 8 * q, 0, 0, 2 * prm.x_gp * q);
        }
    }
    for (int i = 0; i < depth; ++i) {
        if (i < pre) issue(i);
        cp_async_commit();                                            // empty groups keep the count uniform
    }

    const WaitCtl ctl{abort_flag, prm.status, prm.timeout_cycles};
    // (tests) a wait that nothing ends: it runs out, records the timeout and stops this warp
    bool ok = !(prm.test_stall && threadIdx.x == 0) || mbar_wait(stall_bar, 0, ctl);
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;                 // the whole warp stops with it
    int x_piece = -1;                                                 // last activation piece waited for
    // activation piece of the current group, tracked as the groups advance by KS (no division
    // per group): group ks + i KS lies in piece `piece`, which ends before group piece_end
    int piece = ks / prm.x_gp, piece_end = (piece + 1) * prm.x_gp, grp = ks;

    // activation addresses: token row m = 8 nb + g sits at 128-byte row (panel * Mpad + m) whose
    // swizzle key is (row & 7) = g; the lane's 16-byte chunk in a panel is (4 (j & 1) + c) ^ g
    const uint32_t xo_even = g * 128 + ((c ^ g) << 4);
    const uint32_t xo_odd = g * 128 + (((4 + c) ^ g) << 4);
    const uint32_t x_grp_step = static_cast<uint32_t>(KS) * 2 * C::kMpad * 128;
    uint32_t x_grp = s_x + static_cast<uint32_t>(ks) * 2 * C::kMpad * 128;
    const uint32_t a_off = g * 16 + 4 * c;                            // word c of row g in a chunk

    constexpr uint32_t kMagic = BF16 ? 0x43004300u : 0x64006400u;
    for (int i = 0; i < n_my && ok; ++i, grp += KS) {
        while (grp >= piece_end) {
            ++piece;
            piece_end += prm.x_gp;
        }
        if (piece != x_piece) {
            ok = mbar_wait(s_bar + 8 * piece, 0, ctl);
            x_piece = piece;
            if (!ok) break;
        }
        if (depth == 4)
            cp_async_wait<3>();
        else
            cp_async_wait<1>();
        __syncwarp();
        const int slot = i & (depth - 1);
        const uint32_t st = my_ring + slot * kDecStage;
        uint32_t sub_lo, sub_hi;                                      // 128 + z (bf16) per row
        const uint8_t* const stp = sm + (st - sbase);
        if constexpr (ZP) {
            const uint32_t w0 = *reinterpret_cast<const uint32_t*>(stp + 1056);
            const uint32_t w1 = *reinterpret_cast<const uint32_t*>(stp + 1060);
            const uint32_t z0 = (w0 >> (g * 4)) & 0xFu, z1 = (w1 >> (g * 4)) & 0xFu;
            sub_lo = ((BF16 ? 0x4300u : 0x6400u) | z0) * 0x10001u;
            sub_hi = ((BF16 ? 0x4300u : 0x6400u) | z1) * 0x10001u;
        } else {
            sub_lo = sub_hi = BF16 ? 0x43084308u : 0x64086408u;
        }
        const uint8_t* const a_base = stp + a_off;
        const uint8_t* const xe = sm + (x_grp - sbase) + xo_even;
        const uint8_t* const xd = sm + (x_grp - sbase) + xo_odd;
        float p[NB][4], p2[NB][4];                                    // two chains: even / odd chunks
#pragma unroll
        for (int nb = 0; nb < NB; ++nb)
#pragma unroll
            for (int t = 0; t < 4; ++t) p[nb][t] = p2[nb][t] = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            // word c of rows g and g + 8
            const uint32_t wlo = *reinterpret_cast<const uint32_t*>(a_base + j * 256);
            const uint32_t whi = *reinterpret_cast<const uint32_t*>(a_base + j * 256 + 128);
            uint32_t lo[4], hi[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                lo[e] = dec_sub2<BF16>(((wlo >> (4 * e)) & 0x000F000Fu) | kMagic, sub_lo);
                hi[e] = dec_sub2<BF16>(((whi >> (4 * e)) & 0x000F000Fu) | kMagic, sub_hi);
            }
            const uint32_t a0[4] = {lo[0], hi[0], lo[1], hi[1]};
            const uint32_t a1[4] = {lo[2], hi[2], lo[3], hi[3]};
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) {
                const uint4 xb = *reinterpret_cast<const uint4*>(((j & 1) ? xd : xe) +
                                                                 (j >> 1) * C::kMpad * 128 + nb * 8 * 128);
                if (j & 1) {
                    mma16816<BF16>(p2[nb], a0, xb.x, xb.y);
                    mma16816<BF16>(p2[nb], a1, xb.z, xb.w);
                } else {
                    mma16816<BF16>(p[nb], a0, xb.x, xb.y);
                    mma16816<BF16>(p[nb], a1, xb.z, xb.w);
                }
            }
        }
        x_grp += x_grp_step;
        // group scale (rows g and g + 8), then release the stage and fetch the group DEPTH ahead
        const uint32_t sbits_lo = *reinterpret_cast<const uint16_t*>(stp + 1024 + 2 * g);
        const uint32_t sbits_hi = *reinterpret_cast<const uint16_t*>(stp + 1040 + 2 * g);
        float s_lo, s_hi;
        if constexpr (BF16) {
            s_lo = __uint_as_float(sbits_lo << 16);
            s_hi = __uint_as_float(sbits_hi << 16);
        } else {
            s_lo = __half2float(__ushort_as_half(static_cast<uint16_t>(sbits_lo)));
            s_hi = __half2float(__ushort_as_half(static_cast<uint16_t>(sbits_hi)));
        }
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
            acc[nb][0] = fmaf(s_lo, p[nb][0] + p2[nb][0], acc[nb][0]);
            acc[nb][1] = fmaf(s_lo, p[nb][1] + p2[nb][1], acc[nb][1]);
            acc[nb][2] = fmaf(s_hi, p[nb][2] + p2[nb][2], acc[nb][2]);
            acc[nb][3] = fmaf(s_hi, p[nb][3] + p2[nb][3], acc[nb][3]);
        }
        __syncwarp();
        if (i + depth < n_my) issue(slot);
        cp_async_commit();
    }
    cp_async_wait<0>();

    // the epilogue's C values and bias for the rows this warp writes, loaded now so that their
    // latency overlaps the exchange of partials below (each element is read here and written
    // later by the same thread, so C may be Y itself)
    const bool writer = active && ks == 0;
    const int n0 = block * 16 + g;
    uint16_t cv[NB][4];
    float bv[2] = {0.f, 0.f};
#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
        for (int t = 0; t < 4; ++t) cv[nb][t] = 0;
    if (writer && prm.has_epi) {
        if (prm.beta != 0.f) {
            const uint16_t* cp = static_cast<const uint16_t*>(prm.c);
#pragma unroll
            for (int nb = 0; nb < NB; ++nb)
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const int m = nb * 8 + 2 * c + (t & 1);
                    if (m < prm.M) cv[nb][t] = cp[static_cast<size_t>(m) * prm.N + n0 + (t >> 1) * 8];
                }
        }
        if (prm.bias) {
            const uint16_t* bp = static_cast<const uint16_t*>(prm.bias);
            bv[0] = dec_to_float<BF16>(bp[n0]);
            bv[1] = dec_to_float<BF16>(bp[n0 + 8]);
        }
    }

    // slice partials -> shared memory, then slice 0 adds them in slice order and writes Y
#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
        sts128(s_red + ((warp * NB + nb) * 32 + lane) * 16, __float_as_uint(acc[nb][0]), __float_as_uint(acc[nb][1]),
               __float_as_uint(acc[nb][2]), __float_as_uint(acc[nb][3]));
    __syncthreads();
    // A CTA that gave up (the flag is final after the barrier above; a warp waits only for the
    // activation pieces of its own groups) lets every activation copy land before it exits.
    if (threadIdx.x == 0 && *abort_flag) {
        for (int q = 0; q < prm.x_pieces; ++q) mbar_wait_plain(s_bar + 8 * q, 0, drain_limit(prm.timeout_cycles));
    }
    if (writer) {
        uint16_t* y = reinterpret_cast<uint16_t*>(prm.y);
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
            float v[4] = {0.f, 0.f, 0.f, 0.f};
            for (int s = 0; s < KS; ++s) {
                const uint4 q = lds128(s_red + (((s * prm.rb + bl) * NB + nb) * 32 + lane) * 16);
                v[0] += __uint_as_float(q.x);
                v[1] += __uint_as_float(q.y);
                v[2] += __uint_as_float(q.z);
                v[3] += __uint_as_float(q.w);
            }
            // fragment: (row g, tokens 2c, 2c+1), (row g + 8, tokens 2c, 2c+1)
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const int m = nb * 8 + 2 * c + (t & 1);
                const int n = n0 + (t >> 1) * 8;
                if (m < prm.M) {
                    float val = v[t];
                    if (prm.has_epi) {   // alpha acc + beta C + bias in fp32, rounded once below
                        val *= prm.alpha;
                        if (prm.beta != 0.f) val = fmaf(prm.beta, dec_to_float<BF16>(cv[nb][t]), val);
                        if (prm.bias) val += bv[t >> 1];
                    }
                    uint16_t o;
                    if constexpr (BF16) {
                        o = __bfloat16_as_ushort(__float2bfloat16_rn(val));
                    } else {
                        o = __half_as_ushort(__float2half_rn(val));
                    }
                    y[static_cast<size_t>(m) * prm.N + n] = o;
                }
            }
        }
    }
}

// Activation pieces: groups per piece and piece count, 4 to 8 pieces with the least padding (the
// last piece may run past K; the copy fills what lies beyond the tensor with zeros and the kernel
// never reads it, but shared memory must hold it).
static void dec_x_geometry(int K, int* gp, int* pieces) {
    const int kg = K / kTileK;
    int best_gp = kg, best_waste = 1 << 30;
    for (int target = 4; target <= kDecXPieces; ++target) {
        const int g = (kg + target - 1) / target;
        const int waste = g * ((kg + g - 1) / g) - kg;
        if (waste < best_waste) {
            best_waste = waste;
            best_gp = g;
        }
    }
    *gp = best_gp;
    *pieces = (kg + best_gp - 1) / best_gp;
}

static int decode_smem_bytes(int nb, int K, int depth) {
    int gp, pieces;
    dec_x_geometry(K, &gp, &pieces);
    const int x = (8 * nb * gp * pieces * 256 + 1023) & ~1023;
    return 1024 + x + dec_warps(nb) * depth * kDecStage + dec_warps(nb) * nb * 32 * 16 + 8 * kDecXPieces + 32;
}

// Deepest per-warp ring that fits next to the activations.
static int decode_depth(int nb, int K) { return decode_smem_bytes(nb, K, 4) <= 232448 ? 4 : 2; }

bool decode_fits(int M, int K) {
    if (M < 1 || M > 32 || K / 64 > 256) return false;
    const int nb = (M + 7) / 8;
    const int mpad = 8 * (nb == 3 ? 4 : nb);
    return mpad * K * 2 <= kDecMaxX && decode_smem_bytes(mpad / 8, K, 2) <= 232448;
}

template <int NB, bool BF16, bool ZP>
static cudaError_t go_decode(const DecodeParams& p, int grid, bool pdl, cudaStream_t st) {
    auto kern = wq4_decode_kernel<NB, BF16, ZP>;
    const int smem = decode_smem_bytes(NB, p.K, p.depth);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(dec_warps(NB) * 32, 1, 1);
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

template <int NB>
static cudaError_t pick_decode(const DecodeParams& p, bool bf16, bool zp, int grid, bool pdl, cudaStream_t st) {
    if (bf16) return zp ? go_decode<NB, true, true>(p, grid, pdl, st) : go_decode<NB, true, false>(p, grid, pdl, st);
    return zp ? go_decode<NB, false, true>(p, grid, pdl, st) : go_decode<NB, false, false>(p, grid, pdl, st);
}

// Host entry used by wq4_mm: X [M][K], blob, Y [M][N]; the caller has checked decode_fits().
cudaError_t launch_decode(const void* X, const void* Wp, void* Y, int M, int N, int K, int dtype, int qtype,
                          int sm_count, unsigned int* status, long long timeout_cycles, void* encode_fn_ptr,
                          bool pdl, int test_stall, const EpilogueArgs* epi, int* grid_out, int* rb_out,
                          cudaStream_t st) {
    using Enc = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                             const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                             CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
    int nb = (M + 7) / 8;
    if (nb == 3) nb = 4;
    DecodeParams p;
    std::memset(static_cast<void*>(&p), 0, sizeof(p));
    const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(M), static_cast<cuuint64_t>(K / 64)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(K) * 2, 128};
    int gp, pieces;
    dec_x_geometry(K, &gp, &pieces);
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(8 * nb), static_cast<cuuint32_t>(2 * gp)};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = reinterpret_cast<Enc>(encode_fn_ptr)(
        &p.xmap, dtype == 0 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
        const_cast<void*>(X), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    p.wp = static_cast<const uint8_t*>(Wp) + kBlobHeader;
    p.y = Y;
    p.M = M;
    p.N = N;
    p.K = K;
    p.k_groups = K / kTileK;
    p.n_blocks = N / 16;
    // fewest row blocks per CTA that keeps the grid within one wave; each CTA's warps split K into
    // warps / rb slices (warps beyond rb * slices stay idle: at N = 14336, 6 blocks on 150 CTAs
    // beat 8 blocks on 112 CTAs by a quarter less work per SM)
    const int warps = dec_warps(nb);
    int rb = (p.n_blocks + sm_count - 1) / sm_count;
    if (rb > warps) rb = warps;
    p.rb = rb;
    p.depth = decode_depth(nb, K);
    p.x_gp = gp;
    p.x_pieces = pieces;
    p.status = status;
    p.timeout_cycles = timeout_cycles;
    p.test_stall = test_stall;
    if (epi) {
        p.has_epi = 1;
        p.alpha = epi->alpha;
        p.beta = epi->beta;
        p.c = epi->c;
        p.bias = epi->bias;
    }
    const int grid = (p.n_blocks + rb - 1) / rb;
    *grid_out = grid;
    *rb_out = rb;
    const bool bf16 = dtype == 0, zp = qtype == 1;
    switch (nb) {
        case 1: return pick_decode<1>(p, bf16, zp, grid, pdl, st);
        case 2: return pick_decode<2>(p, bf16, zp, grid, pdl, st);
        default: return pick_decode<4>(p, bf16, zp, grid, pdl, st);
    }
}

}  // namespace wq4
