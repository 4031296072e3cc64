// Resident small-M kernel ("gemv"): y = x . W^T for 1 <= M <= 32 activation
// rows (one, two or four 8-column MMA blocks), streaming the packed weights
// once per call; also several projections of one x per launch and the fused
// gate/up + SiLU.  Kernel template, plan types and launch dispatch, shared by
// the translation units that instantiate them (aq_gemv*.cu).
//
// Method (mlx-bun pages, @mlx-bun/inference 1.0.0, kernels/quantization/):
//   * the weight format: 64-value groups, 2*B uint32 words each, LSB-first
//     codes (affine-split-mma.ts affine_unit; affine3/4-mma.ts);
//   * the factored group dot product of affine3-rows.ts / affine4-rows.ts:
//     sum_g [ scale_g * sum_k q_k x_k + bias_g * sum_k x_k ], each weight
//     decoded once and reused for every activation row;
//   * the K-permuted operand layout of affine{3,4}-mma.ts: inside a group
//     any order of k serves, provided x takes the same order;
//   * the gate/up kernel of trellis-shared-m.ts: silu(gate) * up formed in
//     the epilogue of the two products.
//
// GB300 design:
//   * At most one CTA per SM.  CTA c owns a contiguous block of R weight
//     rows over all of K, R = ceil(N / SMs), so every SM streams the same
//     number of bytes; a block taller than 128 rows (96 with two or four
//     column blocks) runs in passes.
//   * A producer warp streams the block through a ring of stages in shared
//     memory: one stage is SG groups of K (SG = 8, 16 or 32) for the R rows,
//     loaded by three TMA boxes issued from three lanes at once - the codes
//     as one 3-D box (SG/4 column blocks of 128 bytes, 96 at 3 bits, times R
//     rows), the scales and the biases as one 3-D box each (blocks of 8
//     groups times R rows, so a row's 8 scales are 16 bytes from the next
//     row's and the loads of 8 rows never share a bank) - with completion
//     counted on an mbarrier.  (On GB300 a TMA op costs ~75 ns of issue time
//     whatever its size, so a stage is a few large boxes.)  A last stage
//     past the end of K reads zero fill and its groups are skipped.  The
//     weights do not depend on the preceding kernel, so the producer fills
//     the ring before the CTA waits on the preceding grid.
//     With one column block a CTA takes at most 112 KB of shared memory and
//     288 threads, so it fits on an SM beside a CTA of the previous call:
//     with programmatic dependent launch a call's weight stream overlaps the
//     previous call's tail.  With two or four blocks the CTA has the SM (and
//     its 227 KB) to itself.
//   * Eight consumer warps.  Warp w takes SG/8 consecutive groups of every
//     stage, for all the block's 16-row tiles and column blocks (template
//     parameters, so the units interleave freely).
//   * x whole (one column block, x and its sums within 48 KB): one bulk copy
//     per activation row once the grid dependency resolves, rewritten in
//     place into B-fragment order with the group sums.  Otherwise
//     ("staged"): a fourth producer lane streams it with the weights, one
//     3-D TMA box of the stage's groups x M rows per stage, and each warp
//     builds its fragments and sums per group.
//   * Codes decode into MMA A fragments (weights are the 16-row A operand)
//     with one shift and one LOP3 per two codes (4-bit fp16: one AND per
//     two codes plus a shift per word, the codes staying in place), each
//     code alone in the bits of a 16-bit half:
//       fp16 MMA: the half is the subnormal q * 2^(p-24) (exact), so
//               y_g = scale * 2^24 * D + bias * sum(x);
//       bf16 MMA: under the exponent of 128 the half is the bf16 value
//               128 + q (exact), so y_g = scale * D + (bias - 128 * scale) * sum(x).
//     At 4 bits with x whole, x is rewritten as fp16 with a power-of-two
//     scale per (group, row) and the fp16 MMA serves either x type; staged
//     x is the B operand in its own type.  mma.sync m16n8k16 accumulates in
//     fp32.
//   * The eight warps' partial tiles meet in shared memory and are added in
//     warp order (deterministic).
#pragma once

#include "aq_internal.h"
#include "aq_ptx.cuh"

#include <cuda.h>

#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <mutex>
#include <type_traits>

namespace aq {
namespace gemv {

constexpr int kConsumers = 8;                     // consumer warps
constexpr int kGemvThreads = (kConsumers + 1) * 32;  // + one producer warp
constexpr int kMaxTiles = 8;                      // 16-row tiles per pass
constexpr int kMaxProj = 4;                       // projections of one x per launch
constexpr int kMaxPassRows = 16 * kMaxTiles;
constexpr int kXPitch = 144;     // bytes per activation row in an x slot (128 + 16: no bank conflicts)
// An x slot holds one group of every activation row (M rows at kXPitch),
// rewritten in place into MMA B-fragment order, then the group's sums of x
// for the 8 MMA columns (32 bytes).
constexpr size_t kSmemBudget = 112 * 1024;  // two CTAs (two calls) per SM

struct GemvParams {
    const void *x;
    void *y;
    uint32_t *err;   // the device error word
    int M, N, K;
    int rows_cta;    // weight rows per CTA (passes * pass_rows)
    int pass_rows;   // rows per pass = TMA box height (<= 128)
    int passes;
    int tiles;       // 16-row tiles per pass
    int sg;          // groups per stage (8 x groups per warp)
    int n_stages;    // G / sg
    int ring;        // weight stages in the ring
    int x_whole;     // 1: all of x in shared memory (one bulk copy per row); 0: staged per stage
    int red_alias;   // 1: the partial-tile buffer reuses the ring (single pass)
    uint32_t slot_bytes, off_sc, off_bi;  // inside a ring slot (codes at 0)
    uint32_t off_x, off_red, off_bar;
    uint32_t x_row_pitch;   // whole x: bytes per activation row (2K + 16)
    uint32_t off_xs;        // whole x: group sums [G][8] floats, then scale factors [G][8]
    uint32_t off_xst;       // staged x: box inside a ring slot
    int x_rows;             // staged x: rows per group in the box (= M)
    uint32_t stage_tx;      // bytes one stage brings in
#ifdef AQ_TEST_HOOKS
    int withhold;           // test builds only: the producer skips its first stage
#endif
};

// Several projections of the same x in one launch (kernels instantiated
// with MP = true only).  Independent outputs: CTAs cta0[j] .. cta0[j+1]-1
// take projection j.  Gate/up (gate_up = 1, two projections of equal N):
// every CTA takes the same rows of both, pass 0 the gate and pass 1 the up
// projection, and writes silu(gate) * up; the gate's rows wait in shared
// memory at off_gu.
struct GemvMulti {
    int nproj;
    int gate_up;
    int cta0[kMaxProj + 1];
    int n_proj[kMaxProj];
    void *y_proj[kMaxProj];
    uint32_t off_gu;
};

// Tensor maps of one launch (host side): x (staged x only) and the codes,
// scales and biases of each projection.  The kernel takes each map as a
// parameter of its own, in the order w0, s0, b0, x, then the other
// projections; the single-projection kernels carry no code for the others.
struct GemvMaps {
    CUtensorMap x;
    CUtensorMap w[kMaxProj], s[kMaxProj], b[kMaxProj];
};

__device__ __forceinline__ void consumers_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumers * 32) : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const void *tm) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(tm) : "memory");
}

__device__ __forceinline__ void gemv_record(volatile int *flag, uint32_t *err, uint32_t code) {
    *flag = 1;
    atomicOr(err, code);
}

// Bounded mbarrier wait; gives up at once if another warp already gave up.
__device__ __forceinline__ bool gemv_wait(uint64_t *bar, uint32_t parity, volatile int *flag,
                                          uint32_t *err, uint32_t code) {
    if (*flag) return false;
    if (mbar_wait(bar, parity)) return true;
    gemv_record(flag, err, code);
    return false;
}

// (Not volatile: the MMA has no side effects, so independent ones may be
// scheduled freely.)
template <bool BF16>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    if constexpr (BF16)
        asm(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
            "{%8,%9}, {%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    else
        asm(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
            "{%8,%9}, {%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// d = A * B (no accumulator input): the zero C comes from one register that
// the compiler keeps for the whole loop, instead of four zeroed registers
// per MMA chain.
template <bool BF16>
__device__ __forceinline__ void mma16816_first(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1, float zero) {
    if constexpr (BF16)
        asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
            "{%8,%9}, {%10,%10,%10,%10};"
            : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(zero));
    else
        asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
            "{%8,%9}, {%10,%10,%10,%10};"
            : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(zero));
}

// A thread holds 16 codes of a group for one row (codes 16c .. 16c+15 of the
// group, c = lane % 4).  They decode into 8 registers P[i] of two 16-bit
// halves holding codes (lo(i), hi(i)):
//   4-bit: (0,4) (1,5) (2,6) (3,7) (8,12) (9,13) (10,14) (11,15)
//   3-bit: (i, i+8)
// The four MMA k-steps of the group take the register pairs
//   4-bit: (P0,P2) (P4,P6) (P1,P3) (P5,P7);  3-bit: (P0,P1) (P2,P3) (P4,P5) (P6,P7).
//
// 4-bit with fp16 x: each code stays where it is inside its half, which is
// then the exact fp16 subnormal q * 2^(p-24) with p = 0 for P0, P2, P4, P6
// and p = 4 for P1, P3, P5, P7 (one shift and four ANDs per word).  Steps
// 0-1 and steps 2-3 therefore accumulate separately (D0 at 2^-24, D4 at
// 2^-20).  Otherwise every code is shifted to bit 0 of its half and or-ed
// with `magic`: zero (fp16 subnormal q * 2^-24) or the bf16 exponent of 128
// (the bf16 value 128 + q).
// (a & b) | c in one LOP3.  Written out because with two immediate operands
// the compiler splits it into two logic operations.
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

template <bool kInPlace, uint32_t kMagic>
__device__ __forceinline__ void decode4(uint32_t w0, uint32_t w1, uint32_t (&P)[8]) {
    constexpr uint32_t m = 0x000F000Fu;
    if constexpr (kInPlace) {
        const uint32_t v0 = w0 >> 8, v1 = w1 >> 8;
        P[0] = w0 & m;
        P[1] = w0 & (m << 4);
        P[2] = v0 & m;
        P[3] = v0 & (m << 4);
        P[4] = w1 & m;
        P[5] = w1 & (m << 4);
        P[6] = v1 & m;
        P[7] = v1 & (m << 4);
    } else {
        P[0] = and_or(w0, m, kMagic);
        P[1] = and_or(w0 >> 4, m, kMagic);
        P[2] = and_or(w0 >> 8, m, kMagic);
        P[3] = and_or(w0 >> 12, m, kMagic);
        P[4] = and_or(w1, m, kMagic);
        P[5] = and_or(w1 >> 4, m, kMagic);
        P[6] = and_or(w1 >> 8, m, kMagic);
        P[7] = and_or(w1 >> 12, m, kMagic);
    }
}

// 3-bit: the thread's 48-bit span (code j at bit 3j) starts at byte bo of
// word wa.  r0 = span bytes {0,1,3,4} has codes 0..4 in its low half and
// 8..12 in its high half, each half starting at bit 0; r2 = span bytes
// {1,2,4,5} has codes 5..7 and 13..15 from bit 7 of each half.
template <uint32_t kMagic>
__device__ __forceinline__ void decode3(uint32_t wa, uint32_t wb, uint32_t sel0, uint32_t sel2,
                                        uint32_t (&P)[8]) {
    constexpr uint32_t m = 0x00070007u;
    const uint32_t r0 = prmt(wa, wb, sel0);
    const uint32_t r2 = prmt(wa, wb, sel2);
    P[0] = and_or(r0, m, kMagic);
    P[1] = and_or(r0 >> 3, m, kMagic);
    P[2] = and_or(r0 >> 6, m, kMagic);
    P[3] = and_or(r0 >> 9, m, kMagic);
    P[4] = and_or(r0 >> 12, m, kMagic);
    P[5] = and_or(r2 >> 7, m, kMagic);
    P[6] = and_or(r2 >> 10, m, kMagic);
    P[7] = and_or(r2 >> 13, m, kMagic);
}

// B fragments of the four k-steps from the thread's 16 raw x values
// (r[j] = (x_2j, x_2j+1)), matching the code pairs of each step.
template <int B>
__device__ __forceinline__ void x_frags(const uint4 &u0, const uint4 &u1, uint32_t (&bx)[4][2]) {
    const uint32_t r[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
    if constexpr (B == 4) {
        // (x0,x4)(x2,x6) | (x8,x12)(x10,x14) | (x1,x5)(x3,x7) | (x9,x13)(x11,x15)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int a = 4 * (q & 1);                     // 0, 4, 0, 4
            const uint32_t sel = q < 2 ? 0x5410u : 0x7632u;  // low or high halves
            bx[q][0] = prmt(r[a], r[a + 2], sel);
            bx[q][1] = prmt(r[a + 1], r[a + 3], sel);
        }
    } else {
        // (x0,x8)(x1,x9) | (x2,x10)(x3,x11) | (x4,x12)(x5,x13) | (x6,x14)(x7,x15)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            bx[q][0] = prmt(r[q], r[q + 4], 0x5410u);
            bx[q][1] = prmt(r[q], r[q + 4], 0x7632u);
        }
    }
}

// Code registers of k-step q (see decode4 / decode3).
template <int B>
__device__ __forceinline__ void step_frags(const uint32_t (&PA)[8], const uint32_t (&PB)[8], int q,
                                           uint32_t (&af)[4]) {
    int i0, i1;
    if constexpr (B == 4) {
        i0 = (q & 1) * 4 + (q >> 1);  // 0, 4, 1, 5
        i1 = i0 + 2;
    } else {
        i0 = 2 * q;
        i1 = i0 + 1;
    }
    af[0] = PA[i0];
    af[1] = PB[i0];
    af[2] = PA[i1];
    af[3] = PB[i1];
}

template <typename T>
__device__ __forceinline__ void store_y(T *p, float v);
template <>
__device__ __forceinline__ void store_y<__half>(__half *p, float v) { *p = __float2half_rn(v); }
template <>
__device__ __forceinline__ void store_y<__nv_bfloat16>(__nv_bfloat16 *p, float v) {
    *p = __float2bfloat16_rn(v);
}

template <int B, bool BF16, int TILES, int WPS, int MB, bool XST, bool MP>
__global__ void __launch_bounds__(kGemvThreads, MB > 1 ? 1 : 2)
    gemv_kernel(const __grid_constant__ GemvParams p, const __grid_constant__ CUtensorMap tm_w0,
                const __grid_constant__ CUtensorMap tm_s0, const __grid_constant__ CUtensorMap tm_b0,
                const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w1,
                const __grid_constant__ CUtensorMap tm_s1, const __grid_constant__ CUtensorMap tm_b1,
                const __grid_constant__ CUtensorMap tm_w2, const __grid_constant__ CUtensorMap tm_s2,
                const __grid_constant__ CUtensorMap tm_b2, const __grid_constant__ CUtensorMap tm_w3,
                const __grid_constant__ CUtensorMap tm_s3, const __grid_constant__ CUtensorMap tm_b3,
                const __grid_constant__ GemvMulti mx) {
    constexpr bool kXStage = XST;  // x streamed per stage by a fourth producer lane
    using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
    constexpr int kBox = B == 4 ? 128 : 96;  // bytes of a row in one column block (4 groups)
    extern __shared__ uint8_t smem_raw[];
    // Align to 1024 bytes by an offset from the __shared__ array itself, so
    // that every access below stays a shared-memory access (32-bit address).
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + p.off_bar);
    uint64_t *empty = full + p.ring;
    uint64_t *x_landed = empty + p.ring;  // one arrival per consumer warp
    uint64_t *x_full = x_landed + 1;      // whole x: the bulk copies of x
    volatile int *flag = reinterpret_cast<volatile int *>(x_full + 1);

    if (threadIdx.x == 0) {
        for (int i = 0; i < p.ring; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kConsumers);
        }
        mbar_init(x_landed, kConsumers);
        mbar_init(x_full, 1);
        *flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    // The next call is allowed to launch (and start streaming its weights)
    // only once this CTA's x has landed: launched earlier, its prefetch
    // would queue in front of this call's x loads.  Every thread that stays
    // alive triggers at that point (consumers after their copy, the
    // producer lanes once x_landed completes).

    int proj = 0;  // this CTA's projection (independent outputs)
    int row_cta = blockIdx.x * p.rows_cta;
    if constexpr (MP) {
        if (!mx.gate_up)
            while (proj + 1 < mx.nproj && (int)blockIdx.x >= mx.cta0[proj + 1]) ++proj;
        row_cta = ((int)blockIdx.x - mx.cta0[proj]) * p.rows_cta;
    }
    const int total = p.passes * p.n_stages;
    const int nb = p.sg / 4;  // column blocks per stage

    if (warp == kConsumers) {
        // ------------------------------------------------------------------
        // Producer: lanes 0, 1, 2 issue the codes, scales and biases boxes of
        // each (pass, stage) in order; lane 0 also posts the byte count.
        // ------------------------------------------------------------------
        if (lane < (kXStage ? 4 : 3)) {
            // the lane's map for projection j (lane 3: x)
            auto map_of = [&](int j) -> const CUtensorMap * {
                if (lane == 3) return &tm_x;
                if (j == 0) return lane == 0 ? &tm_w0 : lane == 1 ? &tm_s0 : &tm_b0;
                if (j == 1) return lane == 0 ? &tm_w1 : lane == 1 ? &tm_s1 : &tm_b1;
                if (j == 2) return lane == 0 ? &tm_w2 : lane == 1 ? &tm_s2 : &tm_b2;
                return lane == 0 ? &tm_w3 : lane == 1 ? &tm_s3 : &tm_b3;
            };
            const CUtensorMap *tm =
                lane == 0 ? &tm_w0 : lane == 1 ? &tm_s0 : lane == 2 ? &tm_b0 : &tm_x;
            if constexpr (MP) tm = map_of(proj);
            prefetch_tmap(tm);
            if constexpr (MP)
                if (mx.gate_up) prefetch_tmap(map_of(1));
            if (lane == 3) grid_dependency_wait();  // x belongs to the stream order
            bool triggered = false;
            int it = 0, slot = 0, lap = 0, pass = 0, s = 0;
            for (; it < total; ++it) {
                if (!triggered && mbar_test_wait(x_landed, 0)) {
                    launch_dependents();
                    triggered = true;
                }
                if (lap > 0 && !mbar_wait_sleep(&empty[slot], (lap - 1) & 1, 128)) {
                    gemv_record(flag, p.err, ERR_GEMV_EMPTY);
                    break;
                }
                int r0 = row_cta + pass * p.pass_rows;
                if constexpr (MP)
                    if (mx.gate_up) {  // the same rows of projection `pass`
                        r0 = row_cta;
                        tm = map_of(pass);
                    }
                uint8_t *dst = smem + (size_t)slot * p.slot_bytes;
#ifdef AQ_TEST_HOOKS
                const bool withheld = p.withhold && it == 0;  // nothing completes full[0]
#else
                constexpr bool withheld = false;
#endif
                if (withheld) {
                } else if (lane == 3) {
                    tma_load_3d(dst + p.off_xst, tm, 0, 0, s * p.sg, &full[slot]);
                } else if (lane == 0) {
                    mbar_arrive_expect_tx(&full[slot], p.stage_tx);
                    tma_load_3d(dst, tm, 0, r0, s * nb, &full[slot]);
                } else {
                    tma_load_3d(dst + (lane == 1 ? p.off_sc : p.off_bi), tm, 0, r0, s * (p.sg / 8),
                                &full[slot]);
                }
                if (++slot == p.ring) {
                    slot = 0;
                    ++lap;
                }
                if (++s == p.n_stages) {
                    s = 0;
                    ++pass;
                }
            }
            if (!triggered) {
                if (!mbar_wait_sleep(x_landed, 0, 512)) gemv_record(flag, p.err, ERR_GEMV_FULL);
                launch_dependents();
            }
            // Copies still in flight must land before the CTA may exit.
            if (lane == 0)
                for (int j = std::max(0, it - p.ring); j < it; ++j)
                    if (!mbar_wait_sleep(&full[j % p.ring], (j / p.ring) & 1, 512))
                        gemv_record(flag, p.err, ERR_GEMV_DRAIN);  // and wait for the others
        }
        return;
    }

    // ----------------------------------------------------------------------
    // Consumers.  Warp w takes groups w*WPS .. w*WPS + WPS-1 of every stage
    // (a stage is 8*WPS groups), for every 16-row tile of the pass; the
    // WPS x TILES units of a stage are unrolled.
    // ----------------------------------------------------------------------
    // Whole x at 4 bits ("converted"): x is rewritten as fp16 with a
    // power-of-two scale per (group, row), 2^(14 - floor(log2 max|x|)), and
    // the x paired with codes at bit 4 carries a further 2^-4; the codes then
    // stay in place (exact fp16 subnormals) and one MMA chain gives
    // scale_x * 2^-24 * sum(q x); the epilogue multiplies by the group's
    // scale times the inverse power of two.  Otherwise fp16 x is used as it
    // is (codes at bit 4 in a second chain) and bf16 x with 128 + q codes.
    constexpr bool kConv = (B == 4) && !XST;
    constexpr bool kMmaBf16 = BF16 && !kConv;
    constexpr bool kInPlace = (B == 4) && !kMmaBf16;
    constexpr uint32_t kMagicDec = kMmaBf16 ? 0x43004300u : 0u;
    // fp16 MMAs: the products carry 2^-24, which the group sums of x take
    // too; y = 2^24 * acc.
    constexpr float kXsScale = kMmaBf16 ? 1.f : 5.9604644775390625e-08f;
    const int g = lane >> 2, c = lane & 3;
    // MMA row g (and g + 8) reads tile row pg (and pg + 8): rows 0,2,4,6 for
    // the lanes of one half-warp and 1,3,5,7 for the other, so that the
    // 8-byte code loads of the 128-byte swizzle never share a bank.
    const int pg = ((g & 3) << 1) | (g >> 2);
    const int M = p.M;
    const int64_t K = p.K;
    const int xrow = min(g, M - 1);     // columns past M repeat row M-1 (never stored)

    // 3-bit: where this lane's 48-bit span starts (word, byte) in a group.
    uint32_t sel0 = 0, sel2 = 0;
    int wi3 = 0;
    if constexpr (B == 3) {
        const uint32_t bo = 2u * (uint32_t)(c & 1);
        sel0 = bo | ((bo + 1) << 4) | ((bo + 3) << 8) | ((bo + 4) << 12);
        sel2 = (bo + 1) | ((bo + 2) << 4) | ((bo + 4) << 8) | ((bo + 5) << 12);
        wi3 = (3 * c) >> 1;
    }

    // x and y belong to the stream order: wait for the preceding grid.
    grid_dependency_wait();

    const T *xg = static_cast<const T *>(p.x);
    const uint32_t one = kMmaBf16 ? 0x3F803F80u : 0x3C003C00u;
    const uint32_t ones[4] = {one, one, one, one};
    // Whole x: one bulk copy per activation row, then all consumer threads
    // rewrite it in place into B-fragment order (one 32-byte quarter of a
    // group each) and take the group sums, [G][8] floats (and, converted,
    // the inverse scales, [G][8] floats).
    uint8_t *xraw = smem + p.off_x;
    float *xsg = reinterpret_cast<float *>(smem + p.off_xs);
    const int G = (int)(K / 64);
    float *xeg = xsg + G * 8;
    if constexpr (!kXStage) {
        if (threadIdx.x == 0) {
            mbar_arrive_expect_tx(x_full, (uint32_t)(M * K * 2));
            for (int m = 0; m < M; ++m)
                bulk_g2s_plain(xraw + m * p.x_row_pitch, xg + (int64_t)m * K, (uint32_t)(K * 2),
                               x_full);
        }
        gemv_wait(x_full, 0, flag, p.err, ERR_GEMV_FULL);
        if (lane == 0) mbar_arrive(x_landed);
        launch_dependents();
        for (int m = 0; m < M; ++m) {
            for (int u = threadIdx.x; u < G * 4; u += kConsumers * 32) {
                const int gg = u >> 2, cq = u & 3;
                uint4 *q = reinterpret_cast<uint4 *>(xraw + m * p.x_row_pitch + gg * 128 + 32 * cq);
                const uint4 u0 = q[0], u1 = q[1];
                const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
                float f[16];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    if constexpr (BF16) {
                        f[2 * i] = __uint_as_float(w[i] << 16);
                        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
                    } else {
                        const float2 v = __half22float2(*reinterpret_cast<const __half2 *>(&w[i]));
                        f[2 * i] = v.x;
                        f[2 * i + 1] = v.y;
                    }
                }
                float part[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) part[i] = f[2 * i] + f[2 * i + 1];
                float sum = ((part[0] + part[1]) + (part[2] + part[3])) +
                            ((part[4] + part[5]) + (part[6] + part[7]));
                // the four quarters of a group are four adjacent lanes
                sum += __shfl_xor_sync(0xffffffffu, sum, 1);
                sum += __shfl_xor_sync(0xffffffffu, sum, 2);
                if constexpr (kConv) {
                    float mx = 0.f;
#pragma unroll
                    for (int i = 0; i < 16; ++i) mx = fmaxf(mx, fabsf(f[i]));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                    // 2^sh with max|x| * 2^sh in [2^14, 2^15): exact, in range
                    const int ex = mx > 0.f ? (int)((__float_as_uint(mx) >> 23) & 0xFF) - 127 : 0;
                    const int sh = 14 - ex;
                    const float sc = __uint_as_float((uint32_t)(127 + sh) << 23);
                    const float s4 = __uint_as_float((uint32_t)(127 + sh - 4) << 23);
                    q[0] = make_uint4(pack_half2(f[0] * sc, f[4] * sc), pack_half2(f[2] * sc, f[6] * sc),
                                      pack_half2(f[8] * sc, f[12] * sc),
                                      pack_half2(f[10] * sc, f[14] * sc));
                    q[1] = make_uint4(pack_half2(f[1] * s4, f[5] * s4), pack_half2(f[3] * s4, f[7] * s4),
                                      pack_half2(f[9] * s4, f[13] * s4),
                                      pack_half2(f[11] * s4, f[15] * s4));
                    if (cq == 0) xeg[gg * 8 + m] = __uint_as_float((uint32_t)(127 - sh) << 23);
                } else {
                    uint32_t bx[4][2];
                    x_frags<B>(u0, u1, bx);
                    q[0] = make_uint4(bx[0][0], bx[0][1], bx[1][0], bx[1][1]);
                    q[1] = make_uint4(bx[2][0], bx[2][1], bx[3][0], bx[3][1]);
                }
                if (cq == 0) xsg[gg * 8 + m] = sum * kXsScale;
            }
        }
        consumers_sync();
    }

    T *y = static_cast<T *>(p.y);
    int Np = p.N;
    float *gbuf = nullptr;  // gate/up: the gate's rows
    if constexpr (MP) {
        y = static_cast<T *>(mx.y_proj[proj]);
        Np = mx.n_proj[proj];
        gbuf = reinterpret_cast<float *>(smem + mx.off_gu);
    }
    float *red = reinterpret_cast<float *>(smem + p.off_red);
    const int pr = p.pass_rows;

    int slot = 0, lap = 0;  // ring position of the current stage
    for (int pass = 0; pass < p.passes; ++pass) {
        float acc[TILES][MB][4];
#pragma unroll
        for (int t = 0; t < TILES; ++t)
#pragma unroll
            for (int mb = 0; mb < MB; ++mb)
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[t][mb][i] = 0.f;

        for (int s = 0; s < p.n_stages; ++s) {
            const uint8_t *st = smem + (size_t)slot * p.slot_bytes;
            // (no check of the error flag here: the wait is bounded by itself)
            if (!mbar_wait(&full[slot], lap & 1)) gemv_record(flag, p.err, ERR_GEMV_FULL);
            if (kXStage && pass == 0 && s == 0) {  // this call's x has started landing
                if (lane == 0) mbar_arrive(x_landed);
                launch_dependents();
            }
            // The warp's WPS groups of the stage sit in column block
            // (warp*WPS) >> 2 and scale block (warp*WPS) >> 3.
            const int j0 = warp * WPS;
            const uint8_t *cb0 = st + (size_t)((j0 >> 2) * pr) * kBox;
            const int q7 = ((j0 >> 2) * pr + pg) & 7;
            const uint8_t *sc0 = st + p.off_sc + ((j0 >> 3) * pr) * 16 + (j0 & 7) * 2;
            const uint8_t *bi0 = st + p.off_bi + ((j0 >> 3) * pr) * 16 + (j0 & 7) * 2;
            const int gg0 = s * (8 * WPS) + j0;  // global group of unit i = 0
#pragma unroll
            for (int i = 0; i < WPS; ++i) {
                if (WPS > 1 && gg0 + i >= G) continue;  // past the end of K (last stage)
                // B fragments and group sums of columns 2c, 2c+1 of each block
                uint32_t bx[MB][4][2];
                float xs0[MB], xs1[MB];
                float e0 = 1.f, e1 = 1.f;  // converted x: inverse scales of columns 2c, 2c+1
                if constexpr (kXStage) {
                    // raw x of the group: [M rows][128 bytes], 128-byte swizzle; the
                    // columns past M take zeros
#pragma unroll
                    for (int mb = 0; mb < MB; ++mb) {
                        const int row = 8 * mb + g;
                        const int seg = (j0 + i) * p.x_rows + row;
                        const uint8_t *xr = st + p.off_xst + seg * 128;
                        uint4 u0 = make_uint4(0u, 0u, 0u, 0u), u1 = u0;
                        if (row < p.x_rows) {
                            u0 = *reinterpret_cast<const uint4 *>(xr + (((2 * c) ^ (seg & 7)) << 4));
                            u1 = *reinterpret_cast<const uint4 *>(xr +
                                                                  (((2 * c + 1) ^ (seg & 7)) << 4));
                        }
                        x_frags<B>(u0, u1, bx[mb]);
                        float xsum[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            mma16816<kMmaBf16>(xsum, ones, bx[mb][q][0], bx[mb][q][1]);
                        xs0[mb] = xsum[0] * kXsScale;
                        xs1[mb] = xsum[1] * kXsScale;
                    }
                } else {
                    const int gg = gg0 + i;
                    const uint8_t *fr = xraw + xrow * p.x_row_pitch + gg * 128 + 32 * c;
                    const uint4 u0 = *reinterpret_cast<const uint4 *>(fr);
                    const uint4 u1 = *reinterpret_cast<const uint4 *>(fr + 16);
                    bx[0][0][0] = u0.x; bx[0][0][1] = u0.y; bx[0][1][0] = u0.z; bx[0][1][1] = u0.w;
                    bx[0][2][0] = u1.x; bx[0][2][1] = u1.y; bx[0][3][0] = u1.z; bx[0][3][1] = u1.w;
                    const float2 xs = *reinterpret_cast<const float2 *>(xsg + gg * 8 + 2 * c);
                    xs0[0] = xs.x;
                    xs1[0] = xs.y;
                    if constexpr (kConv) {
                        const float2 e = *reinterpret_cast<const float2 *>(xeg + gg * 8 + 2 * c);
                        e0 = e.x;
                        e1 = e.y;
                    }
                }
                const int gi = (j0 + i) & 3;  // group within its column block
                // 128-byte swizzle: 16-byte chunk ch of a row segment q sits at
                // ch ^ (q & 7); rows pg and pg + 8 of every tile share q & 7.
                const int off4 = (((2 * gi + (c >> 1)) ^ q7) << 4) + 8 * (c & 1);
#pragma unroll
                for (int t = 0; t < TILES; ++t) {
                    const int ra = 16 * t + pg, rb = ra + 8;
                    uint32_t PA[8], PB[8];
                    if constexpr (B == 4) {
                        const uint2 qa = *reinterpret_cast<const uint2 *>(cb0 + ra * 128 + off4);
                        const uint2 qb = *reinterpret_cast<const uint2 *>(cb0 + rb * 128 + off4);
                        decode4<kInPlace, kMagicDec>(qa.x, qa.y, PA);
                        decode4<kInPlace, kMagicDec>(qb.x, qb.y, PB);
                    } else {
                        const uint32_t *pa =
                            reinterpret_cast<const uint32_t *>(cb0 + ra * 96 + 24 * gi) + wi3;
                        const uint32_t *pb =
                            reinterpret_cast<const uint32_t *>(cb0 + rb * 96 + 24 * gi) + wi3;
                        decode3<kMagicDec>(pa[0], pa[1], sel0, sel2, PA);
                        decode3<kMagicDec>(pb[0], pb[1], sel0, sel2, PB);
                    }
                    const float sa = __half2float(*reinterpret_cast<const __half *>(sc0 + ra * 16 + 2 * i));
                    const float sb = __half2float(*reinterpret_cast<const __half *>(sc0 + rb * 16 + 2 * i));
                    float ba = __half2float(*reinterpret_cast<const __half *>(bi0 + ra * 16 + 2 * i));
                    float bb = __half2float(*reinterpret_cast<const __half *>(bi0 + rb * 16 + 2 * i));
                    if constexpr (kConv) {
                        // one chain: the x of codes at bit 4 already carries 2^-4
                        float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            uint32_t af[4];
                            step_frags<B>(PA, PB, q, af);
                            mma16816<false>(d, af, bx[0][q][0], bx[0][q][1]);
                        }
                        float *a4 = acc[t][0];
                        a4[0] = fmaf(sa * e0, d[0], fmaf(ba, xs0[0], a4[0]));
                        a4[1] = fmaf(sa * e1, d[1], fmaf(ba, xs1[0], a4[1]));
                        a4[2] = fmaf(sb * e0, d[2], fmaf(bb, xs0[0], a4[2]));
                        a4[3] = fmaf(sb * e1, d[3], fmaf(bb, xs1[0], a4[3]));
                    } else {
                        if constexpr (kMmaBf16) {
                            ba = fmaf(-128.f, sa, ba);
                            bb = fmaf(-128.f, sb, bb);
                        }
                        // steps 2-3 hold the codes at bit 4 (16 q * 2^-24) in the in-place decode
                        const float sa4 = kInPlace ? sa * 0.0625f : sa;
                        const float sb4 = kInPlace ? sb * 0.0625f : sb;
#pragma unroll
                        for (int mb = 0; mb < MB; ++mb) {
                            // two independent MMA chains (steps 0-1 and 2-3)
                            float da[4] = {0.f, 0.f, 0.f, 0.f}, db[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                uint32_t af[4];
                                step_frags<B>(PA, PB, q, af);
                                if (q < 2)
                                    mma16816<kMmaBf16>(da, af, bx[mb][q][0], bx[mb][q][1]);
                                else
                                    mma16816<kMmaBf16>(db, af, bx[mb][q][0], bx[mb][q][1]);
                            }
                            float *a4 = acc[t][mb];
                            a4[0] = fmaf(sa, da[0], fmaf(sa4, db[0], fmaf(ba, xs0[mb], a4[0])));
                            a4[1] = fmaf(sa, da[1], fmaf(sa4, db[1], fmaf(ba, xs1[mb], a4[1])));
                            a4[2] = fmaf(sb, da[2], fmaf(sb4, db[2], fmaf(bb, xs0[mb], a4[2])));
                            a4[3] = fmaf(sb, da[3], fmaf(sb4, db[3], fmaf(bb, xs1[mb], a4[3])));
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
            if (++slot == p.ring) {
                slot = 0;
                ++lap;
            }
        }

        // ------------------------------------------------------------------
        // The eight warps' partial tiles, added in warp order.  With a single
        // pass the buffer is the ring itself, free once every warp is done.
        // ------------------------------------------------------------------
        if (p.red_alias) consumers_sync();
#pragma unroll
        for (int t = 0; t < TILES; ++t)
#pragma unroll
            for (int mb = 0; mb < MB; ++mb)
                *reinterpret_cast<float4 *>(&red[(((warp * TILES + t) * MB + mb) * 32 + lane) * 4]) =
                    make_float4(acc[t][mb][0], acc[t][mb][1], acc[t][mb][2], acc[t][mb][3]);
        consumers_sync();
        int r0 = row_cta + pass * pr;
        if constexpr (MP)
            if (mx.gate_up) r0 = row_cta;
        const int rows = std::min(pr, Np - r0);
        for (int e = threadIdx.x; e < rows * M; e += kConsumers * 32) {
            const int m = e / rows, r = e - m * rows;
            const int t = r >> 4, rr = r & 15;
            const int ph = rr & 7;                       // tile row within the half
            const int gl = (ph >> 1) | ((ph & 1) << 2);  // the MMA row that read it
            const int mb = m >> 3, mm = m & 7;           // column block, column in it
            const int ln = 4 * gl + (mm >> 1), i = 2 * (rr >> 3) + (mm & 1);
            float v = 0.f;
            for (int w = 0; w < kConsumers; ++w)
                v += red[(((w * TILES + t) * MB + mb) * 32 + ln) * 4 + i];
            if constexpr (!kMmaBf16) v *= 16777216.f;  // 2^24
            if constexpr (MP)
                if (mx.gate_up) {
                    if (pass == 0) {  // the gate waits for the up projection
                        gbuf[m * pr + r] = v;
                        continue;
                    }
                    const float gt = gbuf[m * pr + r];
                    v = gt / (1.f + expf(-gt)) * v;  // silu(gate) * up
                }
            store_y<T>(&y[(int64_t)m * Np + r0 + r], v);
        }
        consumers_sync();  // the buffer is rewritten by the next pass
    }
}

// ---------------------------------------------------------------------------
// Plan and launch (host)
// ---------------------------------------------------------------------------
struct GemvPlan {
    GemvParams prm;
    GemvMulti mx;
    bool mp;   // several projections or gate/up: the MP = true kernels
    size_t smem;
    int grid;
    int mb;    // 8-column blocks of activation rows
    int wps;   // groups per warp per stage
    int bits;
    bool bf16;
};

constexpr size_t kSmemMax = 227 * 1024;  // one CTA per SM at most

template <int B, bool BF16, int TILES, int WPS, int MB, bool XST, bool MP>
cudaError_t launch_t(const GemvPlan &pl, const GemvMaps &maps, cudaStream_t stream) {
    auto kern = gemv_kernel<B, BF16, TILES, WPS, MB, XST, MP>;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)kSmemMax);
    });
    if (attr_err != cudaSuccess) return attr_err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)pl.grid, 1, 1);
    cfg.blockDim = dim3(kGemvThreads, 1, 1);
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, pl.prm, maps.w[0], maps.s[0], maps.b[0], maps.x,
                              maps.w[1], maps.s[1], maps.b[1], maps.w[2], maps.s[2], maps.b[2],
                              maps.w[3], maps.s[3], maps.b[3], pl.mx);
}

// Dispatch from the plan to an instantiation.  One 8-column block with x
// whole (XST = false) or staged, two blocks (M = 9..16), four (M = 17..32);
// groups per warp by tiles as max_wps allows.
template <int B, bool BF16, int TILES, bool XST, bool MP>
cudaError_t mb1_wps(const GemvPlan &pl, const GemvMaps &m, cudaStream_t s) {
    if constexpr (TILES <= 2)
        if (pl.wps == 4) return launch_t<B, BF16, TILES, 4, 1, XST, MP>(pl, m, s);
    if constexpr (TILES <= 4)
        if (pl.wps == 2) return launch_t<B, BF16, TILES, 2, 1, XST, MP>(pl, m, s);
    return launch_t<B, BF16, TILES, 1, 1, XST, MP>(pl, m, s);
}

template <int B, bool BF16, bool XST, bool MP>
cudaError_t mb1_tiles(const GemvPlan &pl, const GemvMaps &m, cudaStream_t s) {
    switch (pl.prm.tiles) {
        case 1: return mb1_wps<B, BF16, 1, XST, MP>(pl, m, s);
        case 2: return mb1_wps<B, BF16, 2, XST, MP>(pl, m, s);
        case 3: return mb1_wps<B, BF16, 3, XST, MP>(pl, m, s);
        case 4: return mb1_wps<B, BF16, 4, XST, MP>(pl, m, s);
        case 5: return mb1_wps<B, BF16, 5, XST, MP>(pl, m, s);
        case 6: return mb1_wps<B, BF16, 6, XST, MP>(pl, m, s);
        case 7: return mb1_wps<B, BF16, 7, XST, MP>(pl, m, s);
        default: return mb1_wps<B, BF16, 8, XST, MP>(pl, m, s);
    }
}

template <int B, bool BF16, int TILES, bool MP>
cudaError_t mb2_wps(const GemvPlan &pl, const GemvMaps &m, cudaStream_t s) {
    if constexpr (TILES <= 2)
        if (pl.wps == 2) return launch_t<B, BF16, TILES, 2, 2, true, MP>(pl, m, s);
    return launch_t<B, BF16, TILES, 1, 2, true, MP>(pl, m, s);
}

template <int B, bool BF16, bool MP>
cudaError_t mb2_tiles(const GemvPlan &pl, const GemvMaps &m, cudaStream_t s) {
    switch (pl.prm.tiles) {
        case 1: return mb2_wps<B, BF16, 1, MP>(pl, m, s);
        case 2: return mb2_wps<B, BF16, 2, MP>(pl, m, s);
        case 3: return mb2_wps<B, BF16, 3, MP>(pl, m, s);
        case 4: return mb2_wps<B, BF16, 4, MP>(pl, m, s);
        case 5: return mb2_wps<B, BF16, 5, MP>(pl, m, s);
        default: return mb2_wps<B, BF16, 6, MP>(pl, m, s);
    }
}

template <int B, bool BF16, bool MP>
cudaError_t mb4_tiles(const GemvPlan &pl, const GemvMaps &m, cudaStream_t s) {
    switch (pl.prm.tiles) {
        case 1: return launch_t<B, BF16, 1, 1, 4, true, MP>(pl, m, s);
        case 2: return launch_t<B, BF16, 2, 1, 4, true, MP>(pl, m, s);
        case 3: return launch_t<B, BF16, 3, 1, 4, true, MP>(pl, m, s);
        case 4: return launch_t<B, BF16, 4, 1, 4, true, MP>(pl, m, s);
        case 5: return launch_t<B, BF16, 5, 1, 4, true, MP>(pl, m, s);
        default: return launch_t<B, BF16, 6, 1, 4, true, MP>(pl, m, s);
    }
}

// One plan's launch for each (bits, dtype).  Column blocks: 1 (XST says
// whether x is staged), 2 or 4.
template <int MBLK, bool XST, bool MP>
cudaError_t launch_blocks(const GemvPlan &pl, const GemvMaps &m, cudaStream_t s) {
    if constexpr (MBLK == 1) {
        if (pl.bits == 3)
            return pl.bf16 ? mb1_tiles<3, true, XST, MP>(pl, m, s)
                           : mb1_tiles<3, false, XST, MP>(pl, m, s);
        return pl.bf16 ? mb1_tiles<4, true, XST, MP>(pl, m, s)
                       : mb1_tiles<4, false, XST, MP>(pl, m, s);
    } else if constexpr (MBLK == 2) {
        if (pl.prm.tiles > 6) return cudaErrorInvalidValue;
        if (pl.bits == 3)
            return pl.bf16 ? mb2_tiles<3, true, MP>(pl, m, s) : mb2_tiles<3, false, MP>(pl, m, s);
        return pl.bf16 ? mb2_tiles<4, true, MP>(pl, m, s) : mb2_tiles<4, false, MP>(pl, m, s);
    } else {
        if (pl.prm.tiles > 6) return cudaErrorInvalidValue;
        if (pl.bits == 3)
            return pl.bf16 ? mb4_tiles<3, true, MP>(pl, m, s) : mb4_tiles<3, false, MP>(pl, m, s);
        return pl.bf16 ? mb4_tiles<4, true, MP>(pl, m, s) : mb4_tiles<4, false, MP>(pl, m, s);
    }
}

// Each instantiation of launch_blocks lives in one translation unit (the
// library builds in parallel): aq_gemv.cu (1 block, x whole), aq_gemv_xs.cu
// (1 block, x staged), aq_gemv16.cu (2), aq_gemv32.cu (4); the
// several-projection kernels in aq_gemv_mpw.cu (1 block, x whole),
// aq_gemv_mps.cu (1 block, x staged) and aq_gemv_mp24.cu (2 and 4 blocks).
extern template cudaError_t launch_blocks<1, false, false>(const GemvPlan &, const GemvMaps &, cudaStream_t);
extern template cudaError_t launch_blocks<1, true, false>(const GemvPlan &, const GemvMaps &, cudaStream_t);
extern template cudaError_t launch_blocks<2, true, false>(const GemvPlan &, const GemvMaps &, cudaStream_t);
extern template cudaError_t launch_blocks<4, true, false>(const GemvPlan &, const GemvMaps &, cudaStream_t);
extern template cudaError_t launch_blocks<1, false, true>(const GemvPlan &, const GemvMaps &, cudaStream_t);
extern template cudaError_t launch_blocks<1, true, true>(const GemvPlan &, const GemvMaps &, cudaStream_t);
extern template cudaError_t launch_blocks<2, true, true>(const GemvPlan &, const GemvMaps &, cudaStream_t);
extern template cudaError_t launch_blocks<4, true, true>(const GemvPlan &, const GemvMaps &, cudaStream_t);

}  // namespace gemv
}  // namespace aq
