// Large-M kernel ("tc"): y = x . W^T on the 5th-generation tensor cores
// (tcgen05, accumulators in tensor memory), for M large enough that the
// product is a dense contraction.
//
// Method (mlx-bun pages, @mlx-bun/inference 1.0.0, kernels/quantization/):
// affine-split-mma.ts computes any number of activation rows with the
// weights as the A operand (8 weight rows per simdgroup tile) and x^T as B,
// dequantising each weight as fma(q, scale, bias) right before the matrix
// product; the trellis prefill kernels on the same site reconstruct a weight
// tile into threadgroup memory and then run matrix products on it.  Here:
//
//   * A = 128 weight rows x 64 k (one group) per stage, dequantised by eight
//     warps into shared memory as bf16 (x bf16) or fp16 (x fp16) in the
//     128-byte-swizzled K-major layout the tensor core reads directly;
//   * B = x^T, loaded by TMA (tensor map, 128-byte swizzle) in sub-tiles of
//     min(BM, 256) activation rows x 64 k - x is never converted;
//   * one thread issues tcgen05.mma (M=128, N=min(BM,256), K=16) x4 per
//     sub-tile into fp32 accumulators in tensor memory.  A and B have rings
//     of their own: each B sub-tile is released as soon as its four MMAs
//     complete (a 512-row x tile is two sub-tiles sharing one A tile) and
//     each A tile after its last; two accumulators alternate (x tiles up to
//     256 rows) so the epilogue of one tile overlaps the main loop of the
//     next;
//   * four epilogue warps read the accumulator with tcgen05.ld, round to the
//     output type and store y; persistent CTAs (one per SM) walk the tiles.
//
// Roles (448 threads): warp 0 TMA producer, warp 1 MMA issuer and tensor
// memory owner, warps 2-5 epilogue, warps 6-13 dequantisation (each streams
// its 16 weight rows through a cp.async ring of 256-k super-stages).  Every
// mbarrier wait is bounded; a wait that gives up records an error and the
// CTA winds down after the copies and MMAs it issued have completed.
#include "aq_internal.h"
#include "aq_ptx.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdio>
#include <mutex>

namespace aq {

__device__ uint32_t g_tc_error;

namespace {

constexpr int kThreadsTc = 14 * 32;
constexpr int kWarpTma = 0, kWarpMma = 1, kWarpDq = 6, kDqWarps = 8;  // warps 2-5: epilogue
constexpr int kGroups = 4;    // groups per raw super-stage (256 k)
constexpr int kATileBytes = 128 * 128;

// Ring depths by x tile width.  The x tiles come from L2 by TMA in
// sub-tiles of min(BM, 256) rows x 64 k (8 to 32 KB), each in a slot of its
// own and released as soon as its four MMAs complete, so that about a
// microsecond of load latency stays covered at the MMA rate.  A tiles (128
// weight rows x 64 k, 16 KB) have a ring of their own: a tile's slot comes
// back one MMA completion plus one dequantisation after its last use, which
// three or more slots keep off the critical path.
constexpr int b_slots_for(int BM, bool gen = false) {
    // 256-row tiles: three 32 KB x slots, beside four A slots (3/4 bits) or
    // the larger raw rings of the general-width path
    return BM > 256 ? 4 : BM == 256 ? (gen ? 3 : 4) : BM == 128 ? 4 : 8;
}
constexpr int a_slots_for(int BM, bool gen = false) {
    return BM > 256 ? 3 : BM == 256 ? (gen ? 3 : 4) : 4;
}
constexpr int ni_for(int BM) { return BM > 256 ? 256 : BM; }
// Raw super-stages per dequant warp; all but one are in flight while the
// warp dequantises, so that the weight stream keeps enough bytes in flight
// to cover the HBM latency.
constexpr int raw_slots_for(int BM) { return BM <= 128 ? 3 : 2; }

// Raw super-stage of one dequantising warp: 16 rows x 4 groups of codes,
// then their scales and biases.  The row pitch puts the rows in distinct
// banks for the dequantising loads: 4-bit rows (16-byte loads, a quarter
// warp at a time) 40 words apart; 3-bit rows (4-byte loads, two lanes a
// row 3 words apart) 26 words apart, which is not a multiple of 16 bytes,
// so 3-bit rows are copied in 8-byte pieces (at a 32-word pitch all 16 rows
// of a load fell in the same banks).
template <int B>
struct Raw {
    static constexpr int kGroupBytes = 8 * B;
    static constexpr int kRowBytes = kGroups * kGroupBytes;  // 128 / 96
    static constexpr int kChunkBytes = B == 3 ? 8 : 16;      // cp.async piece
    static constexpr int kChunksPerRow = kRowBytes / kChunkBytes;  // 8 / 12
    static constexpr int kRowPitch = B == 3 ? 104 : kRowBytes + 32;  // 160 / 104
    static constexpr int kSbOff = 16 * kRowPitch;  // scales[16][4] then biases[16][4]
    static constexpr int kSlotBytes = kSbOff + 2 * 16 * 8;
    static_assert(kRowPitch % kChunkBytes == 0 && kSbOff % 16 == 0, "raw slot alignment");
};

// Raw super-stage of the general-width path (any code width B, groups of
// 32, 64 or 128): 16 rows x 256 k of codes (32B bytes a row), then up to 8
// scales and 8 biases a row.  Row pitches chosen so that the dequantising
// loads of 16 rows (two lanes a row) fall in distinct banks, or in two.
template <int B>
struct RawG {
    static constexpr int kGroupBytes = 8 * B;                // 64 k of one row
    static constexpr int kRowBytes = kGroups * kGroupBytes;  // 256 k
    static constexpr int kChunkBytes = 16;
    static constexpr int kChunksPerRow = kRowBytes / 16;
    static constexpr int kRowPitch = kRowBytes + (B == 4 ? 32 : 16);
    static constexpr int kSbOff = 16 * kRowPitch;  // scales[16][8] then biases[16][8]
    static constexpr int kSlotBytes = kSbOff + 2 * 16 * 16;
    static_assert(kRowPitch % 16 == 0 && kSbOff % 16 == 0, "raw slot alignment");
};
// Raw slots per dequantising warp on the general-width path (as many as
// shared memory holds next to 64 KB of A tiles and 80 KB of x tiles).
constexpr int raw_slots_g(int B) { return B >= 6 ? 2 : 3; }

// The 32 codes of one lane (B words, code i at bits [iB, iB+B) of the
// little-endian stream) and the float 2048 + q of code i: the code moved to
// mantissa bit 12 under the exponent of 2^11 (exact for q < 2^11).
template <int B>
__device__ __forceinline__ void load_codes(const uint8_t *p, uint32_t (&w)[B]) {
    if constexpr (B == 2) {
        const uint2 v = *reinterpret_cast<const uint2 *>(p);
        w[0] = v.x, w[1] = v.y;
    } else if constexpr (B == 4 || B == 8) {
#pragma unroll
        for (int i = 0; i < B / 4; ++i) {
            const uint4 v = *reinterpret_cast<const uint4 *>(p + 16 * i);
            w[4 * i] = v.x, w[4 * i + 1] = v.y, w[4 * i + 2] = v.z, w[4 * i + 3] = v.w;
        }
    } else if constexpr (B == 6) {
#pragma unroll
        for (int i = 0; i < 3; ++i) {
            const uint2 v = *reinterpret_cast<const uint2 *>(p + 8 * i);
            w[2 * i] = v.x, w[2 * i + 1] = v.y;
        }
    } else {
#pragma unroll
        for (int i = 0; i < B; ++i) w[i] = reinterpret_cast<const uint32_t *>(p)[i];
    }
}
template <int B>
__device__ __forceinline__ float code_f(const uint32_t (&w)[B], int i) {
    const int bit = i * B, wd = bit >> 5, off = bit & 31;
    uint32_t t;
    if (off + B <= 32)
        t = off >= 12 ? (w[wd] >> (off - 12)) : (w[wd] << (12 - off));
    else
        t = __funnelshift_r(w[wd], w[wd + 1], off) << 12;
    return __uint_as_float((t & (((1u << B) - 1u) << 12)) | 0x45000000u);
}

// x tiles of up to 128 rows (3/4-bit path) take the A tiles from tensor
// memory: the dequantising warps write them with tcgen05.st and the MMAs read
// them there, so that the dequantisation needs no shared-memory stores of A
// and no proxy fence.  Eight A stages of 32 columns sit beside the two
// accumulators.
constexpr bool ta_for(int BM, bool gen) { return BM <= 256 && !gen; }
constexpr int kATmemSlots = 8;
// raw super-stages per dequantising warp with A in tensor memory (256-row x
// tiles: two, beside four 32 KB x slots)
constexpr int raw_slots_ta(int BM) { return BM == 256 ? 2 : 3; }

// Raw super-stage of one dequantising warp when A is in tensor memory: the
// 32 rows of its lane quarter, 4 groups.
template <int B>
struct RawT {
    static constexpr int kGroupBytes = 8 * B;
    static constexpr int kRowBytes = kGroups * kGroupBytes;  // 128 / 96
    static constexpr int kChunksPerRow = kRowBytes / 16;    // 8 / 6
    static constexpr int kRowPitch = kRowBytes + 16;         // 144 / 112: rows in distinct banks
    static constexpr int kSbOff = 32 * kRowPitch;            // scales[32][4], then biases[32][4]
    static constexpr int kSlotBytes = kSbOff + 2 * 32 * 8;
};

struct TcParams {
    const uint32_t *Wq;
    const __half *scales;
    const __half *biases;
    void *y;
    int M, N, K, G;
    int n_tiles, m_tiles;
    // Work units: `rounds` rounds of whole tiles (tile = CTA + round * grid),
    // then `tail` tiles split in two K halves between the two CTAs of a
    // cluster (cluster c takes tile rounds * grid + c), added at the end
    // through distributed shared memory.
    int rounds, tail;
    // Few tiles (fewer than SMs, x tiles of at most 128 rows): instead, a
    // cluster of cl_ctas CTAs shares cl_tiles < cl_ctas consecutive tiles
    // (cluster c from tile c * cl_tiles); the cluster's K stages, tile after
    // tile, are dealt out in even runs of whole super-stages, so a CTA holds
    // partial accumulators of one or two tiles, added at the end in rank
    // (that is K) order through distributed shared memory.  0 when unused.
    int cl_ctas, cl_tiles;
    uint32_t off_b, off_raw, off_bar, tmem_cols;
    int lg, NG;  // general-width path: log2 of the group size, groups per row
#ifdef AQ_TEST_HOOKS
    int withhold;  // test builds only: the x producer skips its first stage
#endif
};

__device__ __forceinline__ void tc_record(volatile int *flag, uint32_t code) {
    *flag = 1;
    atomicOr(&g_tc_error, code);
}

// Bounded mbarrier wait; gives up at once if another role already gave up.
__device__ __forceinline__ bool tc_wait(uint64_t *bar, uint32_t parity, volatile int *flag,
                                        uint32_t code) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*flag) return false;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1; it < (1u << 31); ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 0u) {
            if (*flag) return false;
            if (globaltimer_ns() - t0 > AQ_WAIT_LIMIT_NS) break;
        }
    }
    tc_record(flag, code);
    return false;
}

// Bounded wait used while winding down: no error is recorded (it only makes
// sure that copies or MMAs already issued have finished before the CTA
// releases its shared and tensor memory).
__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1; it < (1u << 31); ++it) {
        if (mbar_try_wait(bar, parity)) return;
        if ((it & 255u) == 0u && globaltimer_ns() - t0 > AQ_WAIT_LIMIT_NS) return;
    }
}

__device__ __forceinline__ float h_at(const uint4 &v, int j) {
    const uint32_t w = j < 2 ? v.x : j < 4 ? v.y : j < 6 ? v.z : v.w;
    return __half2float(__ushort_as_half((unsigned short)((j & 1) ? (w >> 16) : (w & 0xFFFFu))));
}

__device__ __forceinline__ uint32_t bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

// ---------------------------------------------------------------------------
// Dequantisation of the tensor-core kernels.  A code q at bit p of a 32-bit word,
// with 12 <= p and p + bits <= 23, becomes the exact float 2^(23-p) + q once
// the word is masked to the code and OR-ed with the exponent of 2^(23-p)
// (the pages' mantissa trick, here with the code at one of a few mantissa
// positions so that one shift serves two codes).  Then w = (2^E + q) s +
// (b - 2^E s) in one fp32 fma per value, two values per packed fma; the bias
// term b - 2^E s is rounded to fp32 once per group (error <= 2^-24 * 2^E s,
// at most 2^-13 s here), and w is rounded once to the operand type.
// ---------------------------------------------------------------------------
constexpr uint32_t kExp11 = 0x45000000u;  // 2048.0f: code at bit 12
constexpr uint32_t kExp8 = 0x43800000u;   // 256.0f: code at bit 15
constexpr uint32_t kExp7 = 0x43000000u;   // 128.0f: code at bit 16
constexpr uint32_t kExp5 = 0x42000000u;   // 32.0f: code at bit 18

__device__ __forceinline__ float code_at(uint32_t t, uint32_t mask, uint32_t expo) {
    return __uint_as_float((t & mask) | expo);
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack_out(float2 w) {
    if constexpr (BF16) {
        return bf16x2(w.x, w.y);
    } else {
        return pack_half2(w.x, w.y);
    }
}

// Per-group constants of one weight row: the scale and the bias terms of the
// code positions used (4-bit: codes at bits 16 and 12 alternate, so every
// pair takes (b - 128 s, b - 2048 s); 3-bit: pairs take (b - 2048 s,
// b - 256 s) or (b - 32 s, b - 2048 s)).
struct GroupConst {
    float2 s2, p1, p2;
};

template <int B>
__device__ __forceinline__ GroupConst group_const(float s, float b) {
    GroupConst c;
    c.s2 = make_float2(s, s);
    const float b11 = fmaf(-2048.f, s, b);
    if constexpr (B == 4) {
        c.p1 = make_float2(fmaf(-128.f, s, b), b11);
        c.p2 = c.p1;
    } else {
        c.p1 = make_float2(b11, fmaf(-256.f, s, b));
        c.p2 = make_float2(fmaf(-32.f, s, b), b11);
    }
    return c;
}

// Eight codes (code i at bits B*i of u; 3-bit: bits 24-31 ignored) -> four
// packed output pairs (k, k+1).
template <int B, bool BF16>
__device__ __forceinline__ uint4 dq8(uint32_t u, const GroupConst &c) {
    float2 f01, f23, f45, f67;
    if constexpr (B == 4) {
        const uint32_t t1 = u << 8, t2 = u >> 8, t3 = prmt(u, u, 0x1032u);  // t3: u rotated by 16
        f01 = make_float2(code_at(t3, 0x000F0000u, kExp7), code_at(t1, 0x0000F000u, kExp11));
        f23 = make_float2(code_at(t1, 0x000F0000u, kExp7), code_at(u, 0x0000F000u, kExp11));
        f45 = make_float2(code_at(u, 0x000F0000u, kExp7), code_at(t2, 0x0000F000u, kExp11));
        f67 = make_float2(code_at(t2, 0x000F0000u, kExp7), code_at(t3, 0x0000F000u, kExp11));
    } else {
        const uint32_t ta = u << 12, tb = u << 3, td = u >> 9;
        f01 = make_float2(code_at(ta, 0x00007000u, kExp11), code_at(ta, 0x00038000u, kExp8));
        f23 = make_float2(code_at(ta, 0x001C0000u, kExp5), code_at(tb, 0x00007000u, kExp11));
        f45 = make_float2(code_at(u, 0x00007000u, kExp11), code_at(u, 0x00038000u, kExp8));
        f67 = make_float2(code_at(u, 0x001C0000u, kExp5), code_at(td, 0x00007000u, kExp11));
    }
    return make_uint4(pack_out<BF16>(__ffma2_rn(f01, c.s2, c.p1)),
                      pack_out<BF16>(__ffma2_rn(f23, c.s2, c.p2)),
                      pack_out<BF16>(__ffma2_rn(f45, c.s2, c.p1)),
                      pack_out<BF16>(__ffma2_rn(f67, c.s2, c.p2)));
}

template <typename T>
__device__ __forceinline__ T cvt_out(float v);
template <>
__device__ __forceinline__ __half cvt_out<__half>(float v) { return __float2half_rn(v); }
template <>
__device__ __forceinline__ __nv_bfloat16 cvt_out<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}

// Clustered K split: the run [s, e) of the cluster's stages (in groups, from
// the cluster's first tile t0) that CTA `cta` takes.  Runs are whole
// 4-group super-stages, as even as that allows.
// (32-bit arithmetic: with K below 2^30 and clusters of at most 8, (r + 1) *
// w4 stays below 2^28.)
__device__ __forceinline__ void cl_range(const TcParams &p, int G, int total, int cta, int &s,
                                         int &e, int &t0) {
    const int C = p.cl_ctas, r = cta % C;
    t0 = (cta / C) * p.cl_tiles;
    const int w4 = min(p.cl_tiles, total - t0) * (G / 4);
    s = 4 * (r * w4 / C);
    e = 4 * ((r + 1) * w4 / C);
}

}  // namespace

template <int B, bool BF16, int BM, bool GEN>
__global__ void __launch_bounds__(kThreadsTc, 1)
    tc_kernel(const __grid_constant__ TcParams p, const __grid_constant__ CUtensorMap tmap_x) {
    using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
    // GEN: any code width and group size (32/64/128, p.lg), codes decoded at
    // compile-time bit offsets; otherwise 3/4 bits at groups of 64.
    using R = typename std::conditional<GEN, RawG<B>, Raw<B>>::type;
    constexpr bool TA = ta_for(BM, GEN);
    constexpr int kA = TA ? kATmemSlots : a_slots_for(BM, GEN);
    constexpr int kB = b_slots_for(BM, GEN);
    constexpr int kRawSlots = TA ? raw_slots_ta(BM) : GEN ? raw_slots_g(B) : raw_slots_for(BM);
    constexpr int kRawSlotBytes = [] {
        if constexpr (TA) return RawT<B>::kSlotBytes;
        else return R::kSlotBytes;
    }();
    // A 512-row x tile is two N = 256 MMAs per k-step into one 512-column
    // accumulator (each weight tile dequantised once for 512 x rows); the
    // narrower tiles double-buffer their accumulator.
    constexpr int kNI = ni_for(BM);  // N of one MMA = rows of one B sub-tile
    constexpr int kH = BM / kNI;     // B sub-tiles per stage
    constexpr int kBTile = kNI * 128;
    // accumulators in tensor memory: one of 512 columns, two of up to 256, or
    // one of 256 beside 256-row tensor-memory A stages
    constexpr int kAcc = (BM > 256 || (BM == 256 && TA)) ? 1 : 2;
    // x tiles of up to 128 rows take two stages per MMA step: one x barrier for both
    // stages' sub-tiles, one wait for both A tiles, 8 MMAs, then one commit
    // for each ring.  The issuing thread pays about 80 cycles for every
    // barrier wait and 100 for every commit, which an N = 128 MMA (64
    // cycles at the full rate) does not hide; measured on GB300, a round of
    // 8 MMAs with two waits and two commits takes 889 cycles against 706
    // for 4 MMAs with the same.
    // 64-row x tiles with A in tensor memory take four stages per step (one
    // dequantising warp's super-stage): 16 MMAs between two waits and two
    // commits, which the probe above puts at ~64 cycles an MMA (GB300, M =
    // 64: 10240x5120 3-bit 25.0 -> 24.2 us, 5120x13824 30.6 -> 29.0).  At
    // 128 rows the eight 16 KB x slots this needs leave two raw slots a warp,
    // which cost the 4-bit weight stream more than the steps gain.
    constexpr int kSP = (BM == 64 && TA) ? 4 : (BM <= 128 || TA) ? 2 : 1;
    constexpr int kBG = kB / kSP;  // x barriers (groups of kSP slots)
    static_assert(kSP == 1 || (kH == 1 && kB % kSP == 0 && kA % kSP == 0 && kBG >= 2),
                  "stage groups");
    extern __shared__ uint8_t smem_dyn[];
    // Align to 1024 bytes by an offset from the __shared__ array itself, so
    // that every access below stays a shared-memory access (32-bit address).
    uint8_t *smem = smem_dyn + ((1024u - (smem_u32(smem_dyn) & 1023u)) & 1023u);
    uint8_t *a_ring = smem;
    uint8_t *b_ring = smem + p.off_b;
    uint8_t *raw = smem + p.off_raw;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + p.off_bar);
    uint64_t *a_full = bars;
    uint64_t *a_empty = a_full + kA;
    uint64_t *b_full = a_empty + kA;
    uint64_t *b_empty = b_full + kB;
    uint64_t *acc_full = b_empty + kB;
    uint64_t *acc_empty = acc_full + 2;
    uint64_t *drain = acc_empty + 2;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *flag = reinterpret_cast<volatile int *>(tmem_holder + 1);
    // Clustered K split: the CTA's two sum segments, worked out by an
    // epilogue warp while the main loop runs (16 ints each: tile, chunk
    // range, contributor ranks, this CTA's unit of the tile, and each
    // contributor's partial as a cluster address).
    int *cl_tab = reinterpret_cast<int *>(reinterpret_cast<uint8_t *>(bars) +
                                          (2 * kA + 2 * kB + 5) * 8 + 16);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int total = p.n_tiles * p.m_tiles;
    const int G = p.G;
    // Unit u of this CTA: its tile and K range [gb, ge) in groups.
    // Clustered K split: this CTA's run [cl_s, cl_e) of its cluster's
    // stages (in groups from the cluster's first tile cl_t0), which starts
    // in the cluster's tile cl_ts.
    int cl_s = 0, cl_e = 0, cl_t0 = 0, cl_ts = 0;
    if (p.cl_ctas > 0) {
        cl_range(p, G, total, (int)blockIdx.x, cl_s, cl_e, cl_t0);
        cl_ts = cl_s / G;
    }
    auto unit_of = [&](int u, int &tile, int &gb, int &ge) -> bool {
        if (p.cl_ctas > 0) {
            const int tt = cl_ts + u;  // the cluster's tile of unit u
            if (cl_s >= cl_e || tt * G >= cl_e) return false;
            tile = cl_t0 + tt;
            gb = u == 0 ? cl_s - tt * G : 0;
            ge = min(G, cl_e - tt * G);
            return true;
        }
        if (u < p.rounds) {
            tile = (int)blockIdx.x + u * (int)gridDim.x;
            gb = 0;
            ge = G;
            return tile < total;
        }
        if (u == p.rounds && p.tail > 0 && ((int)blockIdx.x >> 1) < p.tail) {
            tile = p.rounds * (int)gridDim.x + ((int)blockIdx.x >> 1);
            const int r = (int)blockIdx.x & 1;
            gb = r ? G / 2 : 0;
            ge = r ? G : G / 2;
            return true;
        }
        return false;
    };

    // The clustered K split's sum segments (one warp, converged): this CTA
    // sums an even run [q0, q1) of its cluster's 16-byte output chunks,
    // tile after tile (BM * 32 a tile, [BM][128] floats); with fewer tiles
    // than CTAs a run meets at most two tiles.  For each: the tile, the
    // chunk range, the contributors ra..rb (the ranks whose runs meet the
    // tile, in K order), this CTA's unit index of it (if a contributor) and
    // each contributor's partial as a cluster address.
    auto cl_fill_table = [&]() {
        const int C = p.cl_ctas, r = (int)blockIdx.x % C, cbase = (int)blockIdx.x - r;
        constexpr int E4 = BM * 32;
        int k_s = 0, k_e = 0;  // lane k < C: the run of rank k
        if (lane < C) {
            int t0;
            cl_range(p, G, total, cbase + lane, k_s, k_e, t0);
        }
        const int te = min(p.cl_tiles, total - cl_t0) * E4;
        const int q0 = r * te / C, q1 = (r + 1) * te / C;
        for (int i = 0; i < 2; ++i) {
            int *t = cl_tab + 16 * i;
            const int qs = i == 0 ? q0 : (q0 / E4 + 1) * E4;  // segment i's start
            const int tt = qs / E4;
            const int lo = tt * G, hi = lo + G;
            int ra = -1, rb = -1, own_sl = 0;
            uint32_t src_l = 0;  // lane k: contributor k's partial
            for (int k = 0; k < C; ++k) {
                const int sk = __shfl_sync(0xffffffffu, k_s, k), ek = __shfl_sync(0xffffffffu, k_e, k);
                if (sk < hi && ek > lo) {
                    if (ra < 0) ra = k;
                    rb = k;
                    const int sl = tt - sk / G;  // its unit index of this tile
                    if (k == r) own_sl = sl;
                    const uint32_t a = map_to_rank(smem_u32(smem) + (uint32_t)(sl * BM * 128 * 4),
                                                   (uint32_t)k);
                    if (lane == k) src_l = a;
                }
            }
            if (lane < 8) t[8 + lane] = (int)src_l;
            if (lane == 0) {
                t[0] = qs < q1;
                t[1] = cl_t0 + tt;
                t[2] = qs - tt * E4;
                t[3] = min(E4, q1 - tt * E4);
                t[4] = ra;
                t[5] = rb;
                t[6] = own_sl;
            }
        }
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < kA; ++s) {
            // tensor-memory A: one dequantising warp per lane quarter writes a stage
            mbar_init(&a_full[s], TA ? 4 : kDqWarps);
            mbar_init(&a_empty[s], 1);
        }
        for (int s = 0; s < kB; ++s) {
            mbar_init(&b_full[s], 1);
            mbar_init(&b_empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], 4);
        }
        mbar_init(drain, 1);
        *flag = 0;
        fence_mbar_init();
    }
    if (warp == kWarpMma) {
        tmem_alloc(tmem_holder, p.tmem_cols);
        tmem_relinquish();
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    // Weights do not depend on earlier kernels: only the x loads (TMA warp)
    // and the y stores (epilogue) wait for the preceding grid, and the next
    // kernel may launch once every CTA of this one is running.
    launch_dependents();

    if (warp == kWarpTma) {
        // ------------------------------------------------------------------
        // x sub-tiles: kNI rows x 64 k, 128-byte swizzled, by TMA; kH of
        // them per stage, each into its own slot of the B ring.
        // ------------------------------------------------------------------
        if (lane == 0) {
            grid_dependency_wait();
            uint32_t bi = 0;
            int tile, gb, ge;
            for (int u = 0; unit_of(u, tile, gb, ge); ++u) {
                const int m0 = (tile % p.m_tiles) * BM;
                if constexpr (kSP >= 2) {
                    // the group's kSP stages' sub-tiles on one barrier
                    for (int g = gb; g < ge; g += kSP, ++bi) {
                        const int slot = bi % kBG;
                        const uint32_t ph = (bi / kBG) & 1u;
                        if (bi >= kBG && !tc_wait(&b_empty[slot], ph ^ 1u, flag, 0x0102))
                            goto tma_done;
#ifdef AQ_TEST_HOOKS
                        if (p.withhold && bi == 0) continue;  // nothing will complete b_full[0]
#endif
                        mbar_arrive_expect_tx(&b_full[slot], kSP * kBTile);
#pragma unroll
                        for (int e = 0; e < kSP; ++e)
                            tma_load_2d(b_ring + (kSP * slot + e) * kBTile, &tmap_x, 64 * (g + e),
                                        m0, &b_full[slot]);
                    }
                    continue;
                }
                for (int g = gb; g < ge; ++g) {
#pragma unroll
                    for (int h = 0; h < kH; ++h) {
                        const int slot = bi % kB;
                        const uint32_t ph = (bi / kB) & 1u;
                        if (bi >= kB && !tc_wait(&b_empty[slot], ph ^ 1u, flag, 0x0102))
                            goto tma_done;
#ifdef AQ_TEST_HOOKS
                        if (p.withhold && bi == 0) {  // nothing will complete b_full[0]
                            ++bi;
                            continue;
                        }
#endif
                        mbar_arrive_expect_tx(&b_full[slot], kBTile);
                        tma_load_2d(b_ring + slot * kBTile, &tmap_x, 64 * g, m0 + h * kNI,
                                    &b_full[slot]);
                        ++bi;
                    }
                }
            }
        tma_done:
            // Wind-down: the loads issued for the last sub-tiles land before
            // the CTA goes on (earlier ones were consumed by the MMAs).
            for (uint32_t j = bi > (uint32_t)kBG ? bi - kBG : 0u; j < bi; ++j)
                drain_wait(&b_full[j % kBG], (j / kBG) & 1u);
        }
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------------------
        // MMA issue: per stage, for each B sub-tile h, 4 x (128 x kNI x 16)
        // into columns [h kNI, (h+1) kNI) of accumulator b, then release the
        // sub-tile; after the last, release the A tile.  The whole warp
        // walks the stages (converged, waits taken by every lane and agreed
        // on); lane 0 issues.  Descriptors: those of slot 0, k-step 0, plus
        // the byte offset of the slot and k-step over 16.
        // ------------------------------------------------------------------
        const uint32_t idesc = (1u << 4) | ((BF16 ? 1u : 0u) << 7) | ((BF16 ? 1u : 0u) << 10) |
                               ((uint32_t)(kNI >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
        const uint64_t a_desc0 = sw128_desc(smem_u32(a_ring));
        const uint64_t b_desc0 = sw128_desc(smem_u32(b_ring));
        uint32_t ai = 0, bi = 0, ti = 0;
        int tile, gb, ge;
        bool ok = true, issued = false;  // both warp-uniform
        for (int u = 0; ok && unit_of(u, tile, gb, ge); ++u, ++ti) {
            const uint32_t b = ti % kAcc, use = ti / kAcc;
            const bool free = ti < (uint32_t)kAcc ||
                              tc_wait(&acc_empty[b], (use & 1u) ^ 1u, flag, 0x0202);
            if (!__all_sync(0xffffffffu, free)) break;
            tc_fence_after();
            const uint32_t d = tmem + b * BM;
            if constexpr (kSP >= 2) {
                for (int g = gb; ok && g < ge; g += kSP, ai += kSP, ++bi) {
                    const uint32_t al = ai + kSP - 1;  // the group's last A stage
                    const bool got_a = tc_wait(&a_full[al % kA], (al / kA) & 1u, flag, 0x0302);
                    if (!__all_sync(0xffffffffu, got_a)) {
                        ok = false;
                        break;
                    }
                    const int bs = bi % kBG;
                    const bool got_b = tc_wait(&b_full[bs], (bi / kBG) & 1u, flag, 0x0402);
                    if (!__all_sync(0xffffffffu, got_b)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    issued = true;
                    if (lane == 0) {
#pragma unroll
                        for (int e = 0; e < kSP; ++e) {
                            const uint64_t bd =
                                b_desc0 + (uint64_t)((uint32_t)((kSP * bs + e) * kBTile) >> 4);
                            if constexpr (TA) {
                                // A stage: 32 columns after the accumulators, 8 a k-step
                                const uint32_t at =
                                    tmem + (uint32_t)(kAcc * BM + ((ai + e) % kA) * 32);
#pragma unroll
                                for (int kk = 0; kk < 4; ++kk)
                                    tc_mma_f16_ta(d, at + 8u * kk, bd + 2 * kk, idesc,
                                                  (g + e != gb || kk != 0) ? 1u : 0u);
                            } else {
                                const uint64_t ad = a_desc0 +
                                    (uint64_t)((uint32_t)(((ai + e) % kA) * kATileBytes) >> 4);
#pragma unroll
                                for (int kk = 0; kk < 4; ++kk)
                                    tc_mma_f16(d, ad + 2 * kk, bd + 2 * kk, idesc,
                                               (g + e != gb || kk != 0) ? 1u : 0u);
                            }
                        }
                        tc_commit(&b_empty[bs]);
                        tc_commit(&a_empty[al % kA]);  // frees the group's A slots
                    }
                    __syncwarp();
                }
            } else {
            for (int g = gb; ok && g < ge; ++g, ++ai) {
                const int as = ai % kA;
                const bool got_a = tc_wait(&a_full[as], (ai / kA) & 1u, flag, 0x0302);
                if (!__all_sync(0xffffffffu, got_a)) {
                    ok = false;
                    break;
                }
#pragma unroll
                for (int h = 0; h < kH; ++h, ++bi) {
                    const int bs = bi % kB;
                    const bool got_b = tc_wait(&b_full[bs], (bi / kB) & 1u, flag, 0x0402);
                    if (!__all_sync(0xffffffffu, got_b)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    issued = true;
                    if (lane == 0) {
                        const uint64_t ad = a_desc0 + (uint64_t)((uint32_t)(as * kATileBytes) >> 4);
                        const uint64_t bd = b_desc0 + (uint64_t)((uint32_t)(bs * kBTile) >> 4);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            tc_mma_f16(d + h * kNI, ad + 2 * kk, bd + 2 * kk, idesc,
                                       (g != gb || kk != 0) ? 1u : 0u);
                        tc_commit(&b_empty[bs]);
                    }
                    __syncwarp();
                }
                if (!ok) break;
                if (lane == 0) tc_commit(&a_empty[as]);
                __syncwarp();
            }
            }
            if (!ok) break;
            if (lane == 0) tc_commit(&acc_full[b]);
            __syncwarp();
        }
        // Wind-down: every MMA issued has completed (it reads the rings and
        // writes tensor memory) before the CTA goes on.
        if (issued) {
            if (lane == 0) tc_commit(drain);
            __syncwarp();
            drain_wait(drain, 0);
            __syncwarp();
        }
    } else if (warp < kWarpDq) {
        // ------------------------------------------------------------------
        // Epilogue: TMEM lanes 32q..32q+31 (weight rows), BM columns (x rows).
        // ------------------------------------------------------------------
        const int q = warp & 3;
        T *y = static_cast<T *>(p.y);
        if constexpr (BM <= 128) {
            if (p.cl_ctas > 0 && warp == kWarpMma + 1) cl_fill_table();
        }
        grid_dependency_wait();
        uint32_t ti = 0;
        int tile, gb, ge;
        for (int u = 0; unit_of(u, tile, gb, ge); ++u, ++ti) {
            const uint32_t b = ti % kAcc, use = ti / kAcc;
            if (!tc_wait(&acc_full[b], use & 1u, flag, 0x0502)) break;
            tc_fence_after();
            if (u >= p.rounds) break;  // a split tail tile: added at the end
            const int n = (tile / p.m_tiles) * 128 + 32 * q + lane;
            const int m0 = (tile % p.m_tiles) * BM;
            for (int c0 = 0; c0 < BM && m0 + c0 < p.M; c0 += 16) {
                uint32_t v[16];
                tmem_ld16(tmem + ((uint32_t)(32 * q) << 16) + b * BM + c0, v);
                tmem_wait_ld();
                if (n < p.N) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int m = m0 + c0 + i;
                        if (m < p.M) y[(size_t)m * p.N + n] = cvt_out<T>(__uint_as_float(v[i]));
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[b]);
        }
    } else if constexpr (TA) {
        // ------------------------------------------------------------------
        // Dequantisation into tensor memory.  The warp's lane quarter q is
        // the 32-row block q of each 128-row weight tile (thread = row); the
        // two warps of a quarter take alternate 4-group super-stages.  Each
        // stage (one group) is 64 values of the thread's row: eight words of
        // codes, dequantised and written as 32 columns of the A stage.  The
        // MMA warp takes stages in groups of kSP (2, or 4: a whole
        // super-stage): the group's slots are waited for once and its last
        // stage's arrival stands for all.
        // ------------------------------------------------------------------
        static_assert((kSP == 2 || kSP == 4) && kA % kSP == 0 && kGroups % kSP == 0,
                      "tensor-memory A is consumed in groups of stages");
        using RT = RawT<B>;
        const int dw = warp - kWarpDq;
        const int q = warp & 3;
        const int par = dw >> 2;
        constexpr int kRawSlotsTa = raw_slots_ta(BM);
        uint8_t *ring = raw + dw * kRawSlotsTa * RT::kSlotBytes;
        const int64_t row_bytes = (int64_t)p.K * B / 8;
        const int nlast = p.N - 1;
        auto issue = [&](int tile, int ss, int slot) {
            const int n0 = (tile / p.m_tiles) * 128 + 32 * q;
            uint8_t *dst = ring + slot * RT::kSlotBytes;
            const int64_t kb = (int64_t)ss * kGroups * RT::kGroupBytes;
#pragma unroll
            for (int i = 0; i < RT::kChunksPerRow; ++i) {
                const int c = lane + 32 * i;
                const int r = c / RT::kChunksPerRow, col = c % RT::kChunksPerRow;
                const int64_t n = min(n0 + r, nlast);
                cp_async16(dst + r * RT::kRowPitch + col * 16,
                           reinterpret_cast<const uint8_t *>(p.Wq) + n * row_bytes + kb + col * 16,
                           16u);
            }
            const int64_t n = min(n0 + lane, nlast);
            cp_async8(dst + RT::kSbOff + lane * 8, p.scales + n * p.G + ss * kGroups);
            cp_async8(dst + RT::kSbOff + 256 + lane * 8, p.biases + n * p.G + ss * kGroups);
        };
        // Cursor over the CTA's super-stages in order (gs counts them all);
        // this warp takes those with gs % 2 == par.
        struct Cur {
            int u, tile, gb, ge, ss, gs;
            bool valid;
        };
        auto cur_init = [&](Cur &c) {
            c.u = c.ss = c.gs = 0;
            c.valid = unit_of(0, c.tile, c.gb, c.ge);
        };
        auto cur_next = [&](Cur &c) {
            do {
                if (++c.ss == (c.ge - c.gb) / kGroups) {
                    c.ss = 0;
                    ++c.u;
                    c.valid = unit_of(c.u, c.tile, c.gb, c.ge);
                }
                ++c.gs;
            } while (c.valid && (c.gs & 1) != par);
        };
        Cur ic, cc;
        cur_init(ic);
        if (ic.valid && par == 1) cur_next(ic);
        cc = ic;
        int iss = 0;
        // kRawSlotsTa - 1 super-stages ahead, one commit group each
#pragma unroll 1
        for (int pre = 0; pre < kRawSlotsTa - 1; ++pre) {
            if (ic.valid) {
                issue(ic.tile, ic.gb / kGroups + ic.ss, iss % kRawSlotsTa);
                ++iss;
                cur_next(ic);
            }
            cp_async_commit();
        }
        const uint32_t trow = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(kAcc * BM);
        bool ok = true;
        for (int cnt = 0; cc.valid && ok; ++cnt) {
            if (ic.valid) {
                issue(ic.tile, ic.gb / kGroups + ic.ss, iss % kRawSlotsTa);
                ++iss;
                cur_next(ic);
            }
            cp_async_commit();
            cp_async_wait<kRawSlotsTa - 1>();
            __syncwarp();
            const uint8_t *slotp = ring + (cnt % kRawSlotsTa) * RT::kSlotBytes;
            const uint2 sv2 = *reinterpret_cast<const uint2 *>(slotp + RT::kSbOff + lane * 8);
            const uint2 bv2 = *reinterpret_cast<const uint2 *>(slotp + RT::kSbOff + 256 + lane * 8);
            const uint4 sv = make_uint4(sv2.x, sv2.y, 0u, 0u);
            const uint4 bv = make_uint4(bv2.x, bv2.y, 0u, 0u);
            const uint8_t *rowp = slotp + lane * RT::kRowPitch;
#pragma unroll 1
            for (int j = 0; j < kGroups; ++j) {
                const uint32_t it = 4u * (uint32_t)cc.gs + (uint32_t)j;  // the MMA's stage count
                const int slot = (int)(it % kA);
                if (j % kSP == 0) {  // the group's slots: freed by one commit
                    const uint32_t il = it + kSP - 1;
                    if (il >= (uint32_t)kA &&
                        !tc_wait(&a_empty[il % kA], ((il / kA) & 1u) ^ 1u, flag, 0x0602)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                }
                const GroupConst gc = group_const<B>(h_at(sv, j), h_at(bv, j));
                uint32_t u[8];  // 8 codes per entry, k = 8c .. 8c+7 of the stage
                if constexpr (B == 4) {
                    const uint4 w0 = *reinterpret_cast<const uint4 *>(rowp + 32 * j);
                    const uint4 w1 = *reinterpret_cast<const uint4 *>(rowp + 32 * j + 16);
                    u[0] = w0.x, u[1] = w0.y, u[2] = w0.z, u[3] = w0.w;
                    u[4] = w1.x, u[5] = w1.y, u[6] = w1.z, u[7] = w1.w;
                } else {
                    const uint32_t *wp = reinterpret_cast<const uint32_t *>(rowp + 24 * j);
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const uint32_t x0 = wp[3 * hh], x1 = wp[3 * hh + 1], x2 = wp[3 * hh + 2];
                        u[4 * hh + 0] = x0;
                        u[4 * hh + 1] = __funnelshift_r(x0, x1, 24);
                        u[4 * hh + 2] = __funnelshift_r(x1, x2, 16);
                        u[4 * hh + 3] = x2 >> 8;
                    }
                }
                uint32_t out[32];
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint4 v = dq8<B, BF16>(u[c], gc);
                    out[4 * c + 0] = v.x;
                    out[4 * c + 1] = v.y;
                    out[4 * c + 2] = v.z;
                    out[4 * c + 3] = v.w;
                }
                tmem_st32(trow + (uint32_t)(slot * 32), out);
                if (j % kSP == kSP - 1) {  // the group is complete
                    tmem_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&a_full[slot]);
                }
            }
            __syncwarp();
            cur_next(cc);
        }
        cp_async_wait<0>();
        tmem_wait_st();
    } else {
        // ------------------------------------------------------------------
        // Dequantisation: this warp's 16 rows of each 128-row weight tile.
        // ------------------------------------------------------------------
        const int dw = warp - kWarpDq;
        uint8_t *ring = raw + dw * kRawSlots * R::kSlotBytes;
        const int64_t row_bytes = (int64_t)p.K * B / 8;
        // copy plan: kChunks pieces of 16 rows per super-stage + s/b
        constexpr int kChunks = R::kChunksPerRow / 2;
        uint32_t roff[kChunks], doff[kChunks];
#pragma unroll
        for (int i = 0; i < kChunks; ++i) {
            const int c = lane + 32 * i;
            const int r = c / R::kChunksPerRow, col = c % R::kChunksPerRow;
            roff[i] = (uint32_t)r;
            doff[i] = (uint32_t)(r * R::kRowPitch + col * R::kChunkBytes);
            roff[i] |= (uint32_t)col << 8;
        }
        const int nlast = p.N - 1;
        auto issue = [&](int tile, int ss, int slot) {
            const int n0 = (tile / p.m_tiles) * 128 + 16 * dw;
            uint8_t *dst = ring + slot * R::kSlotBytes;
            const int64_t kb = (int64_t)ss * kGroups * R::kGroupBytes;
#pragma unroll
            for (int i = 0; i < kChunks; ++i) {
                const int r = roff[i] & 0xFF, col = roff[i] >> 8;
                const int64_t n = min(n0 + r, nlast);
                const uint8_t *src = reinterpret_cast<const uint8_t *>(p.Wq) + n * row_bytes + kb +
                                     col * R::kChunkBytes;
                if constexpr (R::kChunkBytes == 16)
                    cp_async16(dst + doff[i], src, 16u);
                else
                    cp_async8(dst + doff[i], src);
            }
            const int sr = lane & 15;
            const int64_t n = min(n0 + sr, nlast);
            const __half *base = (lane < 16) ? p.scales : p.biases;
            if constexpr (GEN) {
                // 256 >> lg scales (or biases) of this row: 16, 8 or 4 bytes
                uint8_t *sd = dst + R::kSbOff + (lane >> 4) * 256 + sr * 16;
                const __half *src = base + n * p.NG + ss * (256 >> p.lg);
                if (p.lg == 5)
                    cp_async16(sd, src, 16u);
                else if (p.lg == 6)
                    cp_async8(sd, src);
                else
                    cp_async4(sd, src);
            } else {
                cp_async8(dst + R::kSbOff + (lane >> 4) * 128 + sr * 8,
                          base + n * p.G + ss * kGroups);
            }
        };
        // flat sequence of (unit, super-stage) for this CTA: the one being
        // dequantised (c...) and the next one to issue (n...)
        int cu = 0, ctile = 0, cgb = 0, cge = 0, css = 0;
        bool cvalid = unit_of(cu, ctile, cgb, cge);
        int nu = 0, ntile = 0, ngb = 0, nge = 0, nss_next = 0;
        bool nvalid = unit_of(nu, ntile, ngb, nge);
        auto advance = [&](int &u, int &t, int &gbv, int &gev, bool &valid, int &ssv) {
            if (++ssv == (gev - gbv) / kGroups) {
                ssv = 0;
                ++u;
                valid = unit_of(u, t, gbv, gev);
            }
        };
        uint32_t it = 0;  // A-stage counter (matches the MMA's)
        int iss = 0;      // super-stages issued
        // kRawSlots - 1 super-stages ahead, one commit group each
#pragma unroll 1
        for (int pre = 0; pre < kRawSlots - 1; ++pre) {
            if (nvalid) {
                issue(ntile, ngb / kGroups + nss_next, iss % kRawSlots);
                ++iss;
                advance(nu, ntile, ngb, nge, nvalid, nss_next);
            }
            cp_async_commit();
        }
        const int rl = lane >> 1, h = lane & 1;
        const int arow = 16 * dw + rl;  // row within the 128-row A tile
        bool ok = true;
        for (int cnt = 0; cvalid && ok; ++cnt) {
            if (nvalid) {
                issue(ntile, ngb / kGroups + nss_next, iss % kRawSlots);
                ++iss;
                advance(nu, ntile, ngb, nge, nvalid, nss_next);
            }
            cp_async_commit();
            cp_async_wait<kRawSlots - 1>();
            __syncwarp();
            const uint8_t *slotp = ring + (cnt % kRawSlots) * R::kSlotBytes;
            uint4 sv, bv;  // this row's scales and biases of the super-stage
            if constexpr (GEN) {
                sv = *reinterpret_cast<const uint4 *>(slotp + R::kSbOff + rl * 16);
                bv = *reinterpret_cast<const uint4 *>(slotp + R::kSbOff + 256 + rl * 16);
            } else {
                const uint2 sv2 = *reinterpret_cast<const uint2 *>(slotp + R::kSbOff + rl * 8);
                const uint2 bv2 =
                    *reinterpret_cast<const uint2 *>(slotp + R::kSbOff + 128 + rl * 8);
                sv = make_uint4(sv2.x, sv2.y, 0u, 0u);
                bv = make_uint4(bv2.x, bv2.y, 0u, 0u);
            }
            const uint8_t *rowp = slotp + rl * R::kRowPitch;
            // kPair groups (A stages) at a time: with a deep enough A ring,
            // two groups give the ALUs twice the independent work and one
            // fence serves both; a shallow ring keeps one.
            constexpr int kPair = kA >= 4 ? 2 : 1;
            static_assert(kSP == 1 || kPair == 2, "stage pairs are dequantised together");
#pragma unroll 1
            for (int j = 0; j < kGroups; j += kPair, it += kPair) {
                bool free2 = true;
                if constexpr (kSP == 2) {
                    // a pair's slots come back together (one commit after the
                    // pair that last used them)
                    const uint32_t il = it + 1;
                    if (il >= (uint32_t)kA &&
                        !tc_wait(&a_empty[il % kA], ((il / kA) & 1u) ^ 1u, flag, 0x0602))
                        free2 = false;
                } else {
#pragma unroll
                    for (int e = 0; e < kPair; ++e) {
                        const uint32_t ie = it + e;
                        if (ie >= (uint32_t)kA &&
                            !tc_wait(&a_empty[ie % kA], ((ie / kA) & 1u) ^ 1u, flag, 0x0602))
                            free2 = false;
                    }
                }
                if (!free2) {
                    ok = false;
                    break;
                }
                if constexpr (GEN) {
                    // this lane's 32 codes of stage j+e: one group (its index
                    // within the super-stage from the group size), w = (2048
                    // + q) s + (b - 2048 s) two at a time
#pragma unroll
                    for (int e = 0; e < kPair; ++e) {
                        const int gi = (64 * (j + e) + 32 * h) >> p.lg;
                        const float sc = h_at(sv, gi), bc = h_at(bv, gi);
                        const float2 s2 = make_float2(sc, sc);
                        const float pb = fmaf(-2048.f, sc, bc);
                        const float2 p2 = make_float2(pb, pb);
                        uint32_t w[B];
                        load_codes<B>(rowp + (j + e) * R::kGroupBytes + h * 4 * B, w);
                        uint8_t *arow_p = a_ring + ((it + e) % kA) * kATileBytes + arow * 128;
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            uint32_t o[4];
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                const int i0 = 8 * c + 2 * q;
                                const float2 f = make_float2(code_f<B>(w, i0), code_f<B>(w, i0 + 1));
                                o[q] = pack_out<BF16>(__ffma2_rn(f, s2, p2));
                            }
                            const int chunk = 4 * h + c;  // k = 8*chunk .. 8*chunk+7
                            *reinterpret_cast<uint4 *>(arow_p + ((chunk ^ (arow & 7)) << 4)) =
                                make_uint4(o[0], o[1], o[2], o[3]);
                        }
                    }
                } else {
                uint32_t u[kPair][4];  // 8 codes per entry, this lane's chunks 4h..4h+3
                GroupConst gc[kPair];
#pragma unroll
                for (int e = 0; e < kPair; ++e) {
                    gc[e] = group_const<B>(h_at(sv, j + e), h_at(bv, j + e));
                    if constexpr (B == 4) {
                        const uint4 w =
                            *reinterpret_cast<const uint4 *>(rowp + (j + e) * 32 + h * 16);
                        u[e][0] = w.x;
                        u[e][1] = w.y;
                        u[e][2] = w.z;
                        u[e][3] = w.w;
                    } else {
                        const uint32_t *wp =
                            reinterpret_cast<const uint32_t *>(rowp + (j + e) * 24 + h * 12);
                        const uint32_t w0 = wp[0], w1 = wp[1], w2 = wp[2];
                        u[e][0] = w0;
                        u[e][1] = __funnelshift_r(w0, w1, 24);
                        u[e][2] = __funnelshift_r(w1, w2, 16);
                        u[e][3] = w2 >> 8;
                    }
                }
#pragma unroll
                for (int e = 0; e < kPair; ++e) {
                    uint8_t *arow_p = a_ring + ((it + e) % kA) * kATileBytes + arow * 128;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int chunk = 4 * h + c;  // k = 8*chunk .. 8*chunk+7
                        const uint4 v = dq8<B, BF16>(u[e][c], gc[e]);
                        *reinterpret_cast<uint4 *>(arow_p + ((chunk ^ (arow & 7)) << 4)) = v;
                    }
                }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    if constexpr (kSP == 2) {
                        mbar_arrive(&a_full[(it + 1) % kA]);  // the MMA waits on the second
                    } else {
#pragma unroll
                        for (int e = 0; e < kPair; ++e) mbar_arrive(&a_full[(it + e) % kA]);
                    }
                }
            }
            __syncwarp();
            advance(cu, ctile, cgb, cge, cvalid, css);
        }
        cp_async_wait<0>();
    }

    // Copies and MMAs issued have completed (the producers and the MMA
    // warp drained them, with bounded waits), so shared and tensor memory
    // may be reused or released from here on, error or not.
    __syncthreads();
    if (p.tail > 0 && ((int)blockIdx.x >> 1) < p.tail) {
        // The split tail tile: rank 1 hands its half of the accumulator to
        // rank 0 through distributed shared memory, up to 256 columns at a
        // time (the idle ring holds them); rank 0 adds it to its own half
        // (rank 0 first) and stores y.  Both CTAs of the cluster take every
        // barrier, error or not.
        constexpr int kCh = BM < 256 ? BM : 256;  // columns per hand-over
        constexpr int kXP = kCh + 4;              // floats per row of the buffer
        // the idle rings: A tiles (in shared memory unless TA), x tiles, raw codes
        static_assert(128 * kXP * 4 <= (TA ? 0 : kA * kATileBytes) + kB * kBTile +
                                           kDqWarps * kRawSlots * kRawSlotBytes,
                      "hand-over buffer");
        const int r = (int)blockIdx.x & 1;
        const int tile = p.rounds * (int)gridDim.x + ((int)blockIdx.x >> 1);
        int nfull = 0;  // whole tiles this CTA took before the tail
        for (int u = 0; u < p.rounds; ++u)
            nfull += ((int)blockIdx.x + u * (int)gridDim.x < total) ? 1 : 0;
        const uint32_t b = (uint32_t)nfull % kAcc;
        float *xbuf = reinterpret_cast<float *>(smem);  // [128][kXP] floats on rank 0
        const bool epi = warp >= kWarpMma + 1 && warp < kWarpDq;
        const int q = warp & 3;
        const int row = 32 * q + lane;  // weight row of the tile
        const int n = (tile / p.m_tiles) * 128 + row;
        const int m0 = (tile % p.m_tiles) * BM;
        T *y = static_cast<T *>(p.y);
        const uint32_t rbuf = map_to_rank(smem_u32(xbuf), 0u) + 4u * (uint32_t)(row * kXP);
        const uint32_t ta = tmem + ((uint32_t)(32 * q) << 16) + b * BM;
        tc_fence_after();
        // rank 0's ring (the buffer) is idle only once its main loop is done
        cluster_sync();
        for (int c0 = 0; c0 < BM; c0 += kCh) {
            if (epi && r == 1) {
                for (int c1 = 0; c1 < kCh; c1 += 16) {
                    uint32_t v[16];
                    tmem_ld16(ta + (uint32_t)(c0 + c1), v);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 16; j += 4)
                        st_dsmem_v4(rbuf + 4u * (uint32_t)(c1 + j), __uint_as_float(v[j]),
                                    __uint_as_float(v[j + 1]), __uint_as_float(v[j + 2]),
                                    __uint_as_float(v[j + 3]));
                }
            }
            cluster_sync();
            if (epi && r == 0) {
                for (int c1 = 0; c1 < kCh; c1 += 16) {
                    uint32_t v[16];
                    tmem_ld16(ta + (uint32_t)(c0 + c1), v);
                    tmem_wait_ld();
                    if (*flag || n >= p.N) continue;
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int m = m0 + c0 + c1 + j;
                        if (m < p.M)
                            y[(size_t)m * p.N + n] =
                                cvt_out<T>(__uint_as_float(v[j]) + xbuf[row * kXP + c1 + j]);
                    }
                }
            }
            cluster_sync();
        }
        tc_fence_before();
    }
    if constexpr (BM <= 128) {
        if (p.cl_ctas > 0) {
            // Clustered K split.  (1) Warps 2..13 copy each of the CTA's one
            // or two partial accumulators into the idle ring as [BM][128]
            // floats (unit i at i * BM * 128).  (2) After a cluster barrier,
            // each CTA sums its segments of the cluster's outputs (the table
            // filled during the main loop): each output is the sum of its
            // tile's partials in rank order, read through distributed shared
            // memory.  (3) A last cluster barrier keeps every partial readable
            // until all sums are done; then y is stored.  Every CTA takes both
            // barriers, error or not.
            static_assert(2 * BM * 128 * 4 <= (TA ? 0 : kA * kATileBytes) + kB * kBTile +
                                                  kDqWarps * kRawSlots * kRawSlotBytes,
                          "partial tiles");
            const int r = (int)blockIdx.x % p.cl_ctas;
            float *part = reinterpret_cast<float *>(smem);
            tc_fence_after();
            if (warp > kWarpMma) {
                // warps 2..13: lane quarter warp % 4, column blocks of 16
                // dealt out over the quarter's three warps
                const int q = warp & 3, h = (warp - kWarpMma - 1) >> 2;
                const int row = 32 * q + lane;
                int tile, gb, ge;
                constexpr int kBlk = (BM / 16 + 2) / 3;  // column blocks a warp, at most
                for (int i = 0; i < 2 && unit_of(i, tile, gb, ge); ++i) {
                    const uint32_t ta = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(i % kAcc) * BM;
                    float *dst = part + i * BM * 128 + row;
                    uint32_t v[kBlk][16];
#pragma unroll
                    for (int bk = 0; bk < kBlk; ++bk)
                        if (16 * h + 48 * bk < BM) tmem_ld16(ta + (uint32_t)(16 * h + 48 * bk), v[bk]);
                    tmem_wait_ld();
#pragma unroll
                    for (int bk = 0; bk < kBlk; ++bk) {
                        const int c0 = 16 * h + 48 * bk;
                        if (c0 >= BM) continue;
#pragma unroll
                        for (int j = 0; j < 16; ++j) dst[(c0 + j) * 128] = __uint_as_float(v[bk][j]);
                    }
                }
            }
            tc_fence_before();
            cluster_sync();
            grid_dependency_wait();  // every thread below stores y
            T *y = static_cast<T *>(p.y);
            // The sums are held in registers (rounded and packed, four
            // outputs a 16-byte chunk) until every partial has been read:
            // then the last cluster barrier orders only those reads, and the
            // y stores follow it.
            constexpr int E4 = BM * 32;                            // chunks a tile
            constexpr int kJ = (E4 + kThreadsTc - 1) / kThreadsTc;  // a thread's, at most
            uint2 outv[2][kJ];
            int u_c0[2] = {0, 0}, u_c1[2] = {0, 0}, u_m0[2] = {0, 0}, u_n0[2] = {0, 0};
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                // segment i of the table filled during the main loop
                const int *t = cl_tab + 16 * i;
                if (!t[0]) break;
                const int tile = t[1], c0 = t[2], c1 = t[3], ra = t[4], rb = t[5];
                const int own_sl = t[6];
                const int *src = t + 8;  // contributor k's partial, a cluster address
                u_c0[i] = c0;
                u_c1[i] = c1;
                u_n0[i] = (tile / p.m_tiles) * 128;
                u_m0[i] = (tile % p.m_tiles) * BM;
                const float4 *own = reinterpret_cast<const float4 *>(part) + own_sl * E4;
#pragma unroll
                for (int jb = 0; jb < kJ; jb += 4) {
                    const int cb = c0 + (int)threadIdx.x + jb * kThreadsTc;
                    if (cb >= c1) break;
                    float4 acc[4];
                    for (int k = ra; k <= rb; ++k) {
                        float4 w[4];
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const int cj = cb + j * kThreadsTc;
                            if (jb + j < kJ && cj < c1)
                                w[j] = k == r ? own[cj]
                                              : ld_dsmem_v4((uint32_t)src[k] + 16u * (uint32_t)cj);
                        }
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            if (jb + j >= kJ || cb + j * kThreadsTc >= c1) continue;
                            if (k == ra) {
                                acc[j] = w[j];
                            } else {
                                acc[j].x += w[j].x;
                                acc[j].y += w[j].y;
                                acc[j].z += w[j].z;
                                acc[j].w += w[j].w;
                            }
                        }
                    }
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        if (jb + j < kJ)
                            outv[i][jb + j] = make_uint2(pack_out<BF16>(make_float2(acc[j].x, acc[j].y)),
                                                         pack_out<BF16>(make_float2(acc[j].z, acc[j].w)));
                    }
                }
            }
            cluster_sync();
            if (!*flag) {
#pragma unroll
                for (int i = 0; i < 2; ++i) {
#pragma unroll
                    for (int jj = 0; jj < kJ; ++jj) {
                        const int c = u_c0[i] + (int)threadIdx.x + jj * kThreadsTc;
                        if (c >= u_c1[i]) continue;
                        const int m = u_m0[i] + c / 32, n = u_n0[i] + 4 * (c & 31);
                        if (m >= p.M || n >= p.N) continue;
                        T *yr = y + (size_t)m * p.N + n;
                        const uint2 v = outv[i][jj];
                        if (n + 3 < p.N && (reinterpret_cast<uintptr_t>(yr) & 7u) == 0) {
                            *reinterpret_cast<uint2 *>(yr) = v;
                        } else {
                            const uint16_t h[4] = {(uint16_t)(v.x & 0xFFFFu), (uint16_t)(v.x >> 16),
                                                   (uint16_t)(v.y & 0xFFFFu), (uint16_t)(v.y >> 16)};
                            uint16_t *yh = reinterpret_cast<uint16_t *>(yr);
                            for (int e = 0; e < 4 && n + e < p.N; ++e) yh[e] = h[e];
                        }
                    }
                }
            }
        }
    }
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, p.tmem_cols);
    }
}

// ---------------------------------------------------------------------------
// "tcw": the same tensor-core path with the roles swapped, for M <= 128.
//
// A chain of tcgen05.mma instructions of kind::f16 into one accumulator
// advances at about the same rate for any N up to 256 (measured on GB300:
// ~118 cycles an instruction for N = 16..128, 128 for N = 256), so with the
// weights as the 128-row A operand a narrow x tile leaves most of each
// instruction's time unused.  Here the x tile is A (128 rows, rows past M
// read as zero) and a 256-row weight tile is B (N = 256): twice the weights
// per instruction.  A weight tile's K range is split over the CTAs of a cluster
// (up to 8) so that narrow outputs still fill the SMs; the partial tiles are
// added in rank order through distributed shared memory (deterministic).
//
// Roles (448 threads): warp 0 TMA producer of x tiles, warp 1 MMA issuer and
// tensor memory owner, warps 2-5 epilogue, warps 6-13 dequantisation (each
// streams 32 weight rows, one per lane, through a two-slot cp.async ring).
// ---------------------------------------------------------------------------
namespace {

constexpr int kWRows = 256;                  // weight rows per tile (MMA N)
constexpr int kWXRows = 128;                 // x rows per tile (MMA M)
constexpr int kWStages = 3;                  // A/B ring depth
constexpr int kWRawSlots = 2;                // raw super-stages per dequant warp
constexpr int kWATile = kWXRows * 128;       // 16 KB
constexpr int kWBTile = kWRows * 128;        // 32 KB
constexpr int kWPitch = kWRows + 4;          // partial tile: floats per x row

// Raw super-stage of one tcw dequantising warp: 32 rows (one per lane) x 4
// groups, then scales and biases.  Rows 36 (4-bit) or 28 (3-bit) words
// apart: the dequantising loads are 16 bytes wide (3-bit: two groups, 48
// bytes, at a time) and a quarter warp's eight rows fall in distinct banks.
template <int B>
struct RawW {
    static constexpr int kGroupBytes = 8 * B;
    static constexpr int kRowBytes = kGroups * kGroupBytes;  // 128 / 96
    static constexpr int kChunksPerRow = kRowBytes / 16;    // 8 / 6
    static constexpr int kRowPitch = kRowBytes + 16;         // 144 / 112
    static constexpr int kSbOff = 32 * kRowPitch;            // scales[32][4], then biases[32][4]
    static constexpr int kSlotBytes = kSbOff + 2 * 32 * 8;
};

}  // namespace

struct TcwParams {
    const uint32_t *Wq;
    const __half *scales;
    const __half *biases;
    void *y;
    int M, N, K, G;
    int splits;   // CTAs of a cluster sharing one weight tile's K range
    int gps;      // groups per split (a multiple of 4)
    uint32_t off_raw, off_bar;
};

template <int B, bool BF16>
__global__ void __launch_bounds__(kThreadsTc, 1)
    tcw_kernel(const __grid_constant__ TcwParams p, const __grid_constant__ CUtensorMap tmap_x) {
    using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
    using R = RawW<B>;
    extern __shared__ uint8_t smem_dyn[];
    uint8_t *smem = smem_dyn + ((1024u - (smem_u32(smem_dyn) & 1023u)) & 1023u);
    uint8_t *a_ring = smem;                           // x tiles
    uint8_t *b_ring = smem + kWStages * kWATile;      // weight tiles
    uint8_t *raw = smem + p.off_raw;
    float *partial = reinterpret_cast<float *>(smem);  // after the main loop
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + p.off_bar);
    uint64_t *a_full = bars;
    uint64_t *b_full = bars + kWStages;
    uint64_t *ab_empty = bars + 2 * kWStages;
    uint64_t *acc_full = bars + 3 * kWStages;
    uint64_t *drain = acc_full + 1;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *flag = reinterpret_cast<volatile int *>(tmem_holder + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = p.splits;
    const int rank = (int)(blockIdx.x % (unsigned)S);
    const int n0 = (int)(blockIdx.x / (unsigned)S) * kWRows;
    const int g0 = rank * p.gps;
    const int ns = min(p.G, g0 + p.gps) - g0;  // stages of this CTA (>= 4 by the plan)

    if (threadIdx.x == 0) {
        for (int s = 0; s < kWStages; ++s) {
            mbar_init(&a_full[s], 1);
            mbar_init(&b_full[s], kDqWarps);
            mbar_init(&ab_empty[s], 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(drain, 1);
        *flag = 0;
        fence_mbar_init();
    }
    if (warp == kWarpMma) {
        tmem_alloc(tmem_holder, kWRows);
        tmem_relinquish();
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    launch_dependents();

    if (warp == kWarpTma) {
        if (lane == 0) {
            grid_dependency_wait();  // x belongs to the stream order
            int i = 0;
            for (; i < ns; ++i) {
                const int slot = i % kWStages;
                const uint32_t ph = (i / kWStages) & 1u;
                if (i >= kWStages && !tc_wait(&ab_empty[slot], ph ^ 1u, flag, 0x0702)) break;
                mbar_arrive_expect_tx(&a_full[slot], kWATile);
                tma_load_2d(a_ring + slot * kWATile, &tmap_x, 64 * (g0 + i), 0, &a_full[slot]);
            }
            // Wind-down: the loads issued for the last stages land first.
            for (int j = i > kWStages ? i - kWStages : 0; j < i; ++j)
                drain_wait(&a_full[j % kWStages], (uint32_t)(j / kWStages) & 1u);
        }
    } else if (warp == kWarpMma) {
        // D[x row][weight row] += x . W^T: 4 x (M=128, N=256, K=16) per stage
        const uint32_t idesc = (1u << 4) | ((BF16 ? 1u : 0u) << 7) | ((BF16 ? 1u : 0u) << 10) |
                               ((uint32_t)(kWRows >> 3) << 17) | ((uint32_t)(kWXRows >> 4) << 24);
        const uint64_t a_desc0 = sw128_desc(smem_u32(a_ring));
        const uint64_t b_desc0 = sw128_desc(smem_u32(b_ring));
        bool ok = true, issued = false;  // both warp-uniform
        for (int i = 0; i < ns; ++i) {
            const int slot = i % kWStages;
            const uint32_t ph = (i / kWStages) & 1u;
            const bool got = tc_wait(&a_full[slot], ph, flag, 0x0802) &&
                             tc_wait(&b_full[slot], ph, flag, 0x0802);
            if (!__all_sync(0xffffffffu, got)) {
                ok = false;
                break;
            }
            tc_fence_after();
            issued = true;
            if (lane == 0) {
                const uint64_t ad = a_desc0 + (uint64_t)((uint32_t)(slot * kWATile) >> 4);
                const uint64_t bd = b_desc0 + (uint64_t)((uint32_t)(slot * kWBTile) >> 4);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    tc_mma_f16(tmem, ad + 2 * kk, bd + 2 * kk, idesc, (i | kk) != 0);
                tc_commit(&ab_empty[slot]);
            }
            __syncwarp();
        }
        if (ok && lane == 0) tc_commit(acc_full);
        __syncwarp();
        // Wind-down: every MMA issued has completed before the CTA goes on.
        if (issued) {
            if (lane == 0) tc_commit(drain);
            __syncwarp();
            drain_wait(drain, 0);
            __syncwarp();
        }
    } else if (warp < kWarpDq) {
        // Epilogue: TMEM lane = x row m = 32q + lane, column = weight row.
        const int q = warp & 3;
        const int m = 32 * q + lane;
        T *y = static_cast<T *>(p.y);
        grid_dependency_wait();  // y belongs to the stream order
        const bool got = tc_wait(acc_full, 0, flag, 0x0902);
        if (__all_sync(0xffffffffu, got)) {
            tc_fence_after();
            for (int c0 = 0; c0 < kWRows; c0 += 16) {
                uint32_t v[16];
                tmem_ld16(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)c0, v);
                tmem_wait_ld();
                if (m >= p.M) continue;
                if (S > 1) {
                    float4 *dst = reinterpret_cast<float4 *>(partial + m * kWPitch + c0);
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        dst[i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                             __uint_as_float(v[4 * i + 2]),
                                             __uint_as_float(v[4 * i + 3]));
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int n = n0 + c0 + i;
                        if (n < p.N) y[(size_t)m * p.N + n] = cvt_out<T>(__uint_as_float(v[i]));
                    }
                }
            }
            tc_fence_before();
        }
    } else {
        // Dequantisation: lane = weight row 32*dw + lane of the tile.
        const int dw = warp - kWarpDq;
        uint8_t *ring = raw + dw * kWRawSlots * R::kSlotBytes;
        const int64_t row_bytes = (int64_t)p.K * B / 8;
        const int row = 32 * dw + lane;
        const int64_t n = min(n0 + row, p.N - 1);  // rows past N repeat the last (never stored)
        const uint8_t *wrow0 = reinterpret_cast<const uint8_t *>(p.Wq);
        const int nss = ns / kGroups;  // super-stages (4 groups each)
        auto issue = [&](int ss, int slot) {
            uint8_t *dst = ring + slot * R::kSlotBytes;
            const int64_t kb = (int64_t)(g0 + ss * kGroups) * R::kGroupBytes;
            // consecutive lanes copy consecutive 16-byte pieces of a row
#pragma unroll
            for (int i = 0; i < R::kChunksPerRow; ++i) {
                const int c = lane + 32 * i;
                const int r = c / R::kChunksPerRow, col = c % R::kChunksPerRow;
                cp_async16(dst + r * R::kRowPitch + col * 16,
                           wrow0 + (int64_t)min(n0 + 32 * dw + r, p.N - 1) * row_bytes + kb +
                               col * 16,
                           16u);
            }
            cp_async8(dst + R::kSbOff + lane * 8, p.scales + n * p.G + g0 + ss * kGroups);
            cp_async8(dst + R::kSbOff + 256 + lane * 8, p.biases + n * p.G + g0 + ss * kGroups);
        };
        for (int pre = 0; pre < kWRawSlots - 1; ++pre) {
            if (pre < nss) issue(pre, pre);
            cp_async_commit();
        }
        int it = 0;  // stage counter (matches the MMA's)
        bool ok = true;
        for (int ss = 0; ss < nss && ok; ++ss) {
            if (ss + kWRawSlots - 1 < nss)
                issue(ss + kWRawSlots - 1, (ss + kWRawSlots - 1) % kWRawSlots);
            cp_async_commit();
            cp_async_wait<kWRawSlots - 1>();
            __syncwarp();
            const uint8_t *slotp = ring + (ss % kWRawSlots) * R::kSlotBytes;
            const uint2 sv2 = *reinterpret_cast<const uint2 *>(slotp + R::kSbOff + lane * 8);
            const uint2 bv2 = *reinterpret_cast<const uint2 *>(slotp + R::kSbOff + 256 + lane * 8);
            const uint4 sv = make_uint4(sv2.x, sv2.y, 0u, 0u);
            const uint4 bv = make_uint4(bv2.x, bv2.y, 0u, 0u);
            const uint8_t *rowp = slotp + lane * R::kRowPitch;
            uint32_t w3[12];  // 3-bit: the codes of two groups
            (void)w3;
#pragma unroll
            for (int j = 0; j < kGroups; ++j, ++it) {
                const int slot = it % kWStages;
                const uint32_t ph = (it / kWStages) & 1u;
                if (it >= kWStages) {
                    const bool got = tc_wait(&ab_empty[slot], ph ^ 1u, flag, 0x0a02);
                    if (!__all_sync(0xffffffffu, got)) {
                        ok = false;
                        break;
                    }
                }
                const GroupConst gc = group_const<B>(h_at(sv, j), h_at(bv, j));
                uint32_t u[8];  // 8 codes per entry
                if constexpr (B == 4) {
                    const uint4 w0 = *reinterpret_cast<const uint4 *>(rowp + j * 32);
                    const uint4 w1 = *reinterpret_cast<const uint4 *>(rowp + j * 32 + 16);
                    u[0] = w0.x; u[1] = w0.y; u[2] = w0.z; u[3] = w0.w;
                    u[4] = w1.x; u[5] = w1.y; u[6] = w1.z; u[7] = w1.w;
                } else {
                    // groups j and j+1 (48 bytes) are loaded together at even j
                    if ((j & 1) == 0) {
                        const uint4 *wp = reinterpret_cast<const uint4 *>(rowp + j * 24);
                        const uint4 q0 = wp[0], q1 = wp[1], q2 = wp[2];
                        w3[0] = q0.x, w3[1] = q0.y, w3[2] = q0.z, w3[3] = q0.w;
                        w3[4] = q1.x, w3[5] = q1.y, w3[6] = q1.z, w3[7] = q1.w;
                        w3[8] = q2.x, w3[9] = q2.y, w3[10] = q2.z, w3[11] = q2.w;
                    }
                    const uint32_t *wv = w3 + 6 * (j & 1);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const uint32_t w0 = wv[3 * h], w1 = wv[3 * h + 1], w2 = wv[3 * h + 2];
                        u[4 * h] = w0;
                        u[4 * h + 1] = __funnelshift_r(w0, w1, 24);
                        u[4 * h + 2] = __funnelshift_r(w1, w2, 16);
                        u[4 * h + 3] = w2 >> 8;
                    }
                }
                uint8_t *brow = b_ring + slot * kWBTile + row * 128;
#pragma unroll
                for (int c = 0; c < 8; ++c) {  // k = 8c .. 8c+7
                    const uint4 v = dq8<B, BF16>(u[c], gc);
                    *reinterpret_cast<uint4 *>(brow + ((c ^ (row & 7)) << 4)) = v;
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&b_full[slot]);
            }
            __syncwarp();
        }
        cp_async_wait<0>();
    }

    // Copies and MMAs issued have completed (the producers and the MMA
    // warp drained them, with bounded waits), so shared and tensor memory
    // may be reused or released from here on, error or not.
    __syncthreads();
    if (S > 1) {
        // Every CTA of the cluster reaches both barriers, error or not.
        // Rank r adds its share of the tile's M x 256 elements over all
        // ranks, rank 0 first, and stores y (every storing thread has waited
        // for the preceding grid).
        grid_dependency_wait();
        cluster_sync();
        if (!*flag) {
            T *y = static_cast<T *>(p.y);
            const int total = p.M * kWRows;
            const int chunk = (total + S - 1) / S;
            const int e1 = min(total, (rank + 1) * chunk);
            const uint32_t base = smem_u32(partial);
            for (int e = rank * chunk + (int)threadIdx.x; e < e1; e += kThreadsTc) {
                const int mm = e / kWRows, nn = e - mm * kWRows;
                if (n0 + nn >= p.N) continue;
                const uint32_t off = base + 4u * (uint32_t)(mm * kWPitch + nn);
                float v = 0.f;
                for (int r = 0; r < S; ++r) v += ld_dsmem_f32(map_to_rank(off, (uint32_t)r));
                y[(size_t)mm * p.N + n0 + nn] = cvt_out<T>(v);
            }
        }
        cluster_sync();
    }
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, kWRows);
    }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
namespace {

constexpr size_t kSmemLimitTc = 227 * 1024;

struct TcPlan {
    int BM;
    TcParams prm;
    size_t smem;
    int grid;
};

// Co-resident clusters of 1..8 CTAs when each CTA has an SM to itself (every
// tc plan does: its shared memory is over half an SM's), queried once.
const int *tc_active_clusters() {
    static int n[9];
    static std::once_flag once;
    std::call_once(once, [] {
        auto kern = tc_kernel<4, true, 64, false>;
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemLimitTc);
        for (int c = 1; c <= 8; ++c) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3((unsigned)c, 1, 1);
            cfg.blockDim = dim3(kThreadsTc, 1, 1);
            cfg.dynamicSmemBytes = kSmemLimitTc;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = (unsigned)c;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int k = 0;
            if (cudaOccupancyMaxActiveClusters(&k, kern, &cfg) != cudaSuccess) k = 0;
            n[c] = k;
        }
        cudaGetLastError();
    });
    return n;
}

// The clustered K split's fixed cost (partials through shared memory, two
// cluster barriers, the sums), in stages of one group: measured on GB300 at
// about 2-3.6 us when a cluster shares one tile and 7-9 us when it shares
// several (two partial tiles a CTA), against ~0.37 us a stage.
constexpr int cluster_split_stages(int tiles) { return tiles == 1 ? 8 : 20; }

// group: 0 for the 3/4-bit group-64 format, else the group size of the
// general-width path (32, 64 or 128; x tiles of at most 128 rows).
bool tc_plan(const MatmulArgs &a, TcPlan &pl, int group = 0) {
    if (a.K % 512 != 0 || a.M < 1 || a.N < 1) return false;
    if (a.M > INT32_MAX / 2 || a.N > INT32_MAX / 2 || a.K > INT32_MAX / 2) return false;
    const bool gen = group != 0;
    if (gen && group != 32 && group != 64 && group != 128) return false;
    if (!gen && a.bits != 3 && a.bits != 4) return false;
    // Past 256 rows, 512-row x tiles: each weight tile is dequantised once
    // for 512 rows (two N = 256 MMAs per k-step).
    pl.BM = a.M <= 64 ? 64 : a.M <= 128 ? 128 : a.M <= 256 ? 256 : 512;
    if (gen) pl.BM = std::min(pl.BM, 256);
    TcParams &q = pl.prm;
    q.M = (int)a.M;
    q.N = (int)a.N;
    q.K = (int)a.K;
    q.G = (int)(a.K / 64);
    q.n_tiles = (int)((a.N + 127) / 128);
    q.m_tiles = (int)((a.M + pl.BM - 1) / pl.BM);
    if ((int64_t)q.n_tiles * q.m_tiles > INT32_MAX) return false;
    const bool ta = ta_for(pl.BM, gen);
    int raw_slot = ta ? (a.bits == 4 ? RawT<4>::kSlotBytes : RawT<3>::kSlotBytes)
                      : (a.bits == 4 ? Raw<4>::kSlotBytes : Raw<3>::kSlotBytes);
    int kRawSlots = ta ? raw_slots_ta(pl.BM) : raw_slots_for(pl.BM);
    if (gen) {
        switch (a.bits) {
            case 2: raw_slot = RawG<2>::kSlotBytes; break;
            case 3: raw_slot = RawG<3>::kSlotBytes; break;
            case 4: raw_slot = RawG<4>::kSlotBytes; break;
            case 5: raw_slot = RawG<5>::kSlotBytes; break;
            case 6: raw_slot = RawG<6>::kSlotBytes; break;
            case 8: raw_slot = RawG<8>::kSlotBytes; break;
            default: return false;
        }
        kRawSlots = raw_slots_g(a.bits);
        int lg = 0;
        while ((1 << lg) < group) ++lg;
        q.lg = lg;
        q.NG = (int)(a.K / group);
    } else {
        q.lg = 6;
        q.NG = (int)(a.K / 64);
    }
    const int kA = ta ? kATmemSlots : a_slots_for(pl.BM, gen), kB = b_slots_for(pl.BM, gen);
    size_t off = ta ? 0 : (size_t)kA * kATileBytes;  // A tiles in shared memory
    q.off_b = (uint32_t)off;
    off += (size_t)kB * ni_for(pl.BM) * 128;
    q.off_raw = (uint32_t)off;
    off += (size_t)kDqWarps * kRawSlots * raw_slot;
    off = (off + 15) / 16 * 16;
    q.off_bar = (uint32_t)off;
    off += (2 * kA + 2 * kB + 5) * 8 + 16 + 128;  // barriers, TMEM address, flag, sum table
    pl.smem = off + 1024;  // room to align the base to 1024 bytes
    if (pl.smem > kSmemLimitTc) return false;
    q.tmem_cols = (pl.BM >= 256 || ta) ? 512 : pl.BM == 128 ? 256 : 128;
    q.Wq = a.Wq;
    q.scales = static_cast<const __half *>(a.scales);
    q.biases = static_cast<const __half *>(a.biases);
    q.y = a.out;
#ifdef AQ_TEST_HOOKS
    q.withhold = g_test_withhold == 2;
#endif
    const int total = q.n_tiles * q.m_tiles;
    int grid = std::min(total, num_sms());
    q.rounds = (total + grid - 1) / grid;
    q.tail = 0;
    // Tiles left over after whole rounds, when they fill at most half of the
    // grid, are split in two K halves over CTA pairs (clusters of two)
    // instead of running a half-empty round; so are all tiles when there are
    // at most half as many as SMs.
    const int g2 = grid & ~1;
    if (q.G % (2 * kGroups) == 0) {
        if (2 * total <= num_sms()) {
            // few tiles: every one split in two K halves
            grid = 2 * total;
            q.rounds = 0;
            q.tail = total;
        } else if (g2 >= 2) {
            const int full = total / g2, rem = total - full * g2;
            if (rem > 0 && rem <= g2 / 2) {
                grid = g2;
                q.rounds = full;
                q.tail = rem;
            }
        }
    }
    // Fewer tiles than SMs, x tiles of at most 128 rows (two accumulators,
    // room for two partial tiles in the idle rings): a clustered K split
    // when its longest run of stages, plus its fixed cost, is shorter than
    // the plan above.  The clusters must all be resident at once.
    q.cl_ctas = q.cl_tiles = 0;
    const bool cl_room = pl.BM <= 128 && q.off_bar >= (uint32_t)(2 * pl.BM * 128 * 4);
    auto cl_valid = [&](int C, int T) {
        const int clusters = (total + T - 1) / T;
        const int last = total - (clusters - 1) * T;
        // all clusters resident at once; every CTA gets a run
        return clusters <= tc_active_clusters()[C] && last * (q.G / 4) >= C;
    };
    if (cl_room && total < num_sms()) {
        const int G = q.G;
        int best = q.rounds * G + (q.tail > 0 ? G / 2 : 0);
        for (int C = 2; C <= 8; ++C) {
            for (int T = 1; T < C; ++T) {
                if (!cl_valid(C, T)) continue;
                const int cost = 4 * ((T * (G / 4) + C - 1) / C) + cluster_split_stages(T);
                if (cost < best) {
                    best = cost;
                    q.cl_ctas = C;
                    q.cl_tiles = T;
                }
            }
        }
    }
#ifdef AQ_TEST_HOOKS
    if (g_test_cluster_split < 0) {
        q.cl_ctas = q.cl_tiles = 0;
    } else if (g_test_cluster_split > 0) {
        const int C = g_test_cluster_split >> 8, T = g_test_cluster_split & 255;
        if (cl_room && C >= 2 && C <= 8 && T >= 1 && T < C && cl_valid(C, T)) {
            q.cl_ctas = C;
            q.cl_tiles = T;
        }
    }
#endif
    {
        if (q.cl_ctas > 0) {
            q.rounds = 0;
            q.tail = 0;
            grid = (total + q.cl_tiles - 1) / q.cl_tiles * q.cl_ctas;
        }
    }
    pl.grid = grid;
    return true;
}

template <int B, bool BF16, int BM, bool GEN>
cudaError_t tc_launch_t(const TcPlan &pl, const CUtensorMap &tm, cudaStream_t stream) {
    auto kern = tc_kernel<B, BF16, BM, GEN>;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)kSmemLimitTc);
    });
    if (attr_err != cudaSuccess) return attr_err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)pl.grid, 1, 1);
    cfg.blockDim = dim3(kThreadsTc, 1, 1);
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = pl.prm.cl_ctas > 0 ? (unsigned)pl.prm.cl_ctas
                                                   : pl.prm.tail > 0 ? 2u : 1u;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, pl.prm, tm);
}

template <int B, bool BF16>
cudaError_t tc_launch_bm(const TcPlan &pl, const CUtensorMap &tm, cudaStream_t s) {
    switch (pl.BM) {
        case 64: return tc_launch_t<B, BF16, 64, false>(pl, tm, s);
        case 128: return tc_launch_t<B, BF16, 128, false>(pl, tm, s);
        case 256: return tc_launch_t<B, BF16, 256, false>(pl, tm, s);
        default: return tc_launch_t<B, BF16, 512, false>(pl, tm, s);
    }
}

// General-width path: x tiles of 64, 128 or 256 rows.
template <int B, bool BF16>
cudaError_t tc_launch_g_bm(const TcPlan &pl, const CUtensorMap &tm, cudaStream_t s) {
    switch (pl.BM) {
        case 64: return tc_launch_t<B, BF16, 64, true>(pl, tm, s);
        case 128: return tc_launch_t<B, BF16, 128, true>(pl, tm, s);
        default: return tc_launch_t<B, BF16, 256, true>(pl, tm, s);
    }
}
template <int B>
cudaError_t tc_launch_g_bits(const TcPlan &pl, const CUtensorMap &tm, bool bf16, cudaStream_t s) {
    return bf16 ? tc_launch_g_bm<B, true>(pl, tm, s) : tc_launch_g_bm<B, false>(pl, tm, s);
}

// The swapped-role kernel's plan: 256-row weight tiles; the K range of a
// tile split over S CTAs of a cluster (S <= 8, groups per split a multiple
// of 4) so that tiles x splits covers the SMs.
struct TcwPlan {
    TcwParams prm;
    size_t smem;
    int grid;
};

bool tcw_plan(const MatmulArgs &a, TcwPlan &pl) {
    if (a.K % 512 != 0 || a.M < 1 || a.M > kWXRows || a.N < 1) return false;
    if (a.N > INT32_MAX / 2 || a.K > INT32_MAX / 2) return false;
    TcwParams &q = pl.prm;
    q.M = (int)a.M;
    q.N = (int)a.N;
    q.K = (int)a.K;
    q.G = (int)(a.K / 64);
    const int tiles = (int)((a.N + kWRows - 1) / kWRows);
    int S = std::max(1, std::min(8, num_sms() / tiles));
    int gps = (q.G + S - 1) / S;
    gps = (gps + kGroups - 1) / kGroups * kGroups;
    S = (q.G + gps - 1) / gps;
    q.splits = S;
    q.gps = gps;
    const int raw_slot = a.bits == 4 ? RawW<4>::kSlotBytes : RawW<3>::kSlotBytes;
    size_t off = (size_t)kWStages * (kWATile + kWBTile);
    q.off_raw = (uint32_t)off;
    off += (size_t)kDqWarps * kWRawSlots * raw_slot;
    off = (off + 15) / 16 * 16;
    q.off_bar = (uint32_t)off;
    off += (3 * kWStages + 2) * 8 + 16;
    pl.smem = off + 1024;  // room to align the base to 1024 bytes
    if (pl.smem > kSmemLimitTc) return false;
    if ((size_t)kWXRows * kWPitch * 4 > (size_t)kWStages * (kWATile + kWBTile)) return false;
    q.Wq = a.Wq;
    q.scales = static_cast<const __half *>(a.scales);
    q.biases = static_cast<const __half *>(a.biases);
    q.y = a.out;
    pl.grid = tiles * S;
    return true;
}

template <int B, bool BF16>
cudaError_t tcw_launch_t(const TcwPlan &pl, const CUtensorMap &tm, cudaStream_t stream) {
    auto kern = tcw_kernel<B, BF16>;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)kSmemLimitTc);
    });
    if (attr_err != cudaSuccess) return attr_err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)pl.grid, 1, 1);
    cfg.blockDim = dim3(kThreadsTc, 1, 1);
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)pl.prm.splits;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, pl.prm, tm);
}

}  // namespace

bool tcw_supported(const MatmulArgs &a) {
    if (!aligned(a.x, 16) || !aligned(a.Wq, 16) || !aligned(a.scales, 16) ||
        !aligned(a.biases, 16))
        return false;
    TcwPlan pl;
    return tcw_plan(a, pl);
}

cudaError_t tcw_launch(const MatmulArgs &a) {
    TcwPlan pl;
    if (!tcw_plan(a, pl)) return cudaErrorInvalidValue;
    CUtensorMap tm;
    if (!tmap_2d(&tm, a.dtype == AQ_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                         : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                 a.x, (uint64_t)a.K, (uint64_t)a.M, (uint64_t)a.K * 2, 64u, (uint32_t)kWXRows,
                 CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    if (a.bits == 3)
        return a.dtype == AQ_BF16 ? tcw_launch_t<3, true>(pl, tm, a.stream)
                                  : tcw_launch_t<3, false>(pl, tm, a.stream);
    return a.dtype == AQ_BF16 ? tcw_launch_t<4, true>(pl, tm, a.stream)
                              : tcw_launch_t<4, false>(pl, tm, a.stream);
}

int tcw_describe(const MatmulArgs &a, char *buf, int len) {
    TcwPlan pl;
    if (!tcw_plan(a, pl)) return snprintf(buf, len, "tcw: unsupported");
    return snprintf(buf, len, "tcw tiles=%d splits=%d groups/split=%d grid=%d smem=%zu",
                    pl.grid / pl.prm.splits, pl.prm.splits, pl.prm.gps, pl.grid, pl.smem);
}

bool tc_supported(const MatmulArgs &a) {
    if (!aligned(a.x, 16) || !aligned(a.Wq, 16) || !aligned(a.scales, 16) ||
        !aligned(a.biases, 16))
        return false;
    TcPlan pl;
    return tc_plan(a, pl);
}

static bool tc_x_map(const MatmulArgs &a, const TcPlan &pl, CUtensorMap *tm) {
    return tmap_2d(tm, a.dtype == AQ_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                          : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                   a.x, (uint64_t)a.K, (uint64_t)a.M, (uint64_t)a.K * 2, 64u,
                   (uint32_t)std::min(pl.BM, 256), CU_TENSOR_MAP_SWIZZLE_128B);
}

bool tc_supported_g(const MatmulArgs &a, int group) {
    if (!aligned(a.x, 16) || !aligned(a.Wq, 16) || !aligned(a.scales, 16) ||
        !aligned(a.biases, 16))
        return false;
    TcPlan pl;
    return tc_plan(a, pl, group);
}

cudaError_t tc_launch_g(const MatmulArgs &a, int group) {
    TcPlan pl;
    if (!tc_plan(a, pl, group)) return cudaErrorInvalidValue;
    CUtensorMap tm;
    if (!tc_x_map(a, pl, &tm)) return cudaErrorInvalidValue;
    const bool bf16 = a.dtype == AQ_BF16;
    switch (a.bits) {
        case 2: return tc_launch_g_bits<2>(pl, tm, bf16, a.stream);
        case 3: return tc_launch_g_bits<3>(pl, tm, bf16, a.stream);
        case 4: return tc_launch_g_bits<4>(pl, tm, bf16, a.stream);
        case 5: return tc_launch_g_bits<5>(pl, tm, bf16, a.stream);
        case 6: return tc_launch_g_bits<6>(pl, tm, bf16, a.stream);
        case 8: return tc_launch_g_bits<8>(pl, tm, bf16, a.stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t tc_launch(const MatmulArgs &a) {
    TcPlan pl;
    if (!tc_plan(a, pl)) return cudaErrorInvalidValue;
    CUtensorMap tm;
    if (!tc_x_map(a, pl, &tm)) return cudaErrorInvalidValue;
    if (a.bits == 3)
        return a.dtype == AQ_BF16 ? tc_launch_bm<3, true>(pl, tm, a.stream)
                                  : tc_launch_bm<3, false>(pl, tm, a.stream);
    return a.dtype == AQ_BF16 ? tc_launch_bm<4, true>(pl, tm, a.stream)
                              : tc_launch_bm<4, false>(pl, tm, a.stream);
}

int tc_describe(const MatmulArgs &a, char *buf, int len) {
    TcPlan pl;
    if (!tc_plan(a, pl)) return snprintf(buf, len, "tc: unsupported");
    return snprintf(buf, len,
                    "tc bm=%d a_slots=%d b_slots=%d raw_slots=%d tiles=%dx%d grid=%d rounds=%d "
                    "split=%d cluster_split=%dx%d smem=%zu tmem=%u",
                    pl.BM, a_slots_for(pl.BM), b_slots_for(pl.BM), raw_slots_for(pl.BM),
                    pl.prm.n_tiles, pl.prm.m_tiles, pl.grid,
                    pl.prm.rounds, pl.prm.tail, pl.prm.cl_ctas, pl.prm.cl_tiles, pl.smem,
                    pl.prm.tmem_cols);
}

#ifdef AQ_TEST_HOOKS
const int *tc_active_clusters_for_tests() { return tc_active_clusters(); }
#endif

cudaError_t tc_read_error(uint32_t *code, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(code, g_tc_error, sizeof(uint32_t));
    if (e != cudaSuccess || !clear) return e;
    const uint32_t zero = 0;
    return cudaMemcpyToSymbol(g_tc_error, &zero, sizeof(uint32_t));
}

}  // namespace aq
