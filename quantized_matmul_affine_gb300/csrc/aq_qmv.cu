// Small-M kernel ("qmv"): y = x . W^T for up to 32 activation rows per launch
// block, streaming the packed weights once per call.
//
// Method (mlx-bun pages, @mlx-bun/inference 1.0.0, kernels/quantization/):
//   * the weight format: 64-value groups, 2*B uint32 words each, LSB-first
//     codes (affine-split-mma.ts affine_unit; affine3/4-mma.ts);
//   * the factored form of the group dot product used by affine3-rows.ts /
//     affine4-rows.ts: sum_g [ scale_g * sum_k q_k x_k + bias_g * sum_k x_k ],
//     each weight decoded once and reused for every activation row;
//   * the K-permuted operand layout of affine{3,4}-mma.ts (any permutation
//     of k inside a group works, provided x is permuted the same way);
//   * a deterministic split-K sum in a fixed order (affine-split-mma.ts adds
//     its SPLITS partial tiles in index order, no atomics).
//
// GB300 design:
//   * A CTA is eight warps covering rt tiles of 16 weight rows, kw = 8/rt
//     warps per tile splitting the CTA's K stages (512 K-values, 8 groups,
//     each).  Every warp streams its tile's rows through its own two-stage
//     ring in shared memory with 16-byte cp.async copies (coalesced rows),
//     queuing the next stage before it waits on the current one.  There is
//     no cross-warp hand-off in the main loop.
//   * All warps share the CTA's K range, so x is prepared once per CTA:
//     permuted into MMA B-fragment order (fp16, pre-scaled per k as below)
//     with per-group sums of x, in shared memory.  The kw partial tiles of a
//     tile are added in warp order at the end.
//   * Codes decode straight into fp16 MMA A-fragments: a code masked in place
//     inside an fp16 whose exponent field is zero is the exact subnormal
//     q * 2^(p-24) (p = its bit position in the half), so decoding is one AND
//     per two codes plus a shift or byte permute per word.  x is pre-scaled
//     by 2^-p for the matching k, making every product q * x * 2^-24 exact;
//     the group's scale is applied to the fp32 result as scale * 2^24.  bf16
//     x is converted to fp16 once per CTA with a per-row power-of-two scale
//     that keeps it inside the fp16 range.
//   * mma.sync m16n8k16 (fp16 in, fp32 accumulate) does the multiply-adds.
//     Each thread holds 16 consecutive codes of a group for two rows, so an
//     MMA k-step never mixes groups; the 8 groups of a stage are independent
//     MMA chains.
//   * Narrow outputs split K over the CTAs of a thread-block cluster; their
//     partial tiles meet in distributed shared memory and are added in rank
//     order (deterministic).
#include "aq_internal.h"
#include "aq_ptx.cuh"

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdio>
#include <mutex>
#include <type_traits>

namespace aq {

__device__ uint32_t g_qmv_error;

namespace {

constexpr int kWarps = 8;               // warps per CTA
constexpr int kThreads = kWarps * 32;
constexpr int kGroupsPerStage = 8;      // 512 values of K per stage
constexpr int kMaxCluster = 16;

template <int B>
struct Fmt {
    static constexpr int kGroupBytes = 8 * B;                             // 2*B words
    static constexpr int kRowStageBytes = kGroupsPerStage * kGroupBytes;  // 256 / 192
    static constexpr int kChunksPerRow = kRowStageBytes / 16;             // 16 / 12
    // Row pitch in a stage, padded so that the eight rows an MMA reads at
    // once start in different bank groups.
    static constexpr int kRowPitch = kRowStageBytes + (B == 4 ? 32 : 16);
    static constexpr int kScalesOff = 16 * kRowPitch;  // then scales[16][8], biases[16][8]
    static constexpr int kStageBytes = kScalesOff + 2 * 16 * 16;
};

struct Params {
    const void *x;
    const uint32_t *Wq;
    const __half *scales;
    const __half *biases;
    void *y;
    int64_t M, N, K;
    int G;             // groups per row
    int stages_total;  // K / 512
    int ks;            // CTAs per cluster splitting K
    int rt;            // 16-row tiles per CTA
    int kw;            // warps sharing one tile (splitting the CTA's stages)
    int mc;            // activation rows per launch block (8*MB)
    int slots;         // ring depth per warp (stages; slots-1 in flight while computing)
    uint32_t xpitch;   // bytes per activation row of x fragments
    uint32_t off_xfrag, off_xs, off_scale, off_red, off_partial;
};

// Pair i of the 8 fp16 pairs decoded from a thread's 16 codes holds codes
// (lo, hi) at bit position p within each half (see decode4 / decode3).
template <int B>
struct PairMap;
template <>
struct PairMap<4> {
    static constexpr __device__ int lo(int i) { return i < 4 ? i : i + 4; }
    static constexpr __device__ int hi(int i) { return lo(i) + 4; }
    static constexpr __device__ int p(int i) { return (i & 1) ? 4 : 0; }
};
template <>
struct PairMap<3> {
    static constexpr __device__ int lo(int i) { return i; }
    static constexpr __device__ int hi(int i) { return i + 8; }
    // positions 0,3,6,0,3,0,3,6
    static constexpr __device__ int p(int i) {
        return (i == 2 || i == 7) ? 6 : (i == 1 || i == 4 || i == 6) ? 3 : 0;
    }
};

// A-fragment registers of the four MMA k-steps of one group: step s takes
// pairs 2s and 2s+1 of the row-g codes (PA) and of the row-(g+8) codes (PB)
// as {PA[2s], PB[2s], PA[2s+1], PB[2s+1]}.
__device__ __forceinline__ void to_frags(const uint32_t (&PA)[8], const uint32_t (&PB)[8],
                                         uint32_t (&a)[4][4]) {
#pragma unroll
    for (int s = 0; s < 4; ++s) {
        a[s][0] = PA[2 * s];
        a[s][1] = PB[2 * s];
        a[s][2] = PA[2 * s + 1];
        a[s][3] = PB[2 * s + 1];
    }
}

// 4-bit: words w0 (codes 0..7) and w1 (codes 8..15).  Masking nibble pairs
// (j, j+4) in place gives two fp16 subnormals per AND.
__device__ __forceinline__ void decode4(uint32_t w0, uint32_t w1, uint32_t (&P)[8]) {
    const uint32_t v0 = w0 >> 8, v1 = w1 >> 8;
    P[0] = w0 & 0x000F000Fu;  // codes 0,4   at p=0
    P[1] = w0 & 0x00F000F0u;  // codes 1,5   at p=4
    P[2] = v0 & 0x000F000Fu;  // codes 2,6   at p=0
    P[3] = v0 & 0x00F000F0u;  // codes 3,7   at p=4
    P[4] = w1 & 0x000F000Fu;  // codes 8,12
    P[5] = w1 & 0x00F000F0u;  // codes 9,13
    P[6] = v1 & 0x000F000Fu;  // codes 10,14
    P[7] = v1 & 0x00F000F0u;  // codes 11,15
}

// 3-bit: the thread's 48-bit span (16 codes, code j at bit 3j) sits in words
// (wa, wb) starting at byte bo in {0, 2}.  r0 = span bytes [0,1,3,4] puts
// codes 0..4 in the low half and 8..12 in the high half, both starting at
// bit 0 of their half; r2 = span bytes [1,2,4,5] does the same for codes
// 5..7 and 13..15 after a shift by 7.
__device__ __forceinline__ void decode3(uint32_t wa, uint32_t wb, uint32_t sel0, uint32_t sel2,
                                        uint32_t (&P)[8]) {
    const uint32_t r0 = prmt(wa, wb, sel0);
    const uint32_t r2 = prmt(wa, wb, sel2);
    const uint32_t r1 = r0 >> 9;
    const uint32_t r3 = r2 >> 7;
    P[0] = r0 & 0x00070007u;  // codes 0,8   p=0
    P[1] = r0 & 0x00380038u;  // codes 1,9   p=3
    P[2] = r0 & 0x01C001C0u;  // codes 2,10  p=6
    P[3] = r1 & 0x00070007u;  // codes 3,11  p=0
    P[4] = r1 & 0x00380038u;  // codes 4,12  p=3
    P[5] = r3 & 0x00070007u;  // codes 5,13  p=0
    P[6] = r3 & 0x00380038u;  // codes 6,14  p=3
    P[7] = r3 & 0x01C001C0u;  // codes 7,15  p=6
}

template <typename T>
__device__ __forceinline__ void store_out(T *p, float v);
template <>
__device__ __forceinline__ void store_out<__half>(__half *p, float v) { *p = __float2half_rn(v); }
template <>
__device__ __forceinline__ void store_out<__nv_bfloat16>(__nv_bfloat16 *p, float v) {
    *p = __float2bfloat16_rn(v);
}

__device__ __forceinline__ float half_lo(uint32_t v) {
    return __half2float(__ushort_as_half((unsigned short)(v & 0xFFFFu)));
}
__device__ __forceinline__ float half_hi(uint32_t v) {
    return __half2float(__ushort_as_half((unsigned short)(v >> 16)));
}
// element j (0..7) of 8 halves held in a uint4
__device__ __forceinline__ float half_at(const uint4 &v, int j) {
    const uint32_t w = j < 2 ? v.x : j < 4 ? v.y : j < 6 ? v.z : v.w;
    return (j & 1) ? half_hi(w) : half_lo(w);
}

}  // namespace

template <int B, typename T, int MB>
__global__ void __launch_bounds__(kThreads, 2) qmv_kernel(const __grid_constant__ Params prm) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int MCP = 8 * MB;  // padded activation rows per launch block
    using F = Fmt<B>;
    constexpr int kChunks = F::kChunksPerRow / 2;  // 16-byte copies per lane per stage

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int ct = threadIdx.x;
    const int ks = prm.ks, kw = prm.kw, rt = prm.rt;
    const int tile = blockIdx.x / ks;  // CTA row block: rt tiles of 16 rows
    const int rank = blockIdx.x % ks;
    const int wt = warp / kw;          // this warp's tile within the CTA
    const int kslot = warp % kw;       // this warp's share of the CTA's stages
    const int64_t nb = (int64_t)tile * 16 * rt;  // first row of the CTA
    const int64_t m0 = (int64_t)blockIdx.y * prm.mc;
    const int Mc = (int)min((int64_t)prm.mc, prm.M - m0);
    const int st_begin = (int)((int64_t)prm.stages_total * rank / ks);
    const int st_end = (int)((int64_t)prm.stages_total * (rank + 1) / ks);
    const int nst = st_end - st_begin;                          // stages of the CTA
    const int nw = kslot < nst ? (nst - kslot + kw - 1) / kw : 0;  // stages of this warp
    const int gb = st_begin * kGroupsPerStage;
    const int gcta = nst * kGroupsPerStage;

    const int slots = prm.slots;
    uint8_t *ring = smem + (size_t)warp * slots * F::kStageBytes;
    uint8_t *xfrag = smem + prm.off_xfrag;
    float *xs = reinterpret_cast<float *>(smem + prm.off_xs);
    float *escale = reinterpret_cast<float *>(smem + prm.off_scale);  // [MCP] x multiplier
    float *oscale = escale + MCP;                                     // [MCP] y multiplier
    unsigned *amax = reinterpret_cast<unsigned *>(oscale + MCP);      // [MCP]
    float *red = reinterpret_cast<float *>(smem + prm.off_red);
    float *partial = reinterpret_cast<float *>(smem + prm.off_partial);

    // ----------------------------------------------------------------------
    // Copy plan of this lane: kChunks 16-byte pieces of the warp's 16 rows
    // per stage, plus one scale or bias row.  A row past N is read from row
    // N-1 instead: it only feeds output rows that are never stored.
    // ----------------------------------------------------------------------
    const int64_t wrow0 = nb + 16 * wt;
    const int64_t row_bytes = prm.K * B / 8;
    const int64_t nlast = prm.N - 1;
    uint32_t soff[kChunks], doff[kChunks];
#pragma unroll
    for (int i = 0; i < kChunks; ++i) {
        const int c = lane + 32 * i;
        const int r = c / F::kChunksPerRow, col = c % F::kChunksPerRow;
        const int64_t n = min(wrow0 + r, nlast) - min(wrow0, nlast);
        soff[i] = (uint32_t)(n * row_bytes + col * 16);
        doff[i] = (uint32_t)(r * F::kRowPitch + col * 16);
    }
    const uint8_t *wbase = reinterpret_cast<const uint8_t *>(prm.Wq) + min(wrow0, nlast) * row_bytes;
    const int sbr = lane & 15;
    const __half *sbbase = ((lane < 16) ? prm.scales : prm.biases) + min(wrow0 + sbr, nlast) * prm.G;
    const uint32_t sbdoff = F::kScalesOff + (lane >> 4) * 256 + sbr * 16;
    auto issue = [&](int i, int slot) {
        const int s = kslot + i * kw;  // stage within the CTA range
        const int gs = gb + s * kGroupsPerStage;
        uint8_t *dst = ring + slot * F::kStageBytes;
        const uint8_t *src = wbase + (int64_t)gs * F::kGroupBytes;
#pragma unroll
        for (int c = 0; c < kChunks; ++c) cp_async16(dst + doff[c], src + soff[c], 16u);
        cp_async16(dst + sbdoff, sbbase + gs, 16u);
    };
    // The weights do not depend on earlier kernels in the stream: their first
    // stages are queued before waiting for the preceding grid, and the next
    // kernel may launch as soon as every CTA of this one is running.
    for (int i = 0; i < slots - 1; ++i) {
        if (i < nw) issue(i, i);
        cp_async_commit();
    }
    launch_dependents();
    grid_dependency_wait();  // x and y belong to the stream order
    // Raw x of this CTA's K range goes to the fragment rows (one more group
    // of copies).
    {
        const T *xg = static_cast<const T *>(prm.x);
        const int per_row = gcta * 8;  // 16-byte chunks per activation row
        for (int c = ct; c < Mc * per_row; c += kThreads) {
            const int m = c / per_row, q = c - m * per_row;
            cp_async16(xfrag + (size_t)m * prm.xpitch + q * 16,
                       xg + (m0 + m) * prm.K + 64 * gb + 8 * q, 16u);
        }
        cp_async_commit();
    }

    // ----------------------------------------------------------------------
    // Prologue (all threads): once the raw x has landed, rewrite it in place
    // into B-fragment order and take per-group sums of x (times 2^-24, the
    // scale of the MMA products).  The four quarters of a group belong to
    // four adjacent lanes, which read the whole group before any writes.
    // ----------------------------------------------------------------------
    if (ct < MCP) {
        escale[ct] = 1.f;
        oscale[ct] = 16777216.f;
        amax[ct] = 0u;
    }
    cp_async_wait<0>();  // x (the youngest group) and the first weight stages
    __syncthreads();
    if constexpr (std::is_same<T, __nv_bfloat16>::value) {
        // Largest |x| per activation row over this CTA's K range; pick 2^-e
        // so that the fp16 copy stays below 2^15 in magnitude.
        for (int m = 0; m < Mc; ++m) {
            const uint4 *row = reinterpret_cast<const uint4 *>(xfrag + (size_t)m * prm.xpitch);
            unsigned a = 0u;  // max of |x| as bits (bf16 in the high half)
            for (int c = ct; c < gcta * 8; c += kThreads) {
                const uint4 v = row[c];
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    a = max(a, (w[i] << 16) & 0x7FFF0000u);
                    a = max(a, w[i] & 0x7FFF0000u);
                }
            }
#pragma unroll
            for (int d = 16; d >= 1; d >>= 1) a = max(a, __shfl_xor_sync(0xffffffffu, a, d));
            if (lane == 0) atomicMax(&amax[m], a);
        }
        __syncthreads();
        if (ct < Mc) {
            const int e = (int)((amax[ct] >> 23) & 0xFF) - 127;  // floor(log2 amax)
            const int sh = e > 14 ? e - 14 : 0;
            escale[ct] = __int_as_float((127 - sh) << 23);
            oscale[ct] = __int_as_float((127 + 24 + sh) << 23);
        }
        __syncthreads();
    }
    for (int m = 0; m < Mc; ++m) {
        uint8_t *xrowp = xfrag + (size_t)m * prm.xpitch;
        const float es = escale[m];
        for (int vb = 0; vb < gcta * 4; vb += kThreads) {
            const int v = vb + ct;  // (group j, quarter t) of row m
            const bool valid = v < gcta * 4;
            const int j = v >> 2, t = v & 3;
            float f[16];
            if (valid) {
                const uint4 *src = reinterpret_cast<const uint4 *>(xrowp + 32 * v);
                const uint4 u0 = src[0], u1 = src[1];
                const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    if constexpr (std::is_same<T, __half>::value) {
                        const float2 fv = __half22float2(*reinterpret_cast<const __half2 *>(&w[i]));
                        f[2 * i] = fv.x;
                        f[2 * i + 1] = fv.y;
                    } else {
                        f[2 * i] = __uint_as_float(w[i] << 16);
                        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
                    }
                }
            } else {
#pragma unroll
                for (int i = 0; i < 16; ++i) f[i] = 0.f;
            }
            float sum = 0.f;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                f[i] *= es;
                sum += f[i];
            }
            sum += __shfl_xor_sync(0xffffffffu, sum, 1);
            sum += __shfl_xor_sync(0xffffffffu, sum, 2);
            __syncwarp();  // the group's four quarters are read before they are overwritten
            if (valid) {
                uint32_t pr[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float sc = __int_as_float((127 - PairMap<B>::p(i)) << 23);  // 2^-p
                    pr[i] = pack_half2(f[PairMap<B>::lo(i)] * sc, f[PairMap<B>::hi(i)] * sc);
                }
                uint4 *dst = reinterpret_cast<uint4 *>(xrowp) + j * 8 + t;
                dst[0] = make_uint4(pr[0], pr[1], pr[2], pr[3]);
                dst[4] = make_uint4(pr[4], pr[5], pr[6], pr[7]);
                if (t == 0) xs[j * MCP + m] = sum * 5.9604644775390625e-08f;  // * 2^-24
            }
        }
    }
    for (int u = ct; u < gcta * MCP; u += kThreads)
        if (u % MCP >= Mc) xs[u] = 0.f;
    __syncthreads();

    // ----------------------------------------------------------------------
    // Main loop: the warp's 16 rows over its stages.  The next stage is
    // queued before waiting on the current one.
    // ----------------------------------------------------------------------
    const int g = lane >> 2, t = lane & 3;
    uint32_t sel0 = 0, sel2 = 0;
    int wi3 = 0;
    if constexpr (B == 3) {
        const uint32_t bo = 2u * (uint32_t)(t & 1);
        sel0 = (bo + 0) | ((bo + 1) << 4) | ((bo + 3) << 8) | ((bo + 4) << 12);
        sel2 = (bo + 1) | ((bo + 2) << 4) | ((bo + 4) << 8) | ((bo + 5) << 12);
        wi3 = (3 * t) >> 1;
    }
    float acc[MB][4];
#pragma unroll
    for (int mb = 0; mb < MB; ++mb)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[mb][i] = 0.f;

    // x-fragment rows of this lane, clamped to the valid rows: a lane whose
    // activation row does not exist reads row Mc-1 instead, which only feeds
    // output columns that are never stored (MMA columns are independent).
    const uint8_t *xrow[MB];
#pragma unroll
    for (int mb = 0; mb < MB; ++mb)
        xrow[mb] = xfrag + (size_t)min(mb * 8 + g, Mc - 1) * prm.xpitch + 16 * t;
    // this lane's first code word of row g in a stage
    const int wlane_off = g * F::kRowPitch + (B == 4 ? 8 * t : 4 * wi3);

    for (int i = 0; i < nw; ++i) {
        if (i + slots - 1 < nw) issue(i + slots - 1, (i + slots - 1) % slots);
        cp_async_commit();
        // stage i has landed once at most slots-1 younger groups are pending
        switch (slots) {
            case 2: cp_async_wait<1>(); break;
            case 3: cp_async_wait<2>(); break;
            case 4: cp_async_wait<3>(); break;
            case 5: cp_async_wait<4>(); break;
            default: cp_async_wait<5>(); break;
        }
        __syncwarp();
        const uint8_t *sb = ring + (i % slots) * F::kStageBytes;
        const int s = kslot + i * kw;
        const uint4 sA = *reinterpret_cast<const uint4 *>(sb + F::kScalesOff + g * 16);
        const uint4 sB = *reinterpret_cast<const uint4 *>(sb + F::kScalesOff + (g + 8) * 16);
        const uint4 bA = *reinterpret_cast<const uint4 *>(sb + F::kScalesOff + 256 + g * 16);
        const uint4 bB = *reinterpret_cast<const uint4 *>(sb + F::kScalesOff + 256 + (g + 8) * 16);
        const uint8_t *wa = sb + wlane_off;
        const uint8_t *xst[MB];
#pragma unroll
        for (int mb = 0; mb < MB; ++mb) xst[mb] = xrow[mb] + (size_t)s * kGroupsPerStage * 128;
        const float *xss = xs + s * kGroupsPerStage * MCP + 2 * t;
#pragma unroll
        for (int j = 0; j < kGroupsPerStage; ++j) {
            uint32_t PA[8], PB[8];
            if constexpr (B == 4) {
                const uint2 qa = *reinterpret_cast<const uint2 *>(wa + j * F::kGroupBytes);
                const uint2 qb =
                    *reinterpret_cast<const uint2 *>(wa + 8 * F::kRowPitch + j * F::kGroupBytes);
                decode4(qa.x, qa.y, PA);
                decode4(qb.x, qb.y, PB);
            } else {
                const uint32_t *pa = reinterpret_cast<const uint32_t *>(wa + j * F::kGroupBytes);
                const uint32_t *pb =
                    reinterpret_cast<const uint32_t *>(wa + 8 * F::kRowPitch + j * F::kGroupBytes);
                decode3(pa[0], pa[1], sel0, sel2, PA);
                decode3(pb[0], pb[1], sel0, sel2, PB);
            }
            uint32_t a[4][4];
            to_frags(PA, PB, a);
            const float sa = half_at(sA, j), sbb = half_at(sB, j);
            const float ba = half_at(bA, j), bb = half_at(bB, j);
#pragma unroll
            for (int mb = 0; mb < MB; ++mb) {
                const uint4 q0 = *reinterpret_cast<const uint4 *>(xst[mb] + j * 128);
                const uint4 q1 = *reinterpret_cast<const uint4 *>(xst[mb] + j * 128 + 64);
                const float2 xv = *reinterpret_cast<const float2 *>(&xss[j * MCP + mb * 8]);
                float d[4] = {0.f, 0.f, 0.f, 0.f};
                mma_f16_16816(d, a[0], q0.x, q0.y, d);
                mma_f16_16816(d, a[1], q0.z, q0.w, d);
                mma_f16_16816(d, a[2], q1.x, q1.y, d);
                mma_f16_16816(d, a[3], q1.z, q1.w, d);
                acc[mb][0] = fmaf(sa, d[0], fmaf(ba, xv.x, acc[mb][0]));
                acc[mb][1] = fmaf(sa, d[1], fmaf(ba, xv.y, acc[mb][1]));
                acc[mb][2] = fmaf(sbb, d[2], fmaf(bb, xv.x, acc[mb][2]));
                acc[mb][3] = fmaf(sbb, d[3], fmaf(bb, xv.y, acc[mb][3]));
            }
        }
        __syncwarp();
    }
    cp_async_wait<0>();

    // ----------------------------------------------------------------------
    // Epilogue: add the kw warps of each tile in warp order, then write y
    // (or this CTA's partial tile when K is split over a cluster).
    // ----------------------------------------------------------------------
#pragma unroll
    for (int mb = 0; mb < MB; ++mb)
        *reinterpret_cast<float4 *>(&red[((warp * MB + mb) * 32 + lane) * 4]) =
            make_float4(acc[mb][0], acc[mb][1], acc[mb][2], acc[mb][3]);
    __syncthreads();
    T *y = static_cast<T *>(prm.y);
    for (int e = ct; e < rt * MB * 128; e += kThreads) {
        const int tl = e / (MB * 128), rem = e % (MB * 128);
        const int mb = rem / 128, ln = (rem / 4) % 32, i = rem % 4;
        float v = 0.f;
        for (int k = 0; k < kw; ++k) v += red[(((tl * kw + k) * MB + mb) * 32 + ln) * 4 + i];
        const int row = 16 * tl + (ln >> 2) + 8 * (i >> 1);
        const int col = mb * 8 + 2 * (ln & 3) + (i & 1);
        v *= oscale[col];
        if (ks == 1) {
            if (col < Mc && nb + row < prm.N) store_out<T>(&y[(m0 + col) * prm.N + nb + row], v);
        } else {
            partial[row * MCP + col] = v;
        }
    }
    if (ks > 1) {
        // Split-K: CTA `rank` adds element e (e % ks == rank) over all ranks
        // of the cluster, rank 0 first.
        cluster_sync();
        const uint32_t base = smem_u32(partial);
        for (int e = rank + ks * ct; e < 16 * rt * MCP; e += ks * kThreads) {
            const int row = e / MCP, col = e % MCP;
            if (col >= Mc || nb + row >= prm.N) continue;
            float v = 0.f;
            for (int r = 0; r < ks; ++r)
                v += ld_dsmem_f32(map_to_rank(base + 4u * (uint32_t)e, (uint32_t)r));
            store_out<T>(&y[(m0 + col) * prm.N + nb + row], v);
        }
        cluster_sync();
    }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
namespace {

struct Plan {
    int MB, ks, rt, kw, mc, m_chunks, blocks;
    size_t smem;
    Params prm;
};

constexpr size_t kSmemLimit = 227 * 1024;

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct Layout {
    size_t smem;
    uint32_t xpitch, off_xfrag, off_xs, off_scale, off_red, off_partial;
};

Layout layout(int B, int MB, int mc_valid, int st_cta, int rt, int ks, int slots) {
    Layout L;
    const int mc = 8 * MB;
    const int stage_bytes = B == 4 ? Fmt<4>::kStageBytes : Fmt<3>::kStageBytes;
    size_t off = (size_t)kWarps * slots * stage_bytes;
    off = align_up(off, 128);
    L.off_xfrag = (uint32_t)off;
    const size_t gmax = (size_t)st_cta * kGroupsPerStage;
    // one row of fragments per activation row; the 64-byte pad puts
    // consecutive rows in different halves of the banks
    L.xpitch = (uint32_t)(gmax * 128 + 64);
    off += (size_t)L.xpitch * mc_valid;
    off = align_up(off, 128);
    L.off_xs = (uint32_t)off;
    off += gmax * mc * 4;
    off = align_up(off, 128);
    L.off_scale = (uint32_t)off;
    off += 3 * mc * 4;
    off = align_up(off, 128);
    L.off_red = (uint32_t)off;
    off += (size_t)kWarps * MB * 128 * 4;
    L.off_partial = (uint32_t)off;
    off += ks > 1 ? (size_t)16 * rt * mc * 4 : 0;
    L.smem = align_up(off, 128);
    return L;
}

std::atomic<int> g_force_rt{0}, g_force_ks{0}, g_force_slots{0};

// Measured geometry for the benchmarked shapes: the fastest (rows per CTA,
// cluster split, ring depth) of a sweep of every combination on GB300, with
// programmatic dependent launch between consecutive calls.
struct TunedShape {
    int bits, N, K, MB;
    int rt, ks, slots;
};
constexpr TunedShape kTuned[] = {
    {4, 4096, 4096, 1, 1, 1, 2},    // decode 4.78 us
    {4, 1024, 512, 1, 1, 1, 2},     // small 2.22 us
    {3, 10240, 5120, 1, 8, 3, 3},   // 3-bit M=1 12.3 us
    {3, 10240, 5120, 2, 8, 1, 3},   // 3-bit M=9..16 (K split grows if x does not fit)
    {4, 5120, 5120, 1, 4, 3, 2},    // q/o projections 7.6 us
    {4, 1024, 5120, 1, 1, 1, 3},    // k/v projections 3.7 us
    {4, 13824, 5120, 1, 4, 1, 2},   // gate/up 12.0 us
    {4, 5120, 13824, 1, 4, 3, 2},   // down 12.5 us
};

// Pick the CTA shape (rt row tiles x kw K-ways, rt*kw = 8 warps), the
// cluster split ks and the ring depth.  Shapes in kTuned use their measured
// geometry.  Otherwise, from the same sweeps: with consecutive calls
// overlapping, the best launches fill about 1.6 CTAs per SM in one resident
// wave (at most 2 per SM), and each extra cluster CTA costs about as much as
// being 30% off that target; among equal scores the larger row block wins.
bool make_plan(const MatmulArgs &a, Plan &p) {
    const int B = a.bits;
    if (a.K % 512 != 0 || a.M < 1 || a.N < 1) return false;
    p.MB = a.M > 16 ? 4 : a.M > 8 ? 2 : 1;
    p.mc = 8 * p.MB;
    p.m_chunks = (int)((a.M + p.mc - 1) / p.mc);
    if (p.m_chunks > 65535) return false;
    const int64_t tiles16 = (a.N + 15) / 16;
    const int S = (int)(a.K / 512);
    const int mc_valid = (int)std::min<int64_t>(a.M, p.mc);
    if (16 * (a.K * B / 8) >= ((int64_t)1 << 31)) return false;  // 32-bit copy offsets
    const int sms = num_sms();
    const int frt = g_force_rt.load(), fks = g_force_ks.load(), fsl = g_force_slots.load();

    int rt = 1, ks = 1, want_slots = 2;
    bool tuned = false;
    for (const TunedShape &t : kTuned)
        if (t.bits == B && t.N == a.N && t.K == a.K && t.MB == p.MB) {
            rt = t.rt;
            ks = t.ks;
            want_slots = t.slots;
            tuned = true;
        }
    if (!tuned) {
        const double target = 1.6 * sms;
        double best = 1e30;
        for (int r = kWarps; r >= 1; r /= 2) {
            const int64_t blocks = (tiles16 + r - 1) / r;
            for (int k = 1; k <= std::min(S, kMaxCluster); ++k) {
                const int64_t ctas = blocks * k * p.m_chunks;
                if (ctas > 2 * (int64_t)sms && !(k == 1 && r == kWarps)) continue;
                const double score = std::fabs((double)ctas - target) / target + 0.3 * (k - 1);
                if (score < best - 1e-9) {
                    best = score;
                    rt = r;
                    ks = k;
                }
            }
        }
    }
    if (frt) rt = frt;
    if (fks) ks = fks;
    if (fsl) want_slots = fsl;
    ks = std::max(1, std::min({ks, S, kMaxCluster}));
    const int kw = kWarps / rt;
    const int64_t blocks = (tiles16 + rt - 1) / rt;
    if (blocks * ks > (int64_t)INT32_MAX) return false;

    bool found = false;
    // the x fragments of the CTA's K range must fit: grow ks until they do
    for (; ks <= std::min(S, kMaxCluster) && !found; ++ks) {
        const int st_cta = (S + ks - 1) / ks;
        const int per_warp_st = (st_cta + kw - 1) / kw;
        int slots = std::max(2, std::min(want_slots, per_warp_st + 1));
        Layout L = layout(B, p.MB, mc_valid, st_cta, rt, ks, slots);
        while (L.smem > kSmemLimit && slots > 2)
            L = layout(B, p.MB, mc_valid, st_cta, rt, ks, --slots);
        if (L.smem > kSmemLimit || (L.off_scale - L.off_xfrag) > 120 * 1024) {
            if (fks) break;
            continue;
        }
        found = true;
        p.rt = rt;
        p.kw = kw;
        p.ks = ks;
        p.prm.slots = slots;
        p.blocks = (int)blocks;
        p.smem = L.smem;
        p.prm.xpitch = L.xpitch;
        p.prm.off_xfrag = L.off_xfrag;
        p.prm.off_xs = L.off_xs;
        p.prm.off_scale = L.off_scale;
        p.prm.off_red = L.off_red;
        p.prm.off_partial = L.off_partial;
    }
    if (!found) return false;
    Params &q = p.prm;
    q.x = a.x;
    q.Wq = a.Wq;
    q.scales = static_cast<const __half *>(a.scales);
    q.biases = static_cast<const __half *>(a.biases);
    q.y = a.out;
    q.M = a.M;
    q.N = a.N;
    q.K = a.K;
    q.G = (int)(a.K / 64);
    q.stages_total = S;
    q.ks = p.ks;
    q.rt = p.rt;
    q.kw = p.kw;
    q.mc = p.mc;
    return true;
}

template <int B, typename T, int MB>
cudaError_t launch_plan(const Plan &p, cudaStream_t stream) {
    auto kern = qmv_kernel<B, T, MB>;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)kSmemLimit);
        if (attr_err == cudaSuccess)
            attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    });
    if (attr_err != cudaSuccess) return attr_err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(p.blocks * p.ks), (unsigned)p.m_chunks, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int na = 0;
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    if (p.ks > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = (unsigned)p.ks;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, kern, p.prm);
}

template <int B, typename T>
cudaError_t launch_mb(const Plan &p, cudaStream_t s) {
    switch (p.MB) {
        case 1: return launch_plan<B, T, 1>(p, s);
        case 2: return launch_plan<B, T, 2>(p, s);
        default: return launch_plan<B, T, 4>(p, s);
    }
}

}  // namespace

bool qmv_supported(const MatmulArgs &a) {
    if (!aligned(a.x, 16) || !aligned(a.Wq, 16) || !aligned(a.scales, 16) ||
        !aligned(a.biases, 16))
        return false;
    Plan p;
    return make_plan(a, p);
}

cudaError_t qmv_launch(const MatmulArgs &a) {
    Plan p;
    if (!make_plan(a, p)) return cudaErrorInvalidValue;
    if (a.bits == 3)
        return a.dtype == AQ_BF16 ? launch_mb<3, __nv_bfloat16>(p, a.stream)
                                  : launch_mb<3, __half>(p, a.stream);
    return a.dtype == AQ_BF16 ? launch_mb<4, __nv_bfloat16>(p, a.stream)
                              : launch_mb<4, __half>(p, a.stream);
}

void qmv_force_geometry(int rt, int ks, int slots) {
    g_force_rt.store(rt);
    g_force_ks.store(ks);
    g_force_slots.store(slots);
}

int qmv_describe(const MatmulArgs &a, char *buf, int len) {
    Plan p;
    if (!make_plan(a, p)) return snprintf(buf, len, "qmv: unsupported");
    return snprintf(buf, len, "qmv rows/cta=%d kways=%d cluster=%d ring=%d grid=%dx%d smem=%zu mb=%d",
                    16 * p.rt, p.kw, p.ks, p.prm.slots, p.blocks * p.ks, p.m_chunks, p.smem, p.MB);
}

cudaError_t qmv_read_error(uint32_t *code, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(code, g_qmv_error, sizeof(uint32_t));
    if (e != cudaSuccess || !clear) return e;
    const uint32_t zero = 0;
    return cudaMemcpyToSymbol(g_qmv_error, &zero, sizeof(uint32_t));
}

}  // namespace aq
