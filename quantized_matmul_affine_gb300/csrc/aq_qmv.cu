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
//   * A CTA is four warps; each warp owns 16 weight rows and streams them,
//     512 K-values (8 groups) per stage, through its own ring of shared-memory
//     stages with 16-byte cp.async copies (coalesced rows).
//     There is no cross-warp hand-off in the main loop: a warp waits only on
//     its own copies.
//   * The four warps share the CTA's K range, so x is prepared once per CTA:
//     permuted into MMA B-fragment order (fp16, pre-scaled per k as below)
//     with per-group sums of x, in shared memory.
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
#include <mutex>
#include <type_traits>

namespace aq {

__device__ uint32_t g_qmv_error;

namespace {

constexpr int kWarps = 4;               // warps per CTA, 16 weight rows each
constexpr int kThreads = kWarps * 32;
constexpr int kRows = 16 * kWarps;      // weight rows per CTA
constexpr int kGroupsPerStage = 8;      // 512 values of K per stage
constexpr int kRing = 3;                // stages per warp ring
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
    int mc;            // activation rows per launch block (8*MB)
    int slots;         // ring slots allocated per warp (<= kRing)
    uint32_t off_xfrag, off_xs, off_scale, off_partial;
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
__device__ __forceinline__ void load16(const T *src, float (&f)[16]) {
    const uint4 u0 = __ldg(reinterpret_cast<const uint4 *>(src));
    const uint4 u1 = __ldg(reinterpret_cast<const uint4 *>(src) + 1);
    const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        if constexpr (std::is_same<T, __half>::value) {
            const float2 v = __half22float2(*reinterpret_cast<const __half2 *>(&w[i]));
            f[2 * i] = v.x;
            f[2 * i + 1] = v.y;
        } else {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    }
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
__global__ void __launch_bounds__(kThreads) qmv_kernel(const __grid_constant__ Params prm) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int MCP = 8 * MB;  // padded activation rows per launch block
    using F = Fmt<B>;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int ct = threadIdx.x;
    const int ks = prm.ks;
    const int tile = blockIdx.x / ks;
    const int rank = blockIdx.x % ks;
    const int64_t n0 = (int64_t)tile * kRows;
    const int64_t m0 = (int64_t)blockIdx.y * prm.mc;
    const int Mc = (int)min((int64_t)prm.mc, prm.M - m0);  // valid activation rows here
    const int st_begin = (int)((int64_t)prm.stages_total * rank / ks);
    const int st_end = (int)((int64_t)prm.stages_total * (rank + 1) / ks);
    const int nst = st_end - st_begin;
    const int gb = st_begin * kGroupsPerStage;  // first group of this CTA
    const int gcta = nst * kGroupsPerStage;     // groups of this CTA

    uint8_t *ring = smem + (size_t)warp * prm.slots * F::kStageBytes;
    uint8_t *xfrag = smem + prm.off_xfrag;
    float *xs = reinterpret_cast<float *>(smem + prm.off_xs);
    float *escale = reinterpret_cast<float *>(smem + prm.off_scale);  // [MCP] x multiplier
    float *oscale = escale + MCP;                                     // [MCP] y multiplier
    unsigned *amax = reinterpret_cast<unsigned *>(oscale + MCP);      // [MCP]
    float *partial = reinterpret_cast<float *>(smem + prm.off_partial);

    // ----------------------------------------------------------------------
    // Stage issue: 16 rows x 8 groups of packed words, plus the rows' 8
    // scales and 8 biases, as 16-byte cp.async copies.
    // ----------------------------------------------------------------------
    const int64_t row_bytes = prm.K * B / 8;
    const int64_t wrow0 = n0 + 16 * warp;  // first weight row of this warp
    const uint8_t *wq8 = reinterpret_cast<const uint8_t *>(prm.Wq);
    auto issue = [&](int s, int slot) {
        uint8_t *dst = ring + slot * F::kStageBytes;
        const int gs = gb + s * kGroupsPerStage;
#pragma unroll
        for (int i = 0; i < F::kChunksPerRow / 2; ++i) {
            const int c = lane + 32 * i;
            const int r = c / F::kChunksPerRow, col = c % F::kChunksPerRow;
            const int64_t n = wrow0 + r;
            const bool ok = n < prm.N;
            const uint8_t *src = ok ? wq8 + n * row_bytes + (int64_t)gs * F::kGroupBytes + col * 16
                                    : wq8;
            cp_async16(dst + r * F::kRowPitch + col * 16, src, ok ? 16u : 0u);
        }
        {
            const int r = lane & 15;
            const int64_t n = wrow0 + r;
            const bool ok = n < prm.N;
            const __half *base = (lane < 16) ? prm.scales : prm.biases;
            const void *src = ok ? (const void *)(base + n * prm.G + gs) : (const void *)base;
            cp_async16(dst + F::kScalesOff + (lane >> 4) * 256 + r * 16, src, ok ? 16u : 0u);
        }
    };
    const int slots = prm.slots;
#pragma unroll
    for (int s = 0; s < kRing - 1; ++s) {
        if (s < nst) issue(s, s);
        cp_async_commit();
    }

    // ----------------------------------------------------------------------
    // Prologue (all threads): x for this CTA's K range, permuted into
    // B-fragment order, and per-group sums of x.
    // ----------------------------------------------------------------------
    const T *xg = static_cast<const T *>(prm.x);
    if (ct < MCP) {
        escale[ct] = 1.f;
        oscale[ct] = 1.f;
        amax[ct] = 0u;
    }
    __syncthreads();
    if constexpr (std::is_same<T, __nv_bfloat16>::value) {
        // Largest |x| per activation row over this CTA's K range; pick 2^-e
        // so that the fp16 copy stays below 2^15 in magnitude.
        const int kc = gcta * 64;
        for (int m = 0; m < Mc; ++m) {
            float a = 0.f;
            for (int k = 16 * ct; k < kc; k += 16 * kThreads) {
                float f[16];
                load16<T>(xg + (m0 + m) * prm.K + 64 * gb + k, f);
#pragma unroll
                for (int i = 0; i < 16; ++i) a = fmaxf(a, fabsf(f[i]));
            }
#pragma unroll
            for (int d = 16; d >= 1; d >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, d));
            if (lane == 0) atomicMax(&amax[m], __float_as_uint(a));
        }
        __syncthreads();
        if (ct < Mc) {
            const int e = (int)((amax[ct] >> 23) & 0xFF) - 127;  // floor(log2 amax)
            const int sh = e > 14 ? e - 14 : 0;
            escale[ct] = __int_as_float((127 - sh) << 23);
            oscale[ct] = __int_as_float((127 + sh) << 23);
        }
        __syncthreads();
    }
    for (int ub = 0; ub < gcta * Mc * 4; ub += kThreads) {
        const int u = ub + ct;
        const bool valid = u < gcta * Mc * 4;
        const int j = valid ? u / (Mc * 4) : 0, m = valid ? (u >> 2) % Mc : 0, t = u & 3;
        float f[16];
        if (valid) {
            load16<T>(xg + (m0 + m) * prm.K + 64 * (gb + j) + 16 * t, f);
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) f[i] = 0.f;
        }
        const float es = valid ? escale[m] : 0.f;
        float sum = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            f[i] *= es;
            sum += f[i];
        }
        sum += __shfl_xor_sync(0xffffffffu, sum, 1);
        sum += __shfl_xor_sync(0xffffffffu, sum, 2);
        if (valid) {
            uint32_t pr[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float sc = __int_as_float((127 - PairMap<B>::p(i)) << 23);  // 2^-p
                pr[i] = pack_half2(f[PairMap<B>::lo(i)] * sc, f[PairMap<B>::hi(i)] * sc);
            }
            uint4 *dst = reinterpret_cast<uint4 *>(xfrag);
            dst[((j * 2 + 0) * Mc + m) * 4 + t] = make_uint4(pr[0], pr[1], pr[2], pr[3]);
            dst[((j * 2 + 1) * Mc + m) * 4 + t] = make_uint4(pr[4], pr[5], pr[6], pr[7]);
            if (t == 0) xs[j * MCP + m] = sum;
        }
    }
    for (int u = ct; u < gcta * MCP; u += kThreads)
        if (u % MCP >= Mc) xs[u] = 0.f;
    __syncthreads();

    // ----------------------------------------------------------------------
    // Main loop: each warp over its 16 rows and all stages of the CTA.
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

    const uint4 *xf4 = reinterpret_cast<const uint4 *>(xfrag);
    for (int si = 0; si < nst; ++si) {
        cp_async_wait<kRing - 2>();
        __syncwarp();
        const int slot = si % slots;
        const uint8_t *sb = ring + slot * F::kStageBytes;
        const uint4 sA = *reinterpret_cast<const uint4 *>(sb + F::kScalesOff + g * 16);
        const uint4 sB = *reinterpret_cast<const uint4 *>(sb + F::kScalesOff + (g + 8) * 16);
        const uint4 bA = *reinterpret_cast<const uint4 *>(sb + F::kScalesOff + 256 + g * 16);
        const uint4 bB = *reinterpret_cast<const uint4 *>(sb + F::kScalesOff + 256 + (g + 8) * 16);
#pragma unroll
        for (int j = 0; j < kGroupsPerStage; ++j) {
            const int grp = si * kGroupsPerStage + j;  // group within the CTA range
            uint32_t PA[8], PB[8];
            if constexpr (B == 4) {
                const uint2 qa = *reinterpret_cast<const uint2 *>(sb + g * F::kRowPitch +
                                                                  j * F::kGroupBytes + 8 * t);
                const uint2 qb = *reinterpret_cast<const uint2 *>(sb + (g + 8) * F::kRowPitch +
                                                                  j * F::kGroupBytes + 8 * t);
                decode4(qa.x, qa.y, PA);
                decode4(qb.x, qb.y, PB);
            } else {
                const uint32_t *pa =
                    reinterpret_cast<const uint32_t *>(sb + g * F::kRowPitch + j * F::kGroupBytes);
                const uint32_t *pb = reinterpret_cast<const uint32_t *>(
                    sb + (g + 8) * F::kRowPitch + j * F::kGroupBytes);
                decode3(pa[wi3], pa[wi3 + 1], sel0, sel2, PA);
                decode3(pb[wi3], pb[wi3 + 1], sel0, sel2, PB);
            }
            const float sa = half_at(sA, j) * 16777216.f, sbb = half_at(sB, j) * 16777216.f;
            const float ba = half_at(bA, j), bb = half_at(bB, j);
#pragma unroll
            for (int mb = 0; mb < MB; ++mb) {
                const int m = mb * 8 + g;
                uint4 q0 = make_uint4(0, 0, 0, 0), q1 = make_uint4(0, 0, 0, 0);
                if (m < Mc) {
                    q0 = xf4[((grp * 2 + 0) * Mc + m) * 4 + t];
                    q1 = xf4[((grp * 2 + 1) * Mc + m) * 4 + t];
                }
                const float2 xv = *reinterpret_cast<const float2 *>(&xs[grp * MCP + mb * 8 + 2 * t]);
                float d[4] = {0.f, 0.f, 0.f, 0.f};
                {
                    const uint32_t a0[4] = {PA[0], PB[0], PA[1], PB[1]};
                    mma_f16_16816(d, a0, q0.x, q0.y, d);
                    const uint32_t a1[4] = {PA[2], PB[2], PA[3], PB[3]};
                    mma_f16_16816(d, a1, q0.z, q0.w, d);
                    const uint32_t a2[4] = {PA[4], PB[4], PA[5], PB[5]};
                    mma_f16_16816(d, a2, q1.x, q1.y, d);
                    const uint32_t a3[4] = {PA[6], PB[6], PA[7], PB[7]};
                    mma_f16_16816(d, a3, q1.z, q1.w, d);
                }
                acc[mb][0] = fmaf(sa, d[0], fmaf(ba, xv.x, acc[mb][0]));
                acc[mb][1] = fmaf(sa, d[1], fmaf(ba, xv.y, acc[mb][1]));
                acc[mb][2] = fmaf(sbb, d[2], fmaf(bb, xv.x, acc[mb][2]));
                acc[mb][3] = fmaf(sbb, d[3], fmaf(bb, xv.y, acc[mb][3]));
            }
        }
        __syncwarp();
        if (si + kRing - 1 < nst) issue(si + kRing - 1, (si + kRing - 1) % slots);
        cp_async_commit();
    }
    cp_async_wait<0>();

    // ----------------------------------------------------------------------
    // Epilogue.
    // ----------------------------------------------------------------------
    T *y = static_cast<T *>(prm.y);
    const int rowA = 16 * warp + g, rowB = rowA + 8;  // within the CTA
#pragma unroll
    for (int mb = 0; mb < MB; ++mb) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int row = (i < 2) ? rowA : rowB;
            const int col = mb * 8 + 2 * t + (i & 1);
            const float v = acc[mb][i] * oscale[col];
            if (ks == 1) {
                if (col < Mc && n0 + row < prm.N) store_out<T>(&y[(m0 + col) * prm.N + n0 + row], v);
            } else {
                partial[row * MCP + col] = v;
            }
        }
    }
    if (ks > 1) {
        // Split-K: CTA `rank` adds element e (e % ks == rank) over all ranks
        // of the cluster, rank 0 first.
        cluster_sync();
        const uint32_t base = smem_u32(partial);
        for (int e = rank + ks * ct; e < kRows * MCP; e += ks * kThreads) {
            const int row = e / MCP, col = e % MCP;
            if (col >= Mc || n0 + row >= prm.N) continue;
            float v = 0.f;
            for (int r = 0; r < ks; ++r)
                v += ld_dsmem_f32(map_to_rank(base + 4u * (uint32_t)e, (uint32_t)r));
            store_out<T>(&y[(m0 + col) * prm.N + n0 + row], v);
        }
        cluster_sync();
    }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
namespace {

struct Plan {
    int MB, ks, mc, m_chunks, tiles;
    size_t smem;
    Params prm;
};

constexpr size_t kSmemLimit = 227 * 1024;

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool make_plan(const MatmulArgs &a, Plan &p) {
    const int B = a.bits;
    if (a.K % 512 != 0 || a.M < 1 || a.N < 1) return false;
    p.MB = a.M > 16 ? 4 : a.M > 8 ? 2 : 1;
    p.mc = 8 * p.MB;
    p.m_chunks = (int)((a.M + p.mc - 1) / p.mc);
    if (p.m_chunks > 65535) return false;
    const int64_t tiles = (a.N + kRows - 1) / kRows;
    if (tiles * kMaxCluster > (int64_t)INT32_MAX) return false;
    p.tiles = (int)tiles;
    const int stages_total = (int)(a.K / 512);
    const int mc_valid = (int)std::min<int64_t>(a.M, p.mc);
    const int sms = num_sms();
    auto xbytes = [&](int k) {
        const size_t g = (size_t)((stages_total + k - 1) / k) * kGroupsPerStage;
        return g * mc_valid * 128 + g * p.mc * 4;
    };
    // Split K over a cluster until there are about two CTAs per SM and x for
    // a CTA's K range fits comfortably in shared memory.
    int ks = 1;
    const int ks_max = std::min(kMaxCluster, stages_total);
    while (ks < ks_max &&
           ((int64_t)tiles * p.m_chunks * ks < 2 * sms || xbytes(ks) > 64 * 1024))
        ++ks;
    if (xbytes(ks) > 100 * 1024) return false;
    p.ks = ks;
    const int st_cta = (stages_total + ks - 1) / ks;
    const int slots = std::min(kRing, st_cta);
    const int stage_bytes = B == 4 ? Fmt<4>::kStageBytes : Fmt<3>::kStageBytes;

    Params &q = p.prm;
    size_t off = (size_t)kWarps * slots * stage_bytes;
    off = align_up(off, 128);
    q.off_xfrag = (uint32_t)off;
    const size_t gmax = (size_t)st_cta * kGroupsPerStage;
    off += gmax * mc_valid * 128;
    off = align_up(off, 128);
    q.off_xs = (uint32_t)off;
    off += gmax * p.mc * 4;
    off = align_up(off, 128);
    q.off_scale = (uint32_t)off;
    off += 3 * p.mc * 4;
    off = align_up(off, 128);
    q.off_partial = (uint32_t)off;
    off += ks > 1 ? (size_t)kRows * p.mc * 4 : 0;
    p.smem = align_up(off, 128);
    if (p.smem > kSmemLimit) return false;

    q.x = a.x;
    q.Wq = a.Wq;
    q.scales = static_cast<const __half *>(a.scales);
    q.biases = static_cast<const __half *>(a.biases);
    q.y = a.out;
    q.M = a.M;
    q.N = a.N;
    q.K = a.K;
    q.G = (int)(a.K / 64);
    q.stages_total = stages_total;
    q.ks = ks;
    q.mc = p.mc;
    q.slots = slots;
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
    cfg.gridDim = dim3((unsigned)(p.tiles * p.ks), (unsigned)p.m_chunks, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)p.ks;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = p.ks > 1 ? 1 : 0;
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

cudaError_t qmv_read_error(uint32_t *code, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(code, g_qmv_error, sizeof(uint32_t));
    if (e != cudaSuccess || !clear) return e;
    const uint32_t zero = 0;
    return cudaMemcpyToSymbol(g_qmv_error, &zero, sizeof(uint32_t));
}

}  // namespace aq
