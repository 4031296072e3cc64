// Small-M kernel ("qmv"): y = x . W^T for 1..32 activation rows per launch
// block, streaming the packed weights once per call.
//
// Method (mlx-bun pages, @mlx-bun/inference 1.0.0, kernels/quantization/):
//   * the weight format: 64-value groups, 2*B uint32 words each, LSB-first
//     codes (affine-split-mma.ts affine_unit; affine3/4-mma.ts);
//   * the factored form of the group dot product used by affine3-rows.ts /
//     affine4-rows.ts: sum_g [ scale_g * sum_k q_k x_k + bias_g * sum_k x_k ],
//     decoding each weight once and reusing it for every activation row;
//   * the K-permuted operand layout of affine{3,4}-mma.ts (any permutation
//     of k inside a group works, provided x is permuted the same way);
//   * a deterministic split-K sum in a fixed order (affine-split-mma.ts
//     adds its SPLITS partial tiles in index order, no atomics).
//
// GB300 design:
//   * One CTA owns 16*RT weight rows and a contiguous range of 512-wide K
//     stages.  A producer warp streams each stage's packed words, scales and
//     biases into a ring of shared-memory buffers with bulk-async copies
//     (cp.async.bulk, L2 evict-first), completion tracked by mbarriers; all
//     of a CTA's stages are in flight at once when they fit in the ring.
//   * Four consumer warps decode codes straight into fp16 MMA A-fragments:
//     a code masked in place inside an fp16 with a zero exponent field is the
//     exact subnormal q * 2^(p-24) (p = its bit position in the half), so the
//     decode is one AND per two codes plus a shift or byte permute per word.
//     x is pre-scaled by 2^-p for the matching k, making every product
//     q * x * 2^-24 exactly; the per-group scale is applied to the fp32
//     accumulator as scale * 2^24.  bf16 x is converted to fp16 once per CTA
//     with a per-row power-of-two scale that keeps it in fp16 range.
//   * mma.sync m16n8k16 (fp16 in, fp32 accumulate) does the multiply-adds:
//     16 weight rows x 8 activation rows x 16 k per instruction.  Each
//     thread holds 16 consecutive codes of a group for two rows, so one
//     MMA k-step never mixes groups and the factored form applies per group.
//   * Split-K across the CTAs of a thread-block cluster: partial tiles meet in
//     distributed shared memory and are added in rank order.
//   * Every mbarrier wait is bounded; a wait that gives up sets the kernel's
//     error word and the CTA winds down without further waits.
#include "aq_internal.h"
#include "aq_ptx.cuh"

#include <algorithm>
#include <mutex>
#include <type_traits>

namespace aq {

__device__ uint32_t g_qmv_error;

namespace {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kGroupsPerStage = 8;  // 512 values of K per stage
constexpr int kGroupsPerWarp = kGroupsPerStage / kConsumerWarps;
constexpr int kMaxStages = 8;

template <int B>
struct Fmt {
    static constexpr int kGroupBytes = 8 * B;                        // 2*B words
    static constexpr int kRowStageBytes = kGroupsPerStage * kGroupBytes;  // 256 / 192
    // Row pitch in the stage buffer, padded against bank conflicts.
    static constexpr int kRowPitch = kRowStageBytes + (B == 4 ? 32 : 16);
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
    int nstage;        // ring depth
    uint32_t stage_bytes, off_scales, off_biases;  // within one stage buffer
    uint32_t off_bars, off_xfrag, off_xs, off_partial, off_escale, off_flag;
};

// Pair i of the 8 fp16 pairs decoded from a thread's 16 codes holds codes
// (lo, hi) at bit position p within each half (see decode4 / decode3).
template <int B>
struct PairMap;
template <>
struct PairMap<4> {
    static __device__ __forceinline__ int lo(int i) { return i < 4 ? i : i + 4; }
    static __device__ __forceinline__ int hi(int i) { return lo(i) + 4; }
    static __device__ __forceinline__ int p(int i) { return (i & 1) ? 4 : 0; }
};
template <>
struct PairMap<3> {
    static __device__ __forceinline__ int lo(int i) { return i; }
    static __device__ __forceinline__ int hi(int i) { return i + 8; }
    static __device__ __forceinline__ int p(int i) {
        // positions 0,3,6,0,3,0,3,6
        return i == 2 || i == 7 ? 6 : (i == 1 || i == 4 || i == 6) ? 3 : 0;
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

__device__ __forceinline__ void record_error(volatile int *flag, uint32_t code) {
    *flag = 1;
    atomicOr(&g_qmv_error, code);
}

// Bounded wait that also gives up at once when another warp of the CTA has
// already given up (so a failing CTA pays the time limit only once).
__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, volatile int *flag,
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
    record_error(flag, code);
    return false;
}

template <typename T>
__device__ __forceinline__ void load16(const T *src, float (&f)[16]) {
    const uint4 u0 = __ldg(reinterpret_cast<const uint4 *>(src));
    const uint4 u1 = __ldg(reinterpret_cast<const uint4 *>(src) + 1);
    const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        if constexpr (sizeof(T) == 2 && std::is_same<T, __half>::value) {
            const __half2 h = *reinterpret_cast<const __half2 *>(&w[i]);
            const float2 v = __half22float2(h);
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

}  // namespace

template <int B, typename T, int MB, int RT>
__global__ void __launch_bounds__(kThreads) qmv_kernel(const __grid_constant__ Params prm) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int R = 16 * RT;   // weight rows per CTA
    constexpr int MCP = 8 * MB;  // padded activation rows per launch block
    using F = Fmt<B>;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int ks = prm.ks;
    const int tile = blockIdx.x / ks;
    const int rank = blockIdx.x % ks;
    const int64_t n0 = (int64_t)tile * R;
    const int64_t m0 = (int64_t)blockIdx.y * prm.mc;
    const int Mc = (int)min((int64_t)prm.mc, prm.M - m0);  // valid activation rows here
    const int st_begin = (int)((int64_t)prm.stages_total * rank / ks);
    const int st_end = (int)((int64_t)prm.stages_total * (rank + 1) / ks);
    const int nst = st_end - st_begin;
    const int gb = st_begin * kGroupsPerStage;  // first group of this CTA
    const int gcta = nst * kGroupsPerStage;     // groups of this CTA

    uint64_t *full = reinterpret_cast<uint64_t *>(smem + prm.off_bars);
    uint64_t *empty = full + kMaxStages;
    uint8_t *xfrag = smem + prm.off_xfrag;
    float *xs = reinterpret_cast<float *>(smem + prm.off_xs);
    float *partial = reinterpret_cast<float *>(smem + prm.off_partial);
    float *escale = reinterpret_cast<float *>(smem + prm.off_escale);  // [MCP] x multiplier
    float *oscale = escale + MCP;                                      // [MCP] y multiplier
    volatile int *flag = reinterpret_cast<volatile int *>(smem + prm.off_flag);

    if (threadIdx.x == 0) {
        for (int s = 0; s < prm.nstage; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        *flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------------------
        // Producer: one lane per weight row issues that row's three copies.
        // ------------------------------------------------------------------
        const uint64_t pol = policy_evict_first();
        const int64_t wpr = prm.K * B / 32;
        const int valid_rows = (int)min((int64_t)R, prm.N - n0);
        const uint32_t row_bytes = F::kRowStageBytes + 2 * 2 * kGroupsPerStage;
        for (int si = 0; si < nst; ++si) {
            const int slot = si % prm.nstage;
            const uint32_t ph = (uint32_t)(si / prm.nstage) & 1u;
            if (si >= prm.nstage && !wait_or_abort(&empty[slot], ph ^ 1u, flag, ERR_QMV_EMPTY))
                break;
            uint8_t *sb = smem + (size_t)slot * prm.stage_bytes;
            if (lane == 0) mbar_arrive_expect_tx(&full[slot], row_bytes * valid_rows);
            __syncwarp();
            if (lane < valid_rows) {
                const int64_t row = n0 + lane;
                const int g0 = gb + si * kGroupsPerStage;
                bulk_g2s(sb + lane * F::kRowPitch,
                         prm.Wq + row * wpr + (int64_t)g0 * (2 * B), F::kRowStageBytes,
                         &full[slot], pol);
                bulk_g2s(sb + prm.off_scales + lane * 16, prm.scales + row * prm.G + g0, 16,
                         &full[slot], pol);
                bulk_g2s(sb + prm.off_biases + lane * 16, prm.biases + row * prm.G + g0, 16,
                         &full[slot], pol);
            }
        }
    } else {
        // ------------------------------------------------------------------
        // Consumers.  Prologue: x of this CTA's K range, permuted into
        // B-fragment order, plus per-group sums of x.
        // ------------------------------------------------------------------
        const int ct = threadIdx.x;  // 0..127
        const T *xg = static_cast<const T *>(prm.x);
        if (ct < MCP) {
            escale[ct] = 1.f;
            oscale[ct] = 1.f;
        }
        if constexpr (std::is_same<T, __nv_bfloat16>::value) {
            // Largest |x| per activation row over this CTA's K range, as
            // ordered float bits; pick 2^-e so that the fp16 copy stays below
            // 2^15 in magnitude.
            unsigned *amax = reinterpret_cast<unsigned *>(partial);  // scratch before use
            if (ct < MCP) amax[ct] = 0u;
            asm volatile("bar.sync 1, 128;" ::: "memory");
            for (int u = ct; u < gcta * Mc * 4; u += 128) {
                const int j = u / (Mc * 4), m = (u >> 2) % Mc, t = u & 3;
                float f[16];
                load16<T>(xg + (m0 + m) * prm.K + 64 * (gb + j) + 16 * t, f);
                float a = 0.f;
#pragma unroll
                for (int i = 0; i < 16; ++i) a = fmaxf(a, fabsf(f[i]));
                atomicMax(&amax[m], __float_as_uint(a));
            }
            asm volatile("bar.sync 1, 128;" ::: "memory");
            if (ct < Mc) {
                const int e = (int)((amax[ct] >> 23) & 0xFF) - 127;  // floor(log2 amax)
                const int sh = e > 14 ? e - 14 : 0;
                escale[ct] = exp2f((float)-sh);
                oscale[ct] = exp2f((float)sh);
            }
            asm volatile("bar.sync 1, 128;" ::: "memory");
        } else {
            asm volatile("bar.sync 1, 128;" ::: "memory");
        }
        for (int ub = 0; ub < gcta * Mc * 4; ub += 128) {
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
        // zero the padding rows of xs
        for (int u = ct; u < gcta * MCP; u += 128)
            if (u % MCP >= Mc) xs[u] = 0.f;
        asm volatile("bar.sync 1, 128;" ::: "memory");

        // ------------------------------------------------------------------
        // Main loop.
        // ------------------------------------------------------------------
        const int g = lane >> 2, t = lane & 3;
        uint32_t sel0 = 0, sel2 = 0;
        int wi3 = 0;
        if constexpr (B == 3) {
            const uint32_t bo = 2u * (uint32_t)(t & 1);
            sel0 = (bo + 0) | ((bo + 1) << 4) | ((bo + 3) << 8) | ((bo + 4) << 12);
            sel2 = (bo + 1) | ((bo + 2) << 4) | ((bo + 4) << 8) | ((bo + 5) << 12);
            wi3 = (3 * t) >> 1;
        }
        float acc[RT][MB][4];
#pragma unroll
        for (int rt = 0; rt < RT; ++rt)
#pragma unroll
            for (int mb = 0; mb < MB; ++mb)
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[rt][mb][i] = 0.f;

        const uint4 *xf4 = reinterpret_cast<const uint4 *>(xfrag);
        for (int si = 0; si < nst; ++si) {
            const int slot = si % prm.nstage;
            const uint32_t ph = (uint32_t)(si / prm.nstage) & 1u;
            const bool ok = wait_or_abort(&full[slot], ph, flag, ERR_QMV_FULL);
            const uint8_t *sb = smem + (size_t)slot * prm.stage_bytes;
            const __half *ss = reinterpret_cast<const __half *>(sb + prm.off_scales);
            const __half *sbias = reinterpret_cast<const __half *>(sb + prm.off_biases);
            if (ok) {
#pragma unroll
                for (int jj = 0; jj < kGroupsPerWarp; ++jj) {
                    const int jl = warp * kGroupsPerWarp + jj;  // group within the stage
                    const int grp = si * kGroupsPerStage + jl;  // group within the CTA range
                    uint4 bf[MB][2];
                    float xs0[MB], xs1[MB];
#pragma unroll
                    for (int mb = 0; mb < MB; ++mb) {
                        const int m = mb * 8 + g;
                        if (m < Mc) {
                            bf[mb][0] = xf4[((grp * 2 + 0) * Mc + m) * 4 + t];
                            bf[mb][1] = xf4[((grp * 2 + 1) * Mc + m) * 4 + t];
                        } else {
                            bf[mb][0] = make_uint4(0, 0, 0, 0);
                            bf[mb][1] = make_uint4(0, 0, 0, 0);
                        }
                        const float2 v =
                            *reinterpret_cast<const float2 *>(&xs[grp * MCP + mb * 8 + 2 * t]);
                        xs0[mb] = v.x;
                        xs1[mb] = v.y;
                    }
#pragma unroll
                    for (int rt = 0; rt < RT; ++rt) {
                        const int ra = rt * 16 + g, rb = ra + 8;
                        uint32_t PA[8], PB[8];
                        if constexpr (B == 4) {
                            const uint2 qa = *reinterpret_cast<const uint2 *>(
                                sb + ra * F::kRowPitch + jl * F::kGroupBytes + 8 * t);
                            const uint2 qb = *reinterpret_cast<const uint2 *>(
                                sb + rb * F::kRowPitch + jl * F::kGroupBytes + 8 * t);
                            decode4(qa.x, qa.y, PA);
                            decode4(qb.x, qb.y, PB);
                        } else {
                            const uint32_t *pa = reinterpret_cast<const uint32_t *>(
                                sb + ra * F::kRowPitch + jl * F::kGroupBytes);
                            const uint32_t *pb = reinterpret_cast<const uint32_t *>(
                                sb + rb * F::kRowPitch + jl * F::kGroupBytes);
                            decode3(pa[wi3], pa[wi3 + 1], sel0, sel2, PA);
                            decode3(pb[wi3], pb[wi3 + 1], sel0, sel2, PB);
                        }
                        const float sa = __half2float(ss[ra * kGroupsPerStage + jl]) * 16777216.f;
                        const float sbb = __half2float(ss[rb * kGroupsPerStage + jl]) * 16777216.f;
                        const float ba = __half2float(sbias[ra * kGroupsPerStage + jl]);
                        const float bb = __half2float(sbias[rb * kGroupsPerStage + jl]);
#pragma unroll
                        for (int mb = 0; mb < MB; ++mb) {
                            float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                            for (int s = 0; s < 4; ++s) {
                                const uint32_t a[4] = {PA[2 * s], PB[2 * s], PA[2 * s + 1],
                                                       PB[2 * s + 1]};
                                const uint4 &q = bf[mb][s >> 1];
                                const uint32_t b0 = (s & 1) ? q.z : q.x;
                                const uint32_t b1 = (s & 1) ? q.w : q.y;
                                mma_f16_16816(d, a, b0, b1, d);
                            }
                            acc[rt][mb][0] = fmaf(sa, d[0], fmaf(ba, xs0[mb], acc[rt][mb][0]));
                            acc[rt][mb][1] = fmaf(sa, d[1], fmaf(ba, xs1[mb], acc[rt][mb][1]));
                            acc[rt][mb][2] = fmaf(sbb, d[2], fmaf(bb, xs0[mb], acc[rt][mb][2]));
                            acc[rt][mb][3] = fmaf(sbb, d[3], fmaf(bb, xs1[mb], acc[rt][mb][3]));
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
        }

        // ------------------------------------------------------------------
        // Add the four warps' partial tiles in warp order.  The stage ring is
        // idle now (every copy has landed and been read), so it holds them.
        // ------------------------------------------------------------------
        asm volatile("bar.sync 1, 128;" ::: "memory");
        float *red = reinterpret_cast<float *>(smem);
        constexpr int E = RT * MB * 32 * 4;  // elements per warp
#pragma unroll
        for (int rt = 0; rt < RT; ++rt)
#pragma unroll
            for (int mb = 0; mb < MB; ++mb)
                *reinterpret_cast<float4 *>(&red[warp * E + ((rt * MB + mb) * 32 + lane) * 4]) =
                    make_float4(acc[rt][mb][0], acc[rt][mb][1], acc[rt][mb][2], acc[rt][mb][3]);
        asm volatile("bar.sync 1, 128;" ::: "memory");
        T *y = static_cast<T *>(prm.y);
        for (int e = ct; e < E; e += 128) {
            float v = 0.f;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) v += red[w * E + e];
            const int i = e & 3, ln = (e >> 2) & 31, rm = e >> 7;
            const int rt = rm / MB, mb = rm % MB;
            const int row = rt * 16 + (ln >> 2) + 8 * (i >> 1);
            const int col = mb * 8 + 2 * (ln & 3) + (i & 1);
            v *= oscale[col];
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
        if (warp < kConsumerWarps) {
            T *y = static_cast<T *>(prm.y);
            const uint32_t base = smem_u32(partial);
            for (int e = rank + ks * (int)threadIdx.x; e < R * MCP; e += ks * 128) {
                const int row = e / MCP, col = e % MCP;
                if (col >= Mc || n0 + row >= prm.N) continue;
                float v = 0.f;
                for (int r = 0; r < ks; ++r)
                    v += ld_dsmem_f32(map_to_rank(base + 4u * (uint32_t)e, (uint32_t)r));
                store_out<T>(&y[(m0 + col) * prm.N + n0 + row], v);
            }
        }
        cluster_sync();
    }
    if (*flag) {
        // A wait gave up.  Copies issued before that may still be landing in
        // this CTA's shared memory: let them finish before the CTA exits.
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 200000ull) {
        }
    }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
namespace {

struct Plan {
    int MB, RT, ks, mc, nstage, m_chunks, tiles;
    size_t smem;
    Params prm;
};

constexpr size_t kSmemLimit = 227 * 1024;

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool make_plan(const MatmulArgs &a, Plan &p) {
    const int B = a.bits;
    if (a.K % 512 != 0 || a.M < 1 || a.N < 1) return false;
    p.MB = a.M >= 25 ? 4 : a.M >= 17 ? 3 : a.M >= 9 ? 2 : 1;
    if (p.MB == 3) p.MB = 4;
    p.RT = 1;
    p.mc = 8 * p.MB;
    p.m_chunks = (int)((a.M + p.mc - 1) / p.mc);
    if (p.m_chunks > 65535) return false;
    const int R = 16 * p.RT;
    const int64_t tiles = (a.N + R - 1) / R;
    if (tiles * 8 > (int64_t)INT32_MAX) return false;
    p.tiles = (int)tiles;
    const int stages_total = (int)(a.K / 512);
    const int mc_valid = (int)std::min<int64_t>(a.M, p.mc);
    // Split K across a cluster until there are about two CTAs per SM, and
    // until x for a CTA's K range fits comfortably in shared memory.
    const int sms = num_sms();
    int ks = 1;
    auto xbytes = [&](int k) {
        const int g = ((stages_total + k - 1) / k) * kGroupsPerStage;
        return (size_t)g * mc_valid * 128 + (size_t)g * p.mc * 4;
    };
    while (ks < 8 && ks * 2 <= stages_total &&
           ((int64_t)tiles * p.m_chunks * ks < 2 * sms || xbytes(ks) > 96 * 1024))
        ks *= 2;
    if (xbytes(ks) > 120 * 1024) return false;
    p.ks = ks;
    const int st_cta = (stages_total + ks - 1) / ks;
    p.nstage = std::min(kMaxStages, std::max(1, st_cta));

    const int row_pitch = B == 4 ? Fmt<4>::kRowPitch : Fmt<3>::kRowPitch;
    Params &q = p.prm;
    q.off_scales = (uint32_t)(R * row_pitch);
    q.off_biases = q.off_scales + R * 16;
    q.stage_bytes = (uint32_t)align_up(q.off_biases + R * 16, 128);
    size_t off = (size_t)p.nstage * q.stage_bytes;
    const size_t red_bytes = (size_t)kConsumerWarps * p.RT * p.MB * 32 * 4 * 4;
    off = std::max(off, red_bytes);
    off = align_up(off, 128);
    q.off_bars = (uint32_t)off;
    off += 2 * kMaxStages * 8;
    off = align_up(off, 128);
    q.off_xfrag = (uint32_t)off;
    const size_t gmax = (size_t)st_cta * kGroupsPerStage;
    off += gmax * mc_valid * 128;
    off = align_up(off, 128);
    q.off_xs = (uint32_t)off;
    off += gmax * p.mc * 4;
    off = align_up(off, 128);
    q.off_partial = (uint32_t)off;
    off += (size_t)R * p.mc * 4;
    q.off_escale = (uint32_t)off;
    off += 2 * p.mc * 4;
    q.off_flag = (uint32_t)off;
    off += 16;
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
    q.nstage = p.nstage;
    return true;
}

template <int B, typename T, int MB, int RT>
cudaError_t launch_plan(const Plan &p, cudaStream_t stream) {
    auto kern = qmv_kernel<B, T, MB, RT>;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)kSmemLimit);
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
        case 1: return launch_plan<B, T, 1, 1>(p, s);
        case 2: return launch_plan<B, T, 2, 1>(p, s);
        default: return launch_plan<B, T, 4, 1>(p, s);
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
