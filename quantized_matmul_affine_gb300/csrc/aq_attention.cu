// Decode attention over a quantised KV cache: for one query row per head,
//   o[h] = softmax(q[h] . Kd[kv]^T) . Vd[kv],   kv = h / (H / KV),
// with K and V stored in the affine format (4 or 8 bits, one fp16 scale and
// bias per group of 32/64/128 values along the head dimension).  The
// operator of the mlx-bun fused decode kernel (@mlx-bun/inference 1.0.0,
// fused-decode-kernel.ts: flash-decoding split over the cached rows, the
// scores taken in the factored form scale * sum(q * code) + bias * sum(q),
// an online softmax per row block, a deterministic merge of the blocks).
//
// GB300 design:
//   * One CTA per (KV head, block of cached rows) takes every query head of
//     that KV head (up to 8), so each K and V row is read once.  The blocks
//     of a KV head form a thread-block cluster; their partial results are
//     merged in rank order through distributed shared memory - no global
//     scratch, no second launch.  The cluster size is picked from the
//     driver's count of co-resident clusters.
//   * A producer warp streams 128-row stages of K and V codes (2-D TMA,
//     swizzled so that the fragment reads below are free of bank conflicts)
//     and their scales and biases (1-D TMA) into a shared-memory ring.
//   * Each of 8 consumer warps takes a 16-row tile of a stage.  Scores on the
//     tensor cores: S^T-free form S[16 rows][8 heads] = codes x q', the codes
//     as the exact fp16 subnormals code * 2^-24 (or 2^-20 where a nibble sits
//     at bit 4), q' = q * 2^e per head in fp16; one m16n8k16 chain per group,
//     then s = scale * sum(q code) + bias * sum(q) in fp32.
//   * Online softmax in base 2 on the fragment; the probabilities, times the
//     value scale of their row and group (and 2^ev, a per-warp power of two
//     lowered as larger scales appear, which keeps them in the fp16 range
//     and mostly out of its subnormals), are transposed in registers
//     (movmatrix) into the B operand of O^T[d][heads] += codes^T x P'; the
//     value biases enter as sum(p * bias) per (head, group) in fp32.
//   * The warps' (max, sum, o) merge through shared memory in warp order, the
//     cluster's CTAs then in rank order; o is rounded once.
#include "aq_internal.h"
#include "aq_ptx.cuh"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <cstdio>
#include <mutex>

namespace aq {

__device__ uint32_t g_attn_error;

namespace {

constexpr int kCWarps = 8;                           // consumer warps
constexpr int kAttnThreads = (kCWarps + 1) * 32;     // + the TMA producer warp
constexpr int kTile = 16;                            // rows per warp tile
constexpr int kStageRows = kTile * kCWarps;          // 128
constexpr int kMaxStages = 8;
constexpr int kRingBudget = 192 * 1024;
constexpr float kLog2e = 1.4426950408889634f;

struct AttnParams {
    const void *q;
    void *out;
    uint32_t *err;
    int KV, N, nrep;
    int block;          // cached rows per CTA (multiple of 16)
    int csize;          // CTAs per cluster (one KV head)
    int stages;         // ring depth
    int bf16;
};

template <int BITS, int D, int GROUP>
struct Shape {
    static constexpr int kRB = D * BITS / 8;            // bytes of one cached row
    static constexpr int kW = kRB < 128 ? kRB : 128;    // TMA box width = swizzle span
    static constexpr int kBoxes = kRB / kW;
    static constexpr uint32_t kSwz = kW == 128 ? 7u : kW == 64 ? 3u : 1u;
    static constexpr int kG = D / GROUP;                // groups per row
    static constexpr int kGB = GROUP * BITS / 8;        // bytes of one group of a row
    static constexpr int kCK = kGB / 4;                 // bytes a lane takes per row (scores)
    static constexpr int kCV = kGB / 8;                 // bytes a lane takes per row (values)
    static constexpr int kSteps = GROUP / 16;           // k-steps / M-tiles per group
    static constexpr int kRegs = GROUP / 8;             // code registers per row per group
    // scales: 128 rows x G halves from a 16-byte aligned start (up to 7
    // before), in boxes of a multiple of 64 halves so that every box lands
    // on a 128-byte boundary of shared memory (the tensor-copy rule)
    static constexpr int kSH = kStageRows * kG + 8;
    static constexpr int kSBoxes = (kSH + 255) / 256;
    static constexpr int kSBox = ((kSH + kSBoxes - 1) / kSBoxes + 63) / 64 * 64;
    static constexpr int kSArr = kSBoxes * kSBox;       // halves per scale array per stage
    static constexpr int kCodeBytes = kStageRows * kRB; // K (or V) codes per stage
    static constexpr int kTx = 2 * kCodeBytes + 4 * kSArr * 2;
    static constexpr int kStageBytes = (kTx + 1023) / 1024 * 1024;
    static_assert(kSBox <= 256 && (2 * kSBox) % 128 == 0 && (2 * kCodeBytes) % 1024 == 0,
                  "tensor-copy boxes must land 128-byte aligned");
};

// Byte offset of (row, byte) inside a stage's K or V code region, with the
// TMA swizzle of a box kW bytes wide (16-byte chunk index XOR row bits).
template <class S>
__device__ __forceinline__ uint32_t swz(int row, int byte) {
    const uint32_t lin = (uint32_t)(row * S::kW + (byte % S::kW));
    return (uint32_t)(byte / S::kW) * (kStageRows * S::kW) + (lin ^ (((lin >> 7) & S::kSwz) << 4));
}

template <int NB>
__device__ __forceinline__ void lds_words(const uint8_t *p, uint32_t (&w)[NB / 4 > 0 ? NB / 4 : 1]) {
    if constexpr (NB == 2) {
        w[0] = *reinterpret_cast<const uint16_t *>(p);
    } else if constexpr (NB == 4) {
        w[0] = *reinterpret_cast<const uint32_t *>(p);
    } else if constexpr (NB == 8) {
        const uint2 v = *reinterpret_cast<const uint2 *>(p);
        w[0] = v.x;
        w[1] = v.y;
    } else {
        const uint4 v = *reinterpret_cast<const uint4 *>(p);
        w[0] = v.x;
        w[1] = v.y;
        w[2] = v.z;
        w[3] = v.w;
    }
}

__device__ __forceinline__ uint32_t movmatrix_t(uint32_t a) {
    uint32_t d;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
    return d;
}

__device__ __forceinline__ void consumer_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kCWarps * 32) : "memory");
}

__device__ __forceinline__ float pow2i(int e) { return __int_as_float((127 + e) << 23); }

// 15 - (the exponent of v as frexp gives it): v * 2^result lies in [2^14, 2^15)
// (clamped to +-100 so that every power of two used stays a normal float).
__device__ __forceinline__ int exp_for(float v) {
    int ex;
    frexpf(v, &ex);
    return v > 0.f ? max(-100, min(100, 15 - ex)) : 0;
}

__device__ __forceinline__ void attn_record(volatile int *flag, uint32_t *err, uint32_t code) {
    *flag = 1;
    atomicOr(err, code);
}

template <int BITS, int D, int GROUP>
__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ CUtensorMap tm_kw,
                const __grid_constant__ CUtensorMap tm_vw, const __grid_constant__ CUtensorMap tm_ks,
                const __grid_constant__ CUtensorMap tm_kb, const __grid_constant__ CUtensorMap tm_vs,
                const __grid_constant__ CUtensorMap tm_vb) {
    using S = Shape<BITS, D, GROUP>;
    constexpr int G = S::kG;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *ring = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int merge_bytes = 4 * ((kCWarps + 1) * p.nrep * (D + 2));
    uint8_t *tail = ring + max(p.stages * S::kStageBytes, merge_bytes);
    uint2 *qfrag = reinterpret_cast<uint2 *>(tail);                 // [D/16][32]
    float *qf = reinterpret_cast<float *>(qfrag + (D / 16) * 32);   // [8][D]  q * 2^e
    float *qs2 = qf + 8 * D;                                        // [8][G]  sum(q) log2 e
    float *qsc = qs2 + 8 * G;                                       // [8]     2^(24-e) log2 e
    float *red = qsc + 8;                                           // [8]
    uint64_t *full = reinterpret_cast<uint64_t *>(red + 8);
    uint64_t *empty = full + kMaxStages;
    int *flag_s = reinterpret_cast<int *>(empty + kMaxStages);
    volatile int *flag = flag_s;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gid = lane >> 2, t = lane & 3;
    const int kv = (int)blockIdx.x / p.csize;
    const int rank = (int)blockIdx.x % p.csize;
    const int n0 = rank * p.block;
    const int n1 = min(p.N, n0 + p.block);
    const int nst = n1 > n0 ? (n1 - n0 + kStageRows - 1) / kStageRows : 0;
    const int nrep = p.nrep;
    const long long row_base = (long long)kv * p.N;

    if (threadIdx.x == 0) {
        for (int i = 0; i < p.stages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kCWarps);
        }
        *flag_s = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == kCWarps) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int issued = 0;
            for (int st = 0; st < nst && !*flag; ++st) {
                const int slot = st % p.stages, lap = st / p.stages;
                if (lap > 0 && !mbar_wait(&empty[slot], (lap - 1) & 1)) {
                    attn_record(flag, p.err, ERR_ATTN_EMPTY);
                    break;
                }
                uint8_t *sb = ring + slot * S::kStageBytes;
                const int row0 = (int)(row_base + n0 + st * kStageRows);
                const int x0 = (row0 * G) & ~7;
                mbar_arrive_expect_tx(&full[slot], (uint32_t)S::kTx);
#pragma unroll
                for (int b = 0; b < S::kBoxes; ++b) {
                    tma_load_2d(sb + b * kStageRows * S::kW, &tm_kw, b * S::kW, row0, &full[slot]);
                    tma_load_2d(sb + S::kCodeBytes + b * kStageRows * S::kW, &tm_vw, b * S::kW, row0,
                                &full[slot]);
                }
                uint8_t *sc = sb + 2 * S::kCodeBytes;
#pragma unroll
                for (int b = 0; b < S::kSBoxes; ++b) {
                    const int off = 2 * b * S::kSBox;
                    tma_load_1d(sc + off, &tm_ks, x0 + b * S::kSBox, &full[slot]);
                    tma_load_1d(sc + 2 * S::kSArr + off, &tm_kb, x0 + b * S::kSBox, &full[slot]);
                    tma_load_1d(sc + 4 * S::kSArr + off, &tm_vs, x0 + b * S::kSBox, &full[slot]);
                    tma_load_1d(sc + 6 * S::kSArr + off, &tm_vb, x0 + b * S::kSBox, &full[slot]);
                }
                issued = st + 1;
            }
            // copies still in flight land before the CTA moves on
            for (int st = max(0, issued - p.stages); st < issued; ++st)
                if (!mbar_wait(&full[st % p.stages], (st / p.stages) & 1)) {
                    attn_record(flag, p.err, ERR_ATTN_FULL);
                    break;
                }
        }
    } else {
        // ------------------------------------------------------------ prologue
        {
            // warp w: query head w of this KV head (zeros past nrep)
            const int h = warp;
            float qv[D / 32];
            float mx = 0.f;
#pragma unroll
            for (int i = 0; i < D / 32; ++i) {
                float v = 0.f;
                if (h < nrep) {
                    const size_t idx = (size_t)(kv * nrep + h) * D + lane + 32 * i;
                    v = p.bf16 ? __bfloat162float(static_cast<const __nv_bfloat16 *>(p.q)[idx])
                               : __half2float(static_cast<const __half *>(p.q)[idx]);
                }
                qv[i] = v;
                mx = fmaxf(mx, fabsf(v));
            }
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(~0u, mx, off));
            const int e = exp_for(mx);
            const float sc = pow2i(e);
#pragma unroll
            for (int i = 0; i < D / 32; ++i) qf[h * D + lane + 32 * i] = qv[i] * sc;
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float sum = 0.f;
#pragma unroll
                for (int i = 0; i < D / 32; ++i)
                    if ((lane + 32 * i) / GROUP == g) sum += qv[i];
#pragma unroll
                for (int off = 16; off >= 1; off >>= 1) sum += __shfl_xor_sync(~0u, sum, off);
                if (lane == 0) qs2[h * G + g] = sum * kLog2e;
            }
            if (lane == 0) qsc[h] = pow2i(24 - e) * kLog2e;
        }
        consumer_sync();
        // B fragments of q': k-step k of group g, lane (gid, t) = head gid,
        // the k of thread t's registers 2s and 2s+1 (their two halves)
        for (int k = 0; k < D / 16; ++k) {
            const int g = k / S::kSteps, s2 = k % S::kSteps;
            uint32_t r[2];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int i = 2 * s2 + j;
                float v[2];
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    int d;
                    float f = 1.f;
                    if constexpr (BITS == 4) {
                        d = g * GROUP + t * (GROUP / 4) + 8 * (i / 4) + (i % 4) + 4 * hf;
                        if (i & 1) f = 0.0625f;
                    } else {
                        d = g * GROUP + t * (GROUP / 4) + 4 * (i / 2) + (i % 2) + 2 * hf;
                    }
                    v[hf] = gid < nrep ? qf[gid * D + d] * f : 0.f;
                }
                r[j] = pack_half2(v[0], v[1]);
            }
            qfrag[k * 32 + lane] = make_uint2(r[0], r[1]);
        }
        const float qsc0 = qsc[2 * t], qsc1 = qsc[2 * t + 1];
        consumer_sync();

        // ------------------------------------------------------------ main loop
        float m2[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
        // p * scale * 2^ev enters the value product: ev keeps the largest
        // |scale| seen so far below 2^15 (fp16 range, few subnormals); it only
        // decreases, and O is rescaled with it like with the running max
        int ev = 127;
        float bt[2][G];
        float O[D / 16][4];
#pragma unroll
        for (int g = 0; g < G; ++g) bt[0][g] = bt[1][g] = 0.f;
#pragma unroll
        for (int i = 0; i < D / 16; ++i) O[i][0] = O[i][1] = O[i][2] = O[i][3] = 0.f;

        for (int st = 0; st < nst; ++st) {
            const int slot = st % p.stages, lap = st / p.stages;
            if (*flag) break;
            if (!mbar_wait(&full[slot], lap & 1)) {
                attn_record(flag, p.err, ERR_ATTN_FULL);
                break;
            }
            const int r0 = n0 + st * kStageRows + warp * kTile;   // first row of the tile
            if (r0 < n1) {
                const uint8_t *kst = ring + slot * S::kStageBytes;
                const uint8_t *vst = kst + S::kCodeBytes;
                const int row0 = (int)(row_base + n0 + st * kStageRows);
                const int soff = row0 * G - ((row0 * G) & ~7);
                const __half *sks = reinterpret_cast<const __half *>(vst + S::kCodeBytes) + soff;
                const __half *skb = sks + S::kSArr;
                const __half *svs = sks + 2 * S::kSArr;
                const __half *svb = sks + 3 * S::kSArr;
                const int tr = warp * kTile;                       // tile row in the stage
                const int ra = tr + gid, rb = tr + gid + 8;

                // scores: rows (gid, gid+8) x heads (2t, 2t+1)
                float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    uint32_t Ra[S::kRegs], Rb[S::kRegs];
#pragma unroll
                    for (int c = 0; c < (S::kCK + 15) / 16; ++c) {
                        constexpr int NB = S::kCK < 16 ? S::kCK : 16;
                        uint32_t wa[NB / 4], wb[NB / 4];
                        const int byte = g * S::kGB + t * S::kCK + c * 16;
                        lds_words<NB>(kst + swz<S>(ra, byte), wa);
                        lds_words<NB>(kst + swz<S>(rb, byte), wb);
#pragma unroll
                        for (int j = 0; j < NB / 4; ++j) {
                            const int base = (c * (NB / 4) + j) * (BITS == 4 ? 4 : 2);
                            if constexpr (BITS == 4) {
                                const uint32_t va = wa[j] >> 8, vb = wb[j] >> 8;
                                Ra[base + 0] = wa[j] & 0x000F000Fu;
                                Ra[base + 1] = wa[j] & 0x00F000F0u;
                                Ra[base + 2] = va & 0x000F000Fu;
                                Ra[base + 3] = va & 0x00F000F0u;
                                Rb[base + 0] = wb[j] & 0x000F000Fu;
                                Rb[base + 1] = wb[j] & 0x00F000F0u;
                                Rb[base + 2] = vb & 0x000F000Fu;
                                Rb[base + 3] = vb & 0x00F000F0u;
                            } else {
                                Ra[base + 0] = wa[j] & 0x00FF00FFu;
                                Ra[base + 1] = (wa[j] >> 8) & 0x00FF00FFu;
                                Rb[base + 0] = wb[j] & 0x00FF00FFu;
                                Rb[base + 1] = (wb[j] >> 8) & 0x00FF00FFu;
                            }
                        }
                    }
                    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int k = 0; k < S::kSteps; ++k) {
                        const uint2 bq = qfrag[(g * S::kSteps + k) * 32 + lane];
                        const uint32_t a[4] = {Ra[2 * k], Rb[2 * k], Ra[2 * k + 1], Rb[2 * k + 1]};
                        mma_f16_16816(acc, a, bq.x, bq.y, acc);
                    }
                    const float ksa = __half2float(sks[ra * G + g]), ksb = __half2float(sks[rb * G + g]);
                    const float kba = __half2float(skb[ra * G + g]), kbb = __half2float(skb[rb * G + g]);
                    const float q0 = qs2[(2 * t) * G + g], q1 = qs2[(2 * t + 1) * G + g];
                    s[0] = fmaf(ksa, acc[0] * qsc0, fmaf(kba, q0, s[0]));
                    s[1] = fmaf(ksa, acc[1] * qsc1, fmaf(kba, q1, s[1]));
                    s[2] = fmaf(ksb, acc[2] * qsc0, fmaf(kbb, q0, s[2]));
                    s[3] = fmaf(ksb, acc[3] * qsc1, fmaf(kbb, q1, s[3]));
                }
                if (r0 + gid >= n1) s[0] = s[1] = -INFINITY;
                if (r0 + gid + 8 >= n1) s[2] = s[3] = -INFINITY;

                // online softmax (base 2) per head column
                float mx0 = fmaxf(s[0], s[2]), mx1 = fmaxf(s[1], s[3]);
#pragma unroll
                for (int off = 4; off <= 16; off <<= 1) {
                    mx0 = fmaxf(mx0, __shfl_xor_sync(~0u, mx0, off));
                    mx1 = fmaxf(mx1, __shfl_xor_sync(~0u, mx1, off));
                }
                const float mn0 = fmaxf(m2[0], mx0), mn1 = fmaxf(m2[1], mx1);
                const float f0 = exp2f(m2[0] - mn0), f1 = exp2f(m2[1] - mn1);
                m2[0] = mn0;
                m2[1] = mn1;
                const float pr[4] = {exp2f(s[0] - mn0), exp2f(s[1] - mn1), exp2f(s[2] - mn0),
                                     exp2f(s[3] - mn1)};
                l[0] = fmaf(l[0], f0, pr[0] + pr[2]);
                l[1] = fmaf(l[1], f1, pr[1] + pr[3]);
                float vsa[G], vsb[G];
                float vmx = 0.f;
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    vsa[g] = __half2float(svs[ra * G + g]);
                    vsb[g] = __half2float(svs[rb * G + g]);
                    vmx = fmaxf(vmx, fmaxf(fabsf(vsa[g]), fabsf(vsb[g])));
                }
#pragma unroll
                for (int off = 4; off <= 16; off <<= 1)
                    vmx = fmaxf(vmx, __shfl_xor_sync(~0u, vmx, off));
                const int ev_new = min(ev, exp_for(vmx));
                const float r = ev_new - ev < -126 ? 0.f : pow2i(ev_new - ev);
                ev = ev_new;
                const float vsc = pow2i(ev);
                if (__any_sync(~0u, f0 != 1.f || f1 != 1.f || r != 1.f)) {
                    const float o0 = f0 * r, o1 = f1 * r;
#pragma unroll
                    for (int i = 0; i < D / 16; ++i) {
                        O[i][0] *= o0;
                        O[i][1] *= o1;
                        O[i][2] *= o0;
                        O[i][3] *= o1;
                    }
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        bt[0][g] *= f0;
                        bt[1][g] *= f1;
                    }
                }

                // values: O^T[d][heads] += codes^T x (p * scale * 2^ev)
                const int va0 = tr + 2 * t, va1 = va0 + 1, va8 = va0 + 8, va9 = va0 + 9;
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const float vsa_ = vsa[g] * vsc, vsb_ = vsb[g] * vsc;
                    const float vba = __half2float(svb[ra * G + g]);
                    const float vbb = __half2float(svb[rb * G + g]);
                    bt[0][g] = fmaf(pr[0], vba, fmaf(pr[2], vbb, bt[0][g]));
                    bt[1][g] = fmaf(pr[1], vba, fmaf(pr[3], vbb, bt[1][g]));
                    const uint32_t b0 = movmatrix_t(pack_half2(pr[0] * vsa_, pr[1] * vsa_));
                    const uint32_t b1 = movmatrix_t(pack_half2(pr[2] * vsb_, pr[3] * vsb_));
                    constexpr int NW = S::kCV >= 4 ? S::kCV / 4 : 1;
                    uint32_t w0[NW], w1[NW], w8[NW], w9[NW];
                    const int byte = g * S::kGB + gid * S::kCV;
                    lds_words<S::kCV>(vst + swz<S>(va0, byte), w0);
                    lds_words<S::kCV>(vst + swz<S>(va1, byte), w1);
                    lds_words<S::kCV>(vst + swz<S>(va8, byte), w8);
                    lds_words<S::kCV>(vst + swz<S>(va9, byte), w9);
#pragma unroll
                    for (int m = 0; m < S::kSteps; ++m) {
                        uint32_t a[4];
                        if constexpr (BITS == 4) {
                            const int wi = m / 4, bi = m % 4;
                            const uint32_t sel = (uint32_t)bi | ((uint32_t)(4 + bi) << 8);
                            const uint32_t x = prmt(w0[wi], w1[wi], sel);
                            const uint32_t y = prmt(w8[wi], w9[wi], sel);
                            a[0] = x & 0x000F000Fu;
                            a[1] = x & 0x00F000F0u;
                            a[2] = y & 0x000F000Fu;
                            a[3] = y & 0x00F000F0u;
                        } else {
                            const int wi = (2 * m) / 4, bi = (2 * m) % 4;
                            const uint32_t sl = (uint32_t)bi | ((uint32_t)(4 + bi) << 8);
                            const uint32_t sh = sl + 0x101u;
                            a[0] = prmt(w0[wi], w1[wi], sl) & 0x00FF00FFu;
                            a[1] = prmt(w0[wi], w1[wi], sh) & 0x00FF00FFu;
                            a[2] = prmt(w8[wi], w9[wi], sl) & 0x00FF00FFu;
                            a[3] = prmt(w8[wi], w9[wi], sh) & 0x00FF00FFu;
                        }
                        mma_f16_16816(O[g * S::kSteps + m], a, b0, b1, O[g * S::kSteps + m]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
        }

        // sums over the eight row lanes of each head column
#pragma unroll
        for (int off = 4; off <= 16; off <<= 1) {
            l[0] += __shfl_xor_sync(~0u, l[0], off);
            l[1] += __shfl_xor_sync(~0u, l[1], off);
#pragma unroll
            for (int g = 0; g < G; ++g) {
                bt[0][g] += __shfl_xor_sync(~0u, bt[0][g], off);
                bt[1][g] += __shfl_xor_sync(~0u, bt[1][g], off);
            }
        }
        consumer_sync();  // every warp is done with the ring
        float *wm = reinterpret_cast<float *>(ring);       // [warps][nrep]
        float *wl = wm + kCWarps * nrep;                   // [warps][nrep]
        float *wo = wl + kCWarps * nrep;                   // [warps][nrep][D]
        const int evf = ev == 127 ? 0 : ev;  // a warp without rows holds zeros
        const float fa = pow2i(24 - evf), fb = BITS == 4 ? pow2i(20 - evf) : fa;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int h = 2 * t + hh;
            if (h < nrep) {
                if (gid == 0) {
                    wm[warp * nrep + h] = m2[hh];
                    wl[warp * nrep + h] = l[hh];
                }
                float *o = wo + (warp * nrep + h) * D;
#pragma unroll
                for (int g = 0; g < G; ++g)
#pragma unroll
                    for (int m = 0; m < S::kSteps; ++m) {
                        const int d = g * GROUP + gid * (GROUP / 8) + 2 * m;
                        o[d] = fmaf(O[g * S::kSteps + m][hh], fa, bt[hh][g]);
                        o[d + 1] = fmaf(O[g * S::kSteps + m][2 + hh], fb, bt[hh][g]);
                    }
            }
        }
    }
    __syncthreads();

    // the eight warps, in warp order (log2 units)
    const float *wm = reinterpret_cast<const float *>(ring);
    const float *wl = wm + kCWarps * nrep;
    const float *wo = wl + kCWarps * nrep;
    float *cm = const_cast<float *>(wo) + kCWarps * nrep * D;   // [nrep]
    float *cl = cm + nrep;                                      // [nrep]
    float *co = cl + nrep;                                      // [nrep][D]
    for (int i = threadIdx.x; i < nrep * D; i += kAttnThreads) {
        const int j = i / D, d = i - j * D;
        float M = -INFINITY;
        for (int w = 0; w < kCWarps; ++w) M = fmaxf(M, wm[w * nrep + j]);
        float L = 0.f, Ov = 0.f;
        for (int w = 0; w < kCWarps; ++w) {
            const float mw = wm[w * nrep + j];
            const float g = mw == -INFINITY ? 0.f : exp2f(mw - M);  // a warp with no rows
            L = fmaf(wl[w * nrep + j], g, L);
            Ov = fmaf(wo[(w * nrep + j) * D + d], g, Ov);
        }
        co[j * D + d] = Ov;
        if (d == 0) {
            cm[j] = M;
            cl[j] = L;
        }
    }
    __syncthreads();

    // the cluster's CTAs, in rank order; rank r writes its share of o
    const int C = p.csize;
    if (C > 1) cluster_sync();
    const int total = nrep * D;
    const int chunk = (total + C - 1) / C;
    const uint32_t bm = smem_u32(cm), bl = smem_u32(cl), bo = smem_u32(co);
    for (int i = rank * chunk + (int)threadIdx.x; i < min(total, (rank + 1) * chunk);
         i += kAttnThreads) {
        const int j = i / D, d = i - j * D;
        float L = 0.f, Ov = 0.f;
        if (C == 1) {
            L = cl[j];
            Ov = co[i];
        } else {
            // every rank's (max, sum, o) loaded at once, then folded in rank order
            float mr[16], lr[16], orr[16];
#pragma unroll
            for (int rr = 0; rr < 16; ++rr)
                if (rr < C) {
                    mr[rr] = ld_dsmem_f32(map_to_rank(bm + 4u * j, (uint32_t)rr));
                    lr[rr] = ld_dsmem_f32(map_to_rank(bl + 4u * j, (uint32_t)rr));
                    orr[rr] = ld_dsmem_f32(map_to_rank(bo + 4u * (uint32_t)i, (uint32_t)rr));
                }
            float M = -INFINITY;
#pragma unroll
            for (int rr = 0; rr < 16; ++rr)
                if (rr < C) M = fmaxf(M, mr[rr]);
#pragma unroll
            for (int rr = 0; rr < 16; ++rr)
                if (rr < C && mr[rr] != -INFINITY) {  // a block with no rows adds nothing
                    const float g = exp2f(mr[rr] - M);
                    L = fmaf(lr[rr], g, L);
                    Ov = fmaf(orr[rr], g, Ov);
                }
        }
        const float v = Ov / L;
        const size_t oi = (size_t)(kv * nrep + j) * D + d;
        if (p.bf16)
            static_cast<__nv_bfloat16 *>(p.out)[oi] = __float2bfloat16_rn(v);
        else
            static_cast<__half *>(p.out)[oi] = __float2half_rn(v);
    }
    if (C > 1) cluster_sync();  // keep this CTA's results until every rank has read them
}

template <int BITS, int D, int GROUP>
size_t attn_smem_t(int stages, int nrep) {
    using S = Shape<BITS, D, GROUP>;
    const size_t merge = 4 * (size_t)((kCWarps + 1) * nrep * (D + 2));
    const size_t ring = std::max((size_t)stages * S::kStageBytes, merge);
    const size_t tail = (size_t)(D / 16) * 32 * 8 + 4 * (size_t)(8 * D + 8 * S::kG + 16) +
                        16 * (size_t)kMaxStages + 16;
    return 1024 + ring + tail;
}

template <int BITS, int D, int GROUP>
int attn_max_stages() {
    using S = Shape<BITS, D, GROUP>;
    return std::max(1, std::min(kMaxStages, kRingBudget / S::kStageBytes));
}

// Co-resident clusters of each size 1..16 for this instantiation (queried once).
template <int BITS, int D, int GROUP>
const int *attn_active_clusters() {
    static int n[17];
    static std::once_flag once;
    std::call_once(once, [] {
        auto kern = attn_kernel<BITS, D, GROUP>;
        const size_t smem = attn_smem_t<BITS, D, GROUP>(attn_max_stages<BITS, D, GROUP>(), 8);
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        for (int c = 1; c <= 16; ++c) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3((unsigned)(c * 8), 1, 1);
            cfg.blockDim = dim3(kAttnThreads, 1, 1);
            cfg.dynamicSmemBytes = smem;
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

// Cluster size: the c minimising (waves of clusters) x (stages per CTA),
// the smaller c on ties.
template <int BITS, int D, int GROUP>
int attn_pick_cluster(int64_t KV, int64_t N) {
    const int *n = attn_active_clusters<BITS, D, GROUP>();
    const int64_t maxc = std::min<int64_t>(16, std::max<int64_t>(1, (N + kStageRows - 1) / kStageRows));
    int best = 1;
    int64_t best_cost = INT64_MAX;
    for (int c = 1; c <= maxc; ++c) {
        if (n[c] < 1) continue;
        const int64_t waves = (KV + n[c] - 1) / n[c];
        const int64_t block = ((N + c - 1) / c + kTile - 1) / kTile * kTile;
        const int64_t cost = waves * ((block + kStageRows - 1) / kStageRows);
        if (cost < best_cost) {
            best_cost = cost;
            best = c;
        }
    }
    return best;
}

struct AttnPlan {
    int cluster, block, stages;
    size_t smem;
};

struct AttnLaunch {
    int dtype;
    const void *q;
    const uint32_t *kw, *vw;
    const void *ks, *kb, *vs, *vb;
    void *out;
    int64_t H, KV, N;
    cudaStream_t stream;
};

template <int BITS, int D, int GROUP>
cudaError_t attn_run(const AttnLaunch &L, AttnPlan *plan) {
    using S = Shape<BITS, D, GROUP>;
    const int C = attn_pick_cluster<BITS, D, GROUP>(L.KV, L.N);
    AttnParams prm;
    prm.q = L.q;
    prm.out = L.out;
    void *err = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&err, g_attn_error);
    if (e != cudaSuccess) return e;
    prm.err = static_cast<uint32_t *>(err);
    prm.KV = (int)L.KV;
    prm.N = (int)L.N;
    prm.nrep = (int)(L.H / L.KV);
    prm.csize = C;
    prm.block = (int)(((L.N + C - 1) / C + kTile - 1) / kTile * kTile);
    const int nst = (prm.block + kStageRows - 1) / kStageRows;
    prm.stages = std::max(1, std::min(attn_max_stages<BITS, D, GROUP>(), nst));
    prm.bf16 = L.dtype == AQ_BF16;
    if (plan) {
        *plan = {C, prm.block, prm.stages, attn_smem_t<BITS, D, GROUP>(prm.stages, prm.nrep)};
        return cudaSuccess;
    }

    const uint64_t rows = (uint64_t)(L.KV * L.N);
    const CUtensorMapSwizzle swz = S::kW == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                                   : S::kW == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                 : CU_TENSOR_MAP_SWIZZLE_32B;
    CUtensorMap m[6];
    if (!tmap_2d(&m[0], CU_TENSOR_MAP_DATA_TYPE_UINT8, L.kw, S::kRB, rows, S::kRB, S::kW,
                 kStageRows, swz) ||
        !tmap_2d(&m[1], CU_TENSOR_MAP_DATA_TYPE_UINT8, L.vw, S::kRB, rows, S::kRB, S::kW,
                 kStageRows, swz))
        return cudaErrorInvalidValue;
    const void *sp[4] = {L.ks, L.kb, L.vs, L.vb};
    for (int i = 0; i < 4; ++i) {
        const uint64_t dims[1] = {rows * S::kG};
        const uint32_t box[1] = {(uint32_t)S::kSBox};
        if (!tmap_encode(&m[2 + i], CU_TENSOR_MAP_DATA_TYPE_UINT16, 1, sp[i], dims, nullptr, box,
                         CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
    }
    auto kern = attn_kernel<BITS, D, GROUP>;
    attn_active_clusters<BITS, D, GROUP>();  // sets the kernel attributes
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(L.KV * C), 1, 1);
    cfg.blockDim = dim3(kAttnThreads, 1, 1);
    cfg.dynamicSmemBytes = attn_smem_t<BITS, D, GROUP>(prm.stages, prm.nrep);
    cfg.stream = L.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, prm, m[0], m[1], m[2], m[3], m[4], m[5]);
}

template <int BITS, int D>
cudaError_t attn_group(int group, const AttnLaunch &L, AttnPlan *c) {
    if constexpr (D == 64) {
        return group == 32 ? attn_run<BITS, D, 32>(L, c) : attn_run<BITS, D, 64>(L, c);
    } else {
        return group == 32   ? attn_run<BITS, D, 32>(L, c)
               : group == 64 ? attn_run<BITS, D, 64>(L, c)
                             : attn_run<BITS, D, 128>(L, c);
    }
}

template <int BITS>
cudaError_t attn_dim(int64_t D, int group, const AttnLaunch &L, AttnPlan *c) {
    switch (D) {
        case 64: return attn_group<BITS, 64>(group, L, c);
        case 128: return attn_group<BITS, 128>(group, L, c);
        default: return attn_group<BITS, 256>(group, L, c);
    }
}

cudaError_t attn_dispatch(int64_t D, int bits, int group, const AttnLaunch &L, AttnPlan *c) {
    return bits == 4 ? attn_dim<4>(D, group, L, c) : attn_dim<8>(D, group, L, c);
}

}  // namespace

bool attention_supported(int64_t H, int64_t KV, int64_t N, int64_t D, int bits, int group) {
    if (H < 1 || KV < 1 || H % KV != 0 || N < 1) return false;
    const int64_t nrep = H / KV;
    if (nrep != 1 && nrep != 2 && nrep != 4 && nrep != 8) return false;
    if (D != 64 && D != 128 && D != 256) return false;
    if (bits != 4 && bits != 8) return false;
    if (group != 32 && group != 64 && group != 128) return false;
    if (D % group != 0) return false;
    // row and scale-element indices stay in int
    return KV * N <= INT32_MAX / 16 && KV * N * (D / group) <= INT32_MAX / 2;
}

int attention_describe(int64_t H, int64_t KV, int64_t N, int64_t D, int bits, int group,
                       char *buf, int len) {
    AttnLaunch L = {};
    L.H = H;
    L.KV = KV;
    L.N = N;
    AttnPlan pl = {};
    if (attn_dispatch(D, bits, group, L, &pl) != cudaSuccess) return snprintf(buf, len, "no device");
    return snprintf(buf, len, "attn cluster=%d block=%d stages=%d smem=%zu grid=%lld", pl.cluster,
                    pl.block, pl.stages, pl.smem, (long long)(KV * pl.cluster));
}

cudaError_t attention_launch(int dtype, const void *q, const uint32_t *kw, const void *ks,
                             const void *kb, const uint32_t *vw, const void *vs, const void *vb,
                             int64_t H, int64_t KV, int64_t N, int64_t D, int bits, int group,
                             void *out, cudaStream_t stream) {
    const AttnLaunch L = {dtype, q, kw, vw, ks, kb, vs, vb, out, H, KV, N, stream};
    return attn_dispatch(D, bits, group, L, nullptr);
}

cudaError_t attn_read_error(uint32_t *code, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(code, g_attn_error, sizeof(uint32_t));
    if (e != cudaSuccess || !clear) return e;
    const uint32_t zero = 0;
    return cudaMemcpyToSymbol(g_attn_error, &zero, sizeof(uint32_t));
}

}  // namespace aq
