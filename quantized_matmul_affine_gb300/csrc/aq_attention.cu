// Decode attention over a quantised KV cache: for one query row per head,
//   o[h] = softmax(q[h] . Kd[kv]^T) . Vd[kv],   kv = h / (H / KV),
// with K and V stored in the affine format (4 or 8 bits, one fp16 scale and
// bias per group of 32/64/128 values along the head dimension).  The
// operator of the fused decode kernel of the mlx-bun 0.0.4 page
// (src/model/fused-decode-kernel.ts: flash-decoding split over the cached rows, the
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
//   * A producer warp streams stages of one tile per consumer warp (or warp
//     pair): 256 rows, 128 when a row is 256 bytes, 96 at D = 512.  K and V
//     codes arrive by 2-D TMA (swizzled so that the fragment reads below are
//     free of bank conflicts), their scales and biases by 1-D TMA, into a
//     shared-memory ring.
//   * Each of 8 consumer warps takes a tile of two 16-row blocks of a stage
//     (one block when a row is 256 bytes or more); at D = 512, 12 consumer
//     warps take 6 tiles in pairs, each warp half of the head dimension.
//     Scores on the tensor cores, per block S[16 rows][8 heads] =
//     codes x q', the codes as the exact fp16 subnormals code * 2^-24 (or
//     2^-20 where a nibble sits at bit 4), q' = q * 2^e per head in fp16;
//     one m16n8k16 chain per group, then s = scale * sum(q code) +
//     bias * sum(q) in fp32.
//   * Online softmax in base 2 on the fragment; the probabilities, times the
//     value scale of their row and group (and 2^ev, a per-warp power of two
//     lowered as larger scales appear, which keeps them in the fp16 range
//     and mostly out of its subnormals), are transposed in registers
//     (movmatrix) into the B operand of O^T[d][heads] += codes^T x P'; the
//     value biases enter as sum(p * bias) per (head, group) in fp32.
//   * The warps' (max, sum, o) merge through shared memory in warp order, the
//     cluster's CTAs then in rank order; o is rounded once.
//   * Launched with programmatic stream serialisation: the next kernel may
//     launch onto the SMs this grid leaves free, and this grid's first reads
//     wait for the previous grid.
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

constexpr int kMaxStages = 8;
constexpr int kRingBudget = 160 * 1024;
constexpr float kLog2e = 1.4426950408889634f;

struct AttnParams {
    const void *q;
    void *out;
    uint32_t *err;
    int KV, N, nrep;
    int block;          // cached rows per CTA (multiple of 16)
    int csize;          // CTAs per cluster
    int nclus;          // clusters per KV head (> 1 only with a workspace)
    int stages;         // ring depth
    int bf16;
    // workspace (nclus > 1): per (KV head, cluster, query head) the
    // cluster's max and sum (log2 units) and its unnormalised o, and one
    // arrival counter per KV head (zero between calls)
    float *ws_m, *ws_l, *ws_o;
    unsigned *cnt;
};

template <int BITS, int D, int GROUP>
struct Shape {
    // kSplit = 2 gives each tile to a pair of warps, each taking half of the
    // head dimension (partial scores cross shared memory every tile).  It
    // measured slower than one warp per tile up to D = 256, so only D = 512
    // takes it: there one warp would need 128 accumulator registers.
    static constexpr int kSplit = D == 512 ? 2 : 1;
    static constexpr int kPairs = kSplit == 2 ? 6 : 8;  // warp tiles per stage
    static constexpr int kCWarps = kSplit * kPairs;     // consumer warps
    static constexpr int kThreads = (kCWarps + 1) * 32; // + the TMA producer warp
    static constexpr int kRB = D * BITS / 8;            // bytes of one cached row
    static constexpr int kW = kRB < 128 ? kRB : 128;    // TMA box width = swizzle span
    static constexpr int kBoxes = kRB / kW;
    static constexpr uint32_t kSwz = kW == 128 ? 7u : kW == 64 ? 3u : 1u;
    static constexpr int kG = D / GROUP;                // groups per row
    static constexpr int kGB = GROUP * BITS / 8;        // bytes of one group of a row
    static constexpr int kCK = kGB / 4;                 // bytes a lane takes per row (scores)
    static constexpr int kCV = kGB / 8;                 // bytes a lane takes per row (values)
    static constexpr int kSteps = GROUP / 16;           // k-steps / M-tiles per group
    // 16-row blocks a warp takes per stage: two (32 rows) unless a row is 256
    // bytes, where a 256-row stage would leave room for only one in the ring
    static constexpr int kRBk = kRB <= 128 ? 2 : 1;
    static constexpr int kTileRows = 16 * kRBk;
    static constexpr int kStageRows = kTileRows * kPairs;
    // with kSplit = 2 each warp of a pair takes half of the head dimension's
    // 16-wide units (k-steps of the scores, M-tiles of the values): whole
    // groups when there are several, else half of the one group's steps
    static constexpr int kGH = kSplit == 1 ? kG : kG >= 2 ? kG / 2 : 1;  // groups per warp
    static constexpr int kHS = kSplit == 1 || kG >= 2 ? kSteps : kSteps / 2;  // steps per group
    static constexpr int kHU = kGH * kHS;               // units per warp (D / 16 / kSplit)
    // scales: kStageRows rows x G halves from a 16-byte aligned start (up to
    // 7 before), in boxes of a multiple of 64 halves so that every box lands
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
    return (uint32_t)(byte / S::kW) * (S::kStageRows * S::kW) + (lin ^ (((lin >> 7) & S::kSwz) << 4));
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

// Neither has side effects, so neither is volatile: the compiler may then
// interleave the independent MMA chains of a tile instead of issuing each
// chain's dependent steps back to back.
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t a) {
    uint32_t d;
    asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
    return d;
}

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

template <int NWARPS>
__device__ __forceinline__ void consumer_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(NWARPS * 32) : "memory");
}

__device__ __forceinline__ float4 ld_dsmem_v4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
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
__global__ void __launch_bounds__(Shape<BITS, D, GROUP>::kThreads, 1)
    attn_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ CUtensorMap tm_kw,
                const __grid_constant__ CUtensorMap tm_vw, const __grid_constant__ CUtensorMap tm_ks,
                const __grid_constant__ CUtensorMap tm_kb, const __grid_constant__ CUtensorMap tm_vs,
                const __grid_constant__ CUtensorMap tm_vb) {
    using S = Shape<BITS, D, GROUP>;
    constexpr int G = S::kG, RB = S::kRBk, SR = S::kStageRows;
    constexpr int kSplit = S::kSplit, kPairs = S::kPairs, kCWarps = S::kCWarps;
    constexpr int kAttnThreads = S::kThreads;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *ring = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int merge_bytes = (4 * p.nrep * ((kPairs + 1) * D + 3 * kPairs + 2) + 1023) & ~1023;
    uint8_t *tail = ring + max(p.stages * S::kStageBytes, merge_bytes);
    float4 *exch = reinterpret_cast<float4 *>(tail);    // [pairs][2 slots][2 halves][32][RB]
    uint2 *qfrag = reinterpret_cast<uint2 *>(exch + (kSplit == 2 ? kPairs * 2 * 2 * 32 * RB : 0));
    float *qf = reinterpret_cast<float *>(qfrag + (D / 16) * 32);   // [8][D]  q * 2^e
    float *qs2 = qf + 8 * D;                                        // [8][G]  sum(q) log2 e
    float *qsc = qs2 + 8 * G;                                       // [8]     2^(24-e) log2 e
    uint64_t *full = reinterpret_cast<uint64_t *>(qsc + 16);
    uint64_t *empty = full + kMaxStages;
    uint64_t *xbar = empty + kMaxStages;     // [pairs][2 slots]: the score exchange
    int *flag_s = reinterpret_cast<int *>(xbar + 2 * kPairs);
    volatile int *flag = flag_s;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gid = lane >> 2, t = lane & 3;
    const int kv = (int)blockIdx.x / (p.csize * p.nclus);
    const int clus = ((int)blockIdx.x / p.csize) % p.nclus;
    const int rank = (int)blockIdx.x % p.csize;
    const int n0 = (clus * p.csize + rank) * p.block;
    const int n1 = min(p.N, n0 + p.block);
    const int nst = n1 > n0 ? (n1 - n0 + SR - 1) / SR : 0;
    const int nrep = p.nrep;
    const long long row_base = (long long)kv * p.N;

    if (threadIdx.x == 0) {
        for (int i = 0; i < p.stages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kCWarps);
        }
        for (int i = 0; i < 2 * kPairs; ++i) mbar_init(&xbar[i], 64);
        *flag_s = 0;
        fence_mbar_init();
    }
    __syncthreads();
    // the next kernel of the stream may launch now (onto SMs this grid does
    // not hold); this grid's reads of q and the caches wait for the previous
    // one to complete
    launch_dependents();

    if (warp == kCWarps) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            grid_dependency_wait();
            int issued = 0;
            for (int st = 0; st < nst && !*flag; ++st) {
                const int slot = st % p.stages, lap = st / p.stages;
                if (lap > 0 && !mbar_wait(&empty[slot], (lap - 1) & 1)) {
                    attn_record(flag, p.err, ERR_ATTN_EMPTY);
                    break;
                }
                uint8_t *sb = ring + slot * S::kStageBytes;
                const int row0 = (int)(row_base + n0 + st * SR);
                const int x0 = (row0 * G) & ~7;
                mbar_arrive_expect_tx(&full[slot], (uint32_t)S::kTx);
#pragma unroll
                for (int b = 0; b < S::kBoxes; ++b) {
                    tma_load_2d(sb + b * SR * S::kW, &tm_kw, b * S::kW, row0, &full[slot]);
                    tma_load_2d(sb + S::kCodeBytes + b * SR * S::kW, &tm_vw, b * S::kW, row0,
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
        grid_dependency_wait();
        if (warp < 8) {
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
        consumer_sync<kCWarps>();
        // B fragments of q' for k-step k, lane (hg, tt): head hg, the k of
        // thread tt's code registers 2s and 2s+1 (both halves)
        for (int e = threadIdx.x; e < (D / 16) * 32; e += kCWarps * 32) {
            const int k = e >> 5, hg = (e >> 2) & 7, tt = e & 3;
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
                        d = g * GROUP + tt * (GROUP / 4) + 8 * (i / 4) + (i % 4) + 4 * hf;
                        if (i & 1) f = 0.0625f;
                    } else {
                        d = g * GROUP + tt * (GROUP / 4) + 4 * (i / 2) + (i % 2) + 2 * hf;
                    }
                    v[hf] = hg < nrep ? qf[hg * D + d] * f : 0.f;
                }
                r[j] = pack_half2(v[0], v[1]);
            }
            qfrag[e] = make_uint2(r[0], r[1]);
        }
        const float qsc0 = qsc[2 * t], qsc1 = qsc[2 * t + 1];
        consumer_sync<kCWarps>();

        // ------------------------------------------------------------ main loop
        // warps w and w + kPairs share a tile when split
        const int pw = warp % kPairs, half = kSplit == 2 ? warp / kPairs : 0;
        const int g0 = G >= 2 ? half * S::kGH : 0;             // first group of this warp
        const int ks0 = G >= 2 ? 0 : half * S::kHS;           // first step within a group
        float m2[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
        // p * scale * 2^ev enters the value product: ev keeps the largest
        // |scale| seen so far below 2^15 (fp16 range, few subnormals); it only
        // decreases, and O is rescaled with it like with the running max
        int ev = 127;
        float bt[2][S::kGH];
        float O[S::kHU][4];
#pragma unroll
        for (int g = 0; g < S::kGH; ++g) bt[0][g] = bt[1][g] = 0.f;
#pragma unroll
        for (int i = 0; i < S::kHU; ++i) O[i][0] = O[i][1] = O[i][2] = O[i][3] = 0.f;

        int tile = 0;
        for (int st = 0; st < nst; ++st) {
            const int slot = st % p.stages, lap = st / p.stages;
            if (*flag) break;
            if (!mbar_wait(&full[slot], lap & 1)) {
                attn_record(flag, p.err, ERR_ATTN_FULL);
                break;
            }
            const int r0 = n0 + st * SR + pw * S::kTileRows;   // first row of the tile
            if (r0 < n1) {
                const uint8_t *kst = ring + slot * S::kStageBytes;
                const uint8_t *vst = kst + S::kCodeBytes;
                const int row0 = (int)(row_base + n0 + st * SR);
                const int soff = row0 * G - ((row0 * G) & ~7);
                const __half *sks = reinterpret_cast<const __half *>(vst + S::kCodeBytes) + soff;
                const __half *skb = sks + S::kSArr;
                const __half *svs = sks + 2 * S::kSArr;
                const __half *svb = sks + 3 * S::kSArr;
                const int tr = pw * S::kTileRows;                  // tile row in the stage

                // this half's part of the scores of block b: rows (16b + gid,
                // 16b + gid + 8) x heads (2t, 2t+1); t1 = sum scale * sum(q'
                // code), t2 = sum bias * sum(q) log2 e (once per group)
                float t1[RB][4], t2[RB][4];
#pragma unroll
                for (int b = 0; b < RB; ++b)
#pragma unroll
                    for (int i = 0; i < 4; ++i) t1[b][i] = t2[b][i] = 0.f;
#pragma unroll
                for (int gg = 0; gg < S::kGH; ++gg) {
                    const int g = g0 + gg;
                    const float q0 = qs2[(2 * t) * G + g], q1 = qs2[(2 * t + 1) * G + g];
#pragma unroll
                    for (int b = 0; b < RB; ++b) {
                        const int ra = tr + 16 * b + gid, rb = ra + 8;
                        constexpr int NBY = S::kHS * BITS / 2;   // bytes of the half's steps
                        uint32_t Ra[2 * S::kHS], Rb[2 * S::kHS];
#pragma unroll
                        for (int c = 0; c < (NBY + 15) / 16; ++c) {
                            constexpr int NB = NBY < 16 ? NBY : 16;
                            uint32_t wa[NB / 4], wb[NB / 4];
                            const int byte = g * S::kGB + t * S::kCK + ks0 * (BITS / 2) + c * 16;
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
                        for (int k = 0; k < S::kHS; ++k) {
                            const uint2 bq = qfrag[(g * S::kSteps + ks0 + k) * 32 + lane];
                            const uint32_t a[4] = {Ra[2 * k], Rb[2 * k], Ra[2 * k + 1],
                                                   Rb[2 * k + 1]};
                            mma16816(acc, a, bq.x, bq.y);
                        }
                        const float ksa = __half2float(sks[ra * G + g]);
                        const float ksb = __half2float(sks[rb * G + g]);
                        t1[b][0] = fmaf(ksa, acc[0], t1[b][0]);
                        t1[b][1] = fmaf(ksa, acc[1], t1[b][1]);
                        t1[b][2] = fmaf(ksb, acc[2], t1[b][2]);
                        t1[b][3] = fmaf(ksb, acc[3], t1[b][3]);
                        if (ks0 == 0) {
                            const float kba = __half2float(skb[ra * G + g]);
                            const float kbb = __half2float(skb[rb * G + g]);
                            t2[b][0] = fmaf(kba, q0, t2[b][0]);
                            t2[b][1] = fmaf(kba, q1, t2[b][1]);
                            t2[b][2] = fmaf(kbb, q0, t2[b][2]);
                            t2[b][3] = fmaf(kbb, q1, t2[b][3]);
                        }
                    }
                }
                // the pair's two parts, exchanged through shared memory: two
                // slots by tile parity, each with an mbarrier that completes
                // when all 64 lanes of the pair have written (a slot is written
                // again only after the partner has passed the next exchange,
                // so after it has read this one)
                float s[RB][4];
#pragma unroll
                for (int b = 0; b < RB; ++b) {
                    s[b][0] = fmaf(qsc0, t1[b][0], t2[b][0]);
                    s[b][1] = fmaf(qsc1, t1[b][1], t2[b][1]);
                    s[b][2] = fmaf(qsc0, t1[b][2], t2[b][2]);
                    s[b][3] = fmaf(qsc1, t1[b][3], t2[b][3]);
                }
                if constexpr (kSplit == 2) {
                    float4 *xs = exch + ((pw * 2 + (tile & 1)) * 2) * 32 * RB;
                    uint64_t *xb = &xbar[pw * 2 + (tile & 1)];
#pragma unroll
                    for (int b = 0; b < RB; ++b)
                        xs[(half * 32 + lane) * RB + b] =
                            make_float4(s[b][0], s[b][1], s[b][2], s[b][3]);
                    mbar_arrive(xb);
                    if (!mbar_wait(xb, (tile >> 1) & 1)) attn_record(flag, p.err, ERR_ATTN_PAIR);
#pragma unroll
                    for (int b = 0; b < RB; ++b) {
                        const float4 o = xs[((1 - half) * 32 + lane) * RB + b];
                        s[b][0] += o.x;   // the same sums in both warps (a + b == b + a)
                        s[b][1] += o.y;
                        s[b][2] += o.z;
                        s[b][3] += o.w;
                    }
                    ++tile;
                }
#pragma unroll
                for (int b = 0; b < RB; ++b) {
                    if (r0 + 16 * b + gid >= n1) s[b][0] = s[b][1] = -INFINITY;
                    if (r0 + 16 * b + gid + 8 >= n1) s[b][2] = s[b][3] = -INFINITY;
                }

                // online softmax (base 2) per head column, once for the tile
                float mx0 = fmaxf(s[0][0], s[0][2]), mx1 = fmaxf(s[0][1], s[0][3]);
#pragma unroll
                for (int b = 1; b < RB; ++b) {
                    mx0 = fmaxf(mx0, fmaxf(s[b][0], s[b][2]));
                    mx1 = fmaxf(mx1, fmaxf(s[b][1], s[b][3]));
                }
#pragma unroll
                for (int off = 4; off <= 16; off <<= 1) {
                    mx0 = fmaxf(mx0, __shfl_xor_sync(~0u, mx0, off));
                    mx1 = fmaxf(mx1, __shfl_xor_sync(~0u, mx1, off));
                }
                const float mn0 = fmaxf(m2[0], mx0), mn1 = fmaxf(m2[1], mx1);
                const float f0 = exp2f(m2[0] - mn0), f1 = exp2f(m2[1] - mn1);
                m2[0] = mn0;
                m2[1] = mn1;
                float pr[RB][4];
                float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
                for (int b = 0; b < RB; ++b) {
                    pr[b][0] = exp2f(s[b][0] - mn0);
                    pr[b][1] = exp2f(s[b][1] - mn1);
                    pr[b][2] = exp2f(s[b][2] - mn0);
                    pr[b][3] = exp2f(s[b][3] - mn1);
                    ls0 += pr[b][0] + pr[b][2];
                    ls1 += pr[b][1] + pr[b][3];
                }
                l[0] = fmaf(l[0], f0, ls0);
                l[1] = fmaf(l[1], f1, ls1);

                // value scales of the lane's rows in this half's groups; their
                // largest |scale| sets ev
                float vsa[RB][S::kGH], vsb[RB][S::kGH];
                float vmx = 0.f;
#pragma unroll
                for (int b = 0; b < RB; ++b)
#pragma unroll
                    for (int gg = 0; gg < S::kGH; ++gg) {
                        vsa[b][gg] = __half2float(svs[(tr + 16 * b + gid) * G + g0 + gg]);
                        vsb[b][gg] = __half2float(svs[(tr + 16 * b + gid + 8) * G + g0 + gg]);
                        vmx = fmaxf(vmx, fmaxf(fabsf(vsa[b][gg]), fabsf(vsb[b][gg])));
                    }
                vmx = __uint_as_float(__reduce_max_sync(~0u, __float_as_uint(vmx)));
                const int ev_new = min(ev, exp_for(vmx));
                const float r = ev_new - ev < -126 ? 0.f : pow2i(ev_new - ev);
                ev = ev_new;
                const float vsc = pow2i(ev);
                if (__any_sync(~0u, f0 != 1.f || f1 != 1.f || r != 1.f)) {
                    const float o0 = f0 * r, o1 = f1 * r;
#pragma unroll
                    for (int i = 0; i < S::kHU; ++i) {
                        O[i][0] *= o0;
                        O[i][1] *= o1;
                        O[i][2] *= o0;
                        O[i][3] *= o1;
                    }
#pragma unroll
                    for (int gg = 0; gg < S::kGH; ++gg) {
                        bt[0][gg] *= f0;
                        bt[1][gg] *= f1;
                    }
                }

                // values: O^T[d][heads] += codes^T x (p * scale * 2^ev), 16 rows per MMA
#pragma unroll
                for (int gg = 0; gg < S::kGH; ++gg) {
                    const int g = g0 + gg;
#pragma unroll
                    for (int b = 0; b < RB; ++b) {
                        const int ra = tr + 16 * b + gid, rb = ra + 8;
                        const float vsa_ = vsa[b][gg] * vsc, vsb_ = vsb[b][gg] * vsc;
                        const float vba = __half2float(svb[ra * G + g]);
                        const float vbb = __half2float(svb[rb * G + g]);
                        bt[0][gg] = fmaf(pr[b][0], vba, fmaf(pr[b][2], vbb, bt[0][gg]));
                        bt[1][gg] = fmaf(pr[b][1], vba, fmaf(pr[b][3], vbb, bt[1][gg]));
                        const uint32_t b0 = movmatrix_t(pack_half2(pr[b][0] * vsa_, pr[b][1] * vsa_));
                        const uint32_t b1 = movmatrix_t(pack_half2(pr[b][2] * vsb_, pr[b][3] * vsb_));
                        // the half's M-tiles: 4-bit one byte each, 8-bit two
                        constexpr int NV = S::kHS * BITS / 4;
                        constexpr int NW = NV >= 4 ? NV / 4 : 1;
                        uint32_t w0[NW], w1[NW], w8[NW], w9[NW];
                        const int byte = g * S::kGB + gid * S::kCV + ks0 * (BITS / 4);
                        const int v0 = tr + 16 * b + 2 * t;
                        lds_words<NV>(vst + swz<S>(v0, byte), w0);
                        lds_words<NV>(vst + swz<S>(v0 + 1, byte), w1);
                        lds_words<NV>(vst + swz<S>(v0 + 8, byte), w8);
                        lds_words<NV>(vst + swz<S>(v0 + 9, byte), w9);
#pragma unroll
                        for (int m = 0; m < S::kHS; ++m) {
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
                            mma16816(O[gg * S::kHS + m], a, b0, b1);
                        }
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
            for (int gg = 0; gg < S::kGH; ++gg) {
                bt[0][gg] += __shfl_xor_sync(~0u, bt[0][gg], off);
                bt[1][gg] += __shfl_xor_sync(~0u, bt[1][gg], off);
            }
        }
        consumer_sync<kCWarps>();  // every warp is done with the ring
        float *wm = reinterpret_cast<float *>(ring);       // [pairs][nrep]
        float *wl = wm + kPairs * nrep;                    // [pairs][nrep]
        float *wo = wl + kPairs * nrep;                    // [pairs][nrep][D]
        const int evf = ev == 127 ? 0 : ev;  // a warp without rows holds zeros
        const float fa = pow2i(24 - evf), fb = BITS == 4 ? pow2i(20 - evf) : fa;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int h = 2 * t + hh;
            if (h < nrep) {
                if (gid == 0 && half == 0) {
                    wm[pw * nrep + h] = m2[hh];
                    wl[pw * nrep + h] = l[hh];
                }
                float *o = wo + (pw * nrep + h) * D;
#pragma unroll
                for (int gg = 0; gg < S::kGH; ++gg)
#pragma unroll
                    for (int m = 0; m < S::kHS; ++m) {
                        const int d = (g0 + gg) * GROUP + gid * (GROUP / 8) + 2 * (ks0 + m);
                        *reinterpret_cast<float2 *>(o + d) =
                            make_float2(fmaf(O[gg * S::kHS + m][hh], fa, bt[hh][gg]),
                                        fmaf(O[gg * S::kHS + m][2 + hh], fb, bt[hh][gg]));
                    }
            }
        }
    }
    __syncthreads();

    // the tiles, in tile order (log2 units): per-(tile, head) factors
    // first, then o four elements at a time
    const float *wm = reinterpret_cast<const float *>(ring);
    const float *wl = wm + kPairs * nrep;
    const float *wo = wl + kPairs * nrep;
    float *co = const_cast<float *>(wo) + kPairs * nrep * D;   // [nrep][D]
    float *cm = co + nrep * D;                                  // [nrep]
    float *cl = cm + nrep;                                      // [nrep]
    float *wg = cl + nrep;                                      // [pairs][nrep]
    if ((int)threadIdx.x < nrep) {
        const int j = threadIdx.x;
        float M = -INFINITY;
        for (int w = 0; w < kPairs; ++w) M = fmaxf(M, wm[w * nrep + j]);
        float L = 0.f;
        for (int w = 0; w < kPairs; ++w) {
            const float mw = wm[w * nrep + j];
            const float g = mw == -INFINITY ? 0.f : exp2f(mw - M);  // a tile with no rows
            wg[w * nrep + j] = g;
            L = fmaf(wl[w * nrep + j], g, L);
        }
        cm[j] = M;
        cl[j] = L;
    }
    __syncthreads();
    for (int i4 = threadIdx.x; i4 < nrep * D / 4; i4 += kAttnThreads) {
        const int j = (4 * i4) / D;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < kPairs; ++w) {
            const float g = wg[w * nrep + j];
            const float4 v = reinterpret_cast<const float4 *>(wo + w * nrep * D)[i4];
            acc.x = fmaf(v.x, g, acc.x);
            acc.y = fmaf(v.y, g, acc.y);
            acc.z = fmaf(v.z, g, acc.z);
            acc.w = fmaf(v.w, g, acc.w);
        }
        reinterpret_cast<float4 *>(co)[i4] = acc;
    }
    __syncthreads();

    // the cluster's CTAs, in rank order; rank r writes its share of o (or,
    // with several clusters a KV head, of the cluster's partial result)
    const int C = p.csize;
    if (C > 1) cluster_sync();
    const int total4 = nrep * D / 4;
    const int chunk4 = (total4 + C - 1) / C;
    const uint32_t bm = smem_u32(cm), bl = smem_u32(cl), bo = smem_u32(co);
    const size_t wpart = (size_t)(kv * p.nclus + clus) * nrep;  // (head, cluster) partials
    for (int i4 = rank * chunk4 + (int)threadIdx.x; i4 < min(total4, (rank + 1) * chunk4);
         i4 += kAttnThreads) {
        const int j = (4 * i4) / D, d = 4 * i4 - j * D;
        float L = 0.f, M = -INFINITY;
        float4 Ov = make_float4(0.f, 0.f, 0.f, 0.f);
        if (C == 1) {
            L = cl[j];
            M = cm[j];
            Ov = reinterpret_cast<const float4 *>(co)[i4];
        } else {
            // every rank's (max, sum, o) loaded at once, then folded in rank order
            float mr[16], lr[16];
            float4 orr[16];
#pragma unroll
            for (int rr = 0; rr < 16; ++rr)
                if (rr < C) {
                    mr[rr] = ld_dsmem_f32(map_to_rank(bm + 4u * j, (uint32_t)rr));
                    lr[rr] = ld_dsmem_f32(map_to_rank(bl + 4u * j, (uint32_t)rr));
                    orr[rr] = ld_dsmem_v4(map_to_rank(bo + 16u * (uint32_t)i4, (uint32_t)rr));
                }
#pragma unroll
            for (int rr = 0; rr < 16; ++rr)
                if (rr < C) M = fmaxf(M, mr[rr]);
#pragma unroll
            for (int rr = 0; rr < 16; ++rr)
                if (rr < C && mr[rr] != -INFINITY) {  // a block with no rows adds nothing
                    const float g = exp2f(mr[rr] - M);
                    L = fmaf(lr[rr], g, L);
                    Ov.x = fmaf(orr[rr].x, g, Ov.x);
                    Ov.y = fmaf(orr[rr].y, g, Ov.y);
                    Ov.z = fmaf(orr[rr].z, g, Ov.z);
                    Ov.w = fmaf(orr[rr].w, g, Ov.w);
                }
        }
        if (p.nclus > 1) {
            reinterpret_cast<float4 *>(p.ws_o + (wpart + j) * D)[d / 4] = Ov;
            if (d == 0) {
                p.ws_m[wpart + j] = M;
                p.ws_l[wpart + j] = L;
            }
            continue;
        }
        const float inv[4] = {Ov.x / L, Ov.y / L, Ov.z / L, Ov.w / L};
        const size_t oi = (size_t)(kv * nrep + j) * D + d;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            if (p.bf16)
                static_cast<__nv_bfloat16 *>(p.out)[oi + k] = __float2bfloat16_rn(inv[k]);
            else
                static_cast<__half *>(p.out)[oi + k] = __float2half_rn(inv[k]);
        }
    }
    if (p.nclus > 1) __threadfence();  // the partials are visible GPU-wide before the count
    if (C > 1) cluster_sync();  // keep this CTA's results until every rank has read them
    if (p.nclus == 1) return;

    // Several clusters a KV head: the cluster that arrives last (one atomic
    // count a cluster, no waiting) adds the clusters' partials in cluster
    // order, writes o and sets the count back to zero for the next call.
    __shared__ int s_last;
    if (rank != 0) return;
    __syncthreads();  // the cluster barrier above covered every rank's writes
    if (threadIdx.x == 0) {
        const unsigned old = atomicAdd(&p.cnt[kv], 1u);
        s_last = old == (unsigned)(p.nclus - 1);
        __threadfence();
    }
    __syncthreads();
    if (!s_last) return;
    for (int i4 = (int)threadIdx.x; i4 < total4; i4 += kAttnThreads) {
        const int j = (4 * i4) / D, d = 4 * i4 - j * D;
        const size_t w0 = (size_t)kv * p.nclus * nrep + j;  // cluster c at w0 + c * nrep
        float M = -INFINITY;
        for (int c = 0; c < p.nclus; ++c) M = fmaxf(M, __ldcg(p.ws_m + w0 + (size_t)c * nrep));
        float L = 0.f;
        float4 Ov = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int c = 0; c < p.nclus; ++c) {
            const float mc = __ldcg(p.ws_m + w0 + (size_t)c * nrep);
            if (mc == -INFINITY) continue;  // a cluster with no rows adds nothing
            const float g = exp2f(mc - M);
            L = fmaf(__ldcg(p.ws_l + w0 + (size_t)c * nrep), g, L);
            const float4 v = __ldcg(reinterpret_cast<const float4 *>(
                                        p.ws_o + (w0 + (size_t)c * nrep) * D) +
                                    d / 4);
            Ov.x = fmaf(v.x, g, Ov.x);
            Ov.y = fmaf(v.y, g, Ov.y);
            Ov.z = fmaf(v.z, g, Ov.z);
            Ov.w = fmaf(v.w, g, Ov.w);
        }
        const float inv[4] = {Ov.x / L, Ov.y / L, Ov.z / L, Ov.w / L};
        const size_t oi = (size_t)(kv * nrep + j) * D + d;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            if (p.bf16)
                static_cast<__nv_bfloat16 *>(p.out)[oi + k] = __float2bfloat16_rn(inv[k]);
            else
                static_cast<__half *>(p.out)[oi + k] = __float2half_rn(inv[k]);
        }
    }
    if (threadIdx.x == 0) p.cnt[kv] = 0u;
}

template <int BITS, int D, int GROUP>
size_t attn_smem_t(int stages, int nrep) {
    using S = Shape<BITS, D, GROUP>;
    constexpr int kSplit = S::kSplit, kPairs = S::kPairs;
    const size_t merge =
        (4 * (size_t)nrep * ((kPairs + 1) * D + 3 * kPairs + 2) + 1023) & ~(size_t)1023;
    const size_t ring = std::max((size_t)stages * S::kStageBytes, merge);
    const size_t tail = (kSplit == 2 ? (size_t)kPairs * 2 * 2 * 32 * S::kRBk * 16 : 0) +
                        (size_t)(D / 16) * 32 * 8 + 4 * (size_t)(8 * D + 8 * S::kG + 16) +
                        16 * (size_t)kMaxStages + 16 * (size_t)kPairs + 16;
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
            cfg.blockDim = dim3(Shape<BITS, D, GROUP>::kThreads, 1, 1);
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

// Workspace of a plan with k clusters a KV head (k > 1): the arrival
// counters, then the partial maxima, sums and o, each 256-byte aligned.
struct AttnWs {
    size_t off_m, off_l, off_o, bytes;
};
inline AttnWs attn_ws_layout(int64_t KV, int k, int64_t nrep, int64_t D) {
    auto up = [](size_t b) { return (b + 255) / 256 * 256; };
    AttnWs w;
    const size_t parts = (size_t)(KV * k * nrep);
    w.off_m = up((size_t)KV * sizeof(unsigned));
    w.off_l = w.off_m + up(parts * sizeof(float));
    w.off_o = w.off_l + up(parts * sizeof(float));
    w.bytes = w.off_o + parts * (size_t)D * sizeof(float);
    return w;
}

struct AttnPick {
    int c, k;  // CTAs a cluster, clusters a KV head
};

// Cluster size c and clusters per KV head k: the pair minimising
// (waves of clusters) x (stages per CTA), plus, for k > 1, the cost of the
// merge across clusters (the partials through global memory, an atomic,
// one CTA's second merge: measured ~2-3 us, about the time of 2.3 stages of
// 64 KB, so charged as 2.3 x 64 KB / stage bytes stages); among equals the
// smaller k, then the smaller c.  k > 1 only when ws_bytes holds its
// workspace.  {0, 0} when no size can run (no device).
template <int BITS, int D, int GROUP>
AttnPick attn_pick(int64_t KV, int64_t N, int64_t nrep, size_t ws_bytes) {
    constexpr int SR = Shape<BITS, D, GROUP>::kStageRows;
    const int *n = attn_active_clusters<BITS, D, GROUP>();
    const int64_t maxc = std::min<int64_t>(16, std::max<int64_t>(1, (N + SR - 1) / SR));
    const int64_t maxct = std::max<int64_t>(1, (N + 15) / 16);  // CTAs of at least 16 rows
    AttnPick best = {0, 0};
    double best_cost = 1e300;
    for (int k = 1; k <= 16; ++k) {
        if (k > 1 && attn_ws_layout(KV, k, nrep, D).bytes > ws_bytes) break;
        for (int c = 1; c <= maxc; ++c) {
            if (n[c] < 1 || (int64_t)k * c > maxct) continue;
            const int64_t waves = (KV * k + n[c] - 1) / n[c];
            const int64_t block = ((N + (int64_t)k * c - 1) / ((int64_t)k * c) + 15) / 16 * 16;
            const double merge = 2.3 * 65536.0 / (double)Shape<BITS, D, GROUP>::kStageBytes;
            const double cost = (double)(waves * ((block + SR - 1) / SR)) + (k > 1 ? merge : 0.0);
            if (cost < best_cost) {
                best_cost = cost;
                best = {c, k};
            }
        }
    }
    return best;
}

struct AttnPlan {
    int cluster, block, stages, nclus;
    size_t smem, ws_bytes;
};

struct AttnLaunch {
    int dtype;
    const void *q;
    const uint32_t *kw, *vw;
    const void *ks, *kb, *vs, *vb;
    void *out;
    int64_t H, KV, N;
    cudaStream_t stream;
    void *ws;         // workspace, 256-byte aligned (may be null)
    size_t ws_bytes;  // its size (0: one cluster a KV head)
};

template <int BITS, int D, int GROUP>
cudaError_t attn_run(const AttnLaunch &L, AttnPlan *plan) {
    using S = Shape<BITS, D, GROUP>;
    const AttnPick pk = attn_pick<BITS, D, GROUP>(L.KV, L.N, L.H / L.KV, L.ws ? L.ws_bytes : 0);
    const int C = pk.c;
    if (C < 1) return cudaErrorNoDevice;
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
    prm.nclus = pk.k;
    const int64_t ctas = (int64_t)C * pk.k;  // CTAs a KV head
    prm.block = (int)(((L.N + ctas - 1) / ctas + 15) / 16 * 16);
    const int nst = (prm.block + S::kStageRows - 1) / S::kStageRows;
    prm.stages = std::max(1, std::min(attn_max_stages<BITS, D, GROUP>(), nst));
    prm.bf16 = L.dtype == AQ_BF16;
    const AttnWs wl = attn_ws_layout(L.KV, pk.k, prm.nrep, D);
    uint8_t *wsb = static_cast<uint8_t *>(L.ws);
    prm.cnt = pk.k > 1 ? reinterpret_cast<unsigned *>(wsb) : nullptr;
    prm.ws_m = pk.k > 1 ? reinterpret_cast<float *>(wsb + wl.off_m) : nullptr;
    prm.ws_l = pk.k > 1 ? reinterpret_cast<float *>(wsb + wl.off_l) : nullptr;
    prm.ws_o = pk.k > 1 ? reinterpret_cast<float *>(wsb + wl.off_o) : nullptr;
    if (plan) {
        *plan = {C, prm.block, prm.stages, pk.k,
                 attn_smem_t<BITS, D, GROUP>(prm.stages, prm.nrep), pk.k > 1 ? wl.bytes : 0};
        return cudaSuccess;
    }

    const uint64_t rows = (uint64_t)(L.KV * L.N);
    const CUtensorMapSwizzle swz = S::kW == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                                   : S::kW == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                 : CU_TENSOR_MAP_SWIZZLE_32B;
    CUtensorMap m[6];
    if (!tmap_2d(&m[0], CU_TENSOR_MAP_DATA_TYPE_UINT8, L.kw, S::kRB, rows, S::kRB, S::kW,
                 S::kStageRows, swz) ||
        !tmap_2d(&m[1], CU_TENSOR_MAP_DATA_TYPE_UINT8, L.vw, S::kRB, rows, S::kRB, S::kW,
                 S::kStageRows, swz))
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
    cfg.gridDim = dim3((unsigned)(L.KV * C * pk.k), 1, 1);
    cfg.blockDim = dim3(S::kThreads, 1, 1);
    cfg.dynamicSmemBytes = attn_smem_t<BITS, D, GROUP>(prm.stages, prm.nrep);
    cfg.stream = L.stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
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
        case 256: return attn_group<BITS, 256>(group, L, c);
        default: return attn_group<BITS, 512>(group, L, c);
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
    if (D != 64 && D != 128 && D != 256 && D != 512) return false;
    if (bits != 4 && bits != 8) return false;
    if (group != 32 && group != 64 && group != 128) return false;
    if (D % group != 0) return false;
    // row and scale-element indices stay in int
    return KV * N <= INT32_MAX / 16 && KV * N * (D / group) <= INT32_MAX / 2;
}

int attention_describe(int64_t H, int64_t KV, int64_t N, int64_t D, int bits, int group,
                       size_t ws_bytes, char *buf, int len) {
    AttnLaunch L = {};
    L.H = H;
    L.KV = KV;
    L.N = N;
    L.ws = ws_bytes ? reinterpret_cast<void *>(256) : nullptr;  // planning only
    L.ws_bytes = ws_bytes;
    AttnPlan pl = {};
    if (attn_dispatch(D, bits, group, L, &pl) != cudaSuccess) return snprintf(buf, len, "no device");
    if (ws_bytes == 0)
        return snprintf(buf, len, "attn cluster=%d block=%d stages=%d smem=%zu grid=%lld",
                        pl.cluster, pl.block, pl.stages, pl.smem, (long long)(KV * pl.cluster));
    return snprintf(buf, len,
                    "attn cluster=%d block=%d stages=%d smem=%zu grid=%lld "
                    "clusters_per_kv_head=%d workspace=%zu",
                    pl.cluster, pl.block, pl.stages, pl.smem,
                    (long long)(KV * pl.cluster * pl.nclus), pl.nclus, pl.ws_bytes);
}

size_t attention_workspace_bytes(int64_t H, int64_t KV, int64_t N, int64_t D, int bits,
                                 int group) {
    AttnLaunch L = {};
    L.H = H;
    L.KV = KV;
    L.N = N;
    L.ws = reinterpret_cast<void *>(256);  // planning only: any size allowed
    L.ws_bytes = (size_t)1 << 40;
    AttnPlan pl = {};
    if (attn_dispatch(D, bits, group, L, &pl) != cudaSuccess) return 0;
    return pl.ws_bytes;
}

cudaError_t attention_launch(int dtype, const void *q, const uint32_t *kw, const void *ks,
                             const void *kb, const uint32_t *vw, const void *vs, const void *vb,
                             int64_t H, int64_t KV, int64_t N, int64_t D, int bits, int group,
                             void *out, void *ws, size_t ws_bytes, cudaStream_t stream) {
    const AttnLaunch L = {dtype, q,  kw, vw, ks, kb, vs, vb, out, H, KV, N, stream,
                          ws,    ws_bytes};
    return attn_dispatch(D, bits, group, L, nullptr);
}

// Scratch for aq_attention_decode_static: the workspace of the several-
// cluster plan in device memory the library owns, for callers that cannot
// allocate per call (plain C hosts without a device allocator at hand, or
// decode loops that must not pay for a synchronising cudaMalloc each step).
// Zero-initialised at module load; the counters at its start are zero again
// after every call.  One array per device context, so calls that overlap in
// time on one device (two streams) would share it and race.
static __device__ __align__(256) uint8_t g_attn_scratch[AQ_ATTENTION_STATIC_SCRATCH_BYTES];

// The device address of g_attn_scratch for the current device, looked up
// once per device (cudaGetSymbolAddress); nullptr if the lookup fails.
void *attention_static_scratch() {
    static std::mutex mu;
    static void *addr[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_attn_scratch) != cudaSuccess) return nullptr;
        addr[dev] = p;
    }
    return addr[dev];
}

cudaError_t attn_read_error(uint32_t *code, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(code, g_attn_error, sizeof(uint32_t));
    if (e != cudaSuccess || !clear) return e;
    const uint32_t zero = 0;
    return cudaMemcpyToSymbol(g_attn_error, &zero, sizeof(uint32_t));
}

}  // namespace aq
