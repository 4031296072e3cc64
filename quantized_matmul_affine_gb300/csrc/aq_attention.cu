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
//     that KV head (NREP = H / KV of them), so each K and V row is read once.
//     The blocks of a KV head form a thread-block cluster (up to 16 CTAs);
//     their partial results are merged in rank order through distributed
//     shared memory - no global scratch, no second launch.
//   * 256 threads: lane l holds head-dimension elements [l*E, l*E + E),
//     E = D / 32 (all inside one quantisation group); warp w takes rows
//     w, w+8, ... of the block.  Per row: the lane's codes (one load of E
//     codes), the factored partial score for each query head, a warp sum,
//     the online softmax update, and the value row dequantised once and
//     accumulated for every query head.
//   * The eight warps' (max, sum, o) merge through shared memory in warp
//     order; the cluster's CTAs then in rank order.  Scores and
//     probabilities stay in fp32 (the pages round the scores to the input
//     type; fp32 is the more exact reading); o is rounded once.
#include "aq_internal.h"
#include "aq_ptx.cuh"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <mutex>
#include <type_traits>

namespace aq {
namespace {

constexpr int kAttnThreads = 256;
constexpr int kAttnWarps = kAttnThreads / 32;

struct AttnParams {
    const void *q;
    const uint8_t *kw, *vw;       // packed rows [KV*N][D*bits/8] bytes
    const __half *ks, *kb, *vs, *vb;  // [KV*N][D/group]
    void *out;
    int H, KV, N, D, group;
    int block;     // cached rows per CTA
    int csize;     // CTAs per cluster (one KV head)
    int row_bytes;
};

template <typename T>
__device__ __forceinline__ float ld_f(const T *p) {
    if constexpr (std::is_same<T, __nv_bfloat16>::value)
        return __bfloat162float(*p);
    else
        return __half2float(*p);
}

// The lane's E codes as one 1/2/4/8-byte load.
template <int BITS, int E>
__device__ __forceinline__ void load_codes(const uint8_t *p, float (&c)[E]) {
    constexpr int kBytes = E * BITS / 8;
    uint64_t w;
    if constexpr (kBytes == 1)
        w = *p;
    else if constexpr (kBytes == 2)
        w = *reinterpret_cast<const uint16_t *>(p);
    else if constexpr (kBytes == 4)
        w = *reinterpret_cast<const uint32_t *>(p);
    else
        w = *reinterpret_cast<const uint64_t *>(p);
#pragma unroll
    for (int e = 0; e < E; ++e) c[e] = (float)((w >> (BITS * e)) & ((1u << BITS) - 1u));
}

template <int BITS, int E, int NREP, bool BF16>
__global__ void __launch_bounds__(kAttnThreads, 1) attn_kernel(const __grid_constant__ AttnParams p) {
    using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
    constexpr int D = 32 * E;
    extern __shared__ float sh[];
    float *wm = sh;                              // [warps][NREP]
    float *wl = wm + kAttnWarps * NREP;          // [warps][NREP]
    float *wo = wl + kAttnWarps * NREP;          // [warps][NREP][D]
    float *cm = wo + kAttnWarps * NREP * D;      // [NREP]   this CTA's merge
    float *cl = cm + NREP;                       // [NREP]
    float *co = cl + NREP;                       // [NREP][D]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int kv = (int)blockIdx.x / p.csize;
    const int rank = (int)blockIdx.x % p.csize;
    const int n0 = rank * p.block;
    const int n1 = min(p.N, n0 + p.block);
    const int gRow = D / p.group;
    const int grp = lane * E / p.group;

    // the query heads of this KV head: the lane's elements and their sums
    const T *q = static_cast<const T *>(p.q);
    float qv[NREP][E], qsum[NREP];
#pragma unroll
    for (int j = 0; j < NREP; ++j) {
        qsum[j] = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            qv[j][e] = ld_f<T>(q + (size_t)(kv * NREP + j) * D + lane * E + e);
            qsum[j] += qv[j][e];
        }
    }
    float m[NREP], l[NREP], o[NREP][E];
#pragma unroll
    for (int j = 0; j < NREP; ++j) {
        m[j] = -INFINITY;
        l[j] = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) o[j][e] = 0.f;
    }

    for (int n = n0 + warp; n < n1; n += kAttnWarps) {
        const size_t r = (size_t)kv * p.N + n;
        float c[E];
        load_codes<BITS, E>(p.kw + r * p.row_bytes + lane * (E * BITS / 8), c);
        const float ksc = __half2float(p.ks[r * gRow + grp]);
        const float kbi = __half2float(p.kb[r * gRow + grp]);
        float s[NREP];
#pragma unroll
        for (int j = 0; j < NREP; ++j) {
            float dot = 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) dot = fmaf(qv[j][e], c[e], dot);
            float part = fmaf(ksc, dot, kbi * qsum[j]);
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
            s[j] = part;
        }
        float cv[E];
        load_codes<BITS, E>(p.vw + r * p.row_bytes + lane * (E * BITS / 8), cv);
        const float vsc = __half2float(p.vs[r * gRow + grp]);
        const float vbi = __half2float(p.vb[r * gRow + grp]);
        float vd[E];
#pragma unroll
        for (int e = 0; e < E; ++e) vd[e] = fmaf(vsc, cv[e], vbi);
#pragma unroll
        for (int j = 0; j < NREP; ++j) {
            const float mn = fmaxf(m[j], s[j]);
            const float f = expf(m[j] - mn);  // 0 on the first row (m = -inf)
            const float pj = expf(s[j] - mn);
            l[j] = fmaf(l[j], f, pj);
            m[j] = mn;
#pragma unroll
            for (int e = 0; e < E; ++e) o[j][e] = fmaf(o[j][e], f, pj * vd[e]);
        }
    }

    // the eight warps, in warp order
#pragma unroll
    for (int j = 0; j < NREP; ++j) {
        if (lane == 0) {
            wm[warp * NREP + j] = m[j];
            wl[warp * NREP + j] = l[j];
        }
#pragma unroll
        for (int e = 0; e < E; ++e) wo[(warp * NREP + j) * D + lane * E + e] = o[j][e];
    }
    __syncthreads();
    for (int i = threadIdx.x; i < NREP * D; i += kAttnThreads) {
        const int j = i / D, d = i - j * D;
        float M = -INFINITY;
        for (int w = 0; w < kAttnWarps; ++w) M = fmaxf(M, wm[w * NREP + j]);
        float L = 0.f, O = 0.f;
        for (int w = 0; w < kAttnWarps; ++w) {
            const float mw = wm[w * NREP + j];
            const float g = mw == -INFINITY ? 0.f : expf(mw - M);  // a warp with no rows
            L = fmaf(wl[w * NREP + j], g, L);
            O = fmaf(wo[(w * NREP + j) * D + d], g, O);
        }
        co[j * D + d] = O;
        if (d == 0) {
            cm[j] = M;
            cl[j] = L;
        }
    }
    __syncthreads();

    // the cluster's CTAs, in rank order; rank r writes its share of o
    T *out = static_cast<T *>(p.out);
    const int C = p.csize;
    if (C > 1) cluster_sync();
    const int total = NREP * D;
    const int chunk = (total + C - 1) / C;
    const uint32_t bm = smem_u32(cm), bl = smem_u32(cl), bo = smem_u32(co);
    for (int i = rank * chunk + (int)threadIdx.x; i < min(total, (rank + 1) * chunk);
         i += kAttnThreads) {
        const int j = i / D, d = i - j * D;
        float M = -INFINITY;
        for (int rr = 0; rr < C; ++rr)
            M = fmaxf(M, C > 1 ? ld_dsmem_f32(map_to_rank(bm + 4u * j, (uint32_t)rr)) : cm[j]);
        float L = 0.f, O = 0.f;
        for (int rr = 0; rr < C; ++rr) {
            const float mr = C > 1 ? ld_dsmem_f32(map_to_rank(bm + 4u * j, (uint32_t)rr)) : cm[j];
            if (mr == -INFINITY) continue;  // a block with no rows
            const float g = expf(mr - M);
            const float lr = C > 1 ? ld_dsmem_f32(map_to_rank(bl + 4u * j, (uint32_t)rr)) : cl[j];
            const float orr =
                C > 1 ? ld_dsmem_f32(map_to_rank(bo + 4u * (uint32_t)i, (uint32_t)rr)) : co[i];
            L = fmaf(lr, g, L);
            O = fmaf(orr, g, O);
        }
        const float v = O / L;
        if constexpr (BF16)
            out[(size_t)(kv * NREP + j) * D + d] = __float2bfloat16_rn(v);
        else
            out[(size_t)(kv * NREP + j) * D + d] = __float2half_rn(v);
    }
    if (C > 1) cluster_sync();  // keep this CTA's results until every rank has read them
}

size_t attn_smem(int nrep, int D) {
    return sizeof(float) * ((size_t)2 * kAttnWarps * nrep + (size_t)kAttnWarps * nrep * D +
                            2 * (size_t)nrep + (size_t)nrep * D);
}

template <int BITS, int E, int NREP, bool BF16>
cudaError_t attn_launch_t(const AttnParams &prm, cudaStream_t stream) {
    auto kern = attn_kernel<BITS, E, NREP, BF16>;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    const size_t smem = attn_smem(NREP, 32 * E);
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)attn_smem(8, 256));
        if (attr_err == cudaSuccess)
            attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    });
    if (attr_err != cudaSuccess) return attr_err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(prm.KV * prm.csize), 1, 1);
    cfg.blockDim = dim3(kAttnThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)prm.csize;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, prm);
}

template <int BITS, int E, bool BF16>
cudaError_t attn_nrep(int nrep, const AttnParams &prm, cudaStream_t s) {
    switch (nrep) {
        case 1: return attn_launch_t<BITS, E, 1, BF16>(prm, s);
        case 2: return attn_launch_t<BITS, E, 2, BF16>(prm, s);
        case 4: return attn_launch_t<BITS, E, 4, BF16>(prm, s);
        default: return attn_launch_t<BITS, E, 8, BF16>(prm, s);
    }
}

template <int BITS, bool BF16>
cudaError_t attn_d(int D, int nrep, const AttnParams &prm, cudaStream_t s) {
    switch (D) {
        case 64: return attn_nrep<BITS, 2, BF16>(nrep, prm, s);
        case 128: return attn_nrep<BITS, 4, BF16>(nrep, prm, s);
        default: return attn_nrep<BITS, 8, BF16>(nrep, prm, s);
    }
}

}  // namespace

bool attention_supported(int64_t H, int64_t KV, int64_t N, int64_t D, int bits, int group) {
    if (H < 1 || KV < 1 || H % KV != 0 || N < 1 || N > INT32_MAX / 2) return false;
    const int64_t nrep = H / KV;
    if (nrep != 1 && nrep != 2 && nrep != 4 && nrep != 8) return false;
    if (D != 64 && D != 128 && D != 256) return false;
    if (bits != 4 && bits != 8) return false;
    if (group != 32 && group != 64 && group != 128) return false;
    if (D % group != 0 || group < D / 32) return false;
    return KV * N <= INT32_MAX / 2;
}

// Cluster size: enough CTAs to cover the SMs (one KV head per cluster, up to
// 16 blocks of at least 64 rows).
int attention_cluster(int64_t KV, int64_t N) {
    const int64_t want = (num_sms() + KV - 1) / KV;
    const int64_t by_rows = (N + 63) / 64;
    return (int)std::max<int64_t>(1, std::min<int64_t>({16, want, by_rows}));
}

cudaError_t attention_launch(int dtype, const void *q, const uint32_t *kw, const void *ks,
                             const void *kb, const uint32_t *vw, const void *vs, const void *vb,
                             int64_t H, int64_t KV, int64_t N, int64_t D, int bits, int group,
                             void *out, cudaStream_t stream) {
    AttnParams prm;
    prm.q = q;
    prm.kw = reinterpret_cast<const uint8_t *>(kw);
    prm.vw = reinterpret_cast<const uint8_t *>(vw);
    prm.ks = static_cast<const __half *>(ks);
    prm.kb = static_cast<const __half *>(kb);
    prm.vs = static_cast<const __half *>(vs);
    prm.vb = static_cast<const __half *>(vb);
    prm.out = out;
    prm.H = (int)H;
    prm.KV = (int)KV;
    prm.N = (int)N;
    prm.D = (int)D;
    prm.group = group;
    prm.csize = attention_cluster(KV, N);
    prm.block = (int)((N + prm.csize - 1) / prm.csize);
    prm.row_bytes = (int)(D * bits / 8);
    const int nrep = (int)(H / KV);
    const bool bf = dtype == AQ_BF16;
    if (bits == 4)
        return bf ? attn_d<4, true>((int)D, nrep, prm, stream)
                  : attn_d<4, false>((int)D, nrep, prm, stream);
    return bf ? attn_d<8, true>((int)D, nrep, prm, stream)
              : attn_d<8, false>((int)D, nrep, prm, stream);
}

}  // namespace aq
