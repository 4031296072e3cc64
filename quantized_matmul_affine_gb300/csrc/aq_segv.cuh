// Small-M kernel for the other code widths and group sizes (aq_matmul_ex):
// y[m][n] = sum_k x[m][k] * (scale[n][g] * q[n][k] + bias[n][g]) for bits in
// {2, 3, 4, 5, 6, 8} and groups of 32/64/128, in the factored form the pages
// use for the affine formats (mlx-bun pages, @mlx-bun/inference 1.0.0,
// kernels/quantization/affine3-rows.ts header: y = scale * sum(x q) +
// bias * sum(x) per group, each decoded weight reused for all M rows).
//
// GB300 design:
//   * One warp per output row n; a lane takes whole 32-code segments of the
//     row: exactly B consecutive words of the LSB-first stream (32 B bits),
//     never straddling a group (groups are multiples of 32).  The decode of a
//     segment is unrolled at compile time (the shifts and word indices are
//     constants): each code is moved to the top B bits of a float mantissa
//     under the exponent of 2^B, which is the float 2^B + q exactly (one
//     shift and one logic operation), and the 2^B * sum(x) this adds to a
//     segment's sum is taken out with the segment sums of x.
//   * The block's activation rows (up to MB) sit in shared memory as fp32,
//     rows interleaved per code ([segment][j][m], 4 floats of pad per
//     segment), so a lane reads the values of four codes (MB = 1), two codes
//     (MB = 2) or one code (MB >= 4) with 16-byte loads and the 32 lanes'
//     segments fall on distinct banks; the products are paired fp32 fmas.
//     The per-segment sums of x for the bias term are taken while staging
//     (16-byte loads, four in flight).  The grid is persistent over the
//     output rows, so a block stages x once for several rows; the weights of
//     a warp's first row are requested before x is staged.
//   * Per segment: sum(x q) over 32 codes for each row, then
//     acc += scale * sum(x q) + bias * sum(x); a fixed xor-butterfly reduces
//     the lanes; lane 0 rounds once to x's dtype.
#pragma once

#include "aq_internal.h"
#include "aq_ptx.cuh"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <type_traits>

namespace aq {
namespace segv_detail {

constexpr int kSegWarps = 8;    // output rows per block
constexpr int kSegUnroll = 4;   // segments per lane in flight (a 4096-wide row at once)

template <typename T>
__device__ __forceinline__ float ld_act(const T *p) {
    if constexpr (std::is_same<T, __nv_bfloat16>::value)
        return __bfloat162float(*p);
    else
        return __half2float(*p);
}

// Code j of a 32-code segment held in w[0..B-1] (LSB-first), as the float
// 2^B + q: the code moved to mantissa bits [23-B, 23) under the exponent of
// 2^B.  j is a constant once the callers' loops are unrolled.
template <int B>
__device__ __forceinline__ float seg_code_rt(const uint32_t (&w)[B], int j) {
    const int bit = j * B, wi = bit >> 5, sh = bit & 31, top = 23 - B;
    const uint32_t mask = ((1u << B) - 1u) << top;
    const uint32_t expo = (uint32_t)(127 + B) << 23;
    uint32_t v;
    if (sh + B > 32)
        v = __funnelshift_r(w[wi], w[wi + 1], sh) << top;
    else if (sh <= top)
        v = w[wi] << (top - sh);
    else
        v = w[wi] >> (sh - top);
    return __uint_as_float((v & mask) | expo);
}

// The block's activation rows for code j of segment sg: MB consecutive
// floats (rows interleaved), one or two vector loads.
template <int MB>
struct XRow {
    float v[MB];
};
template <int MB>
__device__ __forceinline__ XRow<MB> ld_xrow(const float *p) {
    XRow<MB> r;
    if constexpr (MB == 1) {
        r.v[0] = p[0];
    } else if constexpr (MB == 2) {
        const float2 a = *reinterpret_cast<const float2 *>(p);
        r.v[0] = a.x;
        r.v[1] = a.y;
    } else {
#pragma unroll
        for (int i = 0; i < MB; i += 4) {
            const float4 a = *reinterpret_cast<const float4 *>(p + i);
            r.v[i] = a.x;
            r.v[i + 1] = a.y;
            r.v[i + 2] = a.z;
            r.v[i + 3] = a.w;
        }
    }
    return r;
}

// d[m] (as float2 pairs) += sum_j x[m][j] * (2^B + q_j) over the segment's
// 32 codes: the x values of a 16-byte load (4 codes at MB = 1, 2 at MB = 2,
// one code's 4 rows at MB >= 4) times the codes, two products a packed fma.
template <int B, int MB>
__device__ __forceinline__ void seg_dot(const uint32_t (&w)[B], const float *xs,
                                        float2 (&d)[MB == 1 ? 1 : MB / 2]) {
#pragma unroll
    for (int v = 0; v < 8 * MB; ++v) {  // 16-byte vectors of the segment
        const float4 xv = *reinterpret_cast<const float4 *>(xs + 4 * v);
        if constexpr (MB == 1) {
            const int j = 4 * v;
            d[0] = __ffma2_rn(make_float2(xv.x, xv.y),
                              make_float2(seg_code_rt<B>(w, j), seg_code_rt<B>(w, j + 1)), d[0]);
            d[0] = __ffma2_rn(make_float2(xv.z, xv.w),
                              make_float2(seg_code_rt<B>(w, j + 2), seg_code_rt<B>(w, j + 3)),
                              d[0]);
        } else if constexpr (MB == 2) {
            const float q0 = seg_code_rt<B>(w, 2 * v), q1 = seg_code_rt<B>(w, 2 * v + 1);
            d[0] = __ffma2_rn(make_float2(xv.x, xv.y), make_float2(q0, q0), d[0]);
            d[0] = __ffma2_rn(make_float2(xv.z, xv.w), make_float2(q1, q1), d[0]);
        } else {
            const int j = v / (MB / 4), m0 = 4 * (v % (MB / 4));
            const float q = seg_code_rt<B>(w, j);
            d[m0 / 2] = __ffma2_rn(make_float2(xv.x, xv.y), make_float2(q, q), d[m0 / 2]);
            d[m0 / 2 + 1] = __ffma2_rn(make_float2(xv.z, xv.w), make_float2(q, q), d[m0 / 2 + 1]);
        }
    }
}

// Floats per segment in shared memory: 32 codes x MB rows plus a pad of 4
// that keeps the segments 16-byte aligned and puts the 32 lanes' segments on
// distinct banks for 16-byte loads.
template <int MB>
__host__ __device__ constexpr int seg_stride() {
    return 32 * MB + 4;
}

template <int B, int MB, typename T>
__global__ void __launch_bounds__(kSegWarps * 32)
    segv_kernel(const T *__restrict__ x, const uint32_t *__restrict__ Wq,
                const __half *__restrict__ scales, const __half *__restrict__ biases, int M,
                int N, int K, int gshift, T *__restrict__ y) {
    extern __shared__ float sm[];
    constexpr int SS = seg_stride<MB>();
    const int nseg = K / 32;
    float *xs = sm;                         // [nseg][32][MB] (+ pad per segment)
    float *ss = sm + nseg * SS;             // [MB][nseg]  sum of x over a segment
    const int m0 = blockIdx.y * MB;
    const int rows = min(MB, M - m0);
    const int lane = threadIdx.x & 31;
    const int G = K >> gshift;
    constexpr int kD = MB == 1 ? 1 : MB / 2;  // float2 accumulators of a segment

    // This warp's first row's first segments are brought into L2 before x
    // is staged (they do not depend on it), so that their HBM latency
    // overlaps the staging without holding registers.
    int n = blockIdx.x * kSegWarps + (threadIdx.x >> 5);
    if (n < N) {
        const uint32_t *row = Wq + (size_t)n * nseg * B;
#pragma unroll
        for (int u = 0; u < kSegUnroll; ++u) {
            const int sg = min(lane + 32 * u, nseg - 1);
            prefetch_l2(row + (size_t)sg * B);
        }
        if (lane == 0) {
            prefetch_l2(scales + (size_t)n * G);
            prefetch_l2(biases + (size_t)n * G);
        }
    }
    uint32_t w[kSegUnroll][B];
    float sc[kSegUnroll], bi[kSegUnroll];
    auto load_batch = [&](int nn, int s0) {
        const uint32_t *row = Wq + (size_t)nn * nseg * B;
#pragma unroll
        for (int u = 0; u < kSegUnroll; ++u) {
            const int sg = min(s0 + 32 * u, nseg - 1);  // past the row: re-read, unused
#pragma unroll
            for (int i = 0; i < B; ++i) w[u][i] = __ldg(row + (size_t)sg * B + i);
            const int g = (sg * 32) >> gshift;
            sc[u] = __half2float(scales[(size_t)nn * G + g]);
            bi[u] = __half2float(biases[(size_t)nn * G + g]);
        }
    };

    // the block's activation rows: 8 values (16 bytes) per thread and step,
    // four steps' loads in flight; lanes 4j..4j+3 hold one segment and sum it
    {
        const int k8 = K / 8, nv = MB * k8;
        const int nit = (nv + kSegWarps * 32 - 1) / (kSegWarps * 32);
        for (int it0 = 0; it0 < nit; it0 += 4) {
            uint4 raw[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int v = (it0 + u) * kSegWarps * 32 + threadIdx.x;
                const int m = v / k8;
                raw[u] = make_uint4(0u, 0u, 0u, 0u);
                if (it0 + u < nit && v < nv && m < rows)
                    raw[u] = __ldg(reinterpret_cast<const uint4 *>(x + (size_t)(m0 + m) * K) +
                                   (v - m * k8));
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                if (it0 + u >= nit) break;   // uniform across the block
                const int v = (it0 + u) * kSegWarps * 32 + threadIdx.x;
                const int m = v / k8, kk = 8 * (v - m * k8);
                const T *h = reinterpret_cast<const T *>(&raw[u]);
                float part = 0.f;
                if (v < nv) {
                    const int sg = kk >> 5, j0 = kk & 31;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float f = ld_act<T>(h + i);
                        xs[sg * SS + (j0 + i) * MB + m] = f;
                        part += f;
                    }
                }
                part += __shfl_xor_sync(~0u, part, 1);
                part += __shfl_xor_sync(~0u, part, 2);
                if (v < nv && (threadIdx.x & 3) == 0) ss[m * nseg + (kk >> 5)] = part;
            }
        }
    }
    __syncthreads();

    constexpr float kOff = (float)(1 << B);  // each code reads as 2^B + q
    for (; n < N; n += gridDim.x * kSegWarps) {
        float acc[MB];
#pragma unroll
        for (int m = 0; m < MB; ++m) acc[m] = 0.f;

        for (int s0 = lane; s0 < nseg; s0 += 32 * kSegUnroll) {
            load_batch(n, s0);
#pragma unroll
            for (int u = 0; u < kSegUnroll; ++u) {
                const int sg = s0 + 32 * u;
                if (sg >= nseg) break;
                float2 d[kD];
#pragma unroll
                for (int i = 0; i < kD; ++i) d[i] = make_float2(0.f, 0.f);
                seg_dot<B, MB>(w[u], xs + sg * SS, d);
#pragma unroll
                for (int m = 0; m < MB; ++m) {
                    float dm;
                    if constexpr (MB == 1)
                        dm = d[0].x + d[0].y;
                    else
                        dm = (m & 1) ? d[m / 2].y : d[m / 2].x;
                    const float sx = ss[m * nseg + sg];
                    acc[m] = fmaf(sc[u], fmaf(-kOff, sx, dm), fmaf(bi[u], sx, acc[m]));
                }
            }
        }
#pragma unroll
        for (int m = 0; m < MB; ++m)
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) acc[m] += __shfl_xor_sync(~0u, acc[m], off);
        if (lane == 0)
#pragma unroll
            for (int m = 0; m < MB; ++m)
                if (m < rows) {
                    if constexpr (std::is_same<T, __nv_bfloat16>::value)
                        y[(size_t)(m0 + m) * N + n] = __float2bfloat16_rn(acc[m]);
                    else
                        y[(size_t)(m0 + m) * N + n] = __float2half_rn(acc[m]);
                }
    }
}

inline int segv_rows(int64_t M) { return M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : 8; }

inline size_t segv_smem(int mb, int64_t K) {
    return (size_t)(K / 32) * (size_t)(32 * mb + 4 + mb) * sizeof(float);  // x, then sums
}

template <int B, int MB, typename T>
cudaError_t segv_launch_t(const MatmulArgs &a, int gshift) {
    auto kern = segv_kernel<B, MB, T>;
    const size_t smem = segv_smem(MB, a.K);
    if (smem > 48 * 1024) {
        const cudaError_t e =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    // persistent over the output rows: enough blocks to fill the SMs (by
    // shared memory, up to 8 of 256 threads each), each staging its rows of
    // x once
    const int per_sm = (int)std::max<size_t>(1, std::min<size_t>(8, (227 * 1024) / (smem + 1024)));
    const int64_t want = (a.N + kSegWarps - 1) / kSegWarps;
    const int64_t bx = std::min<int64_t>(want, (int64_t)num_sms() * per_sm);
    dim3 grid((unsigned)bx, (unsigned)((a.M + MB - 1) / MB));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kSegWarps * 32, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = a.stream;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<const T *>(a.x), a.Wq,
                              static_cast<const __half *>(a.scales),
                              static_cast<const __half *>(a.biases), (int)a.M, (int)a.N, (int)a.K,
                              gshift, static_cast<T *>(a.out));
}

template <int B, typename T>
cudaError_t segv_rows_t(const MatmulArgs &a, int gshift) {
    switch (segv_rows(a.M)) {
        case 1: return segv_launch_t<B, 1, T>(a, gshift);
        case 2: return segv_launch_t<B, 2, T>(a, gshift);
        case 4: return segv_launch_t<B, 4, T>(a, gshift);
        default: return segv_launch_t<B, 8, T>(a, gshift);
    }
}

template <typename T>
cudaError_t segv_bits_t(const MatmulArgs &a, int gshift) {
    switch (a.bits) {
        case 2: return segv_rows_t<2, T>(a, gshift);
        case 3: return segv_rows_t<3, T>(a, gshift);
        case 4: return segv_rows_t<4, T>(a, gshift);
        case 5: return segv_rows_t<5, T>(a, gshift);
        case 6: return segv_rows_t<6, T>(a, gshift);
        default: return segv_rows_t<8, T>(a, gshift);
    }
}

}  // namespace segv_detail

// One translation unit per activation type instantiates its kernels.
cudaError_t segv_launch_f16(const MatmulArgs &a, int gshift);
cudaError_t segv_launch_bf16(const MatmulArgs &a, int gshift);

}  // namespace aq
