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
//     constants); each code becomes a float as (2^23 | q) - 2^23, two
//     full-rate operations.
//   * The block's activation rows (up to MB) sit in shared memory as fp32,
//     rows interleaved per code ([segment][j][m], a pad per segment), so a
//     lane reads the MB values of its code j with one or two vector loads and
//     the 32 lanes' segments fall on distinct banks; the per-segment sums of
//     x for the bias term are taken while staging (16-byte loads, four in
//     flight).  The grid is persistent over the output rows, so a block
//     stages x once for several rows.
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

// Code j of a 32-code segment held in w[0..B-1] (LSB-first), as a float.
template <int B, int J>
__device__ __forceinline__ float seg_code(const uint32_t (&w)[B]) {
    constexpr int bit = J * B, wi = bit / 32, sh = bit % 32;
    constexpr uint32_t mask = (1u << B) - 1u;
    uint32_t v;
    if constexpr (sh + B <= 32)
        v = (w[wi] >> sh) & mask;
    else
        v = __funnelshift_r(w[wi], w[wi + 1], sh) & mask;
    return __uint_as_float(v | 0x4B000000u) - 8388608.0f;
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

template <int B, int MB, int J>
struct SegDot {
    // d[m] += sum_{j >= J} x[m][j] * code_j
    __device__ __forceinline__ static void run(const uint32_t (&w)[B], const float *xs,
                                               float (&d)[MB]) {
        const float q = seg_code<B, J>(w);
        const XRow<MB> xr = ld_xrow<MB>(xs + J * MB);
#pragma unroll
        for (int m = 0; m < MB; ++m) d[m] = fmaf(xr.v[m], q, d[m]);
        SegDot<B, MB, J + 1>::run(w, xs, d);
    }
};
template <int B, int MB>
struct SegDot<B, MB, 32> {
    __device__ __forceinline__ static void run(const uint32_t (&)[B], const float *,
                                               float (&)[MB]) {}
};

// Floats per segment in shared memory: 32 codes x MB rows plus a pad that
// puts the 32 lanes' segments on distinct banks (8- or 16-byte slots).
template <int MB>
__host__ __device__ constexpr int seg_stride() {
    return 32 * MB + (MB == 1 ? 1 : MB == 2 ? 2 : 4);
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

    const int lane = threadIdx.x & 31;
    const int G = K >> gshift;
    for (int n = blockIdx.x * kSegWarps + (threadIdx.x >> 5); n < N;
         n += gridDim.x * kSegWarps) {
        const uint32_t *row = Wq + (size_t)n * nseg * B;
        const __half *srow = scales + (size_t)n * G;
        const __half *brow = biases + (size_t)n * G;
        float acc[MB];
#pragma unroll
        for (int m = 0; m < MB; ++m) acc[m] = 0.f;

        for (int s0 = lane; s0 < nseg; s0 += 32 * kSegUnroll) {
            uint32_t w[kSegUnroll][B];
            float sc[kSegUnroll], bi[kSegUnroll];
#pragma unroll
            for (int u = 0; u < kSegUnroll; ++u) {
                const int sg = min(s0 + 32 * u, nseg - 1);  // past the row: re-read, unused
#pragma unroll
                for (int i = 0; i < B; ++i) w[u][i] = __ldg(row + (size_t)sg * B + i);
                const int g = (sg * 32) >> gshift;
                sc[u] = __half2float(srow[g]);
                bi[u] = __half2float(brow[g]);
            }
#pragma unroll
            for (int u = 0; u < kSegUnroll; ++u) {
                const int sg = s0 + 32 * u;
                if (sg >= nseg) break;
                float d[MB];
#pragma unroll
                for (int m = 0; m < MB; ++m) d[m] = 0.f;
                SegDot<B, MB, 0>::run(w[u], xs + sg * SS, d);
#pragma unroll
                for (int m = 0; m < MB; ++m)
                    acc[m] = fmaf(sc[u], d[m], fmaf(bi[u], ss[m * nseg + sg], acc[m]));
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
    const int ss = 32 * mb + (mb == 1 ? 1 : mb == 2 ? 2 : 4);
    return (size_t)(K / 32) * (size_t)(ss + mb) * sizeof(float);
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
