// Generic kernel: any K % 64 == 0 (any multiple of the group size for the
// other code widths and group sizes), any N, any M, pointers aligned only to
// their element size.  It serves the shapes and alignments the fast kernels
// do not take, and is deliberately plain: one warp per (output column n,
// block of up to 8 activation rows); lane l walks k = l, l+32, ...;
// each weight is decoded from the bit stream, dequantised in fp32 as
// w = fma(scale, q, bias) (mlx-bun pages, @mlx-bun/inference 1.0.0,
// kernels/quantization/affine4-mma.ts: fma(s, q, b)) and multiplied into up
// to 8 fp32 accumulators; a fixed xor-butterfly of warp shuffles reduces them.
#include "aq_internal.h"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace aq {

template <typename T>
__device__ __forceinline__ float to_f32(T v);
template <>
__device__ __forceinline__ float to_f32<__half>(__half v) { return __half2float(v); }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) {
    return __bfloat162float(v);
}

template <typename T>
__device__ __forceinline__ T from_f32(float v);
template <>
__device__ __forceinline__ __half from_f32<__half>(float v) { return __float2half_rn(v); }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}

constexpr int kGenericRows = 8;     // activation rows per warp
constexpr int kGenericWarps = 8;    // warps (output columns) per block

template <int B, typename T>
__global__ void __launch_bounds__(kGenericWarps * 32)
    generic_kernel(const T *__restrict__ x, const uint32_t *__restrict__ Wq,
                   const __half *__restrict__ scales, const __half *__restrict__ biases, int64_t M,
                   int64_t N, int64_t K, int gshift, T *__restrict__ y) {
    const int lane = threadIdx.x & 31;
    const int64_t n = (int64_t)blockIdx.x * kGenericWarps + (threadIdx.x >> 5);
    const int64_t m0 = (int64_t)blockIdx.y * kGenericRows;
    if (n >= N) return;
    const int64_t wpr = K * B / 32;
    const int64_t G = K >> gshift;  // groups of 2^gshift values
    const uint32_t *row = Wq + n * wpr;
    const int rows = (int)((M - m0) < kGenericRows ? (M - m0) : kGenericRows);
    float acc[kGenericRows];
#pragma unroll
    for (int r = 0; r < kGenericRows; ++r) acc[r] = 0.f;
    // four k per lane per step (k = lane + 32 j, j = 4i..4i+3): the loads of
    // a step are independent and in flight together
    constexpr int kU = 4;
    for (int64_t k0 = lane; k0 < K; k0 += 32 * kU) {
        float w[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int64_t k = k0 + 32 * u;
            w[u] = 0.f;
            if (k < K) {
                const int64_t g = k >> gshift;
                const int64_t bit = k * B;
                const int64_t wi = bit >> 5;
                const int off = (int)(bit & 31);
                uint32_t q = row[wi] >> off;
                if (off + B > 32) q |= row[wi + 1] << (32 - off);
                q &= (1u << B) - 1u;
                w[u] = fmaf(__half2float(scales[n * G + g]), (float)q,
                            __half2float(biases[n * G + g]));
            }
        }
#pragma unroll
        for (int r = 0; r < kGenericRows; ++r) {
            if (r < rows) {
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    const int64_t k = k0 + 32 * u;
                    if (k < K) acc[r] = fmaf(w[u], to_f32<T>(x[(m0 + r) * K + k]), acc[r]);
                }
            }
        }
    }
#pragma unroll
    for (int r = 0; r < kGenericRows; ++r) {
        float v = acc[r];
#pragma unroll
        for (int d = 16; d >= 1; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
        acc[r] = v;
    }
    if (lane == 0) {
#pragma unroll
        for (int r = 0; r < kGenericRows; ++r)
            if (r < rows) y[(m0 + r) * N + n] = from_f32<T>(acc[r]);
    }
}

bool generic_supported(const MatmulArgs &a) {
    return a.M >= 1 && a.N >= 1 && a.K >= 64 && a.K % 64 == 0 && (a.bits == 3 || a.bits == 4) &&
           (a.M + kGenericRows - 1) / kGenericRows <= 65535;
}

bool generic_supported_g(const MatmulArgs &a, int group) {
    const bool width = a.bits == 2 || a.bits == 3 || a.bits == 4 || a.bits == 5 || a.bits == 6 ||
                       a.bits == 8;
    const bool grp = group == 32 || group == 64 || group == 128;
    return a.M >= 1 && a.N >= 1 && width && grp && a.K >= group && a.K % group == 0 &&
           (a.M + kGenericRows - 1) / kGenericRows <= 65535;
}

template <typename T>
static cudaError_t launch_t(const MatmulArgs &a, int group) {
    dim3 grid((unsigned)((a.N + kGenericWarps - 1) / kGenericWarps),
              (unsigned)((a.M + kGenericRows - 1) / kGenericRows));
    const T *x = static_cast<const T *>(a.x);
    const __half *s = static_cast<const __half *>(a.scales);
    const __half *b = static_cast<const __half *>(a.biases);
    T *y = static_cast<T *>(a.out);
    const int gs = group == 32 ? 5 : group == 64 ? 6 : 7;
    const unsigned th = kGenericWarps * 32;
    switch (a.bits) {
        case 2: generic_kernel<2, T><<<grid, th, 0, a.stream>>>(x, a.Wq, s, b, a.M, a.N, a.K, gs, y); break;
        case 3: generic_kernel<3, T><<<grid, th, 0, a.stream>>>(x, a.Wq, s, b, a.M, a.N, a.K, gs, y); break;
        case 4: generic_kernel<4, T><<<grid, th, 0, a.stream>>>(x, a.Wq, s, b, a.M, a.N, a.K, gs, y); break;
        case 5: generic_kernel<5, T><<<grid, th, 0, a.stream>>>(x, a.Wq, s, b, a.M, a.N, a.K, gs, y); break;
        case 6: generic_kernel<6, T><<<grid, th, 0, a.stream>>>(x, a.Wq, s, b, a.M, a.N, a.K, gs, y); break;
        default: generic_kernel<8, T><<<grid, th, 0, a.stream>>>(x, a.Wq, s, b, a.M, a.N, a.K, gs, y); break;
    }
    return cudaGetLastError();
}

cudaError_t generic_launch(const MatmulArgs &a) {
    return a.dtype == AQ_BF16 ? launch_t<__nv_bfloat16>(a, 64) : launch_t<__half>(a, 64);
}

cudaError_t generic_launch_g(const MatmulArgs &a, int group) {
    return a.dtype == AQ_BF16 ? launch_t<__nv_bfloat16>(a, group) : launch_t<__half>(a, group);
}

}  // namespace aq
