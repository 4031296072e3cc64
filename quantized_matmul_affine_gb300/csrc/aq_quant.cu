// aq_quantize: float weights (fp16 or bf16) -> the affine group-64 format
// (packed codes, fp16 scale and fp16 bias per 64-value group).
//
// The format is the one the matmul reads (mlx-bun pages, @mlx-bun/inference
// 1.0.0, kernels/quantization/affine-split-mma.ts, helper affine_unit:
// LSB-first bit stream, 2*B words per group; w = scale*q + bias).  The pages
// give no quantiser, so the rule is this library's plain reading, decided in
// single precision:
//
//   lo = min, hi = max over the group;
//   scale = fp16((hi - lo) / (2^B - 1)), bias = fp16(lo)   (round to nearest even)
//   q = clamp(rint((w - bias) / scale), 0, 2^B - 1), q = 0 when scale == 0.
//
// The work is a flat array of N*G groups (a group's 64 values, its 2*B words
// and its scale and bias are each contiguous in their arrays).  A warp takes
// four groups per step, eight lanes per group, one 16-byte load of 8 values
// per lane; min and max are reduced over the eight lanes with shuffles.  At 4
// bits a lane's 8 codes are one output word; at 3 bits they are 24 bits, and
// word w' of a half-group is (c_j >> 8j') | (c_j+1 << (24 - 8j')).  HBM-bound:
// 2 bytes read per weight, B/8 + 4/64 bytes written.
//
// The quotient (w - bias) / scale is taken as (w - bias) * RN(1/scale), which
// is within 1.5 * 2^-23 relative of the IEEE quotient; the two can round to
// different integers only if a half-integer lies between them, so a product
// within 2^-15 of a half-integer (|quotient| <= 64; beyond that the clamp
// decides) is replaced by the IEEE quotient itself.  The codes are therefore
// exactly those of the IEEE division.
#include "aq_internal.h"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace aq {
namespace {

template <bool BF16>
__device__ __forceinline__ void widen8(const uint4 &u, float (&f)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if constexpr (BF16) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        } else {
            const float2 v = __half22float2(*reinterpret_cast<const __half2 *>(&w[i]));
            f[2 * i] = v.x;
            f[2 * i + 1] = v.y;
        }
    }
}

template <int B, bool BF16>
__global__ void __launch_bounds__(256) quantize_kernel(const uint4 *__restrict__ w, int64_t groups,
                                                       uint32_t *__restrict__ words,
                                                       __half *__restrict__ scales,
                                                       __half *__restrict__ biases) {
    constexpr int kQmax = (1 << B) - 1;
    const int lane = threadIdx.x & 31;
    const int j = lane & 7;  // eighth of the group: values 8j .. 8j+7
    const int64_t warp = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    // the next two steps' 16 bytes are in flight during this step's arithmetic
    const int64_t g0 = warp * 4 + (lane >> 3);
    uint4 next = make_uint4(0u, 0u, 0u, 0u), next2 = next;
    if (g0 < groups) next = w[g0 * 8 + j];
    if (g0 + 4 * nwarps < groups) next2 = w[(g0 + 4 * nwarps) * 8 + j];
    for (int64_t quad = warp; quad * 4 < groups; quad += nwarps) {
        const int64_t gid = quad * 4 + (lane >> 3);
        const bool live = gid < groups;
        const uint4 cur = next;
        next = next2;
        const int64_t gnext = gid + 8 * nwarps;
        if (gnext < groups) next2 = w[gnext * 8 + j];
        float f[8];
        widen8<BF16>(cur, f);  // zeros past the last group
        float lo = f[0], hi = f[0];
#pragma unroll
        for (int i = 1; i < 8; ++i) {
            lo = fminf(lo, f[i]);
            hi = fmaxf(hi, f[i]);
        }
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) {
            lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
            hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
        }
        const __half s16 = __float2half_rn(__fdiv_rn(__fsub_rn(hi, lo), (float)kQmax));
        const __half b16 = __float2half_rn(lo);
        const float s = __half2float(s16), b = __half2float(b16);
        // Rounding to an integer without conversion instructions: for
        // 0 <= t <= 2^B - 1, t + 1.5 * 2^23 rounds (to nearest even) at unit
        // spacing, so its low mantissa bits are rint(t).  Clamping first is
        // the same as clamping after, the bounds being integers.
        constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
        const float r = __frcp_rn(s);
        uint32_t chunk = 0;  // the lane's 8 codes, code i at bit B*i
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float a = __fsub_rn(f[i], b);
            float t = fminf(fmaxf(__fmul_rn(a, r), 0.f), (float)kQmax);
            float m = __fadd_rn(t, kMagic);
            if (fabsf(__fsub_rn(t, __fsub_rn(m, kMagic))) > 0.5f - 3.0517578125e-05f) {
                // near a tie: the IEEE quotient decides
                t = fminf(fmaxf(__fdiv_rn(a, s), 0.f), (float)kQmax);
                m = __fadd_rn(t, kMagic);
            }
            const uint32_t q = s != 0.f ? (__float_as_uint(m) & (uint32_t)kQmax) : 0u;
            chunk |= q << (B * i);
        }
        if constexpr (B == 4) {
            if (live) words[gid * 8 + j] = chunk;
        } else {
            const uint32_t next = __shfl_down_sync(0xffffffffu, chunk, 1);
            const int jj = j & 3;
            if (live && jj < 3)
                words[gid * 6 + (j < 4 ? j : j - 1)] = (chunk >> (8 * jj)) | (next << (24 - 8 * jj));
        }
        if (live && j == 0) {
            scales[gid] = s16;
            biases[gid] = b16;
        }
    }
}

// Other widths and group sizes: one warp per group of 32, 64 or 128 values
// (1, 2 or 4 per lane), min/max over the warp, the codes decided with the
// IEEE quotient itself and rint (ties to even), packed through a per-warp
// shared-memory word buffer (a group is group*B/32 words).
template <int B, bool BF16, int VPL>
__global__ void __launch_bounds__(256) quantize_g_kernel(const uint16_t *__restrict__ w,
                                                         int64_t groups,
                                                         uint32_t *__restrict__ words,
                                                         __half *__restrict__ scales,
                                                         __half *__restrict__ biases) {
    constexpr int kQmax = (1 << B) - 1;
    constexpr int kGroup = 32 * VPL;
    constexpr int kWords = kGroup * B / 32;
    __shared__ uint32_t buf[8][kWords];
    const int lane = threadIdx.x & 31, wl = threadIdx.x >> 5;
    const int64_t warp = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t gid = warp; gid < groups; gid += nwarps) {
        float f[VPL];
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
            const uint16_t h = w[gid * kGroup + lane * VPL + i];
            f[i] = BF16 ? __uint_as_float((uint32_t)h << 16)
                        : __half2float(__ushort_as_half(h));
        }
        float lo = f[0], hi = f[0];
#pragma unroll
        for (int i = 1; i < VPL; ++i) {
            lo = fminf(lo, f[i]);
            hi = fmaxf(hi, f[i]);
        }
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
            hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
        }
        const __half s16 = __float2half_rn(__fdiv_rn(__fsub_rn(hi, lo), (float)kQmax));
        const __half b16 = __float2half_rn(lo);
        const float s = __half2float(s16), b = __half2float(b16);
        for (int i = lane; i < kWords; i += 32) buf[wl][i] = 0u;
        __syncwarp();
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
            uint32_t q = 0;
            if (s != 0.f)
                q = (uint32_t)min(max(__float2int_rn(__fdiv_rn(__fsub_rn(f[i], b), s)), 0), kQmax);
            const int bit = (lane * VPL + i) * B;
            atomicOr(&buf[wl][bit >> 5], q << (bit & 31));
            if ((bit & 31) + B > 32) atomicOr(&buf[wl][(bit >> 5) + 1], q >> (32 - (bit & 31)));
        }
        __syncwarp();
        for (int i = lane; i < kWords; i += 32) words[gid * kWords + i] = buf[wl][i];
        if (lane == 0) {
            scales[gid] = s16;
            biases[gid] = b16;
        }
        __syncwarp();
    }
}

template <int B, bool BF16>
cudaError_t quantize_g_group(int group, const uint16_t *w, int64_t groups, uint32_t *words,
                             __half *s, __half *b, cudaStream_t stream) {
    int64_t blocks = (groups + 7) / 8;
    const int64_t cap = (int64_t)num_sms() * 8;
    if (blocks > cap) blocks = cap;
    if (group == 32)
        quantize_g_kernel<B, BF16, 1><<<(unsigned)blocks, 256, 0, stream>>>(w, groups, words, s, b);
    else if (group == 64)
        quantize_g_kernel<B, BF16, 2><<<(unsigned)blocks, 256, 0, stream>>>(w, groups, words, s, b);
    else
        quantize_g_kernel<B, BF16, 4><<<(unsigned)blocks, 256, 0, stream>>>(w, groups, words, s, b);
    return cudaGetLastError();
}

template <bool BF16>
cudaError_t quantize_g_bits(int bits, int group, const uint16_t *w, int64_t groups,
                            uint32_t *words, __half *s, __half *b, cudaStream_t stream) {
    switch (bits) {
        case 2: return quantize_g_group<2, BF16>(group, w, groups, words, s, b, stream);
        case 3: return quantize_g_group<3, BF16>(group, w, groups, words, s, b, stream);
        case 4: return quantize_g_group<4, BF16>(group, w, groups, words, s, b, stream);
        case 5: return quantize_g_group<5, BF16>(group, w, groups, words, s, b, stream);
        case 6: return quantize_g_group<6, BF16>(group, w, groups, words, s, b, stream);
        default: return quantize_g_group<8, BF16>(group, w, groups, words, s, b, stream);
    }
}

}  // namespace

cudaError_t quantize_launch_g(int dtype, const void *w, int64_t N, int64_t K, int bits, int group,
                              uint32_t *words, void *scales, void *biases, cudaStream_t stream) {
    const int64_t groups = N * (K / group);
    if (groups == 0) return cudaSuccess;
    const uint16_t *wp = static_cast<const uint16_t *>(w);
    __half *sp = static_cast<__half *>(scales), *bp = static_cast<__half *>(biases);
    return dtype == AQ_BF16 ? quantize_g_bits<true>(bits, group, wp, groups, words, sp, bp, stream)
                            : quantize_g_bits<false>(bits, group, wp, groups, words, sp, bp, stream);
}

cudaError_t quantize_launch(int dtype, const void *w, int64_t N, int64_t K, int bits,
                            uint32_t *words, void *scales, void *biases, cudaStream_t stream) {
    const int64_t groups = N * (K / 64);
    if (groups == 0) return cudaSuccess;
    const int threads = 256;
    const int64_t quads = (groups + 3) / 4;
    int64_t blocks = (quads + 7) / 8;
    const int64_t cap = (int64_t)num_sms() * 8;
    if (blocks > cap) blocks = cap;
    const uint4 *wp = static_cast<const uint4 *>(w);
    __half *sp = static_cast<__half *>(scales), *bp = static_cast<__half *>(biases);
    const bool bf = dtype == AQ_BF16;
    if (bits == 3) {
        if (bf)
            quantize_kernel<3, true><<<(unsigned)blocks, threads, 0, stream>>>(wp, groups, words, sp, bp);
        else
            quantize_kernel<3, false><<<(unsigned)blocks, threads, 0, stream>>>(wp, groups, words, sp, bp);
    } else {
        if (bf)
            quantize_kernel<4, true><<<(unsigned)blocks, threads, 0, stream>>>(wp, groups, words, sp, bp);
        else
            quantize_kernel<4, false><<<(unsigned)blocks, threads, 0, stream>>>(wp, groups, words, sp, bp);
    }
    return cudaGetLastError();
}

}  // namespace aq
