// aq_pack: integer codes -> MLX affine bit stream.
//
// Format (mlx-bun pages, @mlx-bun/inference 1.0.0,
// kernels/quantization/affine-split-mma.ts, helper affine_unit): code v of a
// row occupies bits [v*B, v*B+B) of the row's least-significant-first bit
// stream; stream bit i is bit i%32 of uint32 word i/32.  A 64-value group is
// exactly 2*B words, so a row is K*B/32 words.
//
// One thread builds one output word from the (at most 17, at 2 bits) codes
// that touch it, so every word is written exactly once and no atomics are
// needed.  Any width of 2, 3, 4, 5, 6 or 8 bits.
#include "aq_internal.h"

namespace aq {

template <int B>
__global__ void __launch_bounds__(256) pack_kernel(const uint8_t *__restrict__ codes, int64_t N,
                                                   int64_t K, uint32_t *__restrict__ words) {
    const int64_t wpr = K * B / 32;
    const int64_t total = N * wpr;
    const uint32_t mask = (1u << B) - 1u;
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t n = idx / wpr;
        const int64_t wi = idx - n * wpr;
        const uint8_t *row = codes + n * K;
        const int64_t lo_bit = wi * 32;
        const int64_t v_first = lo_bit / B;
        const int64_t v_last = (lo_bit + 31) / B;
        uint32_t w = 0;
        for (int64_t v = v_first; v <= v_last; ++v) {
            const uint32_t q = row[v] & mask;
            const int64_t sh = v * B - lo_bit;  // position of the code's bit 0 in this word
            if (sh >= 0)
                w |= q << sh;  // bits past 31 belong to the next word and drop off
            else
                w |= q >> (-sh);  // code started in the previous word
        }
        words[idx] = w;
    }
}

cudaError_t pack_launch(const uint8_t *codes, int64_t N, int64_t K, int bits, uint32_t *words,
                        cudaStream_t stream) {
    const int64_t total = N * (K * bits / 32);
    if (total == 0) return cudaSuccess;
    const int threads = 256;
    int64_t blocks = (total + threads - 1) / threads;
    const int64_t cap = (int64_t)num_sms() * 16;
    if (blocks > cap) blocks = cap;
    switch (bits) {
        case 2: pack_kernel<2><<<(unsigned)blocks, threads, 0, stream>>>(codes, N, K, words); break;
        case 3: pack_kernel<3><<<(unsigned)blocks, threads, 0, stream>>>(codes, N, K, words); break;
        case 4: pack_kernel<4><<<(unsigned)blocks, threads, 0, stream>>>(codes, N, K, words); break;
        case 5: pack_kernel<5><<<(unsigned)blocks, threads, 0, stream>>>(codes, N, K, words); break;
        case 6: pack_kernel<6><<<(unsigned)blocks, threads, 0, stream>>>(codes, N, K, words); break;
        default: pack_kernel<8><<<(unsigned)blocks, threads, 0, stream>>>(codes, N, K, words); break;
    }
    return cudaGetLastError();
}

}  // namespace aq
