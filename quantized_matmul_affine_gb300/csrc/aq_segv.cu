// Small-M kernel for the other code widths and group sizes: dispatch and the
// fp16 instantiations (the kernel itself is in aq_segv.cuh).
#include "aq_segv.cuh"

namespace aq {

cudaError_t segv_launch_f16(const MatmulArgs &a, int gshift) {
    return segv_detail::segv_bits_t<__half>(a, gshift);
}

// Served: the generic kernel's widths and group sizes, M <= 32, int32 sizes,
// x 16-byte aligned, and the block's activation rows within 200 KB of shared
// memory.
bool segv_supported(const MatmulArgs &a, int group) {
    if (!generic_supported_g(a, group)) return false;
    if (a.M > 32 || a.N > INT32_MAX || a.K > INT32_MAX / 8) return false;
    if (!aligned(a.x, 16)) return false;   // x is staged with 16-byte loads
    return segv_detail::segv_smem(segv_detail::segv_rows(a.M), a.K) <= 200 * 1024;
}

cudaError_t segv_launch(const MatmulArgs &a, int group) {
    const int gshift = group == 32 ? 5 : group == 64 ? 6 : 7;
    return a.dtype == AQ_BF16 ? segv_launch_bf16(a, gshift) : segv_launch_f16(a, gshift);
}

}  // namespace aq
