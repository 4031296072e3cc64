// bf16 instantiations of the small-M kernel for the other code widths and
// group sizes (aq_segv.cuh).
#include "aq_segv.cuh"

namespace aq {

cudaError_t segv_launch_bf16(const MatmulArgs &a, int gshift) {
    return segv_detail::segv_bits_t<__nv_bfloat16>(a, gshift);
}

}  // namespace aq
