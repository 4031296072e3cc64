// Resident small-M kernel, four 8-column blocks of activation rows
// (M = 17..32), x streamed with the weights; one CTA per SM.  The kernel is
// in aq_gemv.cuh.
#include "aq_gemv.cuh"

namespace aq {
namespace gemv {
namespace {

template <int B, bool BF16>
cudaError_t mb4_tiles(const GemvPlan &pl, const GemvMaps &m, cudaStream_t s) {
    switch (pl.prm.tiles) {
        case 1: return launch_t<B, BF16, 1, 1, 4, true>(pl, m, s);
        case 2: return launch_t<B, BF16, 2, 1, 4, true>(pl, m, s);
        case 3: return launch_t<B, BF16, 3, 1, 4, true>(pl, m, s);
        case 4: return launch_t<B, BF16, 4, 1, 4, true>(pl, m, s);
        case 5: return launch_t<B, BF16, 5, 1, 4, true>(pl, m, s);
        default: return launch_t<B, BF16, 6, 1, 4, true>(pl, m, s);
    }
}

}  // namespace

cudaError_t launch_mb4(const GemvPlan &pl, const GemvMaps &m, cudaStream_t stream) {
    if (pl.prm.tiles > 6) return cudaErrorInvalidValue;
    if (pl.bits == 3)
        return pl.bf16 ? mb4_tiles<3, true>(pl, m, stream)
                       : mb4_tiles<3, false>(pl, m, stream);
    return pl.bf16 ? mb4_tiles<4, true>(pl, m, stream)
                   : mb4_tiles<4, false>(pl, m, stream);
}

}  // namespace gemv
}  // namespace aq
