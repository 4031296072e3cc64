// Resident small-M kernel, two 8-column blocks of activation rows (M = 9..16):
// the instantiations live in their own translation unit so that the library
// builds in parallel.  The kernel is in aq_gemv.cuh.
#include "aq_gemv.cuh"

namespace aq {
namespace gemv {
namespace {

template <int B, bool BF16, int TILES>
cudaError_t mb2_wps(const GemvPlan &pl, const GemvMaps &m, cudaStream_t s) {
    if constexpr (TILES <= 2)
        if (pl.wps == 2) return launch_t<B, BF16, TILES, 2, 2, true>(pl, m, s);
    return launch_t<B, BF16, TILES, 1, 2, true>(pl, m, s);
}

template <int B, bool BF16>
cudaError_t mb2_tiles(const GemvPlan &pl, const GemvMaps &m, cudaStream_t s) {
    switch (pl.prm.tiles) {
        case 1: return mb2_wps<B, BF16, 1>(pl, m, s);
        case 2: return mb2_wps<B, BF16, 2>(pl, m, s);
        case 3: return mb2_wps<B, BF16, 3>(pl, m, s);
        default: return mb2_wps<B, BF16, 4>(pl, m, s);
    }
}

}  // namespace

cudaError_t launch_mb2(const GemvPlan &pl, const GemvMaps &m, cudaStream_t stream) {
    if (pl.prm.tiles > 4) return cudaErrorInvalidValue;
    if (pl.bits == 3)
        return pl.bf16 ? mb2_tiles<3, true>(pl, m, stream)
                       : mb2_tiles<3, false>(pl, m, stream);
    return pl.bf16 ? mb2_tiles<4, true>(pl, m, stream)
                   : mb2_tiles<4, false>(pl, m, stream);
}

}  // namespace gemv
}  // namespace aq
