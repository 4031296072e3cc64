// Resident small-M kernel, one 8-column block of activation rows with x
// streamed per stage (M x K too large to keep x whole): the instantiations
// live in their own translation unit so that the library builds in
// parallel.  The kernel is in aq_gemv.cuh.
#include "aq_gemv.cuh"

namespace aq {
namespace gemv {
namespace {

template <int B, bool BF16, int TILES>
cudaError_t st1_wps(const GemvPlan &pl, const GemvMaps &m, cudaStream_t s) {
    if constexpr (TILES <= 2)
        if (pl.wps == 4) return launch_t<B, BF16, TILES, 4, 1, true>(pl, m, s);
    if constexpr (TILES <= 4)
        if (pl.wps == 2) return launch_t<B, BF16, TILES, 2, 1, true>(pl, m, s);
    return launch_t<B, BF16, TILES, 1, 1, true>(pl, m, s);
}

template <int B, bool BF16>
cudaError_t st1_tiles(const GemvPlan &pl, const GemvMaps &m, cudaStream_t s) {
    switch (pl.prm.tiles) {
        case 1: return st1_wps<B, BF16, 1>(pl, m, s);
        case 2: return st1_wps<B, BF16, 2>(pl, m, s);
        case 3: return st1_wps<B, BF16, 3>(pl, m, s);
        case 4: return st1_wps<B, BF16, 4>(pl, m, s);
        case 5: return st1_wps<B, BF16, 5>(pl, m, s);
        case 6: return st1_wps<B, BF16, 6>(pl, m, s);
        case 7: return st1_wps<B, BF16, 7>(pl, m, s);
        default: return st1_wps<B, BF16, 8>(pl, m, s);
    }
}

}  // namespace

cudaError_t launch_staged1(const GemvPlan &pl, const GemvMaps &m, cudaStream_t stream) {
    if (pl.bits == 3)
        return pl.bf16 ? st1_tiles<3, true>(pl, m, stream)
                       : st1_tiles<3, false>(pl, m, stream);
    return pl.bf16 ? st1_tiles<4, true>(pl, m, stream)
                   : st1_tiles<4, false>(pl, m, stream);
}

}  // namespace gemv
}  // namespace aq
