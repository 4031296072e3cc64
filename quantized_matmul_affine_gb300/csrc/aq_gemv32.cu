// Resident small-M kernel, four 8-column blocks of activation rows
// (M = 17..32), x streamed with the weights; one CTA per SM.  The kernel and
// its dispatch are in aq_gemv.cuh; this unit holds their instantiations.
#include "aq_gemv.cuh"

namespace aq {
namespace gemv {

template cudaError_t launch_blocks<4, true, false>(const GemvPlan &, const GemvMaps &, cudaStream_t);

}  // namespace gemv
}  // namespace aq
