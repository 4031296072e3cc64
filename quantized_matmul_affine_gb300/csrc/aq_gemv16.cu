// Resident small-M kernel, two 8-column blocks of activation rows (M = 9..16),
// x streamed per stage.  The kernel and its dispatch are in aq_gemv.cuh; this
// unit holds their instantiations so that the library builds in parallel.
#include "aq_gemv.cuh"

namespace aq {
namespace gemv {

template cudaError_t launch_blocks<2, true, false>(const GemvPlan &, const GemvMaps &, cudaStream_t);

}  // namespace gemv
}  // namespace aq
