// Resident small-M kernel, one 8-column block of activation rows with x
// streamed per stage (M x K too large to keep x whole).  The kernel and its
// dispatch are in aq_gemv.cuh; this unit holds their instantiations so that
// the library builds in parallel.
#include "aq_gemv.cuh"

namespace aq {
namespace gemv {

template cudaError_t launch_blocks<1, true, false>(const GemvPlan &, const GemvMaps &, cudaStream_t);

}  // namespace gemv
}  // namespace aq
