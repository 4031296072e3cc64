// Resident small-M kernel for several projections of one x per launch
// (aq_matmul_multi, aq_matmul_gate_up), one 8-column block with x staged.
// The kernel and its dispatch are in aq_gemv.cuh; this unit holds their
// instantiations.
#include "aq_gemv.cuh"

namespace aq {
namespace gemv {

template cudaError_t launch_blocks<1, true, true>(const GemvPlan &, const GemvMaps &, cudaStream_t);

}  // namespace gemv
}  // namespace aq
