// Large-M kernel (tcgen05 + TMEM): not built yet; the dispatch rule sends
// every shape to the small-M or generic kernels meanwhile.
#include "aq_internal.h"

#include <cstdio>

namespace aq {

bool tc_supported(const MatmulArgs &) { return false; }

cudaError_t tc_launch(const MatmulArgs &) { return cudaErrorNotSupported; }

int tc_describe(const MatmulArgs &, char *buf, int len) {
    return snprintf(buf, len, "tc: not built");
}

cudaError_t tc_read_error(uint32_t *code, bool) {
    *code = 0;
    return cudaSuccess;
}

}  // namespace aq
