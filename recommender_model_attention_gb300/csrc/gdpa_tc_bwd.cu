// tcgen05 backward kernel (placeholder until the tensor-core path lands).
#include "gdpa_internal.h"

namespace gdpa {
gdpa_status launch_tc_bwd(Plan&, const void*, const void*, const void*, const void*, float*,
                          float*, float*, float, int, cudaStream_t) {
    return GDPA_ERR_UNSUPPORTED;
}
}  // namespace gdpa
