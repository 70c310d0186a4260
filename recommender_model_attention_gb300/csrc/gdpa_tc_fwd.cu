// tcgen05 forward kernel (placeholder until the tensor-core path lands).
#include "gdpa_internal.h"

namespace gdpa {
gdpa_status launch_tc_fwd(Plan&, const void*, const void*, const void*, void*, float, int,
                          cudaStream_t) {
    return GDPA_ERR_UNSUPPORTED;
}
}  // namespace gdpa
