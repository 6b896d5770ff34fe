// Tensor-core (tcgen05) launchers: not built in this configuration.
#include <cuda_runtime.h>

#include "cpdr_internal.hpp"

namespace cpdr {
int launch_tc_pre(const cpdr_ctx *, const void *, const void *, const void *, const float *, float *,
                  float *, void *) {
    return (int)cudaErrorNotSupported;
}
int launch_tc_fwd(const cpdr_ctx *, const void *, const void *, const void *, const void *, const float *,
                  const float *, void *, float *, void *) {
    return (int)cudaErrorNotSupported;
}
}  // namespace cpdr
