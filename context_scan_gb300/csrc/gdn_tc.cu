// gdn_tc.cu -- tcgen05 tensor-core kernels (placeholder: routes nothing yet).
#include "gdn_internal.h"

namespace gdn {

bool tc_supported(const ChainParams&) { return false; }
cudaError_t launch_tc_forward(const ChainParams&, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_tc_summary(const ChainParams&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace gdn
