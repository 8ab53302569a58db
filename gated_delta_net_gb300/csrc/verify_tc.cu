// verify_tc.cu -- tcgen05/TMA fast path of tree verification (sm_103a).
#include "internal.cuh"

namespace gdn {

bool verify_tc_supported(const gdn_verify_args &) { return false; }

cudaError_t launch_verify_tc(const gdn_verify_args &, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace gdn
