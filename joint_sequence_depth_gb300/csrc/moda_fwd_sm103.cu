// MoDA forward on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
#include "moda_common.cuh"

namespace moda {

bool fwd_sm103_supported(const Problem&) { return false; }

cudaError_t launch_fwd_sm103(const FwdArgs&, cudaStream_t) { return cudaErrorNotSupported; }

bool bwd_sm103_supported(const Problem&) { return false; }

cudaError_t launch_bwd_sm103(const BwdArgs&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace moda
