// fwd_tc.cu -- tensor-core (tcgen05) fused chunk forward for bf16 inputs.
#include "gcl_internal.cuh"

namespace gcl {

bool fwd_tc_supported(int, int, int, int) { return false; }

cudaError_t launch_fwd_tc(const FwdParams &, int, cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace gcl
