// bwd_simt_f16.cu -- the CUDA-core backward for f16 inputs (fp32 arithmetic).
#include "bwd_simt.cuh"

namespace gcl {
template cudaError_t launch_bwd_simt_t<__half>(const BwdParams &, bool, bool, cudaStream_t);
}  // namespace gcl
