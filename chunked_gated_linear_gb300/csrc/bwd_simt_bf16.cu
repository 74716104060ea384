// bwd_simt_bf16.cu -- the CUDA-core backward for bf16 inputs (fp32 arithmetic).
#include "bwd_simt.cuh"

namespace gcl {
template cudaError_t launch_bwd_simt_t<__nv_bfloat16>(const BwdParams &, bool, bool, cudaStream_t);
}  // namespace gcl
