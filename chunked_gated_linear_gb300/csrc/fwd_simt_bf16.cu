// fwd_simt_bf16.cu -- the CUDA-core forward for bf16 inputs (fp32 arithmetic).
#include "fwd_simt.cuh"

namespace gcl {
template cudaError_t launch_fwd_simt_t<__nv_bfloat16>(const FwdParams &, int, cudaStream_t);
}  // namespace gcl
