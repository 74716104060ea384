// fwd_simt_f16.cu -- the CUDA-core forward for fp16 inputs (fp32 arithmetic).
#include "fwd_simt.cuh"

namespace gcl {
template cudaError_t launch_fwd_simt_t<__half>(const FwdParams &, int, cudaStream_t);
}  // namespace gcl
