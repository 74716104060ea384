// bwd_simt_f32.cu -- the CUDA-core backward for fp32 inputs, and the dispatch over input
// types (the bf16 and fp16 instantiations live in their own files so that they compile in
// parallel).
#include "bwd_simt.cuh"

namespace gcl {

template cudaError_t launch_bwd_simt_t<float>(const BwdParams &, bool, bool, cudaStream_t);
extern template cudaError_t launch_bwd_simt_t<__nv_bfloat16>(const BwdParams &, bool, bool, cudaStream_t);
extern template cudaError_t launch_bwd_simt_t<__half>(const BwdParams &, bool, bool, cudaStream_t);

static cudaError_t dispatch(const BwdParams &p, int dtype, bool kda, bool sweep_done, cudaStream_t s) {
    if (dtype == GCL_BF16) return launch_bwd_simt_t<__nv_bfloat16>(p, kda, sweep_done, s);
    if (dtype == GCL_F16) return launch_bwd_simt_t<__half>(p, kda, sweep_done, s);
    return launch_bwd_simt_t<float>(p, kda, sweep_done, s);
}

cudaError_t launch_bwd_simt(const BwdParams &p, int dtype, bool sweep_done, cudaStream_t s) {
    return dispatch(p, dtype, false, sweep_done, s);
}

cudaError_t launch_bwd_simt_kda(const BwdParams &p, int dtype, bool sweep_done, cudaStream_t s) {
    return dispatch(p, dtype, true, sweep_done, s);
}

}  // namespace gcl
