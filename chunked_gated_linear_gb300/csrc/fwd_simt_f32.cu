// fwd_simt_f32.cu -- the CUDA-core forward for fp32 inputs, and the dispatch over input types
// (the bf16 and fp16 instantiations live in their own files so that they compile in parallel).
#include "fwd_simt.cuh"

namespace gcl {

template cudaError_t launch_fwd_simt_t<float>(const FwdParams &, int, cudaStream_t);
extern template cudaError_t launch_fwd_simt_t<__nv_bfloat16>(const FwdParams &, int, cudaStream_t);
extern template cudaError_t launch_fwd_simt_t<__half>(const FwdParams &, int, cudaStream_t);

// Workspace of the CUDA-core split plan (its records), 0 where it does not apply (K != V).
size_t fwd_simt_split_bytes(int K, int V, int bt, int64_t nt_max, int H) {
    using namespace simt_split;
    if (K != V || (K != 64 && K != 128) || nt_max <= 0 || H <= 0) return 0;
    if (bt == 32) return K == 64 ? record_bytes<64, 64, 32>(nt_max, H) : record_bytes<128, 128, 32>(nt_max, H);
    return K == 64 ? record_bytes<64, 64, 64>(nt_max, H) : record_bytes<128, 128, 64>(nt_max, H);
}

cudaError_t launch_fwd_simt(const FwdParams &p, int variant, int dtype, cudaStream_t s) {
    if (dtype == GCL_BF16) return launch_fwd_simt_t<__nv_bfloat16>(p, variant, s);
    if (dtype == GCL_F16) return launch_fwd_simt_t<__half>(p, variant, s);
    return launch_fwd_simt_t<float>(p, variant, s);
}

}  // namespace gcl
