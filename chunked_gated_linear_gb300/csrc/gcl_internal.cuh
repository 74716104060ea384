// gcl_internal.cuh -- declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "gcl.h"
#include "gcl_bounds.cuh"

namespace gcl {

enum Variant { kGDN = 0, kKDA = 1 };
constexpr int kChunk = 64;   // BT: tokens per chunk of the tensor-core path (the CUDA-core
                             // path also takes 32)

// Host: record a one-line error for gcl_last_error() and return `st`.
gcl_status_t fail(gcl_status_t st, const char *fmt, ...);
gcl_status_t cuda_check(cudaError_t e, const char *what);
int num_sms();   // SMs of the current device (cached per device)

// Launch parameters of the forward kernels (a resolved copy of gcl_fwd_args).
struct FwdParams {
    const void *q, *k, *v;
    const float *g;
    const void *beta;
    const float *h0;
    const int32_t *cu_seqlens, *chunk_indices, *chunk_offsets, *seq_order;
    void *o;
    float *ht, *h_save;
    int32_t *dev_status;
    void *workspace;
    size_t workspace_bytes;
    int64_t t_max, nt_max;
    int32_t n_max, H, K, V, bt;
    float scale;
    int32_t dtype;        // gcl_dtype_t of q, k, v, beta, o
};

struct BwdParams {
    const void *q, *k, *v;
    const float *g;
    const void *beta;
    const float *h0;
    const void *d_o;
    const float *dht;
    const int32_t *cu_seqlens, *chunk_indices, *chunk_offsets;
    const float *h;       // states before every chunk [nt_max, H, K, V]
    float *dh;            // state gradients after every chunk: fp32 [nt_max, H, K, V] on the
                          // CUDA-core path, bf16 tiles of tr::kDsTileBytes on the tensor cores
    float *dq, *dk, *dv, *dg, *dbeta, *dh0;
    int32_t *dev_status;
    int64_t t_max, nt_max;
    int32_t n_max, H, K, V, bt;
    float scale;
};

// Kernel launchers (return a CUDA error code; no host synchronisation).
cudaError_t launch_chunk_meta(const int32_t *cu, int32_t n_max, int64_t t_max, int32_t bt,
                              int64_t nt_max, int32_t *idx, int32_t *off, int32_t *order,
                              int32_t *status, cudaStream_t s);
cudaError_t launch_chunk_meta_i64(const int64_t *cu, int32_t n_max, int64_t t_max, int32_t bt,
                                  int64_t nt_max, int32_t *cu32, int32_t *idx, int32_t *off,
                                  int32_t *order, int32_t *status, cudaStream_t s);
cudaError_t launch_fwd_simt(const FwdParams &p, int variant, int dtype, cudaStream_t s);
// Workspace of the CUDA-core split plan (chunk prep records + chain), 0 where it does not apply.
size_t fwd_simt_split_bytes(int K, int V, int bt, int64_t nt_max, int H);
template <typename Tin>
cudaError_t launch_fwd_simt_t(const FwdParams &p, int variant, cudaStream_t s);
// Tensor-core forward (GDN, bf16, K = V = 128).  Two launch plans: the W form
// (prep + chain, 25 KiB of workspace per chunk and head) and the transition form
// (96 KiB per chunk and head, a shorter serial step), which is taken when the column
// split is 4 or more and the workspace holds it.
cudaError_t launch_fwd_tc(const FwdParams &p, int variant, cudaStream_t s);
cudaError_t launch_fwd_tc_t(const FwdParams &p, int split, cudaStream_t s);
// KDA on the tensor cores: transition-form records with per-channel gates, then the chain.
cudaError_t launch_fwd_tc_kda(const FwdParams &p, int split, cudaStream_t s);
bool fwd_tc_supported(int variant, int dtype, int K, int V, int bt);
bool bwd_tc_supported(int variant, int dtype, int K, int V, int bt);
size_t fwd_tc_workspace_bytes(int64_t nt_max, int H);     // W form (the minimum)
size_t fwd_tc_t_workspace_bytes(int64_t nt_max, int H);   // transition form
// Segment-parallel chain (few long sequences): segments per sequence (0: the plain chain) and
// the buffers it needs after the transition records.
int fwd_seg_count(int64_t nt_max, int n_max, int H);
size_t fwd_seg_workspace_bytes(int64_t nt_max, int n_max, int H);
// Fused plan (fwd_fused.cu): one CTA per (sequence, head) keeps the whole chunk pipeline on
// chip and needs no workspace; GDN forwards with many units, except a training forward whose
// workspace holds the transition records.
int fwd_fused_min_units();
bool fwd_tc_runs_fused(int variant, int n_max, int H, bool h_save, size_t ws_bytes, int64_t nt_max);
cudaError_t launch_fwd_fused(const FwdParams &p, cudaStream_t s);
// The plan a tensor-core forward runs for these sizes and this (aligned) workspace size.
int fwd_tc_plan(int variant, int n_max, int H, bool h_save, size_t ws_bytes, int64_t nt_max, int dtype);
int fwd_tc_split(int n_max, int H);                        // value-column slices per head
bool fwd_tc_prefers_transition(int n_max, int H);
bool fwd_tc_runs_transition(int variant, int n_max, int H, bool h_save, size_t ws_bytes, int64_t nt_max,
                            int dtype = GCL_BF16);

// Encodes a TMA tensor map (cuTensorMapEncodeTiled, looked up once through the runtime).
bool make_tensor_map(CUtensorMap *m, const void *ptr, int rank, const cuuint64_t *dims,
                     const cuuint64_t *strides, const cuuint32_t *box, CUtensorMapSwizzle sw,
                     CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
// CUDA-core backward: the state-gradient sweep (unless sweep_done: dh already holds dS'
// per chunk and dh0 is written) and the chunk gradients.
cudaError_t launch_bwd_simt(const BwdParams &p, int dtype, bool sweep_done, cudaStream_t s);
// KDA backward on the CUDA cores: state-gradient sweep with per-channel decay, then the chunk
// gradients (dg per key channel).
cudaError_t launch_bwd_simt_kda(const BwdParams &p, int dtype, bool sweep_done, cudaStream_t s);
template <typename Tin>
cudaError_t launch_bwd_simt_t(const BwdParams &p, bool kda, bool sweep_done, cudaStream_t s);
// causal_conv1d (short_conv.cu)
struct ConvLaunch {
    const void *x, *w, *bias, *residual, *h0, *dy;
    void *y, *ht;
    const float *dht;
    float *dx, *dw, *dbias, *dh0, *partial;
    const int32_t *cu_seqlens, *chunk_indices;
    int32_t *dev_status;
    int64_t t_max, nt_max;
    int32_t n_max, D, W, activation, dtype;
};
cudaError_t launch_conv_fwd(const ConvLaunch &a, cudaStream_t s);
cudaError_t launch_conv_bwd(const ConvLaunch &a, cudaStream_t s);
size_t conv_bwd_workspace_bytes(int64_t nt_max, int D, int W);
// KDA transition-form records alone (the backward's sweep reads them).
cudaError_t launch_prep_kda(const FwdParams &p, uint8_t *ws, cudaStream_t s);
// Tensor-core state-gradient sweep from transition-form records (GDN, bf16, K = V = 128).
// kda: per-key Gamma_c, and dS' as fp32 rows in p.dh (for the CUDA-core KDA chunk gradients)
// instead of the bf16 tiles of the tensor-core GDN chunk gradients.
cudaError_t launch_bwd_sweep_t(const BwdParams &p, const uint8_t *records, bool kda, cudaStream_t s);
// Tensor-core chunk gradients (dq, dk, dv, dg, dbeta) from p.h and p.dh, with a scratch record
// of bwd_grad_tc_scratch_bytes per launch (GDN, bf16, K = V = 128).
cudaError_t launch_bwd_grad_tc(const BwdParams &p, float *scratch, cudaStream_t s);
size_t bwd_grad_tc_scratch_bytes(int64_t nt_max, int H);

// ---- device helpers -------------------------------------------------------
__device__ __forceinline__ float ld_in(const float *p, int64_t i) { return p[i]; }
__device__ __forceinline__ float ld_in(const __nv_bfloat16 *p, int64_t i) {
    return __bfloat162float(p[i]);
}
__device__ __forceinline__ float ld_in(const __half *p, int64_t i) { return __half2float(p[i]); }
__device__ __forceinline__ void st_out(float *p, int64_t i, float x) { p[i] = x; }
__device__ __forceinline__ void st_out(__half *p, int64_t i, float x) { p[i] = __float2half_rn(x); }
__device__ __forceinline__ void st_out(__nv_bfloat16 *p, int64_t i, float x) {
    p[i] = __float2bfloat16_rn(x);
}

// Programmatic dependent launch: the next kernel on the stream, if launched with
// cudaLaunchAttributeProgrammaticStreamSerialization, may start once every CTA of this grid
// has called launch_dependents or exited; grid_dependency_wait blocks until the previous
// grid on the stream has completed and its memory operations are visible (a no-op for a
// kernel launched without the attribute).
__device__ __forceinline__ void launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Launches kern<<<grid, block, smem, s>>>(args...) as a programmatic dependent of the
// previous kernel on the stream.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_dependent(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                    cudaStream_t s, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// Reads the device status word (if any); true means "do no work".
__device__ __forceinline__ bool status_blocks(const int32_t *st) {
    return st != nullptr && *reinterpret_cast<const volatile int32_t *>(st) != 0;
}
// Block-uniform form of status_blocks: thread 0 reads the word once and every thread of the
// block takes the same answer, so no warp leaves while the others go on to barriers, mbarrier
// set-up or TMEM allocation.  Every thread of the block must call it (block barrier).
__device__ __forceinline__ bool status_blocks_cta(const int32_t *st) {
    __shared__ int s_blocked;
    if (threadIdx.x == 0) s_blocked = status_blocks(st) ? 1 : 0;
    __syncthreads();
    return s_blocked != 0;
}
__device__ __forceinline__ void status_set(int32_t *st, int32_t code) {
    if (st != nullptr) atomicCAS(st, 0, code);
}

}  // namespace gcl
