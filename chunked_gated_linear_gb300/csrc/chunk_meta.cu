// chunk_meta.cu -- device-side chunk metadata for fixed-capacity (graph) execution.
//
// FLA RFC "[RFC] Add Graph Capture Support for FLA Prefill and Training Paths on
// Ascend NPUs", section "Core design / Device-side metadata": a static
// cu_seqlens buffer is turned on the device into chunk_indices [NT_max, 2]
// (sentinel [-1, 0] in unused rows) and chunk_offsets [N_max + 1], so that a
// replayed graph picks up a new sequence layout without any host round trip.
//
// One CTA of 1024 threads does it all: a validity check, a block-wide
// exclusive scan of the per-sequence chunk counts (in tiles of 1024 with a
// running carry), a fill of the index rows by binary search over the offsets,
// and an optional longest-first order of the sequences (rank by counting).
// The RFC's graph infrastructure covers int32 and int64 cu_seqlens ("Improve the
// common graph infrastructure"): an int64 cu_seqlens is checked in int64 and, once
// valid (every entry in [0, t_max], t_max < 2^31), narrowed exactly into the int32
// copy that the compute calls read.
#include "gcl_internal.cuh"

namespace gcl {
namespace {

constexpr int kThreads = 1024;

__device__ __forceinline__ int block_exclusive_scan(int x, int *warp_sums, int *total) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int incl = x;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += y;
    }
    if (lane == 31) warp_sums[wid] = incl;
    __syncthreads();
    if (wid == 0) {
        int s = warp_sums[lane];
        int si = s;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, si, d);
            if (lane >= d) si += y;
        }
        warp_sums[lane] = si - s;   // exclusive prefix of warp totals
        if (lane == 31) *total = si;
    }
    __syncthreads();
    int r = warp_sums[wid] + incl - x;
    __syncthreads();
    return r;
}

template <typename IdxT>
__global__ void __launch_bounds__(kThreads)
chunk_meta_kernel(const IdxT *__restrict__ cu, int32_t n_max, int64_t t_max, int32_t bt,
                  int64_t nt_max, int32_t *__restrict__ cu32, int32_t *__restrict__ idx,
                  int32_t *__restrict__ off, int32_t *__restrict__ order, int32_t *__restrict__ status) {
    __shared__ int s_flags;
    __shared__ int s_warp[32];
    __shared__ int s_total;
    __shared__ int s_carry;
    launch_dependents();          // the forward's first kernel waits for this grid's completion
    if (threadIdx.x == 0) {
        s_flags = 0;
        s_carry = 0;
    }
    __syncthreads();
    // ---- validity: bit0 decreasing, bit1 nonzero start, bit2 over capacity
    int flags = 0;
    if (threadIdx.x == 0) {
        if (cu[0] != 0) flags |= 2;
        if ((int64_t)cu[n_max] > t_max) flags |= 4;
    }
    for (int n = threadIdx.x; n < n_max; n += kThreads)
        if (cu[n + 1] < cu[n]) flags |= 1;
    if (flags) atomicOr(&s_flags, flags);
    __syncthreads();
    const int f = s_flags;
    const int code = (f & 2) ? GCL_DEV_CU_NONZERO_START
                   : (f & 1) ? GCL_DEV_CU_DECREASING
                   : (f & 4) ? GCL_DEV_CU_OVER_CAPACITY : GCL_DEV_OK;
    if (cu32)                     // the int32 copy: exact once valid, zeros otherwise
        for (int n = threadIdx.x; n <= n_max; n += kThreads) cu32[n] = code == GCL_DEV_OK ? (int32_t)cu[n] : 0;
    if (code != GCL_DEV_OK) {
        for (int64_t j = threadIdx.x; j < nt_max; j += kThreads) {
            idx[2 * j] = -1;
            idx[2 * j + 1] = 0;
        }
        for (int n = threadIdx.x; n <= n_max; n += kThreads) off[n] = 0;
        if (order)
            for (int n = threadIdx.x; n < n_max; n += kThreads) order[n] = n;
        if (threadIdx.x == 0) *status = code;
        return;
    }
    // ---- offsets: exclusive scan of ceil(len / bt)
    for (int base = 0; base < n_max; base += kThreads) {
        const int n = base + threadIdx.x;
        const int cnt = (n < n_max) ? (int)(((int64_t)cu[n + 1] - (int64_t)cu[n] + bt - 1) / bt) : 0;
        const int ex = block_exclusive_scan(cnt, s_warp, &s_total);
        if (n < n_max) off[n] = s_carry + ex;
        __syncthreads();
        if (threadIdx.x == 0) s_carry += s_total;
        __syncthreads();
    }
    const int live = s_carry;
    if (threadIdx.x == 0) off[n_max] = live;
    __syncthreads();   // off[] written by this block is visible to it after the barrier
    // ---- rows: binary search for the sequence that owns row j
    for (int64_t j = threadIdx.x; j < nt_max; j += kThreads) {
        if (j < live) {
            int lo = 0, hi = n_max - 1;   // largest n with off[n] <= j and a non-empty sequence
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (off[mid] <= j) lo = mid; else hi = mid - 1;
            }
            // off is non-decreasing; empty sequences share the offset of the next
            // non-empty one, so the largest n with off[n] <= j is the owner.
            idx[2 * j] = lo;
            idx[2 * j + 1] = (int)(j - off[lo]);
        } else {
            idx[2 * j] = -1;
            idx[2 * j + 1] = 0;
        }
    }
    // ---- longest-first order (stable): rank = #longer + #equal with smaller index
    if (order) {
        for (int n = threadIdx.x; n < n_max; n += kThreads) {
            const int ln = (int)(cu[n + 1] - cu[n]);
            int rank = 0;
            for (int m = 0; m < n_max; ++m) {
                const int lm = (int)(cu[m + 1] - cu[m]);
                rank += (lm > ln) || (lm == ln && m < n);
            }
            order[rank] = n;
        }
    }
    if (threadIdx.x == 0) *status = GCL_DEV_OK;
}

}  // namespace

cudaError_t launch_chunk_meta(const int32_t *cu, int32_t n_max, int64_t t_max, int32_t bt,
                              int64_t nt_max, int32_t *idx, int32_t *off, int32_t *order,
                              int32_t *status, cudaStream_t s) {
    chunk_meta_kernel<int32_t><<<1, kThreads, 0, s>>>(cu, n_max, t_max, bt, nt_max, nullptr, idx, off,
                                                      order, status);
    return cudaGetLastError();
}

cudaError_t launch_chunk_meta_i64(const int64_t *cu, int32_t n_max, int64_t t_max, int32_t bt,
                                  int64_t nt_max, int32_t *cu32, int32_t *idx, int32_t *off,
                                  int32_t *order, int32_t *status, cudaStream_t s) {
    chunk_meta_kernel<int64_t><<<1, kThreads, 0, s>>>(cu, n_max, t_max, bt, nt_max, cu32, idx, off,
                                                      order, status);
    return cudaGetLastError();
}

}  // namespace gcl
