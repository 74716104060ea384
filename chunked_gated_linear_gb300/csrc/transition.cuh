// transition.cuh -- the per-chunk record of the transition form, shared by its forward
// (fwd_tc_transition.cu) and backward (bwd_tc_transition.cu) kernels.
//
// For chunk n of a sequence (HA-NPU paper "Empowering Hybrid Attention Models on NPUs",
// section 2.1, Map-Reduce-Map) the state update and the output are affine in the state
// entering the chunk:
//   S' = Gamma_c S + N S + B,      O = Y S + Z,
//   N = -Ktil^T W,  B = Ktil^T U,  Y = scale diag(Gamma) Q - L W,  Z = L U.
// The record holds [Y; N | B | Z] as 384 rows of 128 bf16 (Y rows 0..63, N 64..191,
// B 192..319, Z 320..383; 96 KiB so every record starts on a 1 KiB boundary).  The workspace
// is nt_max * H records, then Gamma_c of every record in 512-byte slots: GDN's scalar in the
// first float, KDA's per-key-channel decay exp(gamma_c) as 128 floats.
#pragma once

#include "op16.cuh"

#include <cuda_bf16.h>
#include <stdint.h>

#include "gcl_internal.cuh"

namespace gcl {
namespace tr {

constexpr int C = 64;
constexpr int KD = 128;
constexpr int VD = 128;
constexpr size_t kYNRows = 192;                      // [Y; N], bf16, 128 columns
constexpr size_t kYNBytes = kYNRows * KD * 2;        // 48 KiB
constexpr size_t kBBytes = (size_t)KD * VD * 2;      // 32 KiB
constexpr size_t kZBytes = (size_t)C * VD * 2;       // 16 KiB
constexpr size_t kUnitBytes = kYNBytes + kBBytes + kZBytes;
constexpr size_t kGBytes = 512;                      // Gamma_c slot (128 floats)
// The backward sweep hands dS' of every chunk to the chunk-gradient kernels as a bf16 tile:
// 128 key rows x 128 value columns in two 64-column blocks, 128-byte swizzle (kmaj16 below).
constexpr size_t kDsTileBytes = (size_t)KD * VD * 2;
static_assert(kUnitBytes % 1024 == 0, "records start on 1 KiB boundaries");

// Address of the Gamma_c slot of record `unit` in a workspace of nt_max * H records.
__host__ __device__ inline size_t gc_offset(int64_t nt_max, int H, int64_t unit) {
    return (size_t)nt_max * H * kUnitBytes + (size_t)unit * kGBytes;
}

__device__ __forceinline__ uint4 pack8(const float *x) {
    uint4 pk;
    __nv_bfloat162 *pp = reinterpret_cast<__nv_bfloat162 *>(&pk);
#pragma unroll
    for (int e = 0; e < 4; ++e) pp[e] = __floats2bfloat162_rn(x[2 * e], x[2 * e + 1]);
    return pk;
}

// Offset of element (k, n) (n < 64) of an MN-major bf16 operand with the 128-byte swizzle:
// 8-row k-groups of 1024 B, 16-byte chunk index XOR (k % 8).
__device__ __forceinline__ uint32_t mn_sw128(int k, int n) {
    return (uint32_t)((k >> 3) * 1024 + (k & 7) * 128 + ((((n >> 3) ^ (k & 7))) << 4) + (n & 7) * 2);
}

__device__ __forceinline__ float warp_scan(float x) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, x, d);
        if (lane >= d) x += y;
    }
    return x;
}

// K-major 128-byte-swizzled bf16 tile of `rows` rows per 64-column block: byte offset
// of the 16-byte chunk that holds columns [col, col + 8) of `row`.
__device__ __forceinline__ uint32_t kmaj16(int rows, int row, int col) {
    return (uint32_t)((col >> 6) * rows * 128 + (row >> 3) * 1024 + (row & 7) * 128 +
                      ((((col & 63) >> 3) ^ (row & 7)) << 4));
}
// MN-major 128-byte-swizzled bf16 operand (8-row k-groups of 1024 B, 64-element atoms
// `atom_bytes` apart): byte offset of the 16-byte chunk holding elements [n, n + 8) of k.
__device__ __forceinline__ uint32_t mnmaj16(uint32_t atom_bytes, int k, int n) {
    return (uint32_t)((n >> 6) * atom_bytes + (k >> 3) * 1024 + (k & 7) * 128 +
                      ((((n & 63) >> 3) ^ (k & 7)) << 4));
}

// ---------------------------------------------------------------- record-producing launches
// Parameters of the persistent kernels that write the records (GDN: g is [t_max, H];
// KDA: g is [t_max, H, K]).
struct PrepTParams {
    const int32_t *chunk_indices, *cu;
    const float *g;
    const void *beta;            // [t_max, H] of the input type (bf16 or fp16)
    uint8_t *ws;                 // nt_max * H records of kUnitBytes, then the Gamma_c slots
    int32_t *status;
    int64_t t_max, nt_max;
    int32_t n_max, H;
    float scale;
};

// One work item per row j of chunk_indices and head h, numbered i = j H + h (the record
// index).  Rows past the live chunks hold the [-1, 0] sentinel, so a CTA that walks its items
// in increasing order stops at the first sentinel.
struct PrepItem {
    int64_t t0;
    int h, len;
};

// Next live item at or after i in steps of `stride` (-1 when there is none); invalid rows set
// the status word and are skipped.  Every thread of the block computes the same answer.
__device__ __forceinline__ int next_item(const PrepTParams &p, int i, int stride, PrepItem *it) {
    const int total = (int)(p.nt_max * p.H);
    for (; i < total; i += stride) {
        const int j = i / p.H;
        const int n = p.chunk_indices[2 * j];
        if (n < 0) return -1;                                  // sentinel: no more live rows
        const int ic = p.chunk_indices[2 * j + 1];
        if (n < p.n_max && ic >= 0) {
            const int64_t bos = p.cu[n], eos = p.cu[n + 1], t0 = bos + (int64_t)ic * C;
            if (bos >= 0 && eos >= bos && eos <= p.t_max && t0 < eos) {
                it->t0 = t0;
                it->h = i - j * p.H;
                it->len = (int)(eos - t0 < C ? eos - t0 : C);
                return i;
            }
        }
        if (threadIdx.x == 0) status_set(p.status, GCL_DEV_BAD_RANGE);
    }
    return -1;
}

}  // namespace tr

// Tensor maps of q, k, v (64 x 64 boxes, 128-byte swizzle) and of the records in ws (64 x 64
// boxes of the 384-row record), and the kernel parameters, for the record-producing launches.
bool make_prep_maps(const FwdParams &p, uint8_t *ws, CUtensorMap *mq, CUtensorMap *mk, CUtensorMap *mv,
                    CUtensorMap *mrec);
tr::PrepTParams make_prep_params(const FwdParams &p, uint8_t *ws);
// Records of every live chunk and head into ws (nt_max * H records + Gamma_c slots).
cudaError_t launch_prep_t(const FwdParams &p, uint8_t *ws, cudaStream_t s);
size_t transition_record_bytes(int64_t nt_max, int H);
// The chain over the records in ws (p.workspace is not used), split value-column slices per
// head; kda selects the per-key-channel Gamma_c.  Launched as a programmatic dependent.
// n_seg >= 2: the segment-parallel plan (summaries, scan, segment outputs) with its buffers at
// seg_ws (fwd_seg_workspace_bytes).
cudaError_t launch_chain_records(const FwdParams &p, const uint8_t *ws, int split, bool kda,
                                 cudaStream_t s, int n_seg = 0, float *seg_ws = nullptr);
// The segment plan for p when its workspace holds the segment buffers after the records.
void fwd_seg_plan(const FwdParams &p, uint8_t *ws, int *n_seg, float **seg_ws);


}  // namespace gcl
