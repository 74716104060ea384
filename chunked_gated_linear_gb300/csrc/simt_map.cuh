// simt_map.cuh -- the chunk-local Map phase on the CUDA cores (fp32).
//
// Shared by the fp32 forward and the backward kernels.  For one chunk of one
// (sequence, head) it loads q, k, g, beta (rows r >= len read as zero), forms
// the in-chunk inclusive cumsum gamma of the log gate (FLA RFC "[RFC] Add
// Graph Capture Support for FLA Prefill and Training Paths on Ascend NPUs",
// section "Step 3": gate / chunk cumsum), the decay-weighted matrices
//   A'[r,i] = exp(gamma_r - gamma_i) (k_r . k_i)            i < r   (A = beta_r A')
//   L[r,i]  = scale exp(gamma_r - gamma_i) (q_r . k_i)     i <= r
// ("forward intra": KK^T and QK^T; per key channel for KDA), and
// T = (I + A)^-1 by row-wise forward substitution ("triangular solve").
// All decay factors are exp of a non-positive number, so nothing overflows.
// C is the chunk size (BT, 32 or 64); C x C tiles use the row stride C + 1.
#pragma once

#include "gcl_internal.cuh"

namespace gcl {

// Shared-memory row strides: +1 float spreads rows over the banks.
template <int K>
struct SimtStrides {
    static constexpr int LK = K + 1;
};

template <int VAR, typename Tin, int K, int NT, int C>
__device__ __forceinline__ void simt_load_chunk(const Tin *q, const Tin *k, const float *g,
                                                const Tin *beta, int64_t t0, int len, int h,
                                                int H, float *sQ, float *sK, float *sG,
                                                float *sB, int64_t t_max, int32_t *st) {
    constexpr int LK = K + 1;
    const int tid = threadIdx.x;
    for (int e = tid; e < C * K; e += NT) {
        const int r = e / K, c = e % K;
        const int64_t gi = ((t0 + r) * H + h) * (int64_t)K + c;
        const bool ok = r < len && GCL_IN_BOUNDS(gi, t_max * H * K, st);
        sQ[r * LK + c] = ok ? ld_in(q, gi) : 0.f;
        sK[r * LK + c] = ok ? ld_in(k, gi) : 0.f;
        if (VAR == kKDA) sG[r * LK + c] = ok ? g[gi] : 0.f;
    }
    for (int r = tid; r < C; r += NT) {
        const bool ok = r < len && GCL_IN_BOUNDS((t0 + r) * H + h, t_max * H, st);
        sB[r] = ok ? ld_in(beta, (t0 + r) * H + h) : 0.f;
        if (VAR == kGDN) sG[r] = ok ? g[(t0 + r) * H + h] : 0.f;
    }
}

// gamma: inclusive cumsum of g down the chunk (per key channel for KDA).
template <int VAR, int K, int NT, int C>
__device__ __forceinline__ void simt_gate_cumsum(float *sG) {
    constexpr int LK = K + 1;
    const int tid = threadIdx.x;
    if (VAR == kGDN) {
        if (tid == 0) {
            float acc = 0.f;
            for (int r = 0; r < C; ++r) { acc += sG[r]; sG[r] = acc; }
        }
    } else {
        for (int c = tid; c < K; c += NT) {
            float acc = 0.f;
            for (int r = 0; r < C; ++r) { acc += sG[r * LK + c]; sG[r * LK + c] = acc; }
        }
    }
}

template <int VAR, int K>
__device__ __forceinline__ float gam(const float *sG, int r, int c) {
    return VAR == kGDN ? sG[r] : sG[r * (K + 1) + c];
}

// A (= beta_r A', strictly lower) into sA and L into sL.  If sAp is not null it
// also receives A' (without beta).  FastExp takes the per-channel decays of KDA with the
// hardware exponential (__expf: about 2^-21 relative error for the arguments that matter,
// |gamma_r - gamma_i| of a few units, far inside the fp32 bar; the gradients take it, the
// forward keeps expf).  LDA: the row stride of sA (the others take C + 1).
template <int VAR, int K, int NT, int C, bool FastExp = false, int LDA = C + 1>
__device__ __forceinline__ void simt_intra(const float *sQ, const float *sK, const float *sG,
                                           const float *sB, float scale, float *sA, float *sL,
                                           float *sAp) {
    constexpr int LK = K + 1, kLC = C + 1;
    if constexpr (VAR == kGDN && (C / 4) * (C / 4) <= NT) {
        // GDN: one 4 x 4 tile of (r, i) pairs per thread, so each loaded key and query
        // element serves four dot products (tiles above the diagonal are all zero)
        constexpr int NTILE = C / 4;
        const int t = threadIdx.x;
        if (t < NTILE * NTILE) {
            const int r0 = (t / NTILE) * 4, i0 = (t % NTILE) * 4;
            float kk[4][4] = {}, qk[4][4] = {};
            if (i0 <= r0 + 3) {
                for (int c = 0; c < K; ++c) {
                    float kr[4], qr[4], ki[4];
#pragma unroll
                    for (int a = 0; a < 4; ++a) {
                        kr[a] = sK[(r0 + a) * LK + c];
                        qr[a] = sQ[(r0 + a) * LK + c];
                        ki[a] = sK[(i0 + a) * LK + c];
                    }
#pragma unroll
                    for (int a = 0; a < 4; ++a)
#pragma unroll
                        for (int b = 0; b < 4; ++b) {
                            kk[a][b] = fmaf(kr[a], ki[b], kk[a][b]);
                            qk[a][b] = fmaf(qr[a], ki[b], qk[a][b]);
                        }
                }
            }
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    const int r = r0 + a, i = i0 + b;
                    const bool on = i <= r;
                    const float d = expf(on ? sG[r] - sG[i] : 0.f);
                    const float ap = (i < r) ? kk[a][b] * d : 0.f;
                    const float l = on ? scale * (qk[a][b] * d) : 0.f;
                    if (sA) sA[r * LDA + i] = sB[r] * ap;
                    if (sAp) sAp[r * kLC + i] = ap;
                    if (sL) sL[r * kLC + i] = l;
                }
        }
        return;
    }
    for (int e = threadIdx.x; e < C * C; e += NT) {
        const int r = e / C, i = e % C;
        float ap = 0.f, l = 0.f;
        if (i <= r) {
            float kk = 0.f, qk = 0.f;
            if (VAR == kGDN) {
                for (int c = 0; c < K; ++c) {
                    kk = fmaf(sK[r * LK + c], sK[i * LK + c], kk);
                    qk = fmaf(sQ[r * LK + c], sK[i * LK + c], qk);
                }
                const float d = expf(sG[r] - sG[i]);
                kk *= d;
                qk *= d;
            } else {
                for (int c = 0; c < K; ++c) {
                    const float x = sG[r * LK + c] - sG[i * LK + c];
                    const float d = FastExp ? __expf(x) : expf(x);
                    kk = fmaf(sK[r * LK + c] * d, sK[i * LK + c], kk);
                    qk = fmaf(sQ[r * LK + c] * d, sK[i * LK + c], qk);
                }
            }
            ap = (i < r) ? kk : 0.f;
            l = scale * qk;
        }
        if (sA) sA[r * LDA + i] = sB[r] * ap;
        if (sAp) sAp[r * kLC + i] = ap;
        if (sL) sL[r * kLC + i] = l;
    }
}

// T = (I + A)^-1 for unit lower-triangular I + A:
//   T[r,r] = 1,  T[r,i] = -A[r,i] - sum_{i<m<r} A[r,m] T[m,i]  (i < r), row by row.
template <int NT, int C>
__device__ __forceinline__ void simt_solve(const float *sA, float *sT) {
    constexpr int kLC = C + 1;
    for (int e = threadIdx.x; e < C * C; e += NT) {
        const int r = e / C, i = e % C;
        sT[r * kLC + i] = (r == i) ? 1.f : 0.f;
    }
    __syncthreads();
    for (int r = 1; r < C; ++r) {
        for (int i = threadIdx.x; i < r; i += NT) {
            float acc = -sA[r * kLC + i];
            for (int m = i + 1; m < r; ++m) acc = fmaf(-sA[r * kLC + m], sT[m * kLC + i], acc);
            sT[r * kLC + i] = acc;
        }
        __syncthreads();
    }
}

// T = (I + A)^-1 by blocked forward substitution over 16-row blocks (the same scheme as the
// tensor-core path's solve: diagonal blocks column by column, one thread per column, then
// the off-diagonal blocks level by level, T_ij = -T_ii sum_{k=j}^{i-1} A_ik T_kj), with the
// row stride of the CUDA-core layouts; 1 + 2 (C / 16 - 1) block barriers instead of C - 1.
// sX: scratch of at least 3 * 16 * 16 floats.  T is written on and below the diagonal and
// zero above it.  All NT threads of the block call it.
template <int NT, int C>
__device__ __forceinline__ void simt_solve_blocked(const float *sA, float *sT, float *sX) {
    constexpr int kLC = C + 1, NB = C / 16;
    static_assert(C % 16 == 0 && NT >= C, "16-row blocks, one thread per column");
    const int tid = threadIdx.x;
    for (int e = tid; e < C * C; e += NT) {          // zeros above the diagonal blocks
        const int r = e / C, i = e % C;
        if ((i >> 4) > (r >> 4)) sT[r * kLC + i] = 0.f;
    }
    if (tid < C) {   // ---- diagonal blocks: thread (block, column jj)
        const int o = (tid >> 4) * 16, jj = tid & 15;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) x[r] = (r == jj) ? 1.f : 0.f;
#pragma unroll
        for (int r = 1; r < 16; ++r) {
            float part[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int m = 0; m < r; ++m)
                part[m & 3] = fmaf(sA[(o + r) * kLC + o + m], x[m], part[m & 3]);
            const float sum = (part[0] + part[1]) + (part[2] + part[3]);
            if (r > jj) x[r] = -sum;
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) sT[(o + r) * kLC + o + jj] = x[r];
    }
    __syncthreads();
#pragma unroll
    for (int d = 1; d < NB; ++d) {
        const int nel = (NB - d) * 256;               // (block, row, column) of level d
        for (int s = tid; s < nel; s += NT) {
            const int blk = s >> 8, rr = (s >> 4) & 15, cc = s & 15;
            const int bi = d + blk, bj = blk;
            float acc = 0.f;
#pragma unroll
            for (int m = 0; m < 16 * d; ++m)
                acc = fmaf(sA[(bi * 16 + rr) * kLC + bj * 16 + m], sT[(bj * 16 + m) * kLC + bj * 16 + cc], acc);
            sX[(blk * 16 + rr) * 16 + cc] = acc;
        }
        __syncthreads();
        for (int s = tid; s < nel; s += NT) {
            const int blk = s >> 8, rr = (s >> 4) & 15, cc = s & 15;
            const int bi = d + blk, bj = blk;
            float acc = 0.f;
#pragma unroll
            for (int m = 0; m < 16; ++m)
                acc = fmaf(sT[(bi * 16 + rr) * kLC + bi * 16 + m], sX[(blk * 16 + m) * 16 + cc], acc);
            sT[(bi * 16 + rr) * kLC + bj * 16 + cc] = -acc;
        }
        __syncthreads();
    }
}

// W = T diag(beta Gamma) K (GDN) or T diag(beta) (K * Gamma) (KDA).
template <int VAR, int K, int NT, int C>
__device__ __forceinline__ void simt_w(const float *sT, const float *sB, const float *sG,
                                       const float *sK, float *sW) {
    constexpr int LK = K + 1, kLC = C + 1;
    for (int e = threadIdx.x; e < C * K; e += NT) {
        const int r = e / K, c = e % K;
        float acc = 0.f;
        if (VAR == kGDN) {   // the row factor beta_i Gamma_i does not depend on the key
            for (int i = 0; i <= r; ++i)
                acc = fmaf(sT[r * kLC + i] * (sB[i] * expf(sG[i])), sK[i * LK + c], acc);
        } else {
            for (int i = 0; i <= r; ++i)
                acc = fmaf(sT[r * kLC + i] * sB[i] * expf(gam<VAR, K>(sG, i, c)), sK[i * LK + c], acc);
        }
        sW[r * LK + c] = acc;
    }
}

}  // namespace gcl
