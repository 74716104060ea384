// fwd_simt.cuh -- fused chunkwise forward on the CUDA cores, all arithmetic in fp32.
// The kernel templates; fwd_simt_{f32,bf16,f16}.cu instantiate them per input type.
//
// This kernel serves fp32 inputs (where a 1e-5 relative bound leaves no room
// for reduced-precision tensor-core operands) and every size the tensor-core
// kernel does not take.  One CTA owns one (sequence, head, value-column slice):
// it walks the chunks of its sequence in order and keeps its slice of the
// state S [K x VS] in shared memory for the whole sequence (HA-NPU paper
// "Empowering Hybrid Attention Models on NPUs", section 4: head-level mapping
// with the Map-Reduce-Map pipeline fused on one core; column-wise split of the
// value dimension, which needs no cross-CTA reduction because column j of S
// depends only on column j of v and h0).
//
// Per chunk of c <= C tokens (C = BT, 32 or 64; Map phase in simt_map.cuh):
//   Map     A, L, T = (I + A)^-1, W = T diag(beta Gamma) K, U = T diag(beta) V
//   Reduce  E = U - W S                                          (state read)
//   Map     O = scale diag(Gamma) Q S + L E                      (chunk output)
//   Reduce  S <- Gamma_c S + (diag(exp(gamma_c - gamma)) K)^T E (in-place update)
// with the per-key-channel gate of KDA in place of the scalar one.  The output
// is computed from the old state before the update overwrites it (HA-NPU
// section 5, chunk-first order).  Rows past the end of the sequence are loaded
// as k = q = v = 0, beta = 0, g = 0, which leaves S unchanged.
#pragma once

#include "simt_map.cuh"
#include "fwd_simt_split.cuh"

namespace gcl {
namespace simt_fwd {

constexpr int kThreads = 256;

template <int K, int VS, int VAR, int C>
struct FwdLayout {
    static constexpr int kLC = C + 1;
    static constexpr int LK = K + 1;
    static constexpr int LV = VS + 1;
    static constexpr int oQ = 0;                     // Q, later scale*Gamma*Q   [C][LK]
    static constexpr int oK = oQ + C * LK;           // K                        [C][LK]
    static constexpr int oW = oK + C * LK;           // W                        [C][LK]
    static constexpr int oV = oW + C * LK;           // V slice                  [C][LV]
    static constexpr int oE = oV + C * LV;           // E                        [C][LV]
    static constexpr int oS = oE + C * LV;           // state slice              [K][LV]
    static constexpr int oA = oS + K * LV;           // A                        [C][kLC]
    static constexpr int oT = oA + C * kLC;          // T = (I + A)^-1           [C][kLC]
    static constexpr int oL = oT + C * kLC;          // L                        [C][kLC]
    static constexpr int oB = oL + C * kLC;          // beta                     [C]
    static constexpr int oG = oB + C;                // gamma [C] or [C][LK]
    static constexpr int total = oG + (VAR == kKDA ? C * LK : C);
    static constexpr size_t bytes = sizeof(float) * total;
};

template <int VAR, typename Tin, int K, int VS, int C>
__global__ void __launch_bounds__(kThreads)
fwd_simt_kernel(FwdParams p) {
    using Lay = FwdLayout<K, VS, VAR, C>;
    constexpr int kLC = C + 1;
    extern __shared__ float sm[];
    float *sQ = sm + Lay::oQ, *sK = sm + Lay::oK, *sW = sm + Lay::oW;
    float *sV = sm + Lay::oV, *sE = sm + Lay::oE, *sS = sm + Lay::oS;
    float *sA = sm + Lay::oA, *sT = sm + Lay::oT, *sL = sm + Lay::oL;
    float *sB = sm + Lay::oB, *sG = sm + Lay::oG;
    constexpr int LK = Lay::LK, LV = Lay::LV;

    if (status_blocks_cta(p.dev_status)) return;
    const int tid = threadIdx.x;
    const int split = blockIdx.x, h = blockIdx.y;
    const int n = p.seq_order ? p.seq_order[blockIdx.z] : (int)blockIdx.z;
    const int H = p.H, V = p.V;
    const int v0 = split * VS;
    if (n < 0 || n >= p.n_max) {              // checked before cu[n] and cu[n + 1] are read
        if (tid == 0) status_set(p.dev_status, GCL_DEV_BAD_RANGE);
        return;
    }
    const int64_t bos = p.cu_seqlens[n], eos = p.cu_seqlens[n + 1];
    if (bos < 0 || eos < bos || eos > p.t_max) {
        if (tid == 0) status_set(p.dev_status, GCL_DEV_BAD_RANGE);
        return;
    }
    const Tin *q = static_cast<const Tin *>(p.q);
    const Tin *k = static_cast<const Tin *>(p.k);
    const Tin *v = static_cast<const Tin *>(p.v);
    const Tin *beta = static_cast<const Tin *>(p.beta);
    Tin *o = static_cast<Tin *>(p.o);
    const int64_t KV = (int64_t)K * V;
    const int64_t state_base = ((int64_t)n * H + h) * KV;

    for (int e = tid; e < K * VS; e += kThreads) {
        const int c = e / VS, j = e % VS;
        sS[c * LV + j] = (p.h0 && GCL_IN_BOUNDS(state_base + (int64_t)c * V + v0 + j,
                                                (int64_t)p.n_max * H * KV, p.dev_status))
                             ? p.h0[state_base + (int64_t)c * V + v0 + j] : 0.f;
    }
    const int nchunks = (int)((eos - bos + C - 1) / C);
    for (int ic = 0; ic < nchunks; ++ic) {
        const int64_t t0 = bos + (int64_t)ic * C;
        const int len = (int)(eos - t0 < C ? eos - t0 : C);
        __syncthreads();   // previous chunk finished with every buffer
        if (p.h_save) {
            const int64_t row = (int64_t)p.chunk_offsets[n] + ic;
            if (row < 0 || row >= p.nt_max) {      // metadata inconsistent with cu_seqlens
                if (tid == 0) status_set(p.dev_status, GCL_DEV_BAD_RANGE);
                return;
            }
            float *dst = p.h_save + (row * H + h) * KV;
            for (int e = tid; e < K * VS; e += kThreads) {
                const int c = e / VS, j = e % VS;
                if (GCL_IN_BOUNDS((row * H + h) * KV + (int64_t)c * V + v0 + j, p.nt_max * H * KV, p.dev_status))
                    dst[(int64_t)c * V + v0 + j] = sS[c * LV + j];
            }
        }
        simt_load_chunk<VAR, Tin, K, kThreads, C>(q, k, p.g, beta, t0, len, h, H, sQ, sK, sG, sB, p.t_max, p.dev_status);
        for (int e = tid; e < C * VS; e += kThreads) {
            const int r = e / VS, j = e % VS;
            sV[r * LV + j] = (r < len && GCL_IN_BOUNDS(((t0 + r) * H + h) * (int64_t)V + v0 + j,
                                                        p.t_max * H * (int64_t)V, p.dev_status))
                                 ? ld_in(v, ((t0 + r) * H + h) * (int64_t)V + v0 + j) : 0.f;
        }
        __syncthreads();
        simt_gate_cumsum<VAR, K, kThreads, C>(sG);
        __syncthreads();
        simt_intra<VAR, K, kThreads, C>(sQ, sK, sG, sB, p.scale, sA, sL, nullptr);
        __syncthreads();
        simt_solve_blocked<kThreads, C>(sA, sT, sE);    // E is formed only after the solve
        simt_w<VAR, K, kThreads, C>(sT, sB, sG, sK, sW);
        __syncthreads();
        // E = T diag(beta) V - W S
        for (int e = tid; e < C * VS; e += kThreads) {
            const int r = e / VS, j = e % VS;
            float acc = 0.f;
            for (int i = 0; i <= r; ++i) acc = fmaf(sT[r * kLC + i] * sB[i], sV[i * LV + j], acc);
            for (int c = 0; c < K; ++c) acc = fmaf(-sW[r * LK + c], sS[c * LV + j], acc);
            sE[r * LV + j] = acc;
        }
        // Q <- scale Gamma Q (in place; A and L no longer need Q)
        for (int e = tid; e < C * K; e += kThreads) {
            const int r = e / K, c = e % K;
            sQ[r * LK + c] *= p.scale * expf(gam<VAR, K>(sG, r, c));
        }
        __syncthreads();
        // O = (scale Gamma Q) S + L E   (old state: read before the update)
        if (o != nullptr) {
            for (int e = tid; e < C * VS; e += kThreads) {
                const int r = e / VS, j = e % VS;
                if (r < len) {
                    float acc = 0.f;
                    for (int c = 0; c < K; ++c) acc = fmaf(sQ[r * LK + c], sS[c * LV + j], acc);
                    for (int i = 0; i <= r; ++i) acc = fmaf(sL[r * kLC + i], sE[i * LV + j], acc);
                    if (GCL_IN_BOUNDS(((t0 + r) * H + h) * (int64_t)V + v0 + j, p.t_max * H * (int64_t)V,
                                      p.dev_status))
                        st_out(o, ((t0 + r) * H + h) * (int64_t)V + v0 + j, acc);
                }
            }
        }
        // K <- K * exp(gamma_c - gamma) in place (K is not read again in this chunk): one
        // exponential per (row, key) instead of one per (row, key, value column) below
        for (int e = tid; e < C * K; e += kThreads) {
            const int i = e / K, c = e % K;
            sK[i * LK + c] = expf(gam<VAR, K>(sG, C - 1, c) - gam<VAR, K>(sG, i, c)) * sK[i * LK + c];
        }
        __syncthreads();
        // S <- Gamma_c S + (K * exp(gamma_c - gamma))^T E   (in place)
        for (int e = tid; e < K * VS; e += kThreads) {
            const int c = e / VS, j = e % VS;
            float acc = expf(gam<VAR, K>(sG, C - 1, c)) * sS[c * LV + j];
            for (int i = 0; i < C; ++i) acc = fmaf(sK[i * LK + c], sE[i * LV + j], acc);
            sS[c * LV + j] = acc;
        }
    }
    __syncthreads();
    if (p.ht) {
        for (int e = tid; e < K * VS; e += kThreads) {
            const int c = e / VS, j = e % VS;
            if (GCL_IN_BOUNDS(state_base + (int64_t)c * V + v0 + j, (int64_t)p.n_max * H * KV, p.dev_status))
                p.ht[state_base + (int64_t)c * V + v0 + j] = sS[c * LV + j];
        }
    }
}

template <int VAR, typename Tin, int K, int VS, int C>
cudaError_t launch_one(const FwdParams &p, cudaStream_t s) {
    using Lay = FwdLayout<K, VS, VAR, C>;
    auto kern = fwd_simt_kernel<VAR, Tin, K, VS, C>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)Lay::bytes);
    if (e != cudaSuccess) return e;
    dim3 grid(p.V / VS, p.H, p.n_max);
    kern<<<grid, kThreads, Lay::bytes, s>>>(p);
    return cudaGetLastError();
}

// Value-column slices: 16 columns per CTA at K = 64 (a 64-wide head in 4 slices, so a few
// (sequence, head) units still spread over the GPU), 32 at K = 128 (the state slice and the
// chunk's K, Q, W tiles then fill the shared memory of two CTAs per SM).
template <int VAR, typename Tin, int C>
cudaError_t launch_chunk(const FwdParams &p, cudaStream_t s) {
    if (p.K == 64) return launch_one<VAR, Tin, 64, 16, C>(p, s);
    return launch_one<VAR, Tin, 128, 32, C>(p, s);
}

}  // namespace simt_fwd

// The split plan (chunk prep + chain) for K = V, chunk C.
template <int VAR, typename Tin, int C>
cudaError_t launch_split(const FwdParams &p, cudaStream_t s) {
    if (p.K == 64) return simt_split::launch<VAR, Tin, 64, 64, C>(p, s);
    return simt_split::launch<VAR, Tin, 128, 128, C>(p, s);
}

// Whether a call runs the split plan: K = V, the chunk metadata given and a workspace that
// holds the records (the single kernel needs neither).
inline bool fwd_simt_runs_split(const FwdParams &p) {
    const size_t need = fwd_simt_split_bytes(p.K, p.V, p.bt, p.nt_max, p.H);
    return need > 0 && p.workspace && p.workspace_bytes >= need && p.chunk_indices && p.chunk_offsets;
}

// The CUDA-core forward for input type Tin: variant, chunk size 32 or 64; the split plan
// where the workspace holds its records, else the single kernel.
template <typename Tin>
cudaError_t launch_fwd_simt_t(const FwdParams &p, int variant, cudaStream_t s) {
    using namespace simt_fwd;
    if (fwd_simt_runs_split(p)) {
        if (variant == kGDN)
            return p.bt == 32 ? launch_split<kGDN, Tin, 32>(p, s) : launch_split<kGDN, Tin, 64>(p, s);
        return p.bt == 32 ? launch_split<kKDA, Tin, 32>(p, s) : launch_split<kKDA, Tin, 64>(p, s);
    }
    if (variant == kGDN)
        return p.bt == 32 ? launch_chunk<kGDN, Tin, 32>(p, s) : launch_chunk<kGDN, Tin, 64>(p, s);
    return p.bt == 32 ? launch_chunk<kKDA, Tin, 32>(p, s) : launch_chunk<kKDA, Tin, 64>(p, s);
}

}  // namespace gcl
