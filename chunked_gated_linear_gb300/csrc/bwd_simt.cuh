// bwd_simt.cuh -- GDN and KDA chunk backward on the CUDA cores (fp32 arithmetic).
// The kernel templates (chunk size C = BT, 32 or 64); bwd_simt_{f32,bf16,f16}.cu instantiate
// them per input type.
//
// FLA RFC "[RFC] Add Graph Capture Support for FLA Prefill and Training Paths
// on Ascend NPUs", section "Step 3": the backward path covers recomputation,
// state, WY, gate and gradient kernels.  Here that is three launches:
//
//  1. (only without saved states) the forward kernel recomputes the state
//     before every chunk, S_n, into the workspace;
//  2. dstate sweep (here unless the caller ran the tensor-core sweep of
//     bwd_tc_transition.cu): per (sequence, head, value-column slice), in reverse chunk
//     order, the gradient w.r.t. the state after chunk n, dS'_n, is saved and
//     carried back through the chunk:
//        dE = L^T dO + Ktil dS'
//        dS = Gamma_c dS' + Qhat^T dO - W^T dE        (dS'_{n-1} = dS)
//     with Qhat = scale diag(Gamma) Q, Ktil = diag(exp(gamma_c - gamma)) K;
//     the last dS is dh0.  It needs no forward state.
//  3. chunk gradients, one CTA per row of chunk_indices (sentinel rows exit):
//     with S = S_n, dS' = dS'_n, R = diag(beta)(V - diag(Gamma) K S), E = T R,
//        dVb = T^T dE,  dv = diag(beta) dVb,   dT = dE R^T,   dL = dO E^T,
//        dA  = -T^T dT T^T (strictly lower),
//        dq  = scale diag(Gamma) dO S^T + P K,            P = scale e^{g_r-g_i} dL
//        dk  = diag(e^{g_c-g}) E dS'^T - diag(beta Gamma) dVb S^T
//              + P^T Q + M K + M^T K,                      M = dA beta_r e^{g_r-g_i}
//        dbeta, dgamma from every beta, Gamma, Gamma_c and exp(gamma_r - gamma_i)
//        factor, dg = reverse cumsum of dgamma inside the chunk.
//     The value dimension is walked in slices of VS columns; products that sum
//     over it accumulate in registers (dq, dk partials) and shared memory
//     (dT, dL, row sums), always in a fixed order, so results are bitwise
//     reproducible (no atomics).
#pragma once

#include "simt_map.cuh"

namespace gcl {
namespace simt_bwd {

// ---------------------------------------------------------------- dstate sweep
constexpr int kSweepThreads = 256;

template <int K, int VS, int VAR, int C>
struct SweepLayout {
    static constexpr int LK = K + 1, LV = VS + 1, kLC = C + 1;
    static constexpr int oQ = 0, oK = oQ + C * LK, oW = oK + C * LK;
    static constexpr int oDO = oW + C * LK, oDE = oDO + C * LV, oDS = oDE + C * LV;
    static constexpr int oA = oDS + K * LV, oT = oA + C * kLC, oL = oT + C * kLC;
    static constexpr int oB = oL + C * kLC, oG = oB + C;
    static constexpr int total = oG + (VAR == kKDA ? C * LK : C);
    static constexpr size_t bytes = sizeof(float) * total;
};

template <int VAR, typename Tin, int K, int VS, int C>
__global__ void __launch_bounds__(kSweepThreads)
dstate_sweep_kernel(BwdParams p) {
    using Lay = SweepLayout<K, VS, VAR, C>;
    constexpr int kLC = C + 1;
    extern __shared__ float sm[];
    float *sQ = sm + Lay::oQ, *sK = sm + Lay::oK, *sW = sm + Lay::oW;
    float *sDO = sm + Lay::oDO, *sDE = sm + Lay::oDE, *sDS = sm + Lay::oDS;
    float *sA = sm + Lay::oA, *sT = sm + Lay::oT, *sL = sm + Lay::oL;
    float *sB = sm + Lay::oB, *sG = sm + Lay::oG;
    constexpr int LK = Lay::LK, LV = Lay::LV;

    if (status_blocks_cta(p.dev_status)) return;
    const int tid = threadIdx.x;
    const int v0 = blockIdx.x * VS, h = blockIdx.y, n = blockIdx.z;
    const int H = p.H, V = p.V;
    const int64_t bos = p.cu_seqlens[n], eos = p.cu_seqlens[n + 1];
    if (bos < 0 || eos < bos || eos > p.t_max) {
        if (tid == 0) status_set(p.dev_status, GCL_DEV_BAD_RANGE);
        return;
    }
    const Tin *q = static_cast<const Tin *>(p.q);
    const Tin *k = static_cast<const Tin *>(p.k);
    const Tin *beta = static_cast<const Tin *>(p.beta);
    const Tin *d_o = static_cast<const Tin *>(p.d_o);
    const int64_t KV = (int64_t)K * V;
    const int64_t state_base = ((int64_t)n * H + h) * KV;

    for (int e = tid; e < K * VS; e += kSweepThreads) {
        const int c = e / VS, j = e % VS;
        sDS[c * LV + j] = p.dht ? p.dht[state_base + (int64_t)c * V + v0 + j] : 0.f;
    }
    const int nchunks = (int)((eos - bos + C - 1) / C);
    for (int ic = nchunks - 1; ic >= 0; --ic) {
        const int64_t t0 = bos + (int64_t)ic * C;
        const int len = (int)(eos - t0 < C ? eos - t0 : C);
        __syncthreads();
        {   // dS' of this chunk: gradient w.r.t. the state after it
            const int64_t row = (int64_t)p.chunk_offsets[n] + ic;
            if (row < 0 || row >= p.nt_max) {      // metadata inconsistent with cu_seqlens
                if (tid == 0) status_set(p.dev_status, GCL_DEV_BAD_RANGE);
                return;
            }
            float *dst = p.dh + (row * H + h) * KV;
            for (int e = tid; e < K * VS; e += kSweepThreads) {
                const int c = e / VS, j = e % VS;
                dst[(int64_t)c * V + v0 + j] = sDS[c * LV + j];
            }
        }
        simt_load_chunk<VAR, Tin, K, kSweepThreads, C>(q, k, p.g, beta, t0, len, h, H, sQ, sK, sG,
                                                    sB, p.t_max, p.dev_status);
        for (int e = tid; e < C * VS; e += kSweepThreads) {
            const int r = e / VS, j = e % VS;
            sDO[r * LV + j] = r < len ? ld_in(d_o, ((t0 + r) * H + h) * (int64_t)V + v0 + j) : 0.f;
        }
        __syncthreads();
        simt_gate_cumsum<VAR, K, kSweepThreads, C>(sG);
        __syncthreads();
        simt_intra<VAR, K, kSweepThreads, C>(sQ, sK, sG, sB, p.scale, sA, sL, nullptr);
        __syncthreads();
        simt_solve_blocked<kSweepThreads, C>(sA, sT, sW);   // W is formed after the solve
        simt_w<VAR, K, kSweepThreads, C>(sT, sB, sG, sK, sW);
        // dE = L^T dO + Ktil dS'
        for (int e = tid; e < C * VS; e += kSweepThreads) {
            const int i = e / VS, j = e % VS;
            float acc = 0.f;
            for (int r = i; r < C; ++r) acc = fmaf(sL[r * kLC + i], sDO[r * LV + j], acc);
            for (int c = 0; c < K; ++c) {
                const float kt = expf(gam<VAR, K>(sG, C - 1, c) - gam<VAR, K>(sG, i, c)) *
                                 sK[i * LK + c];
                acc = fmaf(kt, sDS[c * LV + j], acc);
            }
            sDE[i * LV + j] = acc;
        }
        for (int e = tid; e < C * K; e += kSweepThreads) {
            const int r = e / K, c = e % K;
            sQ[r * LK + c] *= p.scale * expf(gam<VAR, K>(sG, r, c));
        }
        __syncthreads();
        // dS = Gamma_c dS' + Qhat^T dO - W^T dE   (in place: each element reads only itself)
        for (int e = tid; e < K * VS; e += kSweepThreads) {
            const int c = e / VS, j = e % VS;
            float acc = expf(gam<VAR, K>(sG, C - 1, c)) * sDS[c * LV + j];
            for (int r = 0; r < C; ++r) {
                acc = fmaf(sQ[r * LK + c], sDO[r * LV + j], acc);
                acc = fmaf(-sW[r * LK + c], sDE[r * LV + j], acc);
            }
            sDS[c * LV + j] = acc;
        }
    }
    __syncthreads();
    if (p.dh0) {
        for (int e = tid; e < K * VS; e += kSweepThreads) {
            const int c = e / VS, j = e % VS;
            p.dh0[state_base + (int64_t)c * V + v0 + j] = sDS[c * LV + j];
        }
    }
}

// ---------------------------------------------------------------- chunk gradients (GDN)
constexpr int kGradThreads = 512;
constexpr int kVS = 16;   // value columns per slice

template <int K, int C>
struct GradLayout {
    static constexpr int LK = K + 1, LV = kVS + 1, kLC = C + 1;
    static constexpr int oQ = 0, oK = oQ + C * LK;
    static constexpr int oT = oK + C * LK, oL = oT + C * kLC;
    static constexpr int oDL = oL + C * kLC, oDT = oDL + C * kLC;
    static constexpr int oB = oDT + C * kLC, oG = oB + C;
    static constexpr int oRA = oG + C, oRB = oRA + C, oRC = oRB + C, oRD = oRC + C;
    static constexpr int oDG = oRD + C;                // dgamma per row
    static constexpr int oRED = oDG + C;               // 32 floats for a block reduction
    static constexpr int oEG = oRED + 32;              // exp(gamma) per row
    static constexpr int oFR = oEG + C;                // exp(gamma_c - gamma) per row
    static constexpr int oFree = oFR + C;              // slice region
    // slice buffers
    static constexpr int oS = oFree, oDS = oS + K * LV;
    static constexpr int oV = oDS + K * LV, oDO = oV + C * LV, oKS = oDO + C * LV;
    static constexpr int oR = oKS + C * LV, oE = oR + C * LV, oDE = oE + C * LV;
    static constexpr int oDVB = oDE + C * LV, oX1 = oDVB + C * LV, oX2 = oX1 + C * LV;
    static constexpr int oFreeEnd = oX2 + C * LV;
    static_assert(oFreeEnd - oFree >= 2 * C * kLC, "slice region reused for two C x C tiles");
    static constexpr size_t bytes = sizeof(float) * oFreeEnd;
};

template <typename Tin, int K, int C>
__global__ void __launch_bounds__(kGradThreads)
chunk_grad_kernel(BwdParams p) {
    using Lay = GradLayout<K, C>;
    constexpr int kLC = C + 1;
    extern __shared__ float sm[];
    constexpr int LK = Lay::LK, LV = Lay::LV;
    constexpr int TPR = kGradThreads / C;   // threads per chunk row (8 at C = 64, 16 at C = 32)
    constexpr int CPT = K / TPR;            // dq/dk columns owned per thread
    static_assert(TPR * C == kGradThreads && CPT * TPR == K, "one thread group per chunk row");
    float *sQ = sm + Lay::oQ, *sK = sm + Lay::oK, *sT = sm + Lay::oT, *sL = sm + Lay::oL;
    float *sDL = sm + Lay::oDL, *sDT = sm + Lay::oDT, *sB = sm + Lay::oB, *sG = sm + Lay::oG;
    float *sRA = sm + Lay::oRA, *sRB = sm + Lay::oRB, *sRC = sm + Lay::oRC, *sRD = sm + Lay::oRD;
    float *sDG = sm + Lay::oDG, *sRed = sm + Lay::oRED;
    float *sEG = sm + Lay::oEG, *sFR = sm + Lay::oFR;
    float *sS = sm + Lay::oS, *sDS = sm + Lay::oDS, *sV = sm + Lay::oV, *sDO = sm + Lay::oDO;
    float *sKS = sm + Lay::oKS, *sR = sm + Lay::oR, *sE = sm + Lay::oE, *sDE = sm + Lay::oDE;
    float *sDVB = sm + Lay::oDVB, *sX1 = sm + Lay::oX1, *sX2 = sm + Lay::oX2;
    float *sA = sm + Lay::oFree;              // A during the Map; later dT T^T
    float *sAp = sm + Lay::oFree + C * kLC;   // A' at the end

    if (status_blocks_cta(p.dev_status)) return;
    const int n = p.chunk_indices[2 * blockIdx.x];
    if (n < 0) return;                         // sentinel row: nothing to do
    if (n >= p.n_max) {
        if (threadIdx.x == 0) status_set(p.dev_status, GCL_DEV_BAD_RANGE);
        return;
    }
    const int ic = p.chunk_indices[2 * blockIdx.x + 1];
    const int tid = threadIdx.x, h = blockIdx.y;
    const int H = p.H, V = p.V;
    const int64_t bos = p.cu_seqlens[n], eos = p.cu_seqlens[n + 1];
    const int64_t t0 = bos + (int64_t)ic * C;
    if (bos < 0 || eos < bos || eos > p.t_max || t0 >= eos) {
        if (tid == 0) status_set(p.dev_status, GCL_DEV_BAD_RANGE);
        return;
    }
    const int len = (int)(eos - t0 < C ? eos - t0 : C);
    const Tin *q = static_cast<const Tin *>(p.q);
    const Tin *k = static_cast<const Tin *>(p.k);
    const Tin *v = static_cast<const Tin *>(p.v);
    const Tin *beta = static_cast<const Tin *>(p.beta);
    const Tin *d_o = static_cast<const Tin *>(p.d_o);
    const int64_t KV = (int64_t)K * V;
    const int64_t row = (int64_t)p.chunk_offsets[n] + ic;
    if (row < 0 || row >= p.nt_max || ic < 0) {
        if (tid == 0) status_set(p.dev_status, GCL_DEV_BAD_RANGE);
        return;
    }
    const float *Sg = p.h + (row * H + h) * KV;
    const float *dSg = p.dh + (row * H + h) * KV;

    // ---- Map recompute
    simt_load_chunk<kGDN, Tin, K, kGradThreads, C>(q, k, p.g, beta, t0, len, h, H, sQ, sK, sG, sB, p.t_max, p.dev_status);
    __syncthreads();
    simt_gate_cumsum<kGDN, K, kGradThreads, C>(sG);
    __syncthreads();
    simt_intra<kGDN, K, kGradThreads, C>(sQ, sK, sG, sB, p.scale, sA, sL, nullptr);
    for (int e = tid; e < C * kLC; e += kGradThreads) { sDL[e] = 0.f; sDT[e] = 0.f; }
    for (int r = tid; r < C; r += kGradThreads) { sRA[r] = sRB[r] = sRC[r] = sRD[r] = 0.f; }
    __syncthreads();
    simt_solve_blocked<kGradThreads, C>(sA, sT, sAp);   // A' is formed at the end

    const float gC = sG[C - 1];
    // per-row exponentials, once (the loops below only multiply)
    for (int r = tid; r < C; r += kGradThreads) {
        sEG[r] = expf(sG[r]);
        sFR[r] = expf(gC - sG[r]);
    }
    __syncthreads();
    const int my_r = tid / TPR, my_c0 = tid % TPR;    // owner of dq/dk partials
    float dq_p[CPT], dk_p[CPT];
#pragma unroll
    for (int m = 0; m < CPT; ++m) { dq_p[m] = 0.f; dk_p[m] = 0.f; }
    float dgc_part = 0.f;

    for (int s0 = 0; s0 < V; s0 += kVS) {
        __syncthreads();
        for (int e = tid; e < K * kVS; e += kGradThreads) {
            const int c = e / kVS, j = e % kVS;
            const float sv = Sg[(int64_t)c * V + s0 + j], dsv = dSg[(int64_t)c * V + s0 + j];
            sS[c * LV + j] = sv;
            sDS[c * LV + j] = dsv;
            dgc_part = fmaf(sv, dsv, dgc_part);
        }
        for (int e = tid; e < C * kVS; e += kGradThreads) {
            const int r = e / kVS, j = e % kVS;
            const int64_t gi = ((t0 + r) * H + h) * (int64_t)V + s0 + j;
            sV[r * LV + j] = r < len ? ld_in(v, gi) : 0.f;
            sDO[r * LV + j] = r < len ? ld_in(d_o, gi) : 0.f;
        }
        __syncthreads();
        // KS, R = diag(beta)(V - diag(Gamma) KS), X1 = dO * (Q S), X2 = K dS'
        for (int e = tid; e < C * kVS; e += kGradThreads) {
            const int r = e / kVS, j = e % kVS;
            float ks = 0.f, qs = 0.f, kd = 0.f;
            for (int c = 0; c < K; ++c) {
                ks = fmaf(sK[r * LK + c], sS[c * LV + j], ks);
                qs = fmaf(sQ[r * LK + c], sS[c * LV + j], qs);
                kd = fmaf(sK[r * LK + c], sDS[c * LV + j], kd);
            }
            sKS[r * LV + j] = ks;
            sR[r * LV + j] = sB[r] * (sV[r * LV + j] - sEG[r] * ks);
            sX1[r * LV + j] = sDO[r * LV + j] * qs;
            sX2[r * LV + j] = kd;
        }
        __syncthreads();
        // E = T R;  dE = L^T dO + exp(gamma_c - gamma) X2
        for (int e = tid; e < C * kVS; e += kGradThreads) {
            const int r = e / kVS, j = e % kVS;
            float ev = 0.f, de = sFR[r] * sX2[r * LV + j];
            for (int i = 0; i <= r; ++i) ev = fmaf(sT[r * kLC + i], sR[i * LV + j], ev);
            for (int r2 = r; r2 < C; ++r2) de = fmaf(sL[r2 * kLC + r], sDO[r2 * LV + j], de);
            sE[r * LV + j] = ev;
            sDE[r * LV + j] = de;
        }
        __syncthreads();
        // dVb = T^T dE; dv = beta dVb
        for (int e = tid; e < C * kVS; e += kGradThreads) {
            const int i = e / kVS, j = e % kVS;
            float acc = 0.f;
            for (int r = i; r < C; ++r) acc = fmaf(sT[r * kLC + i], sDE[r * LV + j], acc);
            sDVB[i * LV + j] = acc;
            if (i < len) p.dv[((t0 + i) * H + h) * (int64_t)V + s0 + j] = sB[i] * acc;
        }
        // dL += dO E^T (i <= r);  dT += dE R^T (i <= r)
        for (int e = tid; e < C * C; e += kGradThreads) {
            const int r = e / C, i = e % C;
            if (i <= r) {
                float dl = 0.f, dt = 0.f;
                for (int j = 0; j < kVS; ++j) {
                    dl = fmaf(sDO[r * LV + j], sE[i * LV + j], dl);
                    dt = fmaf(sDE[r * LV + j], sR[i * LV + j], dt);
                }
                sDL[r * kLC + i] += dl;
                sDT[r * kLC + i] += dt;
            }
        }
        __syncthreads();
        // register partials: dq_p += dO S^T;  dk_p += e^{g_c-g} E dS'^T - beta Gamma dVb S^T
        {
            const float fe = sFR[my_r];
            const float fb = sB[my_r] * sEG[my_r];
#pragma unroll
            for (int m = 0; m < CPT; ++m) {
                const int c = my_c0 + TPR * m;
                float aq = dq_p[m], ak = dk_p[m];
                for (int j = 0; j < kVS; ++j) {
                    aq = fmaf(sDO[my_r * LV + j], sS[c * LV + j], aq);
                    ak = fmaf(fe * sE[my_r * LV + j], sDS[c * LV + j], ak);
                    ak = fmaf(-fb * sDVB[my_r * LV + j], sS[c * LV + j], ak);
                }
                dq_p[m] = aq;
                dk_p[m] = ak;
            }
        }
        // row sums (one thread per row, fixed order)
        for (int r = tid; r < C; r += kGradThreads) {
            float a = 0.f, b = 0.f, cc = 0.f, d = 0.f;
            for (int j = 0; j < kVS; ++j) {
                a += sX1[r * LV + j];
                b = fmaf(sDVB[r * LV + j], sV[r * LV + j], b);
                cc = fmaf(sDVB[r * LV + j], sKS[r * LV + j], cc);
                d = fmaf(sE[r * LV + j], sX2[r * LV + j], d);
            }
            sRA[r] += a; sRB[r] += b; sRC[r] += cc; sRD[r] += d;
        }
    }
    // <dS', S> over the whole state: fixed-order block reduction
    {
        float x = dgc_part;
        for (int d = 16; d > 0; d >>= 1) x += __shfl_xor_sync(0xffffffffu, x, d);
        if ((tid & 31) == 0) sRed[tid >> 5] = x;
    }
    __syncthreads();
    // dA = -T^T (dT T^T), strictly lower.  X = dT T^T into sA (dT is lower incl. diag).
    for (int e = tid; e < C * C; e += kGradThreads) {
        const int r = e / C, m = e % C;
        float acc = 0.f;
        for (int i = 0; i <= min(r, m); ++i) acc = fmaf(sDT[r * kLC + i], sT[m * kLC + i], acc);
        sA[r * kLC + m] = acc;
    }
    __syncthreads();
    for (int e = tid; e < C * C; e += kGradThreads) {
        const int r = e / C, i = e % C;
        float acc = 0.f;
        if (i < r)
            for (int m = r; m < C; ++m) acc = fmaf(-sT[m * kLC + r], sA[m * kLC + i], acc);
        sDT[r * kLC + i] = acc;      // sDT now holds dA
    }
    __syncthreads();
    simt_intra<kGDN, K, kGradThreads, C>(sQ, sK, sG, sB, p.scale, nullptr, nullptr, sAp);
    __syncthreads();
    const float* sDA = sDT;
    // dgamma and dbeta, one thread per row
    for (int r = tid; r < C; r += kGradThreads) {
        const float gr = sG[r], Gr = expf(gr);
        float dg = p.scale * Gr * sRA[r];
        for (int i = 0; i <= r; ++i) dg = fmaf(sDL[r * kLC + i], sL[r * kLC + i], dg);
        for (int r2 = r; r2 < C; ++r2) dg = fmaf(-sDL[r2 * kLC + r], sL[r2 * kLC + r], dg);
        float da_row = 0.f;
        for (int i = 0; i < r; ++i) da_row = fmaf(sDA[r * kLC + i], sAp[r * kLC + i], da_row);
        dg = fmaf(sB[r], da_row, dg);
        for (int r2 = r + 1; r2 < C; ++r2)
            dg = fmaf(-sDA[r2 * kLC + r] * sB[r2], sAp[r2 * kLC + r], dg);
        dg -= sB[r] * Gr * sRC[r];
        dg -= expf(gC - gr) * sRD[r];
        sDG[r] = dg;
        if (r < len) p.dbeta[(t0 + r) * H + h] = sRB[r] - Gr * sRC[r] + da_row;
    }
    __syncthreads();
    if (tid == 0) {
        // dgamma_c: the Ktil factors and Gamma_c; gamma_c is the last row's gamma
        float dgc = 0.f;
        for (int w = 0; w < kGradThreads / 32; ++w) dgc += sRed[w];
        dgc *= expf(gC);
        for (int i = 0; i < C; ++i) dgc = fmaf(expf(gC - sG[i]), sRD[i], dgc);
        sDG[C - 1] += dgc;
        // dg = reverse cumsum of dgamma
        float acc = 0.f;
        for (int r = C - 1; r >= 0; --r) {
            acc += sDG[r];
            if (r < len) p.dg[(t0 + r) * H + h] = acc;
        }
    }
    // P = scale e^{g_r - g_i} dL (i <= r) and M = dA beta_r e^{g_r - g_i} (i < r), in place of
    // dL and dA (the gate gradient above has read them), zero elsewhere
    __syncthreads();
    for (int e = tid; e < C * C; e += kGradThreads) {
        const int r = e / C, i = e % C;
        const float dec = i <= r ? expf(sG[r] - sG[i]) : 0.f;
        sDL[r * kLC + i] = i <= r ? p.scale * dec * sDL[r * kLC + i] : 0.f;
        sDT[r * kLC + i] = i < r ? sDT[r * kLC + i] * sB[r] * dec : 0.f;
    }
    __syncthreads();
    // dq = scale Gamma dO S^T + P K;  dk = partials + P^T Q + M K + M^T K
    {
        const float *sP = sDL, *sM = sDT;
        const int r = my_r;
        if (r < len) {
#pragma unroll
            for (int m = 0; m < CPT; ++m) {
                const int c = my_c0 + TPR * m;
                float aq = p.scale * sEG[r] * dq_p[m];
                for (int i = 0; i <= r; ++i) aq = fmaf(sP[r * kLC + i], sK[i * LK + c], aq);
                float ak = dk_p[m];
                for (int r2 = r; r2 < C; ++r2) ak = fmaf(sP[r2 * kLC + r], sQ[r2 * LK + c], ak);
                for (int i = 0; i < r; ++i) ak = fmaf(sM[r * kLC + i], sK[i * LK + c], ak);
                for (int r2 = r + 1; r2 < C; ++r2) ak = fmaf(sM[r2 * kLC + r], sK[r2 * LK + c], ak);
                p.dq[((t0 + r) * H + h) * (int64_t)K + c] = aq;
                p.dk[((t0 + r) * H + h) * (int64_t)K + c] = ak;
            }
        }
    }
}

// ---------------------------------------------------------------- KDA chunk gradients
// The decay is a vector over key channels, gamma[r][c].  With Kp = K o exp(gamma),
// Kb = K o exp(gamma_c - gamma), R = diag(beta)(V - Kp S), E = T R:
//   dE = L^T dO + Kb dS',   dR = T^T dE,   dv = diag(beta) dR,   dT = dE R^T,   dL = dO E^T,
//   dA = -T^T dT T^T (strictly lower),   Y1 = dR S^T,   Y2 = dO S^T,   Y3 = E dS'^T,
// and with D[r][i][c] = exp(gamma[r][c] - gamma[i][c]) the sums over the chunk
//   PL[r][c] = sum_{i<=r} dL[r][i] k[i][c] D[r][i][c],   PA[r][c] = sum_{i<r} dA[r][i] k[i][c] D[r][i][c],
//   QL[i][c] = sum_{r>=i} dL[r][i] q[r][c] D[r][i][c],   QA[i][c] = sum_{r>i} beta_r dA[r][i] k[r][c] D[r][i][c],
// give
//   dq = scale (exp(gamma) o Y2 + PL),
//   dk = -beta exp(gamma) o Y1 + exp(gamma_c - gamma) o Y3 + beta PA + scale QL + QA,
//   dgamma = q o dq + k o (-beta exp(gamma) o Y1 - exp(gamma_c - gamma) o Y3 + beta PA - scale QL - QA),
//   dbeta = sum_v dR o (V - Kp S) + sum_i dA o A',
// and the last row's gamma (gamma_c) adds exp(gamma_c) <dS', S> (per channel) and
// sum_r k exp(gamma_c - gamma) o Y3 to every row of dg = reverse in-chunk cumsum of dgamma.
// Exponentials of differences of gammas only, so nothing overflows for gates <= 0.
template <int K, int C>
struct GradKdaLayout {
    static constexpr int LK = K + 1, LV = kVS + 1, kLC = C + 1;
    static constexpr int oQ = 0, oK = oQ + C * LK, oG = oK + C * LK;
    static constexpr int oT = oG + C * LK, oL = oT + C * kLC, oDL = oL + C * kLC, oDT = oDL + C * kLC;
    // T, L, dL, dT are later reused for dgamma and the gamma_c terms (2 C x LK floats)
    static constexpr int kTiles = 4 * C * kLC > 2 * C * LK ? 4 * C * kLC : 2 * C * LK;
    static constexpr int oB = oT + kTiles, oGC = oB + C, oSS = oGC + K, oRB = oSS + K, oRC = oRB + C;
    static constexpr int oFree = oRC + C;
    static constexpr int oS = oFree, oDS = oS + K * LV;
    static constexpr int oV = oDS + K * LV, oDO = oV + C * LV, oKS = oDO + C * LV, oR = oKS + C * LV;
    static constexpr int oE = oR + C * LV, oDE = oE + C * LV, oDR = oDE + C * LV, oX2 = oDR + C * LV;
    static constexpr int oFreeEnd = oX2 + C * LV;
    static_assert(oFreeEnd - oFree >= 2 * C * kLC, "slice region reused for X and A'");
    static_assert(oB - oT >= 2 * C * LK, "T, L, dL, dT reused for dgamma and the gamma_c terms");
    static constexpr size_t bytes = sizeof(float) * oFreeEnd;
    static_assert(bytes <= 232448, "one CTA per SM");
};

template <typename Tin, int K, int C>
__global__ void __launch_bounds__(kGradThreads)
chunk_grad_kda_kernel(BwdParams p) {
    using Lay = GradKdaLayout<K, C>;
    constexpr int kLC = C + 1;
    extern __shared__ float sm[];
    constexpr int LK = Lay::LK, LV = Lay::LV;
    constexpr int TPR = kGradThreads / C;   // threads per chunk row
    constexpr int CPT = K / TPR;            // (row, channel) pairs owned per thread
    static_assert(TPR * C == kGradThreads && CPT * TPR == K, "one thread group per chunk row");
    float *sQ = sm + Lay::oQ, *sK = sm + Lay::oK, *sG = sm + Lay::oG;
    float *sT = sm + Lay::oT, *sL = sm + Lay::oL, *sDL = sm + Lay::oDL, *sDT = sm + Lay::oDT;
    float *sB = sm + Lay::oB, *sGC = sm + Lay::oGC, *sSS = sm + Lay::oSS;
    float *sRB = sm + Lay::oRB, *sRC = sm + Lay::oRC;
    float *sS = sm + Lay::oS, *sDS = sm + Lay::oDS, *sV = sm + Lay::oV, *sDO = sm + Lay::oDO;
    float *sKS = sm + Lay::oKS, *sR = sm + Lay::oR, *sE = sm + Lay::oE, *sDE = sm + Lay::oDE;
    float *sDR = sm + Lay::oDR, *sX2 = sm + Lay::oX2;
    float *sA = sm + Lay::oFree;              // A during the Map; later X = dT T^T
    float *sAp = sm + Lay::oFree + C * kLC;   // A' at the end
    float *sKp = sQ, *sKb = sG;               // in place of Q and gamma during the slice loop
    float *sDGm = sT, *sW3 = sT + C * LK;     // dgamma and the gamma_c terms at the end

    if (status_blocks_cta(p.dev_status)) return;
    const int n = p.chunk_indices[2 * blockIdx.x];
    if (n < 0) return;                         // sentinel row: nothing to do
    if (n >= p.n_max) {
        if (threadIdx.x == 0) status_set(p.dev_status, GCL_DEV_BAD_RANGE);
        return;
    }
    const int ic = p.chunk_indices[2 * blockIdx.x + 1];
    const int tid = threadIdx.x, h = blockIdx.y;
    const int H = p.H, V = p.V;
    const int64_t bos = p.cu_seqlens[n], eos = p.cu_seqlens[n + 1];
    const int64_t t0 = bos + (int64_t)ic * C;
    if (bos < 0 || eos < bos || eos > p.t_max || t0 >= eos) {
        if (tid == 0) status_set(p.dev_status, GCL_DEV_BAD_RANGE);
        return;
    }
    const int len = (int)(eos - t0 < C ? eos - t0 : C);
    const Tin *q = static_cast<const Tin *>(p.q);
    const Tin *k = static_cast<const Tin *>(p.k);
    const Tin *v = static_cast<const Tin *>(p.v);
    const Tin *beta = static_cast<const Tin *>(p.beta);
    const Tin *d_o = static_cast<const Tin *>(p.d_o);
    const int64_t KV = (int64_t)K * V;
    const int64_t row = (int64_t)p.chunk_offsets[n] + ic;
    if (row < 0 || row >= p.nt_max || ic < 0) {
        if (tid == 0) status_set(p.dev_status, GCL_DEV_BAD_RANGE);
        return;
    }
    const float *Sg = p.h + (row * H + h) * KV;
    const float *dSg = p.dh + (row * H + h) * KV;

    // ---- Map recompute
    simt_load_chunk<kKDA, Tin, K, kGradThreads, C>(q, k, p.g, beta, t0, len, h, H, sQ, sK, sG, sB, p.t_max, p.dev_status);
    __syncthreads();
    simt_gate_cumsum<kKDA, K, kGradThreads, C>(sG);
    __syncthreads();
    simt_intra<kKDA, K, kGradThreads, C, true>(sQ, sK, sG, sB, p.scale, sA, sL, nullptr);
    for (int e = tid; e < C * kLC; e += kGradThreads) { sDL[e] = 0.f; sDT[e] = 0.f; }
    for (int r = tid; r < C; r += kGradThreads) { sRB[r] = 0.f; sRC[r] = 0.f; }
    for (int c = tid; c < K; c += kGradThreads) { sSS[c] = 0.f; sGC[c] = sG[(C - 1) * LK + c]; }
    __syncthreads();
    simt_solve_blocked<kGradThreads, C>(sA, sT, sAp);   // A' is formed at the end
    // Kp and Kb in place of Q and gamma (both are reloaded after the slice loop)
    for (int e = tid; e < C * K; e += kGradThreads) {
        const int r = e / K, c = e % K;
        const float gm = sG[r * LK + c], kv = sK[r * LK + c];
        sKp[r * LK + c] = kv * expf(gm);
        sKb[r * LK + c] = kv * expf(sGC[c] - gm);
    }
    const int my_r = tid / TPR, my_c0 = tid % TPR;    // owner of (row, channel) partials
    float y1[CPT], y2[CPT], y3[CPT];
#pragma unroll
    for (int m = 0; m < CPT; ++m) { y1[m] = 0.f; y2[m] = 0.f; y3[m] = 0.f; }

    // the value slice's S, dS', V and dO columns are read into registers one slice ahead, so
    // their global-memory latency overlaps the previous slice's work
    constexpr int KI = K * kVS / kGradThreads, CI = C * kVS / kGradThreads;
    static_assert(KI * kGradThreads == K * kVS && CI * kGradThreads == C * kVS, "whole loads per thread");
    float pS[KI], pD[KI], pV[CI], pO[CI];
    auto fetch = [&](int s0) {
#pragma unroll
        for (int u = 0; u < KI; ++u) {
            const int e = tid + u * kGradThreads, c = e / kVS, j = e % kVS;
            pS[u] = Sg[(int64_t)c * V + s0 + j];
            pD[u] = dSg[(int64_t)c * V + s0 + j];
        }
#pragma unroll
        for (int u = 0; u < CI; ++u) {
            const int e = tid + u * kGradThreads, r = e / kVS, j = e % kVS;
            const int64_t gi = ((t0 + r) * H + h) * (int64_t)V + s0 + j;
            pV[u] = r < len ? ld_in(v, gi) : 0.f;
            pO[u] = r < len ? ld_in(d_o, gi) : 0.f;
        }
    };
    fetch(0);
    for (int s0 = 0; s0 < V; s0 += kVS) {
        __syncthreads();
#pragma unroll
        for (int u = 0; u < KI; ++u) {
            const int e = tid + u * kGradThreads, c = e / kVS, j = e % kVS;
            sS[c * LV + j] = pS[u];
            sDS[c * LV + j] = pD[u];
        }
#pragma unroll
        for (int u = 0; u < CI; ++u) {
            const int e = tid + u * kGradThreads, r = e / kVS, j = e % kVS;
            sV[r * LV + j] = pV[u];
            sDO[r * LV + j] = pO[u];
        }
        if (s0 + kVS < V) fetch(s0 + kVS);
        __syncthreads();
        for (int c = tid; c < K; c += kGradThreads) {   // <dS', S> per key channel
            float a = sSS[c];
            for (int j = 0; j < kVS; ++j) a = fmaf(sS[c * LV + j], sDS[c * LV + j], a);
            sSS[c] = a;
        }
        // KS = Kp S, R = diag(beta)(V - KS), X2 = Kb dS': rows r and r + C/2 per thread, so
        // each S and dS' value read serves two rows
        for (int e = tid; e < (C / 2) * kVS; e += kGradThreads) {
            const int r = e / kVS, j = e % kVS, r2 = r + C / 2;
            float ks0 = 0.f, kd0 = 0.f, ks1 = 0.f, kd1 = 0.f;
            for (int c = 0; c < K; ++c) {
                const float sv = sS[c * LV + j], dv = sDS[c * LV + j];
                ks0 = fmaf(sKp[r * LK + c], sv, ks0);
                kd0 = fmaf(sKb[r * LK + c], dv, kd0);
                ks1 = fmaf(sKp[r2 * LK + c], sv, ks1);
                kd1 = fmaf(sKb[r2 * LK + c], dv, kd1);
            }
            sKS[r * LV + j] = ks0;
            sR[r * LV + j] = sB[r] * (sV[r * LV + j] - ks0);
            sX2[r * LV + j] = kd0;
            sKS[r2 * LV + j] = ks1;
            sR[r2 * LV + j] = sB[r2] * (sV[r2 * LV + j] - ks1);
            sX2[r2 * LV + j] = kd1;
        }
        __syncthreads();
        // E = T R;  dE = L^T dO + X2
        for (int e = tid; e < C * kVS; e += kGradThreads) {
            const int r = e / kVS, j = e % kVS;
            float ev = 0.f, de = sX2[r * LV + j];
            for (int i = 0; i <= r; ++i) ev = fmaf(sT[r * kLC + i], sR[i * LV + j], ev);
            for (int r2 = r; r2 < C; ++r2) de = fmaf(sL[r2 * kLC + r], sDO[r2 * LV + j], de);
            sE[r * LV + j] = ev;
            sDE[r * LV + j] = de;
        }
        __syncthreads();
        // dR = T^T dE; dv = beta dR
        for (int e = tid; e < C * kVS; e += kGradThreads) {
            const int i = e / kVS, j = e % kVS;
            float acc = 0.f;
            for (int r = i; r < C; ++r) acc = fmaf(sT[r * kLC + i], sDE[r * LV + j], acc);
            sDR[i * LV + j] = acc;
            if (i < len) p.dv[((t0 + i) * H + h) * (int64_t)V + s0 + j] = sB[i] * acc;
        }
        // dL += dO E^T (i <= r);  dT += dE R^T (i <= r)
        for (int e = tid; e < C * C; e += kGradThreads) {
            const int r = e / C, i = e % C;
            if (i <= r) {
                float dl = 0.f, dt = 0.f;
                for (int j = 0; j < kVS; ++j) {
                    dl = fmaf(sDO[r * LV + j], sE[i * LV + j], dl);
                    dt = fmaf(sDE[r * LV + j], sR[i * LV + j], dt);
                }
                sDL[r * kLC + i] += dl;
                sDT[r * kLC + i] += dt;
            }
        }
        __syncthreads();
        // (row, channel) partials: Y1 += dR S^T, Y2 += dO S^T, Y3 += E dS'^T (the row's three
        // values read once per column j; each accumulator still adds j in order)
        for (int j = 0; j < kVS; ++j) {
            const float dr = sDR[my_r * LV + j], dov = sDO[my_r * LV + j], ev = sE[my_r * LV + j];
#pragma unroll
            for (int m = 0; m < CPT; ++m) {
                const int c = my_c0 + TPR * m;
                const float sv = sS[c * LV + j];
                y1[m] = fmaf(dr, sv, y1[m]);
                y2[m] = fmaf(dov, sv, y2[m]);
                y3[m] = fmaf(ev, sDS[c * LV + j], y3[m]);
            }
        }
        // row sums for dbeta (one thread per row, fixed order)
        for (int r = tid; r < C; r += kGradThreads) {
            float b = 0.f, cc = 0.f;
            for (int j = 0; j < kVS; ++j) {
                b = fmaf(sDR[r * LV + j], sV[r * LV + j], b);
                cc = fmaf(sDR[r * LV + j], sKS[r * LV + j], cc);
            }
            sRB[r] += b;
            sRC[r] += cc;
        }
    }
    __syncthreads();
    // q and gamma again (the slice loop held Kp and Kb in their buffers)
    simt_load_chunk<kKDA, Tin, K, kGradThreads, C>(q, k, p.g, beta, t0, len, h, H, sQ, sK, sG, sB, p.t_max, p.dev_status);
    __syncthreads();
    simt_gate_cumsum<kKDA, K, kGradThreads, C>(sG);
    // dA = -T^T (dT T^T), strictly lower.  X = dT T^T into sA (dT is lower incl. diag).
    for (int e = tid; e < C * C; e += kGradThreads) {
        const int r = e / C, m = e % C;
        float acc = 0.f;
        for (int i = 0; i <= min(r, m); ++i) acc = fmaf(sDT[r * kLC + i], sT[m * kLC + i], acc);
        sA[r * kLC + m] = acc;
    }
    __syncthreads();
    for (int e = tid; e < C * C; e += kGradThreads) {
        const int r = e / C, i = e % C;
        float acc = 0.f;
        if (i < r)
            for (int m = r; m < C; ++m) acc = fmaf(-sT[m * kLC + r], sA[m * kLC + i], acc);
        sDT[r * kLC + i] = acc;      // sDT now holds dA
    }
    __syncthreads();
    simt_intra<kKDA, K, kGradThreads, C, true>(sQ, sK, sG, sB, p.scale, nullptr, nullptr, sAp);
    __syncthreads();
    const float *sDA = sDT;
    for (int r = tid; r < C; r += kGradThreads) {   // dbeta, one thread per row
        float da_row = 0.f;
        for (int i = 0; i < r; ++i) da_row = fmaf(sDA[r * kLC + i], sAp[r * kLC + i], da_row);
        if (r < len) p.dbeta[(t0 + r) * H + h] = sRB[r] - sRC[r] + da_row;
    }
    // ---- dq, dk and dgamma of (my_r, channel): the row's dL and dA entries are read once
    // per pair and serve eight channels at a time (eight independent sums per loop)
    float dgv[CPT], wv[CPT];
    {
        const int r = my_r;
        const float br = sB[r];
        constexpr int HM = CPT >= 8 ? 8 : CPT;
#pragma unroll
        for (int m0 = 0; m0 < CPT; m0 += HM) {
            float gr[HM], pl[HM], pa[HM], ql[HM], qa[HM];
#pragma unroll
            for (int mm = 0; mm < HM; ++mm) {
                gr[mm] = sG[r * LK + my_c0 + TPR * (m0 + mm)];
                pl[mm] = pa[mm] = ql[mm] = qa[mm] = 0.f;
            }
            for (int i = 0; i <= r; ++i) {
                const float dl = sDL[r * kLC + i], da = sDA[r * kLC + i];
#pragma unroll
                for (int mm = 0; mm < HM; ++mm) {
                    const int c = my_c0 + TPR * (m0 + mm);
                    const float kd = sK[i * LK + c] * __expf(gr[mm] - sG[i * LK + c]);
                    pl[mm] = fmaf(dl, kd, pl[mm]);
                    pa[mm] = fmaf(da, kd, pa[mm]);
                }
            }
            for (int r2 = r; r2 < C; ++r2) {
                const float dl = sDL[r2 * kLC + r], dab = sDA[r2 * kLC + r] * sB[r2];
#pragma unroll
                for (int mm = 0; mm < HM; ++mm) {
                    const int c = my_c0 + TPR * (m0 + mm);
                    const float d = __expf(sG[r2 * LK + c] - gr[mm]);
                    ql[mm] = fmaf(dl, sQ[r2 * LK + c] * d, ql[mm]);
                    qa[mm] = fmaf(dab, sK[r2 * LK + c] * d, qa[mm]);
                }
            }
#pragma unroll
            for (int mm = 0; mm < HM; ++mm) {
                const int m = m0 + mm, c = my_c0 + TPR * m;
                const float eg = expf(gr[mm]), ec = expf(sGC[c] - gr[mm]);
                const float qv = sQ[r * LK + c], kv = sK[r * LK + c];
                const float dq = p.scale * (eg * y2[m] + pl[mm]);
                const float dk = -br * eg * y1[m] + ec * y3[m] + br * pa[mm] + p.scale * ql[mm] + qa[mm];
                dgv[m] = qv * dq + kv * (-br * eg * y1[m] - ec * y3[m] + br * pa[mm] - p.scale * ql[mm] - qa[mm]);
                wv[m] = kv * ec * y3[m];
                if (r < len) {
                    p.dq[((t0 + r) * H + h) * (int64_t)K + c] = dq;
                    p.dk[((t0 + r) * H + h) * (int64_t)K + c] = dk;
                }
            }
        }
    }
    __syncthreads();   // every read of T, L, dL, dA is done: reuse them for dgamma
#pragma unroll
    for (int m = 0; m < CPT; ++m) {
        const int c = my_c0 + TPR * m;
        sDGm[my_r * LK + c] = dgv[m];
        sW3[my_r * LK + c] = wv[m];
    }
    __syncthreads();
    // dg = reverse cumsum of dgamma per channel; the gamma_c terms reach every row
    for (int c = tid; c < K; c += kGradThreads) {
        float acc = expf(sGC[c]) * sSS[c];
        for (int r = 0; r < C; ++r) acc += sW3[r * LK + c];
        for (int r = C - 1; r >= 0; --r) {
            acc += sDGm[r * LK + c];
            if (r < len) p.dg[((t0 + r) * H + h) * (int64_t)K + c] = acc;
        }
    }
}

template <typename Kern>
cudaError_t prep(Kern kern, size_t bytes) {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

template <typename Tin, int K, int VS, int C>
cudaError_t launch_k(const BwdParams &p, bool sweep_done, cudaStream_t s) {
    cudaError_t e;
    if (!sweep_done) {
        auto sweep = dstate_sweep_kernel<kGDN, Tin, K, VS, C>;
        const size_t sb = SweepLayout<K, VS, kGDN, C>::bytes;
        if ((e = prep(sweep, sb)) != cudaSuccess) return e;
        sweep<<<dim3(p.V / VS, p.H, p.n_max), kSweepThreads, sb, s>>>(p);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    auto grad = chunk_grad_kernel<Tin, K, C>;
    const size_t gb = GradLayout<K, C>::bytes;
    if ((e = prep(grad, gb)) != cudaSuccess) return e;
    grad<<<dim3((unsigned)p.nt_max, p.H), kGradThreads, gb, s>>>(p);
    return cudaGetLastError();
}

template <typename Tin, int K, int VS, int C>
cudaError_t launch_kda(const BwdParams &p, bool sweep_done, cudaStream_t s) {
    cudaError_t e;
    if (!sweep_done) {
        auto sweep = dstate_sweep_kernel<kKDA, Tin, K, VS, C>;
        const size_t sb = SweepLayout<K, VS, kKDA, C>::bytes;
        if ((e = prep(sweep, sb)) != cudaSuccess) return e;
        sweep<<<dim3(p.V / VS, p.H, p.n_max), kSweepThreads, sb, s>>>(p);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    auto grad = chunk_grad_kda_kernel<Tin, K, C>;
    const size_t gb = GradKdaLayout<K, C>::bytes;
    if ((e = prep(grad, gb)) != cudaSuccess) return e;
    grad<<<dim3((unsigned)p.nt_max, p.H), kGradThreads, gb, s>>>(p);
    return cudaGetLastError();
}

template <typename Tin, int C>
cudaError_t launch_chunk(const BwdParams &p, bool kda, bool sweep_done, cudaStream_t s) {
    if (kda)
        return p.K == 64 ? launch_kda<Tin, 64, 64, C>(p, sweep_done, s) : launch_kda<Tin, 128, 32, C>(p, sweep_done, s);
    return p.K == 64 ? launch_k<Tin, 64, 64, C>(p, sweep_done, s) : launch_k<Tin, 128, 32, C>(p, sweep_done, s);
}

}  // namespace simt_bwd

// The CUDA-core backward for input type Tin (GDN or KDA), chunk size 32 or 64.
template <typename Tin>
cudaError_t launch_bwd_simt_t(const BwdParams &p, bool kda, bool sweep_done, cudaStream_t s) {
    return p.bt == 32 ? simt_bwd::launch_chunk<Tin, 32>(p, kda, sweep_done, s)
                      : simt_bwd::launch_chunk<Tin, 64>(p, kda, sweep_done, s);
}

}  // namespace gcl
