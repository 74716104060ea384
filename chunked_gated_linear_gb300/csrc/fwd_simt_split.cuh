// fwd_simt_split.cuh -- the CUDA-core forward as two launches (fp32 arithmetic): a chunk
// prep over every chunk of every sequence at once, then a chain over (sequence, head,
// value-column slice) that carries the state through the chunks in order.
//
// HA-NPU paper "Empowering Hybrid Attention Models on NPUs", section 2.1: of Map-Reduce-Map
// only the Reduce is serial; the chunk-local Map runs for all chunks in parallel.  The prep
// (one CTA per row of chunk_indices and head) forms, from the chunk alone (simt_map.cuh),
//   W = T diag(beta Gamma) K (GDN) or T diag(beta) (K o Gamma) (KDA),   U = T diag(beta) V,
//   Q' = scale diag(Gamma) Q (or scale Q o Gamma),   K' = diag(f) K (or K o exp(gamma_c - gamma)),
//   L,   Gamma_c (per key channel; GDN repeats its scalar),
// and writes them as one fp32 record per chunk and head.  The chain then needs only
//   E = U - W S,   O = Q' S + L E,   S <- Gamma_c o S + K'^T E
// per chunk (section 5's chunk-first order: O from the state before the update), with the
// next chunk's record copied into shared memory while the current one is used.  Rows past
// the end of a sequence have zero q, k, beta and g, so their record rows are zero and leave
// S unchanged.
#pragma once

#include "simt_map.cuh"
#include "tc_ptx.cuh"
#include "tc_solve.cuh"

namespace gcl {
namespace simt_split {

constexpr int kThreads = 256;

// One record per (chunk row, head), fp32, rows padded to the chain's shared-memory strides
// (K + 4 and C + 4 floats; the pads are never read):
//   W [C][K+4] | Q' [C][K+4] | K' [C][K+4] | L [C][C+4] | Gamma_c [K] | U [C][V]
// so that everything before U reaches a chain buffer as one bulk copy of `head` floats (U is
// read by value slices, row by row).
template <int K, int V, int C>
struct Rec {
    static constexpr int LW = K + 4, LL = C + 4;
    static constexpr int oW = 0, oQ = C * LW, oKt = 2 * C * LW, oL = 3 * C * LW;
    static constexpr int oGC = oL + C * LL, oU = oGC + K, head = oU;
    static constexpr int floats = oU + C * V;
    static_assert(floats % 4 == 0 && head % 4 == 0, "records keep 16-byte alignment");
};

// ------------------------------------------------------------------------------- prep
// Four consecutive inputs as fp32 (one 16-byte fp32 load, one 8-byte bf16 or fp16 load).
__device__ __forceinline__ float4 ld4_in(const float *p, int64_t i) {
    return *reinterpret_cast<const float4 *>(p + i);
}
__device__ __forceinline__ float4 ld4_in(const __nv_bfloat16 *p, int64_t i) {
    const uint2 u = *reinterpret_cast<const uint2 *>(p + i);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.y));
    return make_float4(a.x, a.y, b.x, b.y);
}
__device__ __forceinline__ float4 ld4_in(const __half *p, int64_t i) {
    const uint2 u = *reinterpret_cast<const uint2 *>(p + i);
    const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&u.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&u.y));
    return make_float4(a.x, a.y, b.x, b.y);
}

// The chunk's [C][W] tile of a [t, H, W] input, four elements per load, held in registers
// (every load of a batch is in flight before the first store); rows r >= len read as zero.
template <typename Tin, int W, int C>
struct Tile4 {
    static constexpr int N4 = C * W / 4, PER = (N4 + kThreads - 1) / kThreads;
    float4 b[PER];
    __device__ __forceinline__ void load(const Tin *x, int64_t t0, int len, int h, int H, int64_t t_max,
                                         int32_t *st) {
#pragma unroll
        for (int u = 0; u < PER; ++u) {
            const int e = threadIdx.x + u * kThreads, r = e / (W / 4), c4 = e % (W / 4);
            const int64_t gi = ((t0 + r) * H + h) * (int64_t)W + 4 * c4;
            b[u] = (e < N4 && r < len && GCL_RANGE_IN_BOUNDS(gi, gi + 3, t_max * H * (int64_t)W, st))
                       ? ld4_in(x, gi) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    __device__ __forceinline__ void store(float *dst, int ld) const {
#pragma unroll
        for (int u = 0; u < PER; ++u) {
            const int e = threadIdx.x + u * kThreads, r = e / (W / 4), c4 = e % (W / 4);
            if (e < N4) {
                float *d = dst + r * ld + 4 * c4;
                d[0] = b[u].x;
                d[1] = b[u].y;
                d[2] = b[u].z;
                d[3] = b[u].w;
            }
        }
    }
};

template <int K, int V, int VAR, int C>
struct PrepLayout {
    static constexpr int LK = K + 1, LV = V + 1, kLC = C + 1;
    static constexpr int LDA = C + 4;                        // A and T: 16-byte aligned rows
    static constexpr int oQ = 0, oK = oQ + C * LK, oV = oK + C * LK;
    static constexpr int oA = oV + C * LV, oT = oA + C * LDA, oL = oT + C * LDA;
    static constexpr int oB = oL + C * kLC, oE1 = oB + C, oE2 = oE1 + C, oG = oE2 + C;
    // GDN, 64-row chunks: Q^T and K^T [K][C + 4] for the intra-chunk products (float4 loads
    // along rows; at 32 rows the copies would cost a CTA per SM and the plain loads are few)
    static constexpr bool kTransposed = VAR == kGDN && C == 64;
    static constexpr int LT = C + 4, oQT = oG + (VAR == kKDA ? C * LK : C);
    static constexpr int oKT = oQT + (kTransposed ? K * LT : 0);
    static constexpr int total = oKT + (kTransposed ? K * LT : 0);
    static constexpr size_t bytes = sizeof(float) * total;
    static_assert(oA % 4 == 0 && oT % 4 == 0 && oQT % 4 == 0 && oKT % 4 == 0, "float4 rows");
    static_assert(bytes <= 232448, "one CTA per SM at most");
};

// T = (I + A)^-1 for a 32 x 32 strictly lower A (row stride LD, 16-byte aligned rows): one
// warp, lane j forms column j of T by forward substitution down the rows (four partial sums
// per row).  T is written in full (zeros above the diagonal).
template <int LD>
__device__ __forceinline__ void solve_lower32_warp(const float *sA, float *sT) {
    const int j = threadIdx.x & 31;
    float x[32];
#pragma unroll
    for (int r = 0; r < 32; ++r) {
        float part[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int m4 = 0; m4 < r; m4 += 4) {
            const float4 a = *reinterpret_cast<const float4 *>(sA + r * LD + m4);
            part[0] = fmaf(a.x, x[m4], part[0]);
            if (m4 + 1 < r) part[1] = fmaf(a.y, x[m4 + 1], part[1]);
            if (m4 + 2 < r) part[2] = fmaf(a.z, x[m4 + 2], part[2]);
            if (m4 + 3 < r) part[3] = fmaf(a.w, x[m4 + 3], part[3]);
        }
        x[r] = (r == j ? 1.f : 0.f) - ((part[0] + part[1]) + (part[2] + part[3]));
    }
#pragma unroll
    for (int r = 0; r < 32; ++r) sT[r * LD + j] = x[r];
}

// GDN's A (strictly lower, times beta_r; row stride LDA) and L (inclusive, times scale; row
// stride C + 1) from transposed copies Q^T, K^T [K][LT]: one 4 x 4 tile of (r, i) pairs per
// thread, whose four rows and four columns come as one float4 each per key channel (the
// same sums as simt_intra in the same order; tiles above the diagonal are skipped).
template <int K, int C, int LDA, int LT>
__device__ __forceinline__ void simt_intra_t(const float *sQT, const float *sKT, const float *sG,
                                             const float *sB, float scale, float *sA, float *sL) {
    constexpr int NTILE = C / 4, kLC = C + 1;
    const int t = threadIdx.x;
    if (t >= NTILE * NTILE) return;
    const int r0 = (t / NTILE) * 4, i0 = (t % NTILE) * 4;
    float kk[4][4] = {}, qk[4][4] = {};
    if (i0 <= r0 + 3) {
#pragma unroll 4
        for (int c = 0; c < K; ++c) {
            const float4 kr4 = *reinterpret_cast<const float4 *>(sKT + c * LT + r0);
            const float4 qr4 = *reinterpret_cast<const float4 *>(sQT + c * LT + r0);
            const float4 ki4 = *reinterpret_cast<const float4 *>(sKT + c * LT + i0);
            const float kr[4] = {kr4.x, kr4.y, kr4.z, kr4.w}, qr[4] = {qr4.x, qr4.y, qr4.z, qr4.w};
            const float ki[4] = {ki4.x, ki4.y, ki4.z, ki4.w};
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
            sA[r * LDA + i] = sB[r] * ((i < r) ? kk[a][b] * d : 0.f);
            sL[r * kLC + i] = on ? scale * (qk[a][b] * d) : 0.f;
        }
}

// Warps 0..3 solve for T while warps 4..7 write the records that do not need it (Q', K', L,
// Gamma_c) and form the operands of W and U in place (HA-NPU section 5: the inversion runs
// beside the other vector work); then all eight form W and U.
template <int VAR, typename Tin, int K, int V, int C>
__global__ void __launch_bounds__(kThreads)
prep_kernel(FwdParams p) {
    using Lay = PrepLayout<K, V, VAR, C>;
    using R = Rec<K, V, C>;
    constexpr int LK = Lay::LK, LV = Lay::LV, kLC = Lay::kLC, LDA = Lay::LDA;
    static_assert(C == 64 ? LDA == kSolveLD : C == 32, "the 64-row solve's stride");
    extern __shared__ float sm[];
    float *sQ = sm + Lay::oQ, *sK = sm + Lay::oK, *sV = sm + Lay::oV;
    float *sA = sm + Lay::oA, *sT = sm + Lay::oT, *sL = sm + Lay::oL;
    float *sB = sm + Lay::oB, *sG = sm + Lay::oG, *sE1 = sm + Lay::oE1, *sE2 = sm + Lay::oE2;
    float *sQT = sm + Lay::oQT, *sKT = sm + Lay::oKT;
    constexpr int LW = R::LW, LL = R::LL, LT = Lay::LT;

    // launched as a dependent of the metadata kernel: nothing it wrote is read before this
    grid_dependency_wait();
    launch_dependents();                 // the chain reads the records after this grid completes
    if (status_blocks_cta(p.dev_status)) return;
    const int tid = threadIdx.x, j = blockIdx.x, h = blockIdx.y, H = p.H;
    const int n = p.chunk_indices[2 * j];
    if (n < 0) return;                   // sentinel row: nothing to do
    const int ic = p.chunk_indices[2 * j + 1];
    if (n >= p.n_max || ic < 0) {
        if (tid == 0) status_set(p.dev_status, GCL_DEV_BAD_RANGE);
        return;
    }
    const int64_t bos = p.cu_seqlens[n], eos = p.cu_seqlens[n + 1];
    const int64_t t0 = bos + (int64_t)ic * C;
    const int64_t row = (int64_t)p.chunk_offsets[n] + ic;
    if (bos < 0 || eos < bos || eos > p.t_max || t0 >= eos || row < 0 || row >= p.nt_max) {
        if (tid == 0) status_set(p.dev_status, GCL_DEV_BAD_RANGE);
        return;
    }
    const int len = (int)(eos - t0 < C ? eos - t0 : C);
    const Tin *q = static_cast<const Tin *>(p.q);
    const Tin *k = static_cast<const Tin *>(p.k);
    const Tin *v = static_cast<const Tin *>(p.v);
    const Tin *beta = static_cast<const Tin *>(p.beta);
    float *rec = static_cast<float *>(p.workspace) + (row * H + h) * (int64_t)R::floats;
    const int64_t n_rec = p.nt_max * H * (int64_t)R::floats;
    const int64_t rec0 = (row * H + h) * (int64_t)R::floats;

    {   // q, k (and KDA's gates) in one batch of loads, v in a second
        Tile4<Tin, K, C> tq, tk;
        tq.load(q, t0, len, h, H, p.t_max, p.dev_status);
        tk.load(k, t0, len, h, H, p.t_max, p.dev_status);
        float gv = 0.f, bv = 0.f;
        if (tid < C) {
            const bool ok = tid < len && GCL_IN_BOUNDS((t0 + tid) * H + h, p.t_max * H, p.dev_status);
            bv = ok ? ld_in(beta, (t0 + tid) * H + h) : 0.f;
            if (VAR == kGDN) gv = ok ? p.g[(t0 + tid) * H + h] : 0.f;
        }
        if constexpr (VAR == kKDA) {
            Tile4<float, K, C> tg;
            tg.load(p.g, t0, len, h, H, p.t_max, p.dev_status);
            tg.store(sG, LK);
        }
        tq.store(sQ, LK);
        tk.store(sK, LK);
        if (tid < C) {
            sB[tid] = bv;
            if (VAR == kGDN) sG[tid] = gv;
        }
    }
    {
        Tile4<Tin, V, C> tv;
        tv.load(v, t0, len, h, H, p.t_max, p.dev_status);
        tv.store(sV, LV);
    }
    __syncthreads();
    if constexpr (Lay::kTransposed) {   // Q^T, K^T (reads down a column, writes along a row)
        for (int e = tid; e < C * K; e += kThreads) {
            const int r = e % C, c = e / C;
            sQT[c * LT + r] = sQ[r * LK + c];
            sKT[c * LT + r] = sK[r * LK + c];
        }
    }
    if constexpr (VAR == kGDN) {   // inclusive cumsum of g over the rows: warp scans + carry
        __shared__ float s_carry;
        float x = tid < C ? sG[tid] : 0.f;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, x, d);
            if ((tid & 31) >= d) x += y;
        }
        if (tid == 31) s_carry = x;
        __syncthreads();
        if (tid >= 32 && tid < C) x += s_carry;
        if (tid < C) sG[tid] = x;
    } else {
        simt_gate_cumsum<VAR, K, kThreads, C>(sG);
    }
    __syncthreads();
    if (VAR == kGDN && tid < C) {      // the row factors Gamma_r and exp(gamma_c - gamma_r)
        sE1[tid] = expf(sG[tid]);
        sE2[tid] = expf(sG[C - 1] - sG[tid]);
    }
    if constexpr (Lay::kTransposed)
        simt_intra_t<K, C, LDA, LT>(sQT, sKT, sG, sB, p.scale, sA, sL);
    else
        simt_intra<VAR, K, kThreads, C, false, LDA>(sQ, sK, sG, sB, p.scale, sA, sL, nullptr);
    __syncthreads();
    if (tid < 128) {
        // ---- T = (I + A)^-1 on warps 0..3 (named barrier 1 inside the 64-row solve)
        if constexpr (C == 64) {
            solve_unit_lower64_r32<128, 1>(sA, sT);
        } else {
            if (tid < 32) solve_lower32_warp<LDA>(sA, sT);
        }
    } else {
        // ---- warps 4..7: Q' = scale Gamma o Q and K' = exp(gamma_c - gamma) o K into the
        // record, then Q's buffer becomes diag(beta) (K o Gamma) (each element read, then
        // overwritten, by one thread); V's rows take beta; L and Gamma_c into the record
        const int t = tid - 128;
        for (int e = t; e < C * K; e += kThreads - 128) {
            const int r = e / K, c = e % K;
            float e1, e2;
            if constexpr (VAR == kGDN) {
                e1 = sE1[r];
                e2 = sE2[r];
            } else {
                const float gr = gam<VAR, K>(sG, r, c);
                e1 = expf(gr);
                e2 = expf(gam<VAR, K>(sG, C - 1, c) - gr);
            }
            const float kv = sK[r * LK + c];
            const int o = r * LW + c;
            if (GCL_RANGE_IN_BOUNDS(rec0 + R::oQ + o, rec0 + R::oKt + o, n_rec, p.dev_status)) {
                rec[R::oQ + o] = p.scale * e1 * sQ[r * LK + c];
                rec[R::oKt + o] = e2 * kv;
            }
            sQ[r * LK + c] = sB[r] * e1 * kv;
        }
        for (int e = t; e < C * V; e += kThreads - 128) sV[(e / V) * LV + e % V] *= sB[e / V];
        for (int e = t; e < C * C; e += kThreads - 128) {
            const int o = (e / C) * LL + e % C;
            if (GCL_IN_BOUNDS(rec0 + R::oL + o, n_rec, p.dev_status)) rec[R::oL + o] = sL[(e / C) * kLC + e % C];
        }
        for (int c = t; c < K; c += kThreads - 128)
            if (GCL_IN_BOUNDS(rec0 + R::oGC + c, n_rec, p.dev_status)) rec[R::oGC + c] = expf(gam<VAR, K>(sG, C - 1, c));
    }
    __syncthreads();
    // ---- W = T (beta Gamma K) and U = T (beta V): 4 x 4 register tiles, i up to the tile's
    // last row (T is zero above the diagonal inside its 32-row diagonal blocks, and i stays in
    // the tile's own block)
    auto tile_product = [&](const float *X, int ldx, int W, int ldo, int oRec) {
        for (int s = tid; s < (C / 4) * (W / 4); s += kThreads) {
            const int r0 = (s / (W / 4)) * 4, c0 = (s % (W / 4)) * 4;
            float acc[4][4] = {};
            for (int i = 0; i <= r0 + 3; ++i) {
                float t[4], x[4];
#pragma unroll
                for (int a = 0; a < 4; ++a) {
                    t[a] = sT[(r0 + a) * LDA + i];
                    x[a] = X[i * ldx + c0 + a];
                }
#pragma unroll
                for (int a = 0; a < 4; ++a)
#pragma unroll
                    for (int b = 0; b < 4; ++b) acc[a][b] = fmaf(t[a], x[b], acc[a][b]);
            }
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                const int64_t o = rec0 + oRec + (int64_t)(r0 + a) * ldo + c0;
                if (GCL_RANGE_IN_BOUNDS(o, o + 3, n_rec, p.dev_status))
                    *reinterpret_cast<float4 *>(rec + oRec + (r0 + a) * ldo + c0) =
                        make_float4(acc[a][0], acc[a][1], acc[a][2], acc[a][3]);
            }
        }
    };
    tile_product(sQ, LK, K, LW, R::oW);
    tile_product(sV, LV, V, V, R::oU);
}

// ------------------------------------------------------------------------------ chain
__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
                 "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// N consecutive floats of shared memory (N = 1, 2 or 4, the address aligned to N floats).
template <int N>
__device__ __forceinline__ void lds_vec(const float *p, float (&v)[N]) {
    if constexpr (N == 4) {
        const float4 t = *reinterpret_cast<const float4 *>(p);
        v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
    } else if constexpr (N == 2) {
        const float2 t = *reinterpret_cast<const float2 *>(p);
        v[0] = t.x; v[1] = t.y;
    } else {
        static_assert(N == 1, "1, 2 or 4 floats");
        v[0] = p[0];
    }
}

// Shared memory of the chain: NB record buffers (two when they fit: the next chunk's record
// arrives while the current one is used), the state slice S [K][VS] and E [C][VS].  A buffer
// holds the record's head (W, Q', K', L, Gamma_c in the record's own padded layout: row
// strides K + 4 and C + 4, consecutive rows 4 banks apart), which one bulk copy brings in,
// then this slice's columns of U [C][VS + 4], copied row by row in 16-byte pieces.
template <int K, int V, int VS, int C>
struct ChainLayout {
    using R = Rec<K, V, C>;
    static constexpr int LW = R::LW, LL = R::LL, LU = VS + 4;
    static constexpr int oW = R::oW, oQ = R::oQ, oKt = R::oKt, oL = R::oL, oGC = R::oGC;
    static constexpr int oU = R::head, buf = oU + C * LU;
    static constexpr int kMaxFloats = 232448 / 4 - 64;           // (the static shared memory)
    static constexpr int fixed = K * LU + C * LU;
    static constexpr int NB = 2 * buf + fixed <= kMaxFloats ? 2 : 1;
    static constexpr int oS = NB * buf, oE = oS + K * LU, total = oE + C * LU;
    static constexpr size_t bytes = sizeof(float) * total;
    static constexpr uint32_t head_bytes = sizeof(float) * R::head;
    static_assert(bytes <= 232448 - 256, "chain shared memory");
    static_assert(LU % 4 == 0 && buf % 4 == 0 && VS % 4 == 0 && head_bytes < (1u << 20),
                  "16-byte aligned rows and copies; one bulk copy's byte count");
};

template <typename Tin, int K, int V, int VS, int C>
__global__ void __launch_bounds__(kThreads)
chain_kernel(FwdParams p) {
    using Lay = ChainLayout<K, V, VS, C>;
    using R = Rec<K, V, C>;
    constexpr int LW = Lay::LW, LL = Lay::LL, LU = Lay::LU;
    // phase 1 / O tiles: 2 rows x TJ columns; state tiles: TC keys x TS columns
    constexpr int RP = C / 2, CG = kThreads / RP, TJ = VS / CG;
    constexpr int TC = K / 32, TS = VS / 8;
    static_assert(RP * CG == kThreads && TJ * CG == VS && TJ >= 1, "output tiles");
    static_assert(TC * 32 == K && TS * 8 == VS, "state tiles");
    extern __shared__ __align__(16) float sm[];
    float *sS = sm + Lay::oS, *sE = sm + Lay::oE;

    // launched as a dependent of the prep: its records are complete after this wait
    grid_dependency_wait();
    if (status_blocks_cta(p.dev_status)) return;
    const int tid = threadIdx.x, h = blockIdx.y, H = p.H, v0 = blockIdx.x * VS;
    const int z = blockIdx.z;
    const int n = (p.seq_order && GCL_IN_BOUNDS(z, p.n_max, p.dev_status)) ? p.seq_order[z] : z;
    if (n < 0 || n >= p.n_max) {
        if (tid == 0) status_set(p.dev_status, GCL_DEV_BAD_RANGE);
        return;
    }
    const int64_t bos = p.cu_seqlens[n], eos = p.cu_seqlens[n + 1];
    if (bos < 0 || eos < bos || eos > p.t_max) {
        if (tid == 0) status_set(p.dev_status, GCL_DEV_BAD_RANGE);
        return;
    }
    const int nch = (int)((eos - bos + C - 1) / C);
    const int64_t row0 = p.chunk_offsets[n];
    if (nch > 0 && (row0 < 0 || row0 + nch > p.nt_max)) {
        if (tid == 0) status_set(p.dev_status, GCL_DEV_BAD_RANGE);
        return;
    }
    const int64_t KV = (int64_t)K * V;
    const int64_t state_base = ((int64_t)n * H + h) * KV;
    const int64_t n_state = (int64_t)p.n_max * H * KV;
    const float *recs = static_cast<const float *>(p.workspace);
    const int64_t n_rec = p.nt_max * H * (int64_t)R::floats;
    Tin *o = static_cast<Tin *>(p.o);

    for (int e = tid; e < K * VS; e += kThreads) {
        const int c = e / VS, jj = e % VS;
        const int64_t gi = state_base + (int64_t)c * V + v0 + jj;
        sS[c * LU + jj] = (p.h0 && GCL_IN_BOUNDS(gi, n_state, p.dev_status)) ? p.h0[gi] : 0.f;
    }
    __shared__ uint64_t bar_rec[2];
    __shared__ int s_err, s_err2;        // (s_err2: the error word of the final drain's waits)
    if (tid == 0) {
        tc::mbar_init(&bar_rec[0], 1);
        tc::mbar_init(&bar_rec[1], 1);
        s_err = 0;
        tc::fence_barrier_init();
    }
    __syncthreads();
    // the record of chunk ic into buffer b: its head in one bulk copy (thread 0, counted on
    // the buffer's mbarrier), this slice's U columns in 16-byte cp.async pieces
    auto issue = [&](int ic, int b) {
        const int64_t r0 = ((row0 + ic) * H + h) * (int64_t)R::floats;
        if (!GCL_RANGE_IN_BOUNDS(r0, r0 + R::floats - 1, n_rec, p.dev_status)) return;
        const float *src = recs + r0;
        float *dst = sm + b * Lay::buf;
        if (tid == 0) {
            tc::fence_async_smem();      // the buffer's last readers are done (block barrier)
            tc::mbar_arrive_expect_tx(&bar_rec[b], Lay::head_bytes);
            tc::bulk_load(dst, src, Lay::head_bytes, &bar_rec[b]);
        }
        for (int e = tid; e < C * VS / 4; e += kThreads) {
            const int r = e / (VS / 4), c4 = e % (VS / 4);
            cp_async16(dst + Lay::oU + r * LU + 4 * c4, src + R::oU + r * V + v0 + 4 * c4);
        }
        cp_async_commit();
    };
    if (nch > 0) issue(0, 0);
    int issued = nch > 0 ? 1 : 0;        // heads issued so far (one per chunk, in order)

    const int rp = tid / CG, r0 = 2 * rp, j0 = (tid % CG) * TJ;      // output tile
    const int c0 = (tid / 8) * TC, s0 = (tid % 8) * TS;              // state tile
    for (int ic = 0; ic < nch; ++ic) {
        const int b = Lay::NB == 2 ? (ic & 1) : 0;
        const float *sW = sm + b * Lay::buf, *sQp = sW + Lay::oQ, *sKt = sW + Lay::oKt;
        const float *sL = sW + Lay::oL, *sU = sW + Lay::oU, *sGC = sW + Lay::oGC;
        const int64_t t0 = bos + (int64_t)ic * C;
        const int len = (int)(eos - t0 < C ? eos - t0 : C);
        // chunk ic's record: the k = ic / NB-th use of buffer b, parity k & 1 (a wait that
        // gives up records GCL_DEV_WAIT_TIMEOUT; later waits return at once and the loop runs out)
        cp_async_wait_all();
        tc::mbar_wait(&bar_rec[b], (uint32_t)(ic / Lay::NB) & 1u, &s_err, 1);
        __syncthreads();              // chunk ic's record and the state are in place
        if (Lay::NB == 2 && ic + 1 < nch) {
            issue(ic + 1, b ^ 1);
            ++issued;
        }
        if (p.h_save) {               // the state entering the chunk
            const int64_t hb = ((row0 + ic) * H + h) * KV;
            for (int e = tid; e < K * VS; e += kThreads) {
                const int c = e / VS, jj = e % VS;
                if (GCL_IN_BOUNDS(hb + (int64_t)c * V + v0 + jj, p.nt_max * H * KV, p.dev_status))
                    p.h_save[hb + (int64_t)c * V + v0 + jj] = sS[c * LU + jj];
            }
        }
        // ---- phase 1: E = U - W S and Y = Q' S on rows r0, r0 + 1, columns j0 ..
        float ae[2][TJ], ay[2][TJ];
#pragma unroll
        for (int x = 0; x < 2; ++x)
#pragma unroll
            for (int y = 0; y < TJ; ++y) {
                ae[x][y] = sU[(r0 + x) * LU + j0 + y];
                ay[x][y] = 0.f;
            }
#pragma unroll 2
        for (int c = 0; c < K; c += 4) {
            const float4 w0 = *reinterpret_cast<const float4 *>(sW + r0 * LW + c);
            const float4 w1 = *reinterpret_cast<const float4 *>(sW + (r0 + 1) * LW + c);
            const float4 q0 = *reinterpret_cast<const float4 *>(sQp + r0 * LW + c);
            const float4 q1 = *reinterpret_cast<const float4 *>(sQp + (r0 + 1) * LW + c);
            const float wa[4] = {w0.x, w0.y, w0.z, w0.w}, wb[4] = {w1.x, w1.y, w1.z, w1.w};
            const float qa[4] = {q0.x, q0.y, q0.z, q0.w}, qb[4] = {q1.x, q1.y, q1.z, q1.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float sv[TJ];
                lds_vec<TJ>(sS + (c + e) * LU + j0, sv);
#pragma unroll
                for (int y = 0; y < TJ; ++y) {
                    ae[0][y] = fmaf(-wa[e], sv[y], ae[0][y]);
                    ae[1][y] = fmaf(-wb[e], sv[y], ae[1][y]);
                    ay[0][y] = fmaf(qa[e], sv[y], ay[0][y]);
                    ay[1][y] = fmaf(qb[e], sv[y], ay[1][y]);
                }
            }
        }
#pragma unroll
        for (int x = 0; x < 2; ++x)
#pragma unroll
            for (int y = 0; y < TJ; ++y) sE[(r0 + x) * LU + j0 + y] = ae[x][y];
        __syncthreads();
        // ---- phase 2: O = Y + L E (L lower triangular: rows r0, r0 + 1 need i <= r0 + 1)
        if (o != nullptr) {
            for (int i = 0; i <= r0 + 1; i += 4) {
                const float4 l0 = *reinterpret_cast<const float4 *>(sL + r0 * LL + i);
                const float4 l1 = *reinterpret_cast<const float4 *>(sL + (r0 + 1) * LL + i);
                const float la[4] = {l0.x, l0.y, l0.z, l0.w}, lb[4] = {l1.x, l1.y, l1.z, l1.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float ev[TJ];
                    lds_vec<TJ>(sE + (i + e) * LU + j0, ev);
#pragma unroll
                    for (int y = 0; y < TJ; ++y) {
                        ay[0][y] = fmaf(la[e], ev[y], ay[0][y]);
                        ay[1][y] = fmaf(lb[e], ev[y], ay[1][y]);
                    }
                }
            }
#pragma unroll
            for (int x = 0; x < 2; ++x) {
                if (r0 + x >= len) continue;
                const int64_t oi = ((t0 + r0 + x) * H + h) * (int64_t)V + v0 + j0;
                if (!GCL_RANGE_IN_BOUNDS(oi, oi + TJ - 1, p.t_max * H * (int64_t)V, p.dev_status)) continue;
#pragma unroll
                for (int y = 0; y < TJ; ++y) st_out(o, oi + y, ay[x][y]);
            }
        }
        // ---- S <- Gamma_c o S + K'^T E on keys c0 .., columns s0 .. (in place: each thread
        // reads and writes only its own entries)
        {
            float as[TC][TS];
#pragma unroll
            for (int x = 0; x < TC; ++x)
#pragma unroll
                for (int y = 0; y < TS; ++y) as[x][y] = sGC[c0 + x] * sS[(c0 + x) * LU + s0 + y];
#pragma unroll 4
            for (int r = 0; r < C; ++r) {
                float kt[TC], ev[TS];
                lds_vec<TC>(sKt + r * LW + c0, kt);
                lds_vec<TS>(sE + r * LU + s0, ev);
#pragma unroll
                for (int x = 0; x < TC; ++x)
#pragma unroll
                    for (int y = 0; y < TS; ++y) as[x][y] = fmaf(kt[x], ev[y], as[x][y]);
            }
#pragma unroll
            for (int x = 0; x < TC; ++x)
#pragma unroll
                for (int y = 0; y < TS; ++y) sS[(c0 + x) * LU + s0 + y] = as[x][y];
        }
        if (Lay::NB == 1 && ic + 1 < nch) {
            __syncthreads();          // every read of the single record buffer is done
            issue(ic + 1, 0);
            ++issued;
        }
    }
    // every issued head has landed before the CTA exits (after a wait that gave up, the last
    // ones get one more bounded wait each, whose failure is already recorded)
    __syncthreads();
    if (s_err != 0 && tid == 0) {
        for (int k = (issued > Lay::NB ? issued - Lay::NB : 0); k < issued; ++k) {
            s_err2 = 0;
            tc::mbar_wait(&bar_rec[k % Lay::NB], (uint32_t)(k / Lay::NB) & 1u, &s_err2, 1);
        }
        status_set(p.dev_status, GCL_DEV_WAIT_TIMEOUT);
    }
    __syncthreads();
    if (p.ht) {
        for (int e = tid; e < K * VS; e += kThreads) {
            const int c = e / VS, jj = e % VS;
            const int64_t gi = state_base + (int64_t)c * V + v0 + jj;
            if (GCL_IN_BOUNDS(gi, n_state, p.dev_status)) p.ht[gi] = sS[c * LU + jj];
        }
    }
}

// Value-column slice of the chain: 16 at K = 64, 32 at K = 128; half of that (where the tiles
// allow: VS >= 512 / C for the output tiles) when the grid of (slot, head, slice) CTAs would
// fill less than the GPU's SMs -- the serial chain then takes half the work per chunk on
// twice the CTAs (HA-NPU section 4: column-wise split of the residual heads).
template <int K, int C>
struct ChainSlice {
    static constexpr int VS = K == 64 ? 16 : 32;
    static constexpr int VS_small = VS / 2 >= 512 / C ? VS / 2 : VS;
};

template <int K, int V, int C>
size_t record_bytes(int64_t nt_max, int H) {
    return sizeof(float) * (size_t)nt_max * H * Rec<K, V, C>::floats;
}

template <typename Tin, int K, int V, int VS, int C>
cudaError_t launch_chain(const FwdParams &p, cudaStream_t s) {
    using CL = ChainLayout<K, V, VS, C>;
    auto chain = chain_kernel<Tin, K, V, VS, C>;
    const cudaError_t e = cudaFuncSetAttribute(chain, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)CL::bytes);
    if (e != cudaSuccess) return e;
    return launch_dependent(chain, dim3(V / VS, p.H, p.n_max), dim3(kThreads), CL::bytes, s, p);
}

template <int VAR, typename Tin, int K, int V, int C>
cudaError_t launch(const FwdParams &p, cudaStream_t s) {
    using PL = PrepLayout<K, V, VAR, C>;
    using CS = ChainSlice<K, C>;
    auto prep = prep_kernel<VAR, Tin, K, V, C>;
    cudaError_t e = cudaFuncSetAttribute(prep, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)PL::bytes);
    if (e != cudaSuccess) return e;
    e = launch_dependent(prep, dim3((unsigned)p.nt_max, p.H), dim3(kThreads), PL::bytes, s, p);
    if (e != cudaSuccess) return e;
    if (CS::VS_small != CS::VS && (int64_t)p.n_max * p.H * (V / CS::VS) < num_sms())
        return launch_chain<Tin, K, V, CS::VS_small, C>(p, s);
    return launch_chain<Tin, K, V, CS::VS, C>(p, s);
}

}  // namespace simt_split

}  // namespace gcl
