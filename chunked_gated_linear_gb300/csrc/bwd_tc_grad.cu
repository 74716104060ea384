// bwd_tc_grad.cu -- chunk gradients of the GDN backward on the tensor cores (bf16 inputs,
// d_k = d_v = 128, chunk 64): dq, dk, dv, dbeta, dg from the state entering every chunk S
// and the gradient of the state after it dS' (the sweep's output).
//
// FLA RFC "[RFC] Add Graph Capture Support for FLA Prefill and Training Paths on Ascend
// NPUs", section "Step 3": recomputation, WY, gate and gradient kernels.  With
// R = diag(beta)(V - diag(Gamma) K S), E = T R, dE = L^T dO + Ktil dS':
//   dv  = diag(beta) T^T dE,               dT = dE R^T (lower),   dL = dO E^T (lower),
//   dq  = scale diag(Gamma) dO S^T + P K,   P = scale D o dL,
//   dk  = diag(e^{g_c - g}) E dS'^T - diag(beta Gamma) (T^T dE) S^T + P^T Q + M K + M^T K,
//   M   = beta_r D o dA,   dA = -T^T dT T^T (strictly lower),   D[r][i] = e^{g_r - g_i},
// and the gate and beta gradients from row sums.  Two launches per chunk and head:
//   grad1  (tensor cores) the recompute (K K^T, Q K^T, the triangular solve) and five MMA
//          rounds: [K; Q][S | dS'], [T; L] R and L^T dO, then T^T dE, [E; dO] S^T,
//          [E; dO] E^T, [dE; E] R^T, then (-diag(beta Gamma) T^T dE) S^T and E dS'^T.
//          It writes dv, the partial dq and dk, and T, D o K K^T, L, dL, dT and four row sums per
//          chunk to a scratch record;
//   grad2  dA on the CUDA cores (fp32), the gate and beta gradients, and one MMA round
//          [M; P] K, M^T K + P^T Q that completes dq and dk.
#include <cudaTypedefs.h>

#include "gcl_internal.cuh"
#include "tc_ptx.cuh"
#include "tc_solve.cuh"
#include "transition.cuh"

namespace gcl {
namespace {

using namespace tc;
using namespace tr;

// scratch record per chunk and head (fp32): T, A' = D o K K^T (strict), L, dL, dT as
// [64][kSolveLD] (the shared-memory layout of the second kernel, so one bulk copy moves
// them), then rows: RA = sum_v dO o QS, RB = sum_v dVb o V, RC = sum_c (dVb S^T) o K,
// RD = sum_v E o K dS', and <dS', S> after them.
constexpr int kScrMat = C * kSolveLD;
constexpr int kScrT = 0, kScrAp = kScrMat, kScrL = 2 * kScrMat, kScrDL = 3 * kScrMat, kScrDT = 4 * kScrMat;
constexpr int kScrRows = 5 * kScrMat;
constexpr int kScrRowFloats = 4 * C + 8;             // a multiple of 4 floats (16 bytes)
constexpr int kScrFloats = kScrRows + kScrRowFloats;
static_assert((kScrFloats * 4) % 16 == 0 && (kScrRows * 4) % 16 == 0, "bulk copies of 16-byte multiples");

struct GradParams {
    const int32_t *chunk_indices, *cu;
    const float *g;
    const __nv_bfloat16 *beta, *v;
    const float *h;                 // the state entering every chunk, fp32 [unit][K][V]
    const uint8_t *dh;              // dS' of every chunk, bf16 tiles of kDsTileBytes
    float *dq, *dk, *dv, *dg, *dbeta;
    float *scratch;
    int32_t *status;
    int64_t t_max, nt_max;
    int32_t n_max, H;
    float scale;
};

constexpr int kThreads = 256;

// metadata of row j of chunk_indices; false for sentinels and invalid rows (reported)
__device__ __forceinline__ bool chunk_of_row(const GradParams &p, int j, int64_t &t0, int &len) {
    const int n = p.chunk_indices[2 * j];
    if (n < 0) return false;
    const int ic = p.chunk_indices[2 * j + 1];
    if (n >= p.n_max || ic < 0) {
        if (threadIdx.x == 0) status_set(p.status, GCL_DEV_BAD_RANGE);
        return false;
    }
    const int64_t bos = p.cu[n], eos = p.cu[n + 1];
    t0 = bos + (int64_t)ic * C;
    if (bos < 0 || eos < bos || eos > p.t_max || t0 >= eos) {
        if (threadIdx.x == 0) status_set(p.status, GCL_DEV_BAD_RANGE);
        return false;
    }
    len = (int)(eos - t0 < C ? eos - t0 : C);
    return true;
}

// gamma (inclusive cumsum of g over the chunk) and beta, for rows 0..63; all threads call it
__device__ __forceinline__ void chunk_gates(const GradParams &p, int64_t t0, int len, int h, float *sG,
                                            float *sB, float *s_carry) {
    const int tid = threadIdx.x;
    const float gv = (tid < len) ? p.g[(t0 + tid) * p.H + h] : 0.f;
    float x = tid < C ? warp_scan(gv) : 0.f;
    if (tid == 31) *s_carry = x;
    __syncthreads();
    if (tid >= 32 && tid < C) x += *s_carry;
    if (tid < C) {
        sG[tid] = x;
        sB[tid] = tid < len ? __bfloat162float(p.beta[(t0 + tid) * p.H + h]) : 0.f;
    }
    __syncthreads();
}

// ============================================================================ grad1
// shared memory (offsets from the 1024-aligned base)
constexpr uint32_t gKQ = 0;          // [K; Q]: 2 column blocks x 128 rows          32 KiB
constexpr uint32_t gV = 32768;       // V, then R: 2 blocks x 64 rows                16 KiB
constexpr uint32_t gS = 49152;       // S bf16: 2 blocks x 128 rows (key x value)    32 KiB
constexpr uint32_t gDS = 81920;      // dS' bf16                                     32 KiB
constexpr uint32_t gT3 = 114688;     // [dE; E; dO]: 2 blocks x 192 rows             48 KiB
constexpr uint32_t gTL = 163840;     // [T; L]: 128 rows x 64 columns, then dVb      16 KiB
constexpr uint32_t gF = 180224;      // fp32 A (-> dL), T (-> dT), solve scratch
// At the start S arrives as fp32 (64 KiB) in staging: keys 0..31 in the [dE; E] rows of
// column block 0 of gT3, keys 32..127 from gTL on (gTL and gF are contiguous).
constexpr uint32_t gStage0 = gT3, gStage1 = gTL;
static_assert(gTL + 16384 == gF && gStage1 + 3 * 16384 <= gF + kSolveFloats * 4, "S staging");
constexpr uint32_t g1End = gF + kSolveFloats * 4;
constexpr int kGrad1Smem = g1End + 1024;
static_assert(kGrad1Smem <= 232448, "grad1 shared memory");

__global__ void __launch_bounds__(kThreads, 1)
tc_grad1_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                GradParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    float *sA = reinterpret_cast<float *>(smem + gF);
    float *sT = sA + C * kSolveLD;
    float *sX = sT + C * kSolveLD;
    float *sDL = sA, *sDT = sT;                 // after the solve
    __shared__ uint64_t bar_tma, bar_mma;
    __shared__ uint32_t s_tmem;
    __shared__ int s_err;
    __shared__ float sG[C], sB[C], sEG[C], sFR[C], sRow[4][C], sRed[kThreads / 32], s_carry;

    if (status_blocks_cta(p.status)) return;
    const int tid = threadIdx.x, warp = tid >> 5;
    const int quarter = warp & 3, half = warp >> 2;
    const int lrow = quarter * 32 + (tid & 31);
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const int j = blockIdx.x, h = blockIdx.y, H = p.H;
    int64_t t0;
    int len;
    if (!chunk_of_row(p, j, t0, len)) return;
    const int unit = j * H + h;
    const uint32_t sbase = smem_u32(smem);
    float *scr = p.scratch + (size_t)unit * kScrFloats;

    if (tid == 0) {
        mbar_init(&bar_tma, 1);
        mbar_init(&bar_mma, 1);
        s_err = 0;
        fence_barrier_init();
        mbar_arrive_expect_tx(&bar_tma, 65536 + (uint32_t)kDsTileBytes + 65536);
        for (int cb = 0; cb < 2; ++cb) {
            tma_load_3d(smem + gKQ + cb * 16384, &tm_k, cb * 64, h, (int)t0, &bar_tma);
            tma_load_3d(smem + gKQ + cb * 16384 + 8192, &tm_q, cb * 64, h, (int)t0, &bar_tma);
            tma_load_3d(smem + gV + cb * 8192, &tm_v, cb * 64, h, (int)t0, &bar_tma);
            tma_load_3d(smem + gT3 + cb * 24576 + 16384, &tm_do, cb * 64, h, (int)t0, &bar_tma);
        }
        bulk_load(smem + gDS, p.dh + (size_t)unit * kDsTileBytes, (uint32_t)kDsTileBytes, &bar_tma);
        const float *Sg = p.h + (int64_t)unit * KD * VD;
        bulk_load(smem + gStage0, Sg, 16384, &bar_tma);
        for (int q = 0; q < 3; ++q) bulk_load(smem + gStage1 + q * 16384, Sg + (q + 1) * 4096, 16384, &bar_tma);
    }
    __syncwarp();
    if (warp == 0) {
        tmem_alloc(&s_tmem, 512);
        tmem_relinquish();
    }
    for (int e = tid; e < 4 * C; e += kThreads) (&sRow[0][0])[e] = 0.f;
    chunk_gates(p, t0, len, h, sG, sB, &s_carry);
    const float gC = sG[C - 1];
    if (tid < C) {
        sEG[tid] = __expf(sG[tid]);
        sFR[tid] = tid < len ? __expf(gC - sG[tid]) : 0.f;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    uint32_t phase = 0;
    auto mma_done = [&](int code) -> bool {
        const bool ok = mbar_wait(&bar_mma, phase, &s_err, code);
        phase ^= 1;
        tc_fence_after();
        return !__syncthreads_or(!ok);
    };
    auto to_async = [&]() {
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    };
    // 16-byte chunk of a K-major tile with `rows` rows per block of 64 columns
    auto kchunk = [&](uint32_t base, int rows, int r, int c) {
        return reinterpret_cast<uint4 *>(smem + base + kmaj16(rows, r, c));
    };
    auto ld64 = [&](uint32_t col, float *x) {        // 64 columns of this thread's TMEM lane
#pragma unroll
        for (int q = 0; q < 4; ++q) tmem_ld16(tmem + lane_off + col + q * 16, x + q * 16);
        tmem_ld_wait();
    };
    auto unpack8 = [](uint4 w, float *x) {
        const __nv_bfloat162 *pp = reinterpret_cast<const __nv_bfloat162 *>(&w);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = __bfloat1622float2(pp[e]);
            x[2 * e] = f.x;
            x[2 * e + 1] = f.y;
        }
    };
    do {
        const bool landed = mbar_wait(&bar_tma, 0, &s_err, 1);
        if (__syncthreads_or(!landed)) break;
        {   // S (fp32 staging) -> bf16 operand tile; <dS', S> against the dS' tile
            float dgc = 0.f;
            for (int e = tid; e < KD * VD / 8; e += kThreads) {
                const int key = e >> 4, c0 = (e & 15) * 8;
                const float *src = reinterpret_cast<const float *>(
                                       smem + (key < 32 ? gStage0 + key * 512 : gStage1 + (key - 32) * 512)) + c0;
                const float4 a0 = *reinterpret_cast<const float4 *>(src);
                const float4 a1 = *reinterpret_cast<const float4 *>(src + 4);
                const float sv[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
                float dv8[8];
                unpack8(*kchunk(gDS, 128, key, c0), dv8);
#pragma unroll
                for (int q = 0; q < 8; ++q) dgc = fmaf(sv[q], dv8[q], dgc);
                *kchunk(gS, 128, key, c0) = pack8(sv);
            }
#pragma unroll
            for (int d = 16; d > 0; d >>= 1) dgc += __shfl_xor_sync(0xffffffffu, dgc, d);
            if ((tid & 31) == 0) sRed[warp] = dgc;
        }
        __syncthreads();                              // the staging (gT3, gTL, gF) is free
        // decay table D[r][c] = exp(g_r - g_c) for c <= r (1 above the diagonal) in the T buffer
        for (int e = tid; e < C * C / 4; e += kThreads) {
            const int r = e >> 4, c = (e & 15) * 4;
            const float gr = sG[r];
            *reinterpret_cast<float4 *>(sT + r * kSolveLD + c) =
                make_float4(__expf(c <= r ? gr - sG[c] : 0.f), __expf(c + 1 <= r ? gr - sG[c + 1] : 0.f),
                            __expf(c + 2 <= r ? gr - sG[c + 2] : 0.f), __expf(c + 3 <= r ? gr - sG[c + 3] : 0.f));
        }
        if (len < C) {   // rows past the end: zero K, Q, V and dO (NaN padding enters MMAs raw)
            const uint4 zero = make_uint4(0, 0, 0, 0);
            for (int t = tid; t < 8 * C * 8; t += kThreads) {
                const int r = (t >> 3) & 63, blk = t >> 9;     // K0 K1 Q0 Q1 V0 V1 dO0 dO1
                if (r >= len) {
                    uint32_t base;
                    if (blk < 4) base = gKQ + (blk & 1) * 16384 + (blk >> 1) * 8192;
                    else if (blk < 6) base = gV + (blk - 4) * 8192;
                    else base = gT3 + (blk - 6) * 24576 + 16384;
                    *reinterpret_cast<uint4 *>(smem + base + r * 128 + (t & 7) * 16) = zero;
                }
            }
        }
        to_async();
        // ---- MMA1: [K; Q] K^T
        if (tid == 0) {
            const uint64_t d = smem_desc(sbase + gKQ, 16, 1024, kSwizzle128B);
            constexpr uint32_t id = idesc_bf16(128, 64);
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                const uint64_t o = (s >> 2) * 1024 + (s & 3) * 2;
                mma_bf16(tmem, d + o, d + o, id, s > 0);
            }
            mma_commit(&bar_mma);
        }
        if (!mma_done(2)) break;
        {   // lanes 0..63: A' = D o K K^T (strict) -> A = beta A' for the solve, A' -> scratch;
            // lanes 64..127: L = scale D o Q K^T (lower) -> [T; L] rows 64.., L -> scratch
            float v[32];
            tmem_ld16(tmem + lane_off + half * 32, v);
            tmem_ld16(tmem + lane_off + half * 32 + 16, v + 16);
            tmem_ld_wait();
            const int r = lrow & 63;
            float dec[32];
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
                const float4 d4 = *reinterpret_cast<const float4 *>(sT + r * kSolveLD + half * 32 + i);
                dec[i] = d4.x; dec[i + 1] = d4.y; dec[i + 2] = d4.z; dec[i + 3] = d4.w;
            }
            if (lrow < C) {
                const float br = sB[r];
#pragma unroll
                for (int i = 0; i < 32; i += 4) {
                    float ap[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int col = half * 32 + i + e;
                        ap[e] = (col < r && r < len) ? dec[i + e] * v[i + e] : 0.f;
                    }
                    *reinterpret_cast<float4 *>(sA + r * kSolveLD + half * 32 + i) =
                        make_float4(br * ap[0], br * ap[1], br * ap[2], br * ap[3]);
                    *reinterpret_cast<float4 *>(scr + kScrAp + r * kSolveLD + half * 32 + i) =
                        make_float4(ap[0], ap[1], ap[2], ap[3]);
                }
            } else {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float l[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int col = half * 32 + q * 8 + e;
                        l[e] = (col <= r && r < len) ? p.scale * dec[q * 8 + e] * v[q * 8 + e] : 0.f;
                    }
                    *kchunk(gTL, 128, C + r, half * 32 + q * 8) = pack8(l);
                    *reinterpret_cast<float4 *>(scr + kScrL + r * kSolveLD + half * 32 + q * 8) =
                        make_float4(l[0], l[1], l[2], l[3]);
                    *reinterpret_cast<float4 *>(scr + kScrL + r * kSolveLD + half * 32 + q * 8 + 4) =
                        make_float4(l[4], l[5], l[6], l[7]);
                }
            }
        }
        __syncthreads();
        solve_unit_lower64<kThreads>(sA, sT, sX);   // T = (I + A)^-1
        {   // T (lower, zero above) -> bf16 rows 0..63 of [T; L] and the scratch record
            const int r = tid >> 2;
#pragma unroll
            for (int qq = 0; qq < 2; ++qq) {
                const int c0 = ((tid & 3) * 2 + qq) * 8;
                float t8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) t8[e] = c0 + e <= r ? sT[r * kSolveLD + c0 + e] : 0.f;
                *kchunk(gTL, 128, r, c0) = pack8(t8);
                *reinterpret_cast<float4 *>(scr + kScrT + r * kSolveLD + c0) = make_float4(t8[0], t8[1], t8[2], t8[3]);
                *reinterpret_cast<float4 *>(scr + kScrT + r * kSolveLD + c0 + 4) = make_float4(t8[4], t8[5], t8[6], t8[7]);
            }
        }
        to_async();
        // ---- R2: [K; Q] S -> cols 0..127, [K; Q] dS' -> cols 128..255 (S, dS' as MN-major B)
        if (tid == 0) {
            const uint64_t a = smem_desc(sbase + gKQ, 16, 1024, kSwizzle128B);
            const uint64_t bs = smem_desc(sbase + gS, 16384, 1024, kSwizzle128B);
            const uint64_t bd = smem_desc(sbase + gDS, 16384, 1024, kSwizzle128B);
            constexpr uint32_t id = idesc_bf16(128, 128, 0, 1);
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                const uint64_t o = (s >> 2) * 1024 + (s & 3) * 2;
                mma_bf16(tmem, a + o, bs + s * 128, id, s > 0);
            }
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                const uint64_t o = (s >> 2) * 1024 + (s & 3) * 2;
                mma_bf16(tmem + 128, a + o, bd + s * 128, id, s > 0);
            }
            mma_commit(&bar_mma);
        }
        if (!mma_done(3)) break;
        {
            float x[64];
            ld64(half * 64, x);                      // K S (lanes 0..63) or Q S (lanes 64..127)
            if (lrow < C) {                          // R = beta (V - Gamma K S), in place of V
                const int r = lrow;
                const float br = sB[r], gr = sEG[r];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const int c = half * 64 + q * 8;
                    float vv[8], rr[8];
                    unpack8(*kchunk(gV, 64, r, c), vv);
#pragma unroll
                    for (int e = 0; e < 8; ++e) rr[e] = br * (vv[e] - gr * x[q * 8 + e]);
                    *kchunk(gV, 64, r, c) = pack8(rr);
                }
            } else {                                  // RA = sum_v dO o Q S
                const int r = lrow - C;
                float ra = 0.f;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    float dd[8];
                    unpack8(*kchunk(gT3, 192, 128 + r, half * 64 + q * 8), dd);
#pragma unroll
                    for (int e = 0; e < 8; ++e) ra = fmaf(dd[e], x[q * 8 + e], ra);
                }
                atomicAdd(&sRow[0][r], ra);
            }
        }
        to_async();
        // ---- R3: [T; L] R -> cols 256..383 (E in lanes 0..63); L^T dO -> cols 384..511
        if (tid == 0) {
            const uint64_t a = smem_desc(sbase + gTL, 16, 1024, kSwizzle128B);
            const uint64_t br = smem_desc(sbase + gV, 8192, 1024, kSwizzle128B);
            const uint64_t al = smem_desc(sbase + gTL + 8192, 8192, 1024, kSwizzle128B);   // L^T
            const uint64_t bo = smem_desc(sbase + gT3 + 16384, 24576, 1024, kSwizzle128B);  // dO
#pragma unroll
            for (int s = 0; s < 4; ++s)
                mma_bf16(tmem + 256, a + s * 2, br + s * 128, idesc_bf16(128, 128, 0, 1), s > 0);
#pragma unroll
            for (int s = 0; s < 4; ++s)
                mma_bf16(tmem + 384, al + s * 128, bo + s * 128, idesc_bf16(128, 128, 1, 1), s > 0);
            mma_commit(&bar_mma);
        }
        if (!mma_done(4)) break;
        if (lrow < C) {   // dE = Ktil dS' + L^T dO -> [dE; ..] rows 0..63, E -> rows 64..127; RD
            const int r = lrow;
            const float fr = sFR[r];
            float e64[64], x[64];
            ld64(256 + half * 64, e64);
            ld64(128 + half * 64, x);                // K dS'
            float rd = 0.f;
#pragma unroll
            for (int q = 0; q < 64; ++q) rd = fmaf(e64[q], x[q], rd);
            atomicAdd(&sRow[3][r], rd);
#pragma unroll
            for (int q = 0; q < 8; ++q) *kchunk(gT3, 192, C + r, half * 64 + q * 8) = pack8(e64 + q * 8);
            ld64(384 + half * 64, e64);               // L^T dO
#pragma unroll
            for (int q = 0; q < 64; ++q) x[q] = fmaf(fr, x[q], e64[q]);
            // dE as bf16 (hi) and its rounding remainder as bf16 (lo, in the [K; Q] tiles, free
            // since R2): T^T dE and dE R^T take both, so dE enters them with 16 bits
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const uint4 hi = pack8(x + q * 8);
                float hv[8], lo[8];
                unpack8(hi, hv);
#pragma unroll
                for (int e = 0; e < 8; ++e) lo[e] = x[q * 8 + e] - hv[e];
                *kchunk(gT3, 192, r, half * 64 + q * 8) = hi;
                *kchunk(gKQ, 64, r, half * 64 + q * 8) = pack8(lo);
            }
        }
        to_async();
        // ---- R4: dVb = T^T (dE_hi + dE_lo) -> cols 256..383; [E; dO] S^T -> 128..255 (dO S^T in lanes 64..);
        // [E; dO] E^T -> 384..447 (dO E^T in lanes 64..); [dE; E] R^T -> 448..511 (dE R^T in lanes
        // 0..63).  Columns 0..127 keep K S from R2 (lanes 0..63) for the dbeta and gate sums.
        if (tid == 0) {
            const uint64_t at = smem_desc(sbase + gTL, 8192, 1024, kSwizzle128B);          // T^T
            const uint64_t bde = smem_desc(sbase + gT3, 24576, 1024, kSwizzle128B);        // dE
#pragma unroll
            for (int s = 0; s < 4; ++s)
                mma_bf16(tmem + 256, at + s * 128, bde + s * 128, idesc_bf16(128, 128, 1, 1), s > 0);
            const uint64_t aeo = smem_desc(sbase + gT3 + 8192, 16, 1024, kSwizzle128B);    // [E; dO]
            const uint64_t ade = smem_desc(sbase + gT3, 16, 1024, kSwizzle128B);           // [dE; E]
            const uint64_t bs = smem_desc(sbase + gS, 16, 1024, kSwizzle128B);             // S^T
            const uint64_t be = smem_desc(sbase + gT3 + 8192, 16, 1024, kSwizzle128B);     // E^T
            const uint64_t brr = smem_desc(sbase + gV, 16, 1024, kSwizzle128B);            // R^T
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                const uint64_t oa = (s >> 2) * (24576 >> 4) + (s & 3) * 2;
                const uint64_t os = (s >> 2) * (16384 >> 4) + (s & 3) * 2;
                const uint64_t orr = (s >> 2) * (8192 >> 4) + (s & 3) * 2;
                mma_bf16(tmem + 128, aeo + oa, bs + os, idesc_bf16(128, 128), s > 0);
                mma_bf16(tmem + 384, aeo + oa, be + oa, idesc_bf16(128, 64), s > 0);
                mma_bf16(tmem + 448, ade + oa, brr + orr, idesc_bf16(128, 64), s > 0);
            }
            // the dE remainder: T^T dE_lo, and [dE_lo; -] R^T (lanes 64.. of that product unused)
            const uint64_t bdl = smem_desc(sbase + gKQ, 8192, 1024, kSwizzle128B);        // dE_lo
            const uint64_t adl = smem_desc(sbase + gKQ, 16, 1024, kSwizzle128B);
#pragma unroll
            for (int s = 0; s < 4; ++s)
                mma_bf16(tmem + 256, at + s * 128, bdl + s * 128, idesc_bf16(128, 128, 1, 1), true);
#pragma unroll
            for (int s = 0; s < 8; ++s)
                mma_bf16(tmem + 448, adl + (s >> 2) * (8192 >> 4) + (s & 3) * 2,
                         brr + (s >> 2) * (8192 >> 4) + (s & 3) * 2, idesc_bf16(128, 64), true);
            mma_commit(&bar_mma);
        }
        // the v row of this thread (dbeta needs V, whose tile now holds R), while R4 runs
        uint4 vrow8[8];
        if (lrow < C && lrow < len) {
            const uint4 *vrow = reinterpret_cast<const uint4 *>(p.v + ((t0 + lrow) * H + h) * (int64_t)VD + half * 64);
#pragma unroll
            for (int q = 0; q < 8; ++q) vrow8[q] = vrow[q];
        } else {
#pragma unroll
            for (int q = 0; q < 8; ++q) vrow8[q] = make_uint4(0, 0, 0, 0);
        }
        if (!mma_done(5)) break;
        if (lrow < C) {
            // dv = beta dVb; RB = sum_v dVb o V; RC = sum_v dVb o (K S); the R5 operand
            // -beta Gamma dVb (in place of [T; L])
            const int r = lrow;
            const bool live = r < len &&
                              GCL_RANGE_IN_BOUNDS(((t0 + r) * H + h) * (int64_t)VD + half * 64,
                                                  ((t0 + r) * H + h) * (int64_t)VD + half * 64 + 63,
                                                  p.t_max * H * (int64_t)VD, p.status);
            float *dvrow = p.dv + ((t0 + r) * H + h) * (int64_t)VD + half * 64;
            const float br = sB[r], fb = -sB[r] * sEG[r];
            float rb = 0.f, rc = 0.f;
#pragma unroll
            for (int q2 = 0; q2 < 4; ++q2) {          // 16 value columns at a time
                float x[16], ks[16];
                tmem_ld16(tmem + lane_off + 256 + half * 64 + q2 * 16, x);
                tmem_ld16(tmem + lane_off + half * 64 + q2 * 16, ks);
                tmem_ld_wait();
#pragma unroll
                for (int hq = 0; hq < 2; ++hq) {
                    const int q = q2 * 2 + hq, c = half * 64 + q * 8;
                    const float *xx = x + hq * 8;
                    float vv[8], sc[8];
                    unpack8(vrow8[q], vv);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        rb = fmaf(xx[e], vv[e], rb);
                        rc = fmaf(xx[e], ks[hq * 8 + e], rc);
                        sc[e] = fb * xx[e];
                    }
                    *kchunk(gTL, 64, r, c) = pack8(sc);
                    if (live) {
                        *reinterpret_cast<float4 *>(dvrow + q * 8) =
                            make_float4(br * xx[0], br * xx[1], br * xx[2], br * xx[3]);
                        *reinterpret_cast<float4 *>(dvrow + q * 8 + 4) =
                            make_float4(br * xx[4], br * xx[5], br * xx[6], br * xx[7]);
                    }
                }
            }
            atomicAdd(&sRow[1][r], rb);
            atomicAdd(&sRow[2][r], rc);
            {   // dT = dE R^T (32 columns of this half)
                float t32[32];
                tmem_ld16(tmem + lane_off + 448 + half * 32, t32);
                tmem_ld16(tmem + lane_off + 448 + half * 32 + 16, t32 + 16);
                tmem_ld_wait();
#pragma unroll
                for (int q = 0; q < 32; q += 4)
                    *reinterpret_cast<float4 *>(sDT + r * kSolveLD + half * 32 + q) =
                        make_float4(t32[q], t32[q + 1], t32[q + 2], t32[q + 3]);
            }
        } else {
            const int r = lrow - C;
            float x[64];
            ld64(128 + half * 64, x);                // dO S^T
            if (r < len && GCL_RANGE_IN_BOUNDS(((t0 + r) * H + h) * (int64_t)KD + half * 64,
                                               ((t0 + r) * H + h) * (int64_t)KD + half * 64 + 63,
                                               p.t_max * H * (int64_t)KD, p.status)) {
                float *dqrow = p.dq + ((t0 + r) * H + h) * (int64_t)KD + half * 64;
                const float fq = p.scale * sEG[r];
#pragma unroll
                for (int q = 0; q < 64; q += 4)
                    *reinterpret_cast<float4 *>(dqrow + q) =
                        make_float4(fq * x[q], fq * x[q + 1], fq * x[q + 2], fq * x[q + 3]);
            }
            float t32[32];                           // dL = dO E^T (32 columns of this half)
            tmem_ld16(tmem + lane_off + 384 + half * 32, t32);
            tmem_ld16(tmem + lane_off + 384 + half * 32 + 16, t32 + 16);
            tmem_ld_wait();
#pragma unroll
            for (int q = 0; q < 32; q += 4)
                *reinterpret_cast<float4 *>(sDL + r * kSolveLD + half * 32 + q) =
                    make_float4(t32[q], t32[q + 1], t32[q + 2], t32[q + 3]);
        }
        to_async();
        // ---- R5: (-beta Gamma dVb) S^T -> cols 0..127 and [E; dO] dS'^T -> cols 128..255
        // (lanes 0..63); dk = the first + exp(g_c - g) the second
        if (tid == 0) {
            const uint64_t a1 = smem_desc(sbase + gTL, 16, 1024, kSwizzle128B);
            const uint64_t a2 = smem_desc(sbase + gT3 + 8192, 16, 1024, kSwizzle128B);
            const uint64_t bs = smem_desc(sbase + gS, 16, 1024, kSwizzle128B);
            const uint64_t bd = smem_desc(sbase + gDS, 16, 1024, kSwizzle128B);
#pragma unroll
            for (int s = 0; s < 8; ++s)
                mma_bf16(tmem, a1 + (s >> 2) * (8192 >> 4) + (s & 3) * 2, bs + (s >> 2) * (16384 >> 4) + (s & 3) * 2,
                         idesc_bf16(128, 128), s > 0);
#pragma unroll
            for (int s = 0; s < 8; ++s)
                mma_bf16(tmem + 128, a2 + (s >> 2) * (24576 >> 4) + (s & 3) * 2,
                         bd + (s >> 2) * (16384 >> 4) + (s & 3) * 2, idesc_bf16(128, 128), s > 0);
            mma_commit(&bar_mma);
        }
        if (!mma_done(6)) break;
        if (lrow < C) {   // the first part of dk
            const int r = lrow;
            const float fr = sFR[r];
            float *dkrow = p.dk + ((t0 + r) * H + h) * (int64_t)KD + half * 64;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float x[16], y[16];
                tmem_ld16(tmem + lane_off + half * 64 + q * 16, x);
                tmem_ld16(tmem + lane_off + 128 + half * 64 + q * 16, y);
                tmem_ld_wait();
                if (r < len) {
#pragma unroll
                    for (int e = 0; e < 16; e += 4)
                        *reinterpret_cast<float4 *>(dkrow + q * 16 + e) =
                            make_float4(fmaf(fr, y[e], x[e]), fmaf(fr, y[e + 1], x[e + 1]),
                                        fmaf(fr, y[e + 2], x[e + 2]), fmaf(fr, y[e + 3], x[e + 3]));
                }
            }
        }
        __syncthreads();
        // scratch: dL, dT (as computed, full; the consumer masks them), row sums, <dS', S>
        for (int e = tid; e < C * C / 4; e += kThreads) {
            const int r = e >> 4, c = (e & 15) * 4;
            *reinterpret_cast<float4 *>(scr + kScrDL + r * kSolveLD + c) = *reinterpret_cast<const float4 *>(sDL + r * kSolveLD + c);
            *reinterpret_cast<float4 *>(scr + kScrDT + r * kSolveLD + c) = *reinterpret_cast<const float4 *>(sDT + r * kSolveLD + c);
        }
        for (int e = tid; e < 4 * C; e += kThreads) scr[kScrRows + e] = (&sRow[0][0])[e];
        if (tid == 0) {
            float t = 0.f;
            for (int w = 0; w < kThreads / 32; ++w) t += sRed[w];
            scr[kScrRows + 4 * C] = t;
        }
    } while (0);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
    if (tid == 0 && s_err != 0) status_set(p.status, GCL_DEV_WAIT_TIMEOUT);
}

// ============================================================================ grad2
// Two CTAs per SM (104 KiB of shared memory each, at most 128 registers per thread), so one
// CTA's copies overlap the other's arithmetic.  Shared memory, in the order of use:
//   hMP  [M; P] bf16, 128 rows x 64 columns (the MN-major P^T view reads 8 KiB past it, into
//        the T buffer: rows of junk that land in TMEM lanes nobody reads)
//   hF   fp32 T, A', L (later X = dT T^T), dL, dT (later dA), [64][kSolveLD] each (one bulk
//        copy of the scratch record); the K and Q tiles arrive late, over T and A'.
constexpr uint32_t hMP = 0;
constexpr uint32_t hF = 16384;
constexpr uint32_t hKQ = hF;                  // [K; Q] tiles (TMA), once T and A' are consumed
constexpr uint32_t h2End = hF + 5 * C * kSolveLD * 4;
constexpr int kGrad2Smem = h2End + 1024;
static_assert(hF % 1024 == 0 && hKQ + 32768 <= hF + 3 * C * kSolveLD * 4, "K, Q over T, A', L");
static_assert(hMP + 16384 + 8192 <= h2End, "the P^T view's second atom stays inside the allocation");
static_assert(2 * (kGrad2Smem + 4096) <= 233472, "two CTAs per SM");

__global__ void __launch_bounds__(kThreads, 2)
tc_grad2_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                GradParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    float *fT = reinterpret_cast<float *>(smem + hF);
    float *fAp = fT + C * kSolveLD, *fL = fAp + C * kSolveLD, *fDL = fL + C * kSolveLD;
    float *fDT = fDL + C * kSolveLD;
    float *fX = fL;                           // X replaces L once the dL o L sums are taken
    const float *fDA = fDT;                   // dA replaces dT
    __shared__ uint64_t bar_in, bar_kq, bar_mma;
    __shared__ uint32_t s_tmem;
    __shared__ int s_err;
    __shared__ __align__(16) float sRows[kScrRowFloats];   // RA, RB, RC, RD, <dS', S>
    __shared__ float sG[C], sB[C], sDG[C], sPart[4][C], sRed2[2], s_carry;
    const float *sRA = sRows, *sRB = sRows + C, *sRC = sRows + 2 * C, *sRD = sRows + 3 * C;

    if (status_blocks_cta(p.status)) return;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3, half = warp >> 2;
    const int lrow = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const int j = blockIdx.x, h = blockIdx.y, H = p.H;
    int64_t t0;
    int len;
    if (!chunk_of_row(p, j, t0, len)) return;
    const int unit = j * H + h;
    const uint32_t sbase = smem_u32(smem);
    const float *scr = p.scratch + (size_t)unit * kScrFloats;

    if (tid == 0) {   // the five matrices and the row sums of the first kernel
        mbar_init(&bar_in, 1);
        mbar_init(&bar_kq, 1);
        mbar_init(&bar_mma, 1);
        s_err = 0;
        fence_barrier_init();
        mbar_arrive_expect_tx(&bar_in, kScrRows * 4 + kScrRowFloats * 4);
        bulk_load(fT, scr, kScrRows * 4, &bar_in);
        bulk_load(sRows, scr + kScrRows, kScrRowFloats * 4, &bar_in);
    }
    __syncwarp();
    if (warp == 0) {
        tmem_alloc(&s_tmem, 256);
        tmem_relinquish();
    }
    chunk_gates(p, t0, len, h, sG, sB, &s_carry);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    const float gC = sG[C - 1];
    // row (parts 0, 2) and column (parts 1, 3) sums over a [64][kSolveLD] pair, rows
    // 32 (w & 1) + lane for the warp pair of the part; column sums weight row r2 by wc[r2]
    auto row_sum = [&](const float *x, const float *y, int r) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
        for (int i = 0; i < C; i += 4) {
            const float4 a4 = *reinterpret_cast<const float4 *>(x + r * kSolveLD + i);
            const float4 b4 = *reinterpret_cast<const float4 *>(y + r * kSolveLD + i);
            acc[0] = fmaf(a4.x, b4.x, acc[0]);
            acc[1] = fmaf(a4.y, b4.y, acc[1]);
            acc[2] = fmaf(a4.z, b4.z, acc[2]);
            acc[3] = fmaf(a4.w, b4.w, acc[3]);
        }
        return (acc[0] + acc[1]) + (acc[2] + acc[3]);
    };
    auto col_sum = [&](const float *x, const float *y, const float *wc, int r) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
        for (int r2 = 0; r2 < C; ++r2)
            acc[r2 & 3] = fmaf(x[r2 * kSolveLD + r] * (wc ? wc[r2] : 1.f), y[r2 * kSolveLD + r], acc[r2 & 3]);
        return (acc[0] + acc[1]) + (acc[2] + acc[3]);
    };
    do {
        const bool landed = mbar_wait(&bar_in, 0, &s_err, 1);
        if (__syncthreads_or(!landed)) break;
        // ---- gate sums of dL o L (L is zero above the diagonal and past the end):
        // warps 0..3 the row sums, warps 4..7 the column sums
        {
            const int r = (warp & 1) * 32 + lane;
            if (warp < 2) sPart[0][r] = row_sum(fDL, fL, r);
            else if (warp < 4) sPart[1][r] = col_sum(fDL, fL, nullptr, r);
        }
        __syncthreads();
        // ---- dA = -T^T (dT T^T), strictly lower; dT counts only on and below the diagonal.
        // Both products in 4 x 4 register tiles with float4 loads (T is zero above its diagonal).
        // X = dT T^T: X[r][m] = sum_{i <= min(r, m)} dT[r][i] T[m][i]; rows r0 .. r0 + 3, columns
        // mb + 16 a (interleaved, so the T rows a quarter warp loads sit in distinct banks)
        {
            const int r0 = (tid >> 4) * 4, mb = tid & 15;
            float acc[4][4] = {};
            for (int i4 = 0; i4 <= r0 / 4; ++i4) {
                float dt[4][4], tt[4][4];
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    const float4 v = *reinterpret_cast<const float4 *>(fDT + (r0 + x) * kSolveLD + 4 * i4);
                    const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) dt[x][e] = 4 * i4 + e <= r0 + x ? vv[e] : 0.f;
                }
#pragma unroll
                for (int a = 0; a < 4; ++a) {
                    const float4 v = *reinterpret_cast<const float4 *>(fT + (mb + 16 * a) * kSolveLD + 4 * i4);
                    tt[a][0] = v.x;
                    tt[a][1] = v.y;
                    tt[a][2] = v.z;
                    tt[a][3] = v.w;
                }
#pragma unroll
                for (int e = 0; e < 4; ++e)
#pragma unroll
                    for (int x = 0; x < 4; ++x)
#pragma unroll
                        for (int a = 0; a < 4; ++a) acc[x][a] = fmaf(dt[x][e], tt[a][e], acc[x][a]);
            }
#pragma unroll
            for (int x = 0; x < 4; ++x)
#pragma unroll
                for (int a = 0; a < 4; ++a) fX[(r0 + x) * kSolveLD + mb + 16 * a] = acc[x][a];
        }
        __syncthreads();
        // dA[r][i] = -sum_{m >= r} T[m][r] X[m][i] for i < r, else 0 (over dT, which is consumed);
        // rows r0 .. r0 + 3, columns i0 .. i0 + 3
        {
            const int r0 = (tid >> 4) * 4, i0 = (tid & 15) * 4;
            float acc[4][4] = {};
            if (i0 < r0 + 3) {
                for (int m = r0; m < C; ++m) {
                    const float4 t = *reinterpret_cast<const float4 *>(fT + m * kSolveLD + r0);
                    const float4 xv = *reinterpret_cast<const float4 *>(fX + m * kSolveLD + i0);
                    const float tv[4] = {t.x, t.y, t.z, t.w}, xx[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
                    for (int x = 0; x < 4; ++x)
#pragma unroll
                        for (int y = 0; y < 4; ++y) acc[x][y] = fmaf(-tv[x], xx[y], acc[x][y]);
                }
            }
#pragma unroll
            for (int x = 0; x < 4; ++x)
                *reinterpret_cast<float4 *>(fDT + (r0 + x) * kSolveLD + i0) =
                    make_float4(i0 < r0 + x ? acc[x][0] : 0.f, i0 + 1 < r0 + x ? acc[x][1] : 0.f,
                                i0 + 2 < r0 + x ? acc[x][2] : 0.f, i0 + 3 < r0 + x ? acc[x][3] : 0.f);
        }
        __syncthreads();
        // ---- gate sums of dA o A' (both strictly lower): row sums, beta-weighted column sums
        {
            const int r = (warp & 1) * 32 + lane;
            if (warp < 2) sPart[2][r] = row_sum(fDA, fAp, r);
            else if (warp < 4) sPart[3][r] = col_sum(fDA, fAp, sB, r);
        }
        __syncthreads();
        if (tid == 0) {   // T, A' and L are consumed: the K and Q tiles of the last MMA round
            fence_async_smem();
            mbar_arrive_expect_tx(&bar_kq, 32768);
            for (int cb = 0; cb < 2; ++cb) {
                tma_load_3d(smem + hKQ + cb * 16384, &tm_k, cb * 64, h, (int)t0, &bar_kq);
                tma_load_3d(smem + hKQ + cb * 16384 + 8192, &tm_q, cb * 64, h, (int)t0, &bar_kq);
            }
        }
        if (tid < C) {   // dgamma and dbeta of row tid
            const int r = tid;
            const float Gr = __expf(sG[r]);
            const float fr = r < len ? __expf(gC - sG[r]) : 0.f;
            const float da_row = sPart[2][r];
            float frd = fr * sRD[r];
            sDG[r] = p.scale * Gr * sRA[r] + (sPart[0][r] - sPart[1][r]) + sB[r] * da_row - sPart[3][r] -
                     sB[r] * Gr * sRC[r] - frd;
            if (r < len && GCL_IN_BOUNDS((t0 + r) * H + h, p.t_max * H, p.status))
                p.dbeta[(t0 + r) * H + h] = sRB[r] - Gr * sRC[r] + da_row;
            // the last row's gamma also carries the Ktil factors of every row: their sum
#pragma unroll
            for (int d = 16; d > 0; d >>= 1) frd += __shfl_xor_sync(0xffffffffu, frd, d);
            if (lane == 0) sRed2[warp] = frd;
        }
        // ---- P = scale D o dL (i <= r) -> rows 64..127, M = beta_r D o dA (i < r) -> rows 0..63
        // of the [M; P] operand (bf16, K-major over i)
        {
            const int r = tid >> 2;
#pragma unroll
            for (int qq = 0; qq < 2; ++qq) {
                const int c0 = ((tid & 3) * 2 + qq) * 8;
                float m8[8], p8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int i = c0 + e;
                    const float dec = i <= r ? __expf(sG[r] - sG[i]) : 0.f;
                    p8[e] = i <= r ? p.scale * dec * fDL[r * kSolveLD + i] : 0.f;
                    m8[e] = i < r ? sB[r] * dec * fDA[r * kSolveLD + i] : 0.f;
                }
                *reinterpret_cast<uint4 *>(smem + hMP + kmaj16(128, r, c0)) = pack8(m8);
                *reinterpret_cast<uint4 *>(smem + hMP + kmaj16(128, C + r, c0)) = pack8(p8);
            }
        }
        __syncthreads();
        {   // dg = reverse in-chunk cumsum of dgamma (thread t: row 63 - t), gamma_c at the last row
            float x = 0.f;
            if (tid < C) {
                x = sDG[C - 1 - tid];
                if (tid == 0) x += sRows[4 * C] * __expf(gC) + (sRed2[0] + sRed2[1]);
                x = warp_scan(x);
                if (tid == 31) s_carry = x;
            }
            __syncthreads();
            if (tid >= 32 && tid < C) x += s_carry;
            const int r = C - 1 - tid;
            if (tid < C && r < len && GCL_IN_BOUNDS((t0 + r) * H + h, p.t_max * H, p.status))
                p.dg[(t0 + r) * H + h] = x;
        }
        {
            const bool kq = mbar_wait(&bar_kq, 0, &s_err, 3);
            if (__syncthreads_or(!kq)) break;
        }
        if (len < C) {   // K and Q rows past the end (NaN padding) enter the MMAs raw
            const uint4 zero = make_uint4(0, 0, 0, 0);
            for (int t = tid; t < 4 * C * 8; t += kThreads) {
                const int r = (t >> 3) & 63, blk = t >> 9;
                if (r >= len)
                    *reinterpret_cast<uint4 *>(smem + hKQ + (blk & 1) * 16384 + (blk >> 1) * 8192 + r * 128 +
                                               (t & 7) * 16) = zero;
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        // ---- [M; P] K -> cols 0..127 (M K in lanes 0..63, P K in lanes 64..127);
        //      M^T K + P^T Q -> cols 128..255 (lanes 0..63)
        if (tid == 0) {
            const uint64_t amp = smem_desc(sbase + hMP, 16, 1024, kSwizzle128B);
            const uint64_t amt = smem_desc(sbase + hMP, 8192, 1024, kSwizzle128B);          // M^T
            const uint64_t apt = smem_desc(sbase + hMP + 8192, 8192, 1024, kSwizzle128B);   // P^T
            const uint64_t bk = smem_desc(sbase + hKQ, 16384, 1024, kSwizzle128B);
            const uint64_t bq = smem_desc(sbase + hKQ + 8192, 16384, 1024, kSwizzle128B);
#pragma unroll
            for (int s = 0; s < 4; ++s) mma_bf16(tmem, amp + s * 2, bk + s * 128, idesc_bf16(128, 128, 0, 1), s > 0);
#pragma unroll
            for (int s = 0; s < 4; ++s)
                mma_bf16(tmem + 128, amt + s * 128, bk + s * 128, idesc_bf16(128, 128, 1, 1), s > 0);
#pragma unroll
            for (int s = 0; s < 4; ++s)
                mma_bf16(tmem + 128, apt + s * 128, bq + s * 128, idesc_bf16(128, 128, 1, 1), 1);
            mma_commit(&bar_mma);
        }
        // dk += M K + M^T K + P^T Q (lanes 0..63), dq += P K (lanes 64..127), 16 columns at a
        // time; the first kernel's partial rows are read ahead (two groups of 16 columns in
        // flight), so their latency overlaps the MMA round and the additions
        const bool isk = lrow < C;
        const int r = isk ? lrow : lrow - C;
        float *grow = (isk ? p.dk : p.dq) + ((t0 + r) * H + h) * (int64_t)KD + half * 64;
        const bool live = r < len;
        float4 part[2][4];
        auto fetch = [&](int q, float4 (&dst)[4]) {
#pragma unroll
            for (int e = 0; e < 4; ++e)
                dst[e] = live ? *reinterpret_cast<const float4 *>(grow + q * 16 + 4 * e) : make_float4(0.f, 0.f, 0.f, 0.f);
        };
        fetch(0, part[0]);
        fetch(1, part[1]);
        const bool ok = mbar_wait(&bar_mma, 0, &s_err, 2);
        tc_fence_after();
        if (__syncthreads_or(!ok)) break;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            float x[16], y[16];
            tmem_ld16(tmem + lane_off + half * 64 + q * 16, x);
            if (isk) tmem_ld16(tmem + lane_off + 128 + half * 64 + q * 16, y);
            tmem_ld_wait();
            float4 cur[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) cur[e] = part[q & 1][e];
            if (q + 2 < 4) fetch(q + 2, part[q & 1]);
            if (live) {
#pragma unroll
                for (int e = 0; e < 16; e += 4) {
                    float4 d = cur[e >> 2];
                    d.x += x[e] + (isk ? y[e] : 0.f);
                    d.y += x[e + 1] + (isk ? y[e + 1] : 0.f);
                    d.z += x[e + 2] + (isk ? y[e + 2] : 0.f);
                    d.w += x[e + 3] + (isk ? y[e + 3] : 0.f);
                    *reinterpret_cast<float4 *>(grow + q * 16 + e) = d;
                }
            }
        }
    } while (0);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 256);
    if (tid == 0 && s_err != 0) status_set(p.status, GCL_DEV_WAIT_TIMEOUT);
}

}  // namespace

size_t bwd_grad_tc_scratch_bytes(int64_t nt_max, int H) {
    return (size_t)nt_max * H * kScrFloats * sizeof(float);
}

cudaError_t launch_bwd_grad_tc(const BwdParams &p, float *scratch, cudaStream_t s) {
    const int H = p.H;
    CUtensorMap mq, mk, mv, mdo;
    const cuuint64_t dqk[3] = {(cuuint64_t)KD, (cuuint64_t)H, (cuuint64_t)p.t_max};
    const cuuint64_t sqk[2] = {(cuuint64_t)KD * 2, (cuuint64_t)H * KD * 2};
    const cuuint32_t b64[3] = {64, 1, 64};
    const cuuint64_t dv[3] = {(cuuint64_t)VD, (cuuint64_t)H, (cuuint64_t)p.t_max};
    const cuuint64_t sv[2] = {(cuuint64_t)VD * 2, (cuuint64_t)H * VD * 2};
    if (!make_tensor_map(&mq, p.q, 3, dqk, sqk, b64, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tensor_map(&mk, p.k, 3, dqk, sqk, b64, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tensor_map(&mv, p.v, 3, dv, sv, b64, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tensor_map(&mdo, p.d_o, 3, dv, sv, b64, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    GradParams gp{};
    gp.chunk_indices = p.chunk_indices;
    gp.cu = p.cu_seqlens;
    gp.g = p.g;
    gp.beta = static_cast<const __nv_bfloat16 *>(p.beta);
    gp.v = static_cast<const __nv_bfloat16 *>(p.v);
    gp.h = p.h;
    gp.dh = reinterpret_cast<const uint8_t *>(p.dh);
    gp.dq = p.dq;
    gp.dk = p.dk;
    gp.dv = p.dv;
    gp.dg = p.dg;
    gp.dbeta = p.dbeta;
    gp.scratch = scratch;
    gp.status = p.dev_status;
    gp.t_max = p.t_max;
    gp.nt_max = p.nt_max;
    gp.n_max = p.n_max;
    gp.H = H;
    gp.scale = p.scale;
    cudaError_t e = cudaFuncSetAttribute(tc_grad1_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kGrad1Smem);
    if (e != cudaSuccess) return e;
    tc_grad1_kernel<<<dim3((unsigned)p.nt_max, H), kThreads, kGrad1Smem, s>>>(mq, mk, mv, mdo, gp);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if ((e = cudaFuncSetAttribute(tc_grad2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kGrad2Smem)) !=
        cudaSuccess)
        return e;
    tc_grad2_kernel<<<dim3((unsigned)p.nt_max, H), kThreads, kGrad2Smem, s>>>(mq, mk, gp);
    return cudaGetLastError();
}

}  // namespace gcl
