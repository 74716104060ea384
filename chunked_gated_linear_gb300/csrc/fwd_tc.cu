// fwd_tc.cu -- tensor-core (tcgen05 + TMA) chunk forward of the gated delta rule,
// bf16 inputs, d_k = d_v = 128, chunk 64.
//
// HA-NPU paper "Empowering Hybrid Attention Models on NPUs": section 2.1
// (Map-Reduce-Map: the Map phases are independent across chunks, only the
// Reduce is serial), section 4 (one (head, column slice) per core, tail heads
// split along the value columns), section 5 (chunk-first in-place state update;
// grouped GEMMs KK^T, QK^T, KS, QS; W = A^-1 K with the inversion decoupled from
// the GEMMs).  FLA RFC "[RFC] Add Graph Capture Support for FLA Prefill and
// Training Paths on Ascend NPUs", "Core design": fixed grids over NT_max chunk
// rows with the [-1, 0] sentinel checked before any pointer arithmetic.
//
// Two launches:
//
//  prep   one CTA per row of chunk_indices and head (chunk-parallel Map):
//         D1 = [K; Q] K^T on the tensor cores (M = 128: KK^T and QK^T stacked),
//         then on the CUDA cores
//           A[r,i] = beta_r exp(g_r - g_i) (k_r . k_i)       i < r
//           L[r,i] = scale exp(g_r - g_i) (q_r . k_i)        i <= r
//         and T = (I + A)^-1 by blocked forward substitution (16 x 16 diagonal
//         blocks, then three levels of off-diagonal blocks).  [T; L] goes to the
//         workspace as bf16 (128 x 64 per chunk and head).
//
//  chain  one CTA per (sequence, head, column slice of width VS) walks the
//         chunks in order with its state slice S [128 x VS] in fp32 registers
//         (thread c owns key row c) and a bf16 copy in shared memory:
//           P1  W^T   = (diag(beta Gamma) K)^T T^T          -> TMEM, stored as -W
//           P2  D2    = [T; L] (diag(beta) V)               =  [U; L diag(beta) V]
//           C1  D2   += [-W; scale diag(Gamma) Q] S         =  [E; L beta V + Qhat S]
//           C2  D3    = (diag(exp(g_c - g)) K)^T E          (state increment)
//           C3  D2   += [T; L] E                            -> bottom: L beta V + O
//         S <- Gamma_c S + D3 (fp32), O = bottom - L beta V.  E = U - W S comes
//         out of the accumulator directly; every operand is either loaded by TMA
//         or a row-scaled copy of a TMA tile (the transposed views use MN-major
//         shared-memory descriptors), so no operand is transposed by hand except
//         the small E and S slices.
//
// Rows past the end of a sequence are zeroed (selected, not multiplied) in every
// operand the CUDA cores build, so NaN padding never reaches an MMA.
#include <cudaTypedefs.h>

#include "gcl_internal.cuh"
#include "tc_ptx.cuh"
#include "tc_solve.cuh"

namespace gcl {
namespace {

using namespace tc;
constexpr int C = 64;
constexpr int KD = 128;
constexpr int VD = 128;
constexpr int kThreads = 128;
constexpr int kTLRows = 192;   // [T diag(beta Gamma); T diag(beta); L] rows per chunk and head
constexpr int kFRows = 4;      // per-chunk factors (fp32 rows of 64): exp(g_c - g), scale exp(g),
                               // exp(g_c) (broadcast), unused

__device__ __forceinline__ float bf2f(__nv_bfloat16 x) { return __bfloat162float(x); }

// Inclusive scan of one float per lane across a warp.
__device__ __forceinline__ float warp_incl_scan(float x) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, x, d);
        if (lane >= d) x += y;
    }
    return x;
}

// gamma = inclusive cumsum of the 64 gate values of a chunk, by warps 0 and 1 (threads
// 0..63 each hold g of their row); the total of warp 0 is handed over through shared
// memory.  All threads of the block must call it (it contains a block barrier).
__device__ __forceinline__ float chunk_cumsum(float g, float *s_carry) {
    const int tid = threadIdx.x;
    float x = 0.f;
    if (tid < 64) x = warp_incl_scan(g);
    if (tid == 31) *s_carry = x;
    __syncthreads();
    if (tid >= 32 && tid < 64) x += *s_carry;
    return x;
}


// ============================================================================ prep
struct PrepParams {
    const int32_t *chunk_indices, *cu;
    const float *g;
    const __nv_bfloat16 *beta;
    __nv_bfloat16 *tl;          // [nt_max, H, 192, 64]
    float *fac;                 // [nt_max, H, 4, 64]
    int32_t *status;
    int64_t t_max;
    int32_t n_max, H;
    float scale;
};

// The fp32 solve buffers reuse the K/Q tile once the MMA has consumed it.
constexpr int kPrepSmem = 1024 + (kSolveFloats + C * kSolveLD) * 4;   // + decay table
static_assert(kSolveFloats * 4 >= 32768, "the K/Q tile fits under the solve buffers");

__global__ void __launch_bounds__(kThreads)
tc_prep_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               PrepParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    uint8_t *sKQ = smem;                                         // [2 cb][128 rows][128 B]
    float *sA = reinterpret_cast<float *>(smem);                 // [64][kSolveLD], after the MMA
    float *sT = sA + C * kSolveLD;                               // [64][kSolveLD], after the MMA
    float *sX = sT + C * kSolveLD;                               // solve scratch
    float *sD = sA + kSolveFloats;                               // [64][kSolveLD] decay table
    __shared__ uint64_t bar_tma, bar_mma;
    __shared__ uint32_t s_tmem;
    __shared__ int s_err;
    __shared__ float sG[C], sB[C], sEG[C];

    if (status_blocks_cta(p.status)) return;
    const int tid = threadIdx.x, warp = tid >> 5, j = blockIdx.x, h = blockIdx.y;
    const int n = p.chunk_indices[2 * j];
    if (n < 0) return;                              // sentinel: unused chunk slot
    const int ic = p.chunk_indices[2 * j + 1];
    if (n >= p.n_max || ic < 0) {
        if (tid == 0) status_set(p.status, GCL_DEV_BAD_RANGE);
        return;
    }
    const int64_t bos = p.cu[n], eos = p.cu[n + 1], t0 = bos + (int64_t)ic * C;
    if (bos < 0 || eos < bos || eos > p.t_max || t0 >= eos) {
        if (tid == 0) status_set(p.status, GCL_DEV_BAD_RANGE);
        return;
    }
    const int len = (int)(eos - t0 < C ? eos - t0 : C);
    const int H = p.H;

    if (tid == 0) {
        mbar_init(&bar_tma, 1);
        mbar_init(&bar_mma, 1);
        s_err = 0;
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc(&s_tmem, 64);
        tmem_relinquish();
    }
    __shared__ float s_carry;
    {
        const float gv = (tid < len && GCL_IN_BOUNDS((t0 + tid) * H + h, p.t_max * H, p.status))
                             ? p.g[(t0 + tid) * H + h] : 0.f;
        const float gam = chunk_cumsum(gv, &s_carry);
        if (tid < C) {
            sG[tid] = gam;
            sB[tid] = tid < len ? bf2f(p.beta[(t0 + tid) * H + h]) : 0.f;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    if (tid == 0) {
        mbar_arrive_expect_tx(&bar_tma, 32768);
        for (int cb = 0; cb < 2; ++cb) {
            tma_load_3d(sKQ + cb * 16384, &tm_k, cb * 64, h, (int)t0, &bar_tma);
            tma_load_3d(sKQ + cb * 16384 + 8192, &tm_q, cb * 64, h, (int)t0, &bar_tma);
        }
    }
    // while the tiles load: Gamma per column and the decay table D[r][c] = exp(g_r - g_c) for
    // c <= r (1 above the diagonal; the exponent is selected, so no lane branches around the
    // exponential)
    if (tid < C) sEG[tid] = __expf(sG[tid]);
    for (int e = tid; e < C * C / 4; e += kThreads) {
        const int r = e >> 4, c = (e & 15) * 4;
        const float gr = sG[r];
        *reinterpret_cast<float4 *>(sD + r * kSolveLD + c) =
            make_float4(__expf(c <= r ? gr - sG[c] : 0.f), __expf(c + 1 <= r ? gr - sG[c + 1] : 0.f),
                        __expf(c + 2 <= r ? gr - sG[c + 2] : 0.f), __expf(c + 3 <= r ? gr - sG[c + 3] : 0.f));
    }
    if (tid == 0) {
        if (mbar_wait(&bar_tma, 0, &s_err, 1)) {
            tc_fence_after();
            const uint32_t base = smem_u32(sKQ);
            constexpr uint32_t idesc = idesc_bf16(128, 64);
            for (int s = 0; s < KD / 16; ++s) {
                const uint32_t off = (s >> 2) * 16384 + (s & 3) * 32;
                mma_bf16(tmem, smem_desc(base + off, 16, 1024, kSwizzle128B),
                         smem_desc(base + off, 16, 1024, kSwizzle128B), idesc, s > 0);
            }
            mma_commit(&bar_mma);
        }
    }
    __syncthreads();
    mbar_wait(&bar_mma, 0, &s_err, 2);
    tc_fence_after();
    __syncthreads();
    if (s_err == 0) {
        float v[64];
#pragma unroll
        for (int q = 0; q < 4; ++q) tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + q * 16, v + q * 16);
        tmem_ld_wait();
        __nv_bfloat16 *tl = p.tl + ((size_t)j * H + h) * kTLRows * C;
        if (tid < C) {
            const int r = tid;
            const float gr = sG[r], br = sB[r], gc = sG[C - 1];
            const bool live = r < len;
            float *fac = p.fac + ((size_t)j * H + h) * kFRows * C;
            fac[r] = live ? __expf(gc - gr) : 0.f;               // state-update decay of row r
            fac[C + r] = live ? p.scale * __expf(gr) : 0.f;     // read-out factor of row r
            fac[2 * C + r] = __expf(gc);                         // chunk decay Gamma_c
#pragma unroll
            for (int i = 0; i < C; i += 4) {
                const float4 d4 = *reinterpret_cast<const float4 *>(sD + r * kSolveLD + i);
                const float dec[4] = {d4.x, d4.y, d4.z, d4.w};
                float a[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) a[e] = (i + e < r && r < len) ? br * dec[e] * v[i + e] : 0.f;
                *reinterpret_cast<float4 *>(sA + r * kSolveLD + i) = make_float4(a[0], a[1], a[2], a[3]);
            }
        } else {
            const int r = tid - C;
            uint4 *dst = reinterpret_cast<uint4 *>(tl + (size_t)(2 * C + r) * C);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float4 da = *reinterpret_cast<const float4 *>(sD + r * kSolveLD + q * 8);
                const float4 db = *reinterpret_cast<const float4 *>(sD + r * kSolveLD + q * 8 + 4);
                const float dec[8] = {da.x, da.y, da.z, da.w, db.x, db.y, db.z, db.w};
                uint4 pk;
                __nv_bfloat162 *pp = reinterpret_cast<__nv_bfloat162 *>(&pk);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int i0 = q * 8 + 2 * e, i1 = i0 + 1;
                    const float l0 = (i0 <= r && r < len) ? p.scale * dec[2 * e] * v[i0] : 0.f;
                    const float l1 = (i1 <= r && r < len) ? p.scale * dec[2 * e + 1] * v[i1] : 0.f;
                    pp[e] = __floats2bfloat162_rn(l0, l1);
                }
                dst[q] = pk;
            }
        }
        __syncthreads();
        solve_unit_lower64<kThreads>(sA, sT, sX);   // T = (I + A)^-1
        // ---- T diag(beta Gamma) -> rows 0..63, T diag(beta) -> rows 64..127 (bf16)
        {
            const int r = tid >> 1, half = tid & 1;
            uint4 *dst_s = reinterpret_cast<uint4 *>(tl + (size_t)r * C + half * 32);
            uint4 *dst_t = reinterpret_cast<uint4 *>(tl + (size_t)(C + r) * C + half * 32);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint4 pt, ps;
                __nv_bfloat162 *ppt = reinterpret_cast<__nv_bfloat162 *>(&pt);
                __nv_bfloat162 *pps = reinterpret_cast<__nv_bfloat162 *>(&ps);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int i0 = half * 32 + q * 8 + 2 * e;
                    const float t0v = i0 <= r ? sT[r * kSolveLD + i0] : 0.f;
                    const float t1v = i0 + 1 <= r ? sT[r * kSolveLD + i0 + 1] : 0.f;
                    ppt[e] = __floats2bfloat162_rn(t0v * sB[i0], t1v * sB[i0 + 1]);
                    pps[e] = __floats2bfloat162_rn(t0v * sB[i0] * sEG[i0], t1v * sB[i0 + 1] * sEG[i0 + 1]);
                }
                dst_t[q] = pt;
                dst_s[q] = ps;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 64);
    if (tid == 0 && s_err != 0) status_set(p.status, GCL_DEV_WAIT_TIMEOUT);
}

// ============================================================================ chain
struct ChainParams {
    const int32_t *cu, *chunk_offsets, *seq_order;
    const float *h0;
    __nv_bfloat16 *o;
    float *ht, *h_save;
    int32_t *status;
    int64_t t_max, nt_max;
    int32_t n_max, H;
};

// Shared memory of the chain kernel.  Per stage (two stages, chunk n in stage n & 1):
// K tile, [-W; Q], [T diag(bG); T diag(b); L], the 64-column V tile holding this
// slice, and the chunk's factors.  Then the MN-major B operands S, E and f E
// (VS used columns of 64-element swizzle atoms).
struct ChainLayout {
    static constexpr uint32_t kK = 16384, kWQ = 32768, kTL = 24576, kV = 8192, kF = 1024;
    static constexpr uint32_t kStage = kK + kWQ + kTL + kV + kF;          // 82944 (1024-aligned)
    static constexpr uint32_t oK = 0, oWQ = kK, oTL = oWQ + kWQ, oV = oTL + kTL, oF = oV + kV;
    static constexpr uint32_t oSB = 2 * kStage;                          // S, 16 k-groups
    static constexpr uint32_t oET = oSB + 16384;                         // E, 8 k-groups
    static constexpr uint32_t oFT = oET + 8192;                          // exp(g_c - g) E
    static constexpr uint32_t total = oFT + 8192;
    static constexpr uint32_t bytes = total + 1024;                      // + alignment slack
    // bytes TMA delivers per stage: K, the Q half of [-W; Q], [T..; L], V, factors
    // (the -W half is written by the threads)
    static constexpr uint32_t kTmaBytes = kK + kWQ / 2 + kTL + kV + kF;
};

// Offset of element (k, n) of an MN-major bf16 operand with the 128-byte swizzle and
// n < 64: 8-row k-groups of 1024 B, 16-byte chunk index XOR (k % 8).
__device__ __forceinline__ uint32_t mn_sw128(int k, int n) {
    return (uint32_t)((k >> 3) * 1024 + (k & 7) * 128 + ((((n >> 3) ^ (k & 7))) << 4) + (n & 7) * 2);
}

constexpr int kComputeThreads = 256;                  // warps 0..7
constexpr int kChainThreads = kComputeThreads + 32;   // + warp 8: TMA and MMA issue

__device__ __forceinline__ void compute_barrier() {   // named barrier over warps 0..7
    asm volatile("bar.sync 1, %0;" ::"n"(kComputeThreads) : "memory");
}

// Named barrier over warps 0..7 that returns the OR of every thread's flag, so all
// compute threads take the same branch on it.
__device__ __forceinline__ bool compute_barrier_or(bool flag) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, 1, %2, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)flag), "n"(kComputeThreads)
        : "memory");
    return r != 0;
}

// Per-(sequence, head, column slice) state recurrence, warp-specialised.
// Warps 0..7 compute: thread t owns TMEM lane / row 32 (w & 3) + (t & 31) of warp w and
// the column half (w >> 2) of the slice.  Warp 8 (one lane) issues every TMA and MMA.
// Per chunk n, with stage n & 1 holding its tiles:
//   issuer:  C1(n) = [-W; Q] S  |  P(n+1)  |  C2(n) = K^T (f E), C3(n) = [T diag(b); L] E  |  TMA(n+2)
//   compute: land(n+1)  |  E(n)  |  -W(n+1)  |  S, O(n)
// Hand-offs use mbarriers; the compute side arrives from one thread after a named
// barrier over its 256 threads (each of which fenced its shared writes first).
template <int VS>
__global__ void __launch_bounds__(kChainThreads, 1)
tc_chain_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_tl,
                const __grid_constant__ CUtensorMap tm_f, ChainParams p) {
    using Lay = ChainLayout;
    constexpr int HV = VS / 2;                              // columns per compute thread
    // TMEM: D_W 128 | U (2 stages) | [-W S; Q S] | K^T (f E) | [. ; L E]
    constexpr uint32_t tD2p = 128, tD2c = 128 + 2 * VS, tD3 = 128 + 3 * VS, tD4 = 128 + 4 * VS;
    constexpr uint32_t kTmemCols = 128 + 5 * VS <= 256 ? 256 : 512;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    __shared__ uint64_t bar_tma[2], bar_ops[2], bar_c1, bar_c23, bar_p, bar_sb, bar_w, bar_e;
    __shared__ uint32_t s_tmem;
    __shared__ int s_err;

    if (status_blocks_cta(p.status)) return;
    const int tid = threadIdx.x, warp = tid >> 5;
    const bool compute = warp < 8;
    const int quarter = warp & 3, half = (warp >> 2) & 1;
    const int row = quarter * 32 + (tid & 31);
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const int split = blockIdx.x, h = blockIdx.y;
    const int n = p.seq_order ? p.seq_order[blockIdx.z] : (int)blockIdx.z;
    const int H = p.H, v0 = split * VS;
    if (n < 0 || n >= p.n_max) {              // checked before cu[n] and cu[n + 1] are read
        if (tid == 0) status_set(p.status, GCL_DEV_BAD_RANGE);
        return;
    }
    const int64_t bos = p.cu[n], eos = p.cu[n + 1];
    if (bos < 0 || eos < bos || eos > p.t_max) {
        if (tid == 0) status_set(p.status, GCL_DEV_BAD_RANGE);
        return;
    }
    const int nch = (int)((eos - bos + C - 1) / C);
    const int64_t row0 = p.chunk_offsets[n];
    if (nch > 0 && (row0 < 0 || row0 + nch > p.nt_max)) {
        if (tid == 0) status_set(p.status, GCL_DEV_BAD_RANGE);
        return;
    }
    const uint32_t sbase = smem_u32(smem);
    const int64_t KV = (int64_t)KD * VD;
    const int64_t state_base = ((int64_t)n * H + h) * KV;
    const int c0 = half * HV;

    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bar_tma[i], 1);
            mbar_init(&bar_ops[i], 1);
        }
        mbar_init(&bar_c1, 1);
        mbar_init(&bar_c23, 1);
        mbar_init(&bar_p, 1);
        mbar_init(&bar_sb, 1);
        mbar_init(&bar_w, 1);
        mbar_init(&bar_e, 1);
        s_err = 0;
        fence_barrier_init();
    }
    if (warp == 8) {
        tmem_alloc(&s_tmem, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;

    auto chunk_len = [&](int ic) -> int {
        const int64_t t0 = bos + (int64_t)ic * C;
        return (int)(eos - t0 < C ? eos - t0 : C);
    };

    if (!compute) {
        // ======================================================= issuer (warp 8, lane 0)
        if ((tid & 31) == 0) {
            const uint64_t dSB = smem_desc(sbase + Lay::oSB, 8192, 1024, kSwizzle128B);
            const uint64_t dET = smem_desc(sbase + Lay::oET, 8192, 1024, kSwizzle128B);
            const uint64_t dFT = smem_desc(sbase + Lay::oFT, 8192, 1024, kSwizzle128B);
            auto dK = [&](int st) {
                return smem_desc(sbase + st * Lay::kStage + Lay::oK, 8192, 1024, kSwizzle128B);
            };
            auto dKmaj = [&](uint32_t off) { return smem_desc(sbase + off, 16, 1024, kSwizzle128B); };
            auto issue_tma = [&](int ic) {
                const int st = ic & 1;
                const int t0 = (int)(bos + (int64_t)ic * C);
                const int unit = (int)((row0 + ic) * H + h);
                uint64_t *bar = &bar_tma[st];
                uint8_t *b = smem + st * Lay::kStage;
                mbar_arrive_expect_tx(bar, Lay::kTmaBytes);
                tma_load_3d(b + Lay::oK, &tm_k, 0, h, t0, bar);
                tma_load_3d(b + Lay::oK + 8192, &tm_k, 64, h, t0, bar);
                tma_load_3d(b + Lay::oWQ + 8192, &tm_q, 0, h, t0, bar);      // Q rows of [-W; Q]
                tma_load_3d(b + Lay::oWQ + 16384 + 8192, &tm_q, 64, h, t0, bar);
                tma_load_2d(b + Lay::oTL, &tm_tl, 0, unit * kTLRows, bar);
                tma_load_3d(b + Lay::oV, &tm_v, v0 & ~63, h, t0, bar);
                tma_load_2d(b + Lay::oF, &tm_f, 0, unit * kFRows, bar);
            };
            // P1: [W; .] = [T diag(bG); T diag(b)] K;  P2: [U; .] = [T diag(b); L] V
            auto issue_p = [&](int ic) {
                const int st = ic & 1;
                const uint32_t b = st * Lay::kStage;
                constexpr uint32_t id_w = idesc_bf16(128, 128, 0, 1);
                constexpr uint32_t id_v = idesc_bf16(128, VS, 0, 1);
                const uint64_t a1 = dKmaj(b + Lay::oTL), b1 = dK(st);
                const uint64_t a2 = dKmaj(b + Lay::oTL + 8192);
                const uint64_t b2 =
                    smem_desc(sbase + b + Lay::oV + (v0 & 63) * 2, 8192, 1024, kSwizzle128B);
#pragma unroll
                for (int s = 0; s < 4; ++s) mma_bf16(tmem, a1 + s * 2, b1 + s * 128, id_w, s > 0);
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    mma_bf16(tmem + tD2p + st * VS, a2 + s * 2, b2 + s * 128, id_v, s > 0);
                mma_commit(&bar_p);
            };
            if (nch > 0) issue_tma(0);
            if (nch > 1) issue_tma(1);
            if (nch > 0 && mbar_wait(&bar_ops[0], 0, &s_err, 7)) {
                tc_fence_after();
                issue_p(0);
            }
            for (int ic = 0; ic < nch && !s_err; ++ic) {
                const int st = ic & 1;
                const uint32_t sb = st * Lay::kStage;
                if (!mbar_wait(&bar_sb, ic & 1, &s_err, 8) || !mbar_wait(&bar_w, ic & 1, &s_err, 9)) break;
                tc_fence_after();
                {   // C1: [-W S; Q S] = [-W; Q] S
                    constexpr uint32_t id = idesc_bf16(128, VS, 0, 1);
                    const uint64_t a = dKmaj(sb + Lay::oWQ);
#pragma unroll
                    for (int s = 0; s < 8; ++s)
                        mma_bf16(tmem + tD2c, a + (s >> 2) * 1024 + (s & 3) * 2, dSB + s * 128, id, s > 0);
                    mma_commit(&bar_c1);
                }
                if (ic + 1 < nch) {
                    if (!mbar_wait(&bar_ops[(ic + 1) & 1], ((ic + 1) >> 1) & 1, &s_err, 10)) break;
                    tc_fence_after();
                    issue_p(ic + 1);
                }
                if (!mbar_wait(&bar_e, ic & 1, &s_err, 11)) break;
                tc_fence_after();
                {   // C2: K^T (f E);  C3: [T diag(b); L] E
                    constexpr uint32_t id_s = idesc_bf16(128, VS, 1, 1);
                    constexpr uint32_t id_o = idesc_bf16(128, VS, 0, 1);
                    const uint64_t a2 = dK(st), a3 = dKmaj(sb + Lay::oTL + 8192);
#pragma unroll
                    for (int s = 0; s < 4; ++s) mma_bf16(tmem + tD3, a2 + s * 128, dFT + s * 128, id_s, s > 0);
#pragma unroll
                    for (int s = 0; s < 4; ++s) mma_bf16(tmem + tD4, a3 + s * 2, dET + s * 128, id_o, s > 0);
                    mma_commit(&bar_c23);
                }
                if (ic + 2 < nch) {          // stage st is free once S, O(ic) are done
                    if (!mbar_wait(&bar_sb, (ic + 1) & 1, &s_err, 12)) break;
                    issue_tma(ic + 2);
                }
            }
        }
    } else {
        // ======================================================= compute (warps 0..7)
        auto st_mn8 = [&](uint32_t base, int k, int n0, const float *x) {
            uint4 pk;
            __nv_bfloat162 *pp = reinterpret_cast<__nv_bfloat162 *>(&pk);
#pragma unroll
            for (int e = 0; e < 4; ++e) pp[e] = __floats2bfloat162_rn(x[2 * e], x[2 * e + 1]);
            *reinterpret_cast<uint4 *>(smem + base + mn_sw128(k, n0)) = pk;
        };
        // hand-off to the issuer: every compute thread has fenced its writes
        auto handoff = [&](uint64_t *bar) {
            fence_async_smem();
            tc_fence_before();
            compute_barrier();
            if (tid == 0) mbar_arrive(bar);
        };
        // chunk ic's tiles have landed; K and V rows past the end of a partial chunk are
        // zeroed (they may hold the next sequence or NaN padding and enter the MMAs raw)
        auto land_chunk = [&](int ic) {
            const int st = ic & 1, len = chunk_len(ic);
            mbar_wait(&bar_tma[st], (ic >> 1) & 1, &s_err, 3);
            if (len < C) {
                uint8_t *kt = smem + st * Lay::kStage + Lay::oK;
                uint8_t *vt = smem + st * Lay::kStage + Lay::oV;
                const uint4 zero = make_uint4(0, 0, 0, 0);
                for (int t = tid; t < 3 * C * 8; t += kComputeThreads) {
                    const int r = (t >> 3) & 63, blk = t >> 9;
                    if (r >= len) {
                        uint8_t *base = blk < 2 ? kt + blk * 8192 : vt;
                        *reinterpret_cast<uint4 *>(base + r * 128 + (t & 7) * 16) = zero;
                    }
                }
            }
            handoff(&bar_ops[st]);
        };
        // -W (D_W lanes 0..63) into rows 0..63 of [-W; Q] of the chunk's stage
        auto write_w = [&](int ic) {
            mbar_wait(&bar_p, ic & 1, &s_err, 4);
            tc_fence_after();
            if (quarter < 2) {
                uint8_t *wq = smem + (ic & 1) * Lay::kStage + Lay::oWQ;
                const uint32_t rbase = (row >> 3) * 1024 + (row & 7) * 128;
                float w[64];
#pragma unroll
                for (int q = 0; q < 4; ++q) tmem_ld16(tmem + lane_off + half * 64 + q * 16, w + q * 16);
                tmem_ld_wait();
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const int key0 = half * 64 + q * 8;
                    uint4 pk;
                    __nv_bfloat162 *pp = reinterpret_cast<__nv_bfloat162 *>(&pk);
#pragma unroll
                    for (int e2 = 0; e2 < 4; ++e2)
                        pp[e2] = __floats2bfloat162_rn(-w[q * 8 + 2 * e2], -w[q * 8 + 2 * e2 + 1]);
                    const int cb = key0 >> 6, ch = (key0 & 63) >> 3;
                    *reinterpret_cast<uint4 *>(wq + cb * 16384 + rbase + ((ch ^ (row & 7)) << 4)) = pk;
                }
            }
            handoff(&bar_w);
        };

        float S[HV];
        {
            const float *src = (p.h0 && GCL_RANGE_IN_BOUNDS(state_base + (int64_t)row * VD + v0 + c0,
                                                            state_base + (int64_t)row * VD + v0 + c0 + HV - 1,
                                                            (int64_t)p.n_max * H * KV, p.status))
                                   ? p.h0 + state_base + (int64_t)row * VD + v0 + c0 : nullptr;
#pragma unroll
            for (int j = 0; j < HV; ++j) S[j] = src ? src[j] : 0.f;
#pragma unroll
            for (int j = 0; j < HV; j += 8) st_mn8(Lay::oSB, row, c0 + j, S + j);
        }
        handoff(&bar_sb);
        if (nch > 0) {
            land_chunk(0);
            write_w(0);
        }
        bool failed = false;
        for (int ic = 0; ic < nch; ++ic) {
            const int st = ic & 1, len = chunk_len(ic);
            const int64_t t0 = bos + (int64_t)ic * C;
            const float *fac = reinterpret_cast<const float *>(smem + st * Lay::kStage + Lay::oF);
            if (p.h_save &&
                GCL_RANGE_IN_BOUNDS(((row0 + ic) * H + h) * KV + (int64_t)row * VD + v0 + c0,
                                    ((row0 + ic) * H + h) * KV + (int64_t)row * VD + v0 + c0 + HV - 1,
                                    p.nt_max * H * KV, p.status)) {
                float *dst = p.h_save + ((row0 + ic) * H + h) * KV + (int64_t)row * VD + v0 + c0;
#pragma unroll
                for (int j = 0; j < HV; j += 4)
                    *reinterpret_cast<float4 *>(dst + j) = make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
            }
            if (ic + 1 < nch) land_chunk(ic + 1);          // while C1 runs
            // E = U - W S (rows 0..63) -> E and exp(g_c - g) E;  Q S (rows 64..127) kept
            mbar_wait(&bar_c1, ic & 1, &s_err, 5);
            tc_fence_after();
            float qs[HV];
            if (quarter < 2) {
                const float f = fac[row];
#pragma unroll
                for (int q = 0; q < HV / 8; ++q) {
                    float u[8], ws[8], e[8], fe[8];
                    tmem_ld8(tmem + lane_off + tD2p + st * VS + c0 + q * 8, u);
                    tmem_ld8(tmem + lane_off + tD2c + c0 + q * 8, ws);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        e[j] = u[j] + ws[j];
                        fe[j] = f * e[j];
                    }
                    st_mn8(Lay::oET, row, c0 + q * 8, e);
                    st_mn8(Lay::oFT, row, c0 + q * 8, fe);
                }
            } else {
#pragma unroll
                for (int q = 0; q < HV / 8; ++q) tmem_ld8(tmem + lane_off + tD2c + c0 + q * 8, qs + q * 8);
                tmem_ld_wait();
            }
            handoff(&bar_e);
            if (ic + 1 < nch) write_w(ic + 1);             // while C2/C3 run
            // S <- Gamma_c S + K^T (f E);  O = scale Gamma Q S + L E
            mbar_wait(&bar_c23, ic & 1, &s_err, 6);
            tc_fence_after();
            {
                const float GC = fac[2 * C];
#pragma unroll
                for (int q = 0; q < HV / 8; ++q) {
                    float d3[8];
                    tmem_ld8(tmem + lane_off + tD3 + c0 + q * 8, d3);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 8; ++j) S[q * 8 + j] = fmaf(GC, S[q * 8 + j], d3[j]);
                    st_mn8(Lay::oSB, row, c0 + q * 8, S + q * 8);
                }
                if (quarter >= 2) {
                    const int r = row - C;
                    float d4[HV];
#pragma unroll
                    for (int q = 0; q < HV / 8; ++q) tmem_ld8(tmem + lane_off + tD4 + c0 + q * 8, d4 + q * 8);
                    tmem_ld_wait();
                    if (r < len && p.o != nullptr &&
                        GCL_RANGE_IN_BOUNDS(((t0 + r) * H + h) * (int64_t)VD + v0 + c0,
                                            ((t0 + r) * H + h) * (int64_t)VD + v0 + c0 + HV - 1,
                                            p.t_max * H * (int64_t)VD, p.status)) {
                        const float fq = fac[C + r];
                        __nv_bfloat16 *dst = p.o + ((t0 + r) * H + h) * (int64_t)VD + v0 + c0;
#pragma unroll
                        for (int j = 0; j < HV; j += 8) {
                            uint4 pk;
                            __nv_bfloat162 *pp = reinterpret_cast<__nv_bfloat162 *>(&pk);
#pragma unroll
                            for (int e2 = 0; e2 < 4; ++e2)
                                pp[e2] = __floats2bfloat162_rn(fmaf(fq, qs[j + 2 * e2], d4[j + 2 * e2]),
                                                               fmaf(fq, qs[j + 2 * e2 + 1], d4[j + 2 * e2 + 1]));
                            *reinterpret_cast<uint4 *>(dst + j) = pk;
                        }
                    }
                }
            }
            handoff(&bar_sb);
            // the issuer may record a timeout at any moment: decide on it uniformly
            if (compute_barrier_or(*reinterpret_cast<volatile int *>(&s_err) != 0)) {
                failed = true;
                break;
            }
        }
        if (!failed && p.ht &&
            GCL_RANGE_IN_BOUNDS(state_base + (int64_t)row * VD + v0 + c0,
                                state_base + (int64_t)row * VD + v0 + c0 + HV - 1,
                                (int64_t)p.n_max * H * KV, p.status)) {
            float *dst = p.ht + state_base + (int64_t)row * VD + v0 + c0;
#pragma unroll
            for (int j = 0; j < HV; j += 4)
                *reinterpret_cast<float4 *>(dst + j) = make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 8) tmem_dealloc(tmem, kTmemCols);
    if (tid == 0 && s_err != 0) status_set(p.status, GCL_DEV_WAIT_TIMEOUT);
}

// ============================================================================ host
template <int VS>
cudaError_t launch_chain(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                         const CUtensorMap &mtl, const CUtensorMap &mf, const ChainParams &cp,
                         int n_split, int H, int n_max, cudaStream_t s) {
    auto kern = tc_chain_kernel<VS>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)ChainLayout::bytes);
    if (e != cudaSuccess) return e;
    kern<<<dim3(n_split, H, n_max), kChainThreads, ChainLayout::bytes, s>>>(mq, mk, mv, mtl, mf, cp);
    return cudaGetLastError();
}

}  // namespace

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }
    return fn;
}

bool make_tensor_map(CUtensorMap *m, const void *ptr, int rank, const cuuint64_t *dims,
                     const cuuint64_t *strides, const cuuint32_t *box, CUtensorMapSwizzle sw,
                     CUtensorMapDataType dt) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, dt, rank, const_cast<void *>(ptr), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// bf16 inputs for GDN and KDA; fp16 inputs for the GDN forward (the transition and fused
// plans, with every MMA operand and record in fp16).  The backward takes bf16 only
// (bwd_tc_supported).
bool fwd_tc_supported(int variant, int dtype, int K, int V, int bt) {
    const bool type_ok = dtype == GCL_BF16 || (dtype == GCL_F16 && variant == kGDN);
    return (variant == kGDN || variant == kKDA) && type_ok && K == KD && V == VD && bt == kChunk;
}
bool bwd_tc_supported(int variant, int dtype, int K, int V, int bt) {
    return dtype == GCL_BF16 && fwd_tc_supported(variant, dtype, K, V, bt);
}

size_t fwd_tc_workspace_bytes(int64_t nt_max, int H) {
    return (size_t)nt_max * H * (kTLRows * C * sizeof(__nv_bfloat16) + kFRows * C * sizeof(float));
}

// Value-column split: the most CTAs per head that still fit one wave on the GPU,
// between 2 (VS = 64, the shared-memory limit) and 8 (VS = 16).
int fwd_tc_split(int n_max, int H) {
    const int sms = num_sms();
    int split = 2;
    for (int cand : {4, 8})
        if ((int64_t)n_max * H * cand <= sms) split = cand;
    return split;
}

bool fwd_tc_prefers_transition(int n_max, int H) { return fwd_tc_split(n_max, H) >= 4; }

// The transition plan runs for few units (split 4 or 8: a shorter serial step) and for every
// training forward (h_save: its records are what the backward's sweep reads, so the backward
// can take them instead of recomputing them), whenever the workspace holds the records.  KDA
// has the transition plan only.
bool fwd_tc_runs_transition(int variant, int n_max, int H, bool h_save, size_t ws_bytes, int64_t nt_max,
                            int dtype) {
    if (variant == kKDA || dtype == GCL_F16) return true;    // (the W form is bf16 only)
    return (fwd_tc_prefers_transition(n_max, H) || h_save) && ws_bytes >= fwd_tc_t_workspace_bytes(nt_max, H);
}

int fwd_tc_plan(int variant, int n_max, int H, bool h_save, size_t ws_bytes, int64_t nt_max, int dtype) {
    if (fwd_tc_runs_fused(variant, n_max, H, h_save, ws_bytes, nt_max)) return GCL_PLAN_FUSED;
    if (fwd_tc_runs_transition(variant, n_max, H, h_save, ws_bytes, nt_max, dtype)) {
        const size_t rec = fwd_tc_t_workspace_bytes(nt_max, H);
        const size_t seg = fwd_seg_workspace_bytes(nt_max, n_max, H);
        return seg > 0 && ws_bytes >= rec + seg ? GCL_PLAN_SEGMENTED : GCL_PLAN_TRANSITION;
    }
    return GCL_PLAN_W_FORM;
}

cudaError_t launch_fwd_tc(const FwdParams &p, int variant, cudaStream_t s) {
    const int H = p.H;
    if (fwd_tc_runs_fused(variant, p.n_max, H, p.h_save != nullptr, p.workspace_bytes, p.nt_max))
        return launch_fwd_fused(p, s);
    if (variant == kKDA) {   // KDA has the transition form only
        if (p.workspace_bytes < fwd_tc_t_workspace_bytes(p.nt_max, H)) return cudaErrorInvalidValue;
        return launch_fwd_tc_kda(p, fwd_tc_split(p.n_max, H), s);
    }
    if (fwd_tc_runs_transition(variant, p.n_max, H, p.h_save != nullptr, p.workspace_bytes, p.nt_max,
                               p.dtype)) {
        if (p.workspace_bytes < fwd_tc_t_workspace_bytes(p.nt_max, H)) return cudaErrorInvalidValue;
        return launch_fwd_tc_t(p, fwd_tc_split(p.n_max, H), s);
    }
    const int64_t units = p.nt_max * H;              // chunk-head slots of the workspace
    __nv_bfloat16 *tl = static_cast<__nv_bfloat16 *>(p.workspace);
    float *fac = reinterpret_cast<float *>(tl + (size_t)units * kTLRows * C);
    CUtensorMap mq, mk, mv, mtl, mf;
    const cuuint64_t dqk[3] = {(cuuint64_t)KD, (cuuint64_t)H, (cuuint64_t)p.t_max};
    const cuuint64_t sqk[2] = {(cuuint64_t)KD * 2, (cuuint64_t)H * KD * 2};
    const cuuint32_t b64[3] = {64, 1, 64};
    const cuuint64_t dv[3] = {(cuuint64_t)VD, (cuuint64_t)H, (cuuint64_t)p.t_max};
    const cuuint64_t sv[2] = {(cuuint64_t)VD * 2, (cuuint64_t)H * VD * 2};
    const cuuint64_t dtl[2] = {(cuuint64_t)C, (cuuint64_t)units * kTLRows};
    const cuuint64_t stl[1] = {(cuuint64_t)C * 2};
    const cuuint32_t btl[2] = {64, (cuuint32_t)kTLRows};
    const cuuint64_t df[2] = {(cuuint64_t)C, (cuuint64_t)units * kFRows};
    const cuuint64_t sf[1] = {(cuuint64_t)C * 4};
    const cuuint32_t bf[2] = {64, (cuuint32_t)kFRows};
    if (!make_tensor_map(&mq, p.q, 3, dqk, sqk, b64, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tensor_map(&mk, p.k, 3, dqk, sqk, b64, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tensor_map(&mv, p.v, 3, dv, sv, b64, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tensor_map(&mtl, tl, 2, dtl, stl, btl, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tensor_map(&mf, fac, 2, df, sf, bf, CU_TENSOR_MAP_SWIZZLE_NONE,
                         CU_TENSOR_MAP_DATA_TYPE_FLOAT32))
        return cudaErrorInvalidValue;

    PrepParams pp{};
    pp.chunk_indices = p.chunk_indices;
    pp.cu = p.cu_seqlens;
    pp.g = p.g;
    pp.beta = static_cast<const __nv_bfloat16 *>(p.beta);
    pp.tl = tl;
    pp.fac = fac;
    pp.status = p.dev_status;
    pp.t_max = p.t_max;
    pp.n_max = p.n_max;
    pp.H = H;
    pp.scale = p.scale;
    cudaError_t e = cudaFuncSetAttribute(tc_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kPrepSmem);
    if (e != cudaSuccess) return e;
    tc_prep_kernel<<<dim3((unsigned)p.nt_max, H), kThreads, kPrepSmem, s>>>(mq, mk, pp);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;

    ChainParams cp{};
    cp.cu = p.cu_seqlens;
    cp.chunk_offsets = p.chunk_offsets;
    cp.seq_order = p.seq_order;
    cp.h0 = p.h0;
    cp.o = static_cast<__nv_bfloat16 *>(p.o);
    cp.ht = p.ht;
    cp.h_save = p.h_save;
    cp.status = p.dev_status;
    cp.t_max = p.t_max;
    cp.nt_max = p.nt_max;
    cp.n_max = p.n_max;
    cp.H = H;
    const int split = fwd_tc_split(p.n_max, H);
    switch (VD / split) {
        case 16: return launch_chain<16>(mq, mk, mv, mtl, mf, cp, split, H, p.n_max, s);
        case 32: return launch_chain<32>(mq, mk, mv, mtl, mf, cp, split, H, p.n_max, s);
        default: return launch_chain<64>(mq, mk, mv, mtl, mf, cp, split, H, p.n_max, s);
    }
}

}  // namespace gcl
