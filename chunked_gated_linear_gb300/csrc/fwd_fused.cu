// fwd_fused.cu -- the fused tensor-core GDN chunk forward: one CTA per (sequence, head)
// carries the whole Map-Reduce-Map of its chunks on chip (bf16 or fp16 inputs, d_k = d_v = 128,
// chunk 64; every MMA operand in the input type, "bf16" below standing for either).  Nothing but q, k, v, g, beta, h0 is read and nothing but o, ht (and h_save)
// is written: no per-chunk records go through HBM.
//
// HA-NPU paper "Empowering Hybrid Attention Models on NPUs": section 2.1 (Map-Reduce-Map),
// section 4 (head-per-core mapping with every intermediate kept on the core, the first
// scheduling tier when there are at least as many heads as cores), section 5 (GEMM-first
// grouping: KS and QS before the inverse is applied; chunk-first in-place state update).
// FLA RFC "[RFC] Add Graph Capture Support for FLA Prefill and Training Paths on Ascend NPUs",
// "Core design": a fixed grid over the N_max sequence slots; a zero-length slot passes h0 to ht.
//
// Per chunk, with gamma the in-chunk cumsum of g, Gamma = exp(gamma), Gamma_c = Gamma at the
// last row, f = exp(gamma_c - gamma), D[r][i] = exp(gamma_r - gamma_i):
//   A = beta D o (K K^T) (strict),  T = (I + A)^-1,  L = scale D o (Q K^T) (inclusive)
//   R = diag(beta) (V - diag(Gamma) K S),  E = T R          (= U - W S, GEMM-first)
//   O = scale diag(Gamma) Q S + L E,        S' = Gamma_c S + (diag(f) K)^T E.
// The state is held transposed: thread lane v owns row v of S^T (fp32 registers, the key
// columns split over two warps); its bf16 copy sits in TMEM as the A operand of S^T K^T and
// S^T Q^T, so every state-side product has the value index on the 128 MMA rows:
//   MMA1  [K; Q] K^T          -> D1 [128 x 64]   (A = [K; Q] smem, B = K smem)
//   MMA2  S^T [K; Q]^T        -> [X | Y] [128 x 128]  (A = S^T TMEM, B = [K; Q] smem)
//         (Y is then scaled to scale diag(Gamma) Q S in place, giving O^T's first term)
//   MMA3  R^T T^T             -> E^T [128 x 64]  (A = R^T TMEM,   B = T smem)
//   MMA4  (E^T diag f) K      -> dS^T [128x128]  (A TMEM,          B = K MN-major smem)
//   MMA5  O^T += E^T L^T                         (A = E^T TMEM,   B = L smem)
// The triangular solve runs in fp32 on the CUDA cores of warps 0..3 while warps 4..7 form R;
// one lane of warp 4 issues every copy and MMA, and warp 5 forms the next chunk's gate vectors
// (double-buffered) after its share of R.  Two CTAs share an SM (about 100 KB of shared memory
// and 256 TMEM columns each), so one CTA's MMAs, copies and waits overlap the other's CUDA-core
// phases.  Rows past the end of a sequence are selected to zero in every
// operand the threads build and zeroed in the K tile, so NaN padding never reaches an MMA.
#include <cudaTypedefs.h>

#include "gcl_internal.cuh"
#include "op16.cuh"
#include "tc_ptx.cuh"
#include "tc_solve.cuh"

namespace gcl {
namespace {

using namespace tc;
constexpr int C = 64;
constexpr int KD = 128;
constexpr int VD = 128;
constexpr int kThreads = 256;
constexpr int kIssuer = 128;      // lane 0 of warp 4
constexpr int kGateWarp = 5;      // forms the gate vectors, one chunk ahead

struct FusedParams {
    const int32_t *cu, *chunk_offsets, *seq_order;
    const float *g;
    const void *beta;             // [t_max, H] of the input type
    const float *h0;
    void *o;                      // [t_max, H, V] of the input type
    float *ht, *h_save;
    int32_t *status;
    int64_t t_max, nt_max;
    int32_t n_max, H;
    float scale;
};

// Shared memory (offsets from a 1024-byte aligned base).
struct FusedLayout {
    static constexpr uint32_t oKQ = 0;                 // [2 key blocks][K rows 0..63 | Q rows 64..127][128 B]
    static constexpr uint32_t oV = 32768;              // [2 value blocks][64 rows][128 B]
    static constexpr uint32_t oT = oV + 16384;         // T bf16 [64 x 64], K-major, 128-byte swizzle
    static constexpr uint32_t oL = oT + 8192;          // L bf16 [64 x 64]
    static constexpr uint32_t oA = oL + 8192;          // solve: A fp32 [64][kSolveLD]
    static constexpr uint32_t oTf = oA + 64 * kSolveLD * 4;   // solve: T fp32
    static constexpr uint32_t oO = oA;                 // O staging [64][kOLD] bf16, after the solve
    static constexpr uint32_t total = oTf + 64 * kSolveLD * 4;
    static constexpr uint32_t bytes = total + 1024;    // + alignment slack
};
constexpr int kOLD = 136;                              // O staging row stride (bf16 elements)
static_assert(64 * kOLD * 2 <= 2 * 64 * kSolveLD * 4, "O staging fits in the solve buffers");
static_assert(FusedLayout::bytes <= 110 * 1024, "two CTAs per SM");

// TMEM columns (256 per CTA).  Phases of one chunk reuse them:
//   S^T bf16 [0, 64) until MMA2 completes; then the fp32 state slice of warps 0..3 while they
//   run the solve (taken back while MMA3 runs); then D4 (dS^T) [0, 128)
//   X = (K S)^T [64, 128) until R is formed, then E^T (MMA3) [64, 128)
//   Y = (Q S)^T [128, 192): MMA2, scaled in place, then MMA5 accumulates onto it (O^T)
//   D1 [192, 256) until the A / L epilogue; then R^T bf16 [192, 224), then E^T f bf16 [192, 224);
//   E^T bf16 [224, 256)
constexpr uint32_t cS = 0, cD4 = 0, cX = 64, cE32 = 64, cO = 128, cD1 = 192, cR = 192, cEF = 192,
                   cEB = 224;
constexpr uint32_t kTmemCols = 256;


__device__ __forceinline__ float warp_incl_scan(float x) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, x, d);
        if (lane >= d) x += y;
    }
    return x;
}

// T: the input type (bf16, or fp16), which every MMA operand the kernel forms shares (one
// kind::f16 instruction takes A and B of the same type).
template <typename T>
__global__ void __launch_bounds__(kThreads, 2)
tc_fused_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, FusedParams p) {
    using Lay = FusedLayout;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    __shared__ uint64_t bar_kq, bar_v, bar_m1, bar_m2, bar_m3, bar_m45;
    __shared__ uint32_t s_tmem;
    __shared__ int s_err;
    // per-chunk gate vectors, double-buffered by chunk parity (the next chunk's are formed
    // while the current chunk's are still read)
    __shared__ __align__(16) float sGb[2][C], sBb[2][C], sGamb[2][C], sFb[2][C], sF2b[2][4 * C];

    if (status_blocks_cta(p.status)) return;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3, half = warp >> 2;
    const int m = quarter * 32 + lane;                         // TMEM lane: value row v
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const int h = blockIdx.x, z = blockIdx.y, H = p.H;
    const int n = (p.seq_order && GCL_IN_BOUNDS(z, p.n_max, p.status)) ? p.seq_order[z] : z;
    if (n < 0 || n >= p.n_max) {
        if (tid == 0) status_set(p.status, GCL_DEV_BAD_RANGE);
        return;
    }
    if (!GCL_RANGE_IN_BOUNDS(n, n + 1, (int64_t)p.n_max + 1, p.status)) return;
    const int64_t bos = p.cu[n], eos = p.cu[n + 1];
    if (bos < 0 || eos < bos || eos > p.t_max) {
        if (tid == 0) status_set(p.status, GCL_DEV_BAD_RANGE);
        return;
    }
    const int nch = (int)((eos - bos + C - 1) / C);
    const int64_t row0 = p.chunk_offsets ? p.chunk_offsets[n] : 0;
    if (p.h_save && nch > 0 && (row0 < 0 || row0 + nch > p.nt_max)) {
        if (tid == 0) status_set(p.status, GCL_DEV_BAD_RANGE);
        return;
    }
    const int64_t KV = (int64_t)KD * VD;
    const int64_t state_base = ((int64_t)n * H + h) * KV;
    const int k0 = half * 64;                                  // this thread's key columns
    // [first, last] element of this thread's strided state column (h0, ht), and the sizes
    const int64_t st_lo = state_base + (int64_t)k0 * VD + m, st_hi = st_lo + 63 * (int64_t)VD;
    const int64_t n_state = (int64_t)p.n_max * H * KV;

    // S^T row m, keys k0 .. k0 + 63 (S[k][v] at h0[k * V + v])
    float S[64];
    {
        const float *src = (p.h0 && GCL_RANGE_IN_BOUNDS(st_lo, st_hi, n_state, p.status))
                               ? p.h0 + state_base + (int64_t)k0 * VD + m : nullptr;
#pragma unroll
        for (int j = 0; j < 64; ++j) S[j] = src ? src[(int64_t)j * VD] : 0.f;
    }
    if (nch == 0) {                                            // zero-length slot: ht = h0
        if (p.ht && GCL_RANGE_IN_BOUNDS(st_lo, st_hi, n_state, p.status)) {
            float *dst = p.ht + state_base + (int64_t)k0 * VD + m;
#pragma unroll
            for (int j = 0; j < 64; ++j) dst[(int64_t)j * VD] = S[j];
        }
        return;
    }

    if (tid == 0) {
        mbar_init(&bar_kq, 1);
        mbar_init(&bar_v, 1);
        mbar_init(&bar_m1, 1);
        mbar_init(&bar_m2, 1);
        mbar_init(&bar_m3, 1);
        mbar_init(&bar_m45, 1);
        s_err = 0;
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc(&s_tmem, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    const uint32_t sbase = smem_u32(smem);

    auto chunk_t0 = [&](int ic) -> int64_t { return bos + (int64_t)ic * C; };
    auto chunk_len = [&](int ic) -> int {
        const int64_t t0 = chunk_t0(ic);
        return (int)(eos - t0 < C ? eos - t0 : C);
    };
    auto issue_kq = [&](int ic) {
        const int t0 = (int)chunk_t0(ic);
        (void)GCL_IN_BOUNDS(t0, p.t_max, p.status);           // (rows past t_max read zeros)
        mbar_arrive_expect_tx(&bar_kq, 32768);
        for (int cb = 0; cb < 2; ++cb) {
            tma_load_3d(smem + Lay::oKQ + cb * 16384, &tm_k, cb * 64, h, t0, &bar_kq);
            tma_load_3d(smem + Lay::oKQ + cb * 16384 + 8192, &tm_q, cb * 64, h, t0, &bar_kq);
        }
    };
    auto issue_v = [&](int ic) {
        const int t0 = (int)chunk_t0(ic);
        (void)GCL_IN_BOUNDS(t0, p.t_max, p.status);
        mbar_arrive_expect_tx(&bar_v, 16384);
        for (int cb = 0; cb < 2; ++cb)
            tma_load_3d(smem + Lay::oV + cb * 8192, &tm_v, cb * 64, h, t0, &bar_v);
    };
    // S^T (bf16) of this thread's lane and keys into TMEM columns cS + half * 32 ..
    auto store_state_bf16 = [&]() {
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            uint32_t pk[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) pk[j] = Op16<T>::pack2(S[q * 32 + 2 * j], S[q * 32 + 2 * j + 1]);
            tmem_st16_b32(tmem + lane_off + cS + half * 32 + q * 16, pk);
        }
        tmem_st_wait();
    };

    store_state_bf16();
    // one thread issues every copy and MMA: a lane of warp 4, whose warps form R while
    // warps 0..3 run the triangular solve (the longer of the two)
    const bool issuer = tid == kIssuer;
    if (issuer) {
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        issue_kq(0);
        issue_v(0);
    }
    // Gates and betas, rows 2l and 2l + 1 in lane l of warp kGateWarp, loaded one chunk ahead;
    // that warp forms each chunk's gate vectors one chunk ahead too (after its share of R),
    // so no barrier of the chunk waits for them.
    float g_next[2] = {0.f, 0.f}, b_next[2] = {0.f, 0.f};
    auto load_gates = [&](int ic) {
        const int len1 = chunk_len(ic);
        const int64_t t = chunk_t0(ic);
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int r = 2 * lane + e;
            const bool ok = r < len1 && GCL_IN_BOUNDS((t + r) * H + h, p.t_max * H, p.status);
            g_next[e] = ok ? p.g[(t + r) * H + h] : 0.f;
            b_next[e] = ok ? Op16<T>::to_float(static_cast<const T *>(p.beta)[(t + r) * H + h]) : 0.f;
        }
    };
    // gamma (inclusive cumsum; rows past the end have g = 0), beta, Gamma = exp(gamma),
    // f = exp(gamma_c - gamma), and the cross-block decay factors
    // F2[b][c] = exp(gamma_{16 b} - gamma_c) for c < 16 b, of chunk ic into buffer ic & 1
    auto form_gates = [&](int ic) {
        const int len1 = chunk_len(ic), gb = ic & 1;
        float *G = sGb[gb];
        const float a1 = g_next[0] + g_next[1];
        const float x = warp_incl_scan(a1);                    // through row 2l + 1
        const float g1 = x, g0 = x - g_next[1];
        const float gc = __shfl_sync(0xffffffffu, x, 31);
        const int r0 = 2 * lane;
        G[r0] = g0;
        G[r0 + 1] = g1;
        sBb[gb][r0] = b_next[0];
        sBb[gb][r0 + 1] = b_next[1];
        sGamb[gb][r0] = r0 < len1 ? __expf(g0) : 0.f;
        sGamb[gb][r0 + 1] = r0 + 1 < len1 ? __expf(g1) : 0.f;
        sFb[gb][r0] = r0 < len1 ? __expf(gc - g0) : 0.f;
        sFb[gb][r0 + 1] = r0 + 1 < len1 ? __expf(gc - g1) : 0.f;
        __syncwarp();
#pragma unroll
        for (int b = 1; b < 4; ++b) {
            const float rho = G[16 * b];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int c = r0 + e;
                sF2b[gb][b * C + c] = __expf(c < 16 * b ? rho - G[c] : 0.f);
            }
        }
    };
    if (warp == kGateWarp) {
        load_gates(0);
        form_gates(0);
        if (nch > 1) load_gates(1);
    }

    // T and L (bf16) start as zeros: the blocks above their block diagonal are never written
    // again (T is zero there, L too), so the epilogues and the T write-out skip them
    for (int e = tid; e < (8192 + 8192) / 16; e += kThreads)
        *reinterpret_cast<uint4 *>(smem + Lay::oT + e * 16) = make_uint4(0, 0, 0, 0);

    float *sAf = reinterpret_cast<float *>(smem + Lay::oA);
    float *sTf = reinterpret_cast<float *>(smem + Lay::oTf);
    T *sO = reinterpret_cast<T *>(smem + Lay::oO);
    // the valid rows of a chunk's O from the staging tile, 16 threads x 16 bytes per row; run
    // during the next chunk's first MMA wait (the tile lives in the solve buffers, which that
    // chunk's A / L epilogue rewrites only after the wait), or after the last chunk
    auto store_o = [&](int64_t ot0, int olen) {
        if (p.o == nullptr) return;
        const int rsub = tid >> 4, cc = (tid & 15) * 8;
        for (int r = rsub; r < olen; r += kThreads / 16) {
            const int64_t oi = ((ot0 + r) * H + h) * (int64_t)VD + cc;
            if (!GCL_RANGE_IN_BOUNDS(oi, oi + 7, p.t_max * H * VD, p.status) ||
                !GCL_RANGE_IN_BOUNDS(r * kOLD + cc, r * kOLD + cc + 7, C * kOLD, p.status))
                continue;
            const uint4 val = *reinterpret_cast<const uint4 *>(sO + r * kOLD + cc);
            *reinterpret_cast<uint4 *>(static_cast<T *>(p.o) + ((ot0 + r) * H + h) * (int64_t)VD + cc) = val;
        }
    };
    int64_t prev_t0 = 0;
    int prev_len = 0;                  // rows of the previous chunk's O still staged

    for (int ic = 0; ic < nch; ++ic) {
        const int len = chunk_len(ic);
        const int64_t t0 = chunk_t0(ic);
        const uint32_t ph = ic & 1;
        const int gb = ic & 1;
        const float *sG = sGb[gb], *sB = sBb[gb], *sGam = sGamb[gb], *sF = sFb[gb], *sF2 = sF2b[gb];
        // ---- the chunk's K, Q, V tiles; K rows past the end are zeroed (they enter MMA1 and
        // MMA4 raw and may hold the next sequence or NaN padding)
        mbar_wait(&bar_kq, ph, &s_err, 1);
        mbar_wait(&bar_v, ph, &s_err, 2);
        if (len < C) {
            const uint4 zero = make_uint4(0, 0, 0, 0);
            for (int e = tid; e < 2 * C * 8; e += kThreads) {
                const int cb = e >> 9, r = (e >> 3) & 63, j = e & 7;
                if (r >= len) *reinterpret_cast<uint4 *>(smem + Lay::oKQ + cb * 16384 + r * 128 + j * 16) = zero;
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (issuer) {
            // MMA1: D1 = [K; Q] K^T (M = 128, N = 64, K = 128)
            constexpr uint32_t id1 = idesc_f16kind(128, 64, 0, 0, Op16<T>::fmt);
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                const uint32_t off = (s >> 2) * 16384 + (s & 3) * 32;
                const uint64_t dkq = smem_desc(sbase + Lay::oKQ + off, 16, 1024, kSwizzle128B);
                mma_bf16(tmem + cD1, dkq, dkq, id1, s > 0);
            }
            mma_commit(&bar_m1);
            // MMA2: [X | Y] = S^T [K; Q]^T (N = 128): X = (K S)^T, Y = (Q S)^T
            constexpr uint32_t id2 = idesc_f16kind(128, 128, 0, 0, Op16<T>::fmt);
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                const uint32_t off = (s >> 2) * 16384 + (s & 3) * 32;
                mma_bf16_ta(tmem + cX, tmem + cS + s * 8,
                            smem_desc(sbase + Lay::oKQ + off, 16, 1024, kSwizzle128B), id2, s > 0);
            }
            mma_commit(&bar_m2);
        }
        store_o(prev_t0, prev_len);                         // the previous chunk's O
        __syncthreads();                                    // read before the A / L epilogue
        mbar_wait(&bar_m1, ph, &s_err, 3);
        tc_fence_after();
        // ---- A (fp32, for the solve) and L (bf16) from D1, with the decay
        // D[r][c] = exp(gamma_r - gamma_c): inside a 16-row block one exponential per pair; for
        // c in an earlier block, exp(gamma_r - gamma_{16 b}) F2[b][c] (both factors <= 1, so
        // nothing overflows; their product underflows only where the decay itself does).
        // (warps whose rows 0..31 meet columns 32..63 only, all above the diagonal, skip it)
        if (half == 0 || (quarter & 1) == 1) {
            const int r = m & 63, br = r >> 4;
            const bool live = r < len;
            const float gr = sG[r];
            const float f1 = __expf(gr - sG[16 * br]);
            const float rowf = quarter < 2 ? sB[r] : p.scale;      // beta_r (A) or scale (L)
#pragma unroll
            for (int cb = 0; cb < 2; ++cb) {          // the thread's two 16-column blocks
                const int c0 = half * 32 + cb * 16, bc = c0 >> 4;
                float d[16];
                tmem_ld16(tmem + lane_off + cD1 + c0, d);
                tmem_ld_wait();
                float dec[16];
                if (bc < br) {
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        dec[j] = GCL_IN_BOUNDS(br * C + c0 + j, 4 * C, p.status) ? f1 * sF2[br * C + c0 + j] : 0.f;
                } else if (bc == br) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) dec[j] = __expf(c0 + j <= r ? gr - sG[c0 + j] : 0.f);
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j) dec[j] = 0.f;
                }
                if (quarter < 2) {                             // A row r = m: strictly lower
#pragma unroll
                    for (int j = 0; j < 16; j += 4) {
                        float a[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            a[e] = (live && c0 + j + e < r) ? rowf * dec[j + e] * d[j + e] : 0.f;
                        if (GCL_RANGE_IN_BOUNDS(r * kSolveLD + c0 + j, r * kSolveLD + c0 + j + 3, C * kSolveLD, p.status))
                            *reinterpret_cast<float4 *>(sAf + r * kSolveLD + c0 + j) = make_float4(a[0], a[1], a[2], a[3]);
                    }
                } else {                                       // L row r = m - 64: inclusive
#pragma unroll
                    for (int j = 0; j < 16; j += 8) {
                        uint4 pk;
                        uint32_t *pw = reinterpret_cast<uint32_t *>(&pk);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int c = c0 + j + 2 * e;
                            const float l0 = (live && c <= r) ? rowf * dec[j + 2 * e] * d[j + 2 * e] : 0.f;
                            const float l1 = (live && c + 1 <= r) ? rowf * dec[j + 2 * e + 1] * d[j + 2 * e + 1] : 0.f;
                            pw[e] = Op16<T>::pack2(l0, l1);
                        }
                        if (GCL_RANGE_IN_BOUNDS(sw128_offset(C, r, c0 + j), sw128_offset(C, r, c0 + j) + 15, 8192, p.status))
                            *reinterpret_cast<uint4 *>(smem + Lay::oL + sw128_offset(C, r, c0 + j)) = pk;
                    }
                }
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (warp < 4) {
            // ---- T = (I + A)^-1 (fp32) on warps 0..3, then bf16 rows (zeros above the diagonal)
            // the state slice of warps 0..3 waits in TMEM columns [0, 64) (its bf16 copy there
            // is no longer read once MMA2 completes), so the solve has the registers
            mbar_wait(&bar_m2, ph, &s_err, 6);
            tc_fence_after();
#pragma unroll
            for (int q = 0; q < 4; ++q) tmem_st16(tmem + lane_off + cS + q * 16, S + q * 16);
            tmem_st_wait();
            solve_unit_lower64_r32<128, 1>(sAf, sTf);
            const int r = tid >> 1, cq = (tid & 1) * 32;
#pragma unroll
            for (int j = 0; j < 32; j += 8) {
                if (cq + j > r) continue;                  // all above the diagonal: zeros kept
                uint4 pk;
                uint32_t *pw = reinterpret_cast<uint32_t *>(&pk);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int c = cq + j + 2 * e;
                    pw[e] = Op16<T>::pack2(c <= r ? sTf[r * kSolveLD + c] : 0.f,
                                      c + 1 <= r ? sTf[r * kSolveLD + c + 1] : 0.f);
                }
                if (GCL_RANGE_IN_BOUNDS(sw128_offset(C, r, cq + j), sw128_offset(C, r, cq + j) + 15, 8192, p.status))
                    *reinterpret_cast<uint4 *>(smem + Lay::oT + sw128_offset(C, r, cq + j)) = pk;
            }
            // (the parked state slice comes back during MMA3, which does not touch its columns)
        } else {
            // ---- R^T[v][r] = beta_r (V[r][v] - Gamma_r X[v][r]) -> bf16 A operand in TMEM,
            // lane v = m, all 64 rows r, on warps 4..7
            mbar_wait(&bar_m2, ph, &s_err, 6);
            tc_fence_after();
            const int v = m, vb = v >> 6, vc = v & 63;
            const uint8_t *vcol = smem + Lay::oV + vb * 8192 + (vc & 7) * 2;
#pragma unroll
            for (int hh = 0; hh < 4; ++hh) {
                float x[16];
                tmem_ld16(tmem + lane_off + cX + hh * 16, x);
                tmem_ld_wait();
                uint32_t pk[8];
#pragma unroll
                for (int j = 0; j < 16; j += 4) {
                    const int r0 = hh * 16 + j;
                    const float4 b4 = *reinterpret_cast<const float4 *>(sB + r0);
                    const float4 g4 = *reinterpret_cast<const float4 *>(sGam + r0);
                    const float bb[4] = {b4.x, b4.y, b4.z, b4.w}, gg[4] = {g4.x, g4.y, g4.z, g4.w};
                    float rr[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int r = r0 + e;
                        const int voff = vb * 8192 + (vc & 7) * 2 + (r >> 3) * 1024 + (r & 7) * 128 +
                                         ((((vc >> 3) ^ (r & 7))) << 4);
                        const float vv = GCL_IN_BOUNDS(voff, 16384, p.status)
                                             ? Op16<T>::to_float(*reinterpret_cast<const T *>(
                                                   vcol + (r >> 3) * 1024 + (r & 7) * 128 + ((((vc >> 3) ^ (r & 7))) << 4)))
                                             : 0.f;
                        rr[e] = r < len ? bb[e] * (vv - gg[e] * x[j + e]) : 0.f;
                    }
                    pk[j >> 1] = Op16<T>::pack2(rr[0], rr[1]);
                    pk[(j >> 1) + 1] = Op16<T>::pack2(rr[2], rr[3]);
                }
                tmem_st8_b32(tmem + lane_off + cR + hh * 8, pk);
            }
            tmem_st_wait();
            if (warp == kGateWarp && ic + 1 < nch) {      // the next chunk's gate vectors
                form_gates(ic + 1);
                if (ic + 2 < nch) load_gates(ic + 2);
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (issuer) {
            // MMA3: E^T = R^T T^T (M = 128, N = 64, K = 64)
            constexpr uint32_t id = idesc_f16kind(128, 64, 0, 0, Op16<T>::fmt);
#pragma unroll
            for (int s = 0; s < 4; ++s)
                mma_bf16_ta(tmem + cE32, tmem + cR + s * 8,
                            smem_desc(sbase + Lay::oT + s * 32, 16, 1024, kSwizzle128B), id, s > 0);
            mma_commit(&bar_m3);
            if (ic + 1 < nch) issue_v(ic + 1);              // the V tile is no longer read
        }
        if (warp < 4) {                                     // the state slice parked for the solve
#pragma unroll
            for (int q = 0; q < 4; ++q) tmem_ld16(tmem + lane_off + cS + q * 16, S + q * 16);
            tmem_ld_wait();
        }
        mbar_wait(&bar_m3, ph, &s_err, 4);
        tc_fence_after();
        // ---- E^T -> bf16 (for O) and E^T diag(f) -> bf16 (for the state), TMEM A operands
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int c0 = half * 32 + hh * 16;
            float e16[16];
            tmem_ld16(tmem + lane_off + cE32 + c0, e16);
            tmem_ld_wait();
            uint32_t pe[8], pf[8];
#pragma unroll
            for (int j = 0; j < 16; j += 4) {
                const float4 f4 = *reinterpret_cast<const float4 *>(sF + c0 + j);
                pe[j >> 1] = Op16<T>::pack2(e16[j], e16[j + 1]);
                pe[(j >> 1) + 1] = Op16<T>::pack2(e16[j + 2], e16[j + 3]);
                pf[j >> 1] = Op16<T>::pack2(f4.x * e16[j], f4.y * e16[j + 1]);
                pf[(j >> 1) + 1] = Op16<T>::pack2(f4.z * e16[j + 2], f4.w * e16[j + 3]);
            }
            tmem_st8_b32(tmem + lane_off + cEB + (c0 >> 1), pe);
            tmem_st8_b32(tmem + lane_off + cEF + (c0 >> 1), pf);
            // Y -> scale Gamma_r Y (O^T before MMA5 adds E^T L^T); rows past the end selected to 0
            float y16[16];
            tmem_ld16(tmem + lane_off + cO + c0, y16);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 16; j += 4) {
                const float4 g4 = *reinterpret_cast<const float4 *>(sGam + c0 + j);
                const float gg[4] = {g4.x, g4.y, g4.z, g4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    y16[j + e] = c0 + j + e < len ? p.scale * gg[e] * y16[j + e] : 0.f;
            }
            tmem_st16(tmem + lane_off + cO + c0, y16);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (issuer) {
            // MMA4: dS^T = (E^T diag f) K (M = 128, N = 128 keys, K = 64 rows; K MN-major)
            constexpr uint32_t id4 = idesc_f16kind(128, 128, 0, 1, Op16<T>::fmt);
            const uint64_t dk = smem_desc(sbase + Lay::oKQ, 16384, 1024, kSwizzle128B);
#pragma unroll
            for (int s = 0; s < 4; ++s) mma_bf16_ta(tmem + cD4, tmem + cEF + s * 8, dk + s * 128, id4, s > 0);
            // MMA5: O^T += E^T L^T (N = 64, K = 64)
            constexpr uint32_t id5 = idesc_f16kind(128, 64, 0, 0, Op16<T>::fmt);
#pragma unroll
            for (int s = 0; s < 4; ++s)
                mma_bf16_ta(tmem + cO, tmem + cEB + s * 8,
                            smem_desc(sbase + Lay::oL + s * 32, 16, 1024, kSwizzle128B), id5, 1);
            mma_commit(&bar_m45);
        }
        mbar_wait(&bar_m45, ph, &s_err, 5);
        tc_fence_after();
        if (issuer && ic + 1 < nch) issue_kq(ic + 1);       // K and Q are no longer read
        // ---- state: h_save (the state entering the chunk), S <- Gamma_c S + dS; O staging
        {
            const int64_t hs_lo = ((row0 + ic) * H + h) * KV + (int64_t)k0 * VD + m;
            if (p.h_save && GCL_RANGE_IN_BOUNDS(hs_lo, hs_lo + 63 * (int64_t)VD, p.nt_max * H * KV, p.status)) {
                float *dst = p.h_save + ((row0 + ic) * H + h) * KV + (int64_t)k0 * VD + m;
#pragma unroll
                for (int j = 0; j < 64; ++j) dst[(int64_t)j * VD] = S[j];
            }
            const float GC = __expf(sG[C - 1]);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float d4[16];
                tmem_ld16(tmem + lane_off + cD4 + k0 + q * 16, d4);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; ++j) S[q * 16 + j] = fmaf(GC, S[q * 16 + j], d4[j]);
            }
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                float ov[16];
                tmem_ld16(tmem + lane_off + cO + half * 32 + hh * 16, ov);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    if (GCL_IN_BOUNDS((half * 32 + hh * 16 + j) * kOLD + m, C * kOLD, p.status))
                        sO[(half * 32 + hh * 16 + j) * kOLD + m] = Op16<T>::from_float(ov[j]);
            }
        }
        tc_fence_before();
        __syncthreads();        // every read of D4 and O^T is done; O staged
        tc_fence_after();
        store_state_bf16();     // S^T bf16 for the next chunk's MMA2 (over D4's first columns)
        prev_t0 = t0;
        prev_len = len;
        // a wait that gave up (s_err) ends every thread's loop at the same chunk
        if (__syncthreads_or(*reinterpret_cast<volatile int *>(&s_err) != 0)) break;
    }
    if (s_err == 0) store_o(prev_t0, prev_len);             // the last chunk's O
    if (s_err == 0 && p.ht && GCL_RANGE_IN_BOUNDS(st_lo, st_hi, n_state, p.status)) {
        float *dst = p.ht + state_base + (int64_t)k0 * VD + m;
#pragma unroll
        for (int j = 0; j < 64; ++j) dst[(int64_t)j * VD] = S[j];
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
    if (tid == 0 && s_err != 0) status_set(p.status, GCL_DEV_WAIT_TIMEOUT);
}

}  // namespace

// Units (sequence slots x heads) from which the fused plan runs: at least one CTA per SM.
// The fused kernel's step per chunk is long (the whole Map-Reduce-Map of a chunk), so it
// pays only where many units fill the GPU; fewer units keep the split plans, whose serial
// step is short and whose value-column slices put several CTAs on every head (HA-NPU
// section 4: head-per-core while heads fill the cores, column-wise split for the rest).
int fwd_fused_min_units() { return num_sms(); }

// A training forward (h_save) whose workspace holds the transition records runs the
// transition plan instead: the backward's state-gradient sweep reads those records.
bool fwd_tc_runs_fused(int variant, int n_max, int H, bool h_save, size_t ws_bytes, int64_t nt_max) {
    if (variant != kGDN || (int64_t)n_max * H < fwd_fused_min_units() || n_max > 65535)
        return false;                                           // (grid.y holds the slots)
    return !(h_save && ws_bytes >= fwd_tc_t_workspace_bytes(nt_max, H));
}

cudaError_t launch_fwd_fused(const FwdParams &p, cudaStream_t s) {
    const int H = p.H;
    CUtensorMap mq, mk, mv;
    const cuuint64_t dqk[3] = {(cuuint64_t)KD, (cuuint64_t)H, (cuuint64_t)p.t_max};
    const cuuint64_t sqk[2] = {(cuuint64_t)KD * 2, (cuuint64_t)H * KD * 2};
    const cuuint32_t b64[3] = {64, 1, 64};
    const cuuint64_t dv[3] = {(cuuint64_t)VD, (cuuint64_t)H, (cuuint64_t)p.t_max};
    const cuuint64_t sv[2] = {(cuuint64_t)VD * 2, (cuuint64_t)H * VD * 2};
    const CUtensorMapDataType dt = p.dtype == GCL_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                      : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    if (!make_tensor_map(&mq, p.q, 3, dqk, sqk, b64, CU_TENSOR_MAP_SWIZZLE_128B, dt) ||
        !make_tensor_map(&mk, p.k, 3, dqk, sqk, b64, CU_TENSOR_MAP_SWIZZLE_128B, dt) ||
        !make_tensor_map(&mv, p.v, 3, dv, sv, b64, CU_TENSOR_MAP_SWIZZLE_128B, dt))
        return cudaErrorInvalidValue;
    FusedParams fp{};
    fp.cu = p.cu_seqlens;
    fp.chunk_offsets = p.chunk_offsets;
    fp.seq_order = p.seq_order;
    fp.g = p.g;
    fp.beta = p.beta;
    fp.h0 = p.h0;
    fp.o = p.o;
    fp.ht = p.ht;
    fp.h_save = p.h_save;
    fp.status = p.dev_status;
    fp.t_max = p.t_max;
    fp.nt_max = p.nt_max;
    fp.n_max = p.n_max;
    fp.H = H;
    fp.scale = p.scale;
    auto kern = p.dtype == GCL_F16 ? tc_fused_kernel<__half> : tc_fused_kernel<__nv_bfloat16>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)FusedLayout::bytes);
    if (e != cudaSuccess) return e;
    kern<<<dim3(H, p.n_max), kThreads, FusedLayout::bytes, s>>>(mq, mk, mv, fp);
    return cudaGetLastError();
}

}  // namespace gcl
