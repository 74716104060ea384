// fwd_tc_kda.cu -- KDA chunk forward on the tensor cores (bf16, d_k = d_v = 128, chunk 64):
// the transition form of the GDN path with the per-key-channel gate of KDA.
//
// FLA RFC "[RFC] Add Graph Capture Support for FLA Prefill and Training Paths on Ascend NPUs",
// section "Step 3" (gate / chunk cumsum, intra KK^T and triangular solve, recompute_w_u, h, o)
// and HA-NPU paper "Empowering Hybrid Attention Models on NPUs", section 2.1 (Map-Reduce-Map,
// the same pipeline for GDN and KDA).  With gamma_r the in-chunk prefix sum of the log gate,
// a vector over the key channels for KDA,
//   A[r][i] = beta_r sum_c k_r[c] k_i[c] exp(gamma_r[c] - gamma_i[c])   (i < r),
//   L[r][i] = scale sum_c q_r[c] k_i[c] exp(gamma_r[c] - gamma_i[c])    (i <= r),
//   T = (I + A)^-1,   W = T diag(beta) (K o exp(gamma)),   U = T diag(beta) V,
// and from E = U - W S, S' = Diag(exp(gamma_c)) S + Kbar^T E, O = scale (Q o exp(gamma)) S + L E:
//   S' = Diag(exp(gamma_c)) S + N S + B,   O = Y S + Z,
//   N = -Kbar^T W,  B = Kbar^T U,  Y = scale (Q o exp(gamma)) - L W,  Z = L U,
//   Kbar = K o exp(gamma_c - gamma),  gamma_c = gamma of the last row,
// which is the record of the transition form with a vector Gamma_c (one entry per key row).
//
// The decayed K K^T and Q K^T are not one GEMM of pre-scaled operands over the chunk:
// exp(gamma_r) and exp(-gamma_i) on their own leave the fp32 / bf16 range for strong gates.
// Between 16-row blocks they factor through the first row of the later block,
//   exp(gamma_r - gamma_i) = exp(gamma_r - rho_b) exp(rho_b - gamma_i),   rho_b = gamma_{16 b},
// for r in block b and i in an earlier block: with gates <= 0 both exponents are <= 0, so both
// factors lie in (0, 1] and the product is exact up to the bf16 rounding of the operands.
// Those entries come from three GEMMs (block rows b = 1, 2, 3) on the tensor cores; inside the
// 16 x 16 diagonal blocks the factors are not bounded, so those entries take one exponential
// per (pair, channel) on the CUDA cores in fp32, while the GEMMs run.
//
// prep (persistent, one CTA per SM, 256 threads), per chunk and head:
//   gamma     per-channel prefix sums of g (fp32, shared memory)
//   MMA1      [Kt; Qt] Khat_b^T, b = 1..3           -> A, L between blocks
//   diagonal  A, L inside the diagonal blocks       (CUDA cores, during MMA1)
//   solve     T = (I + A)^-1                        (blocked forward substitution)
//   MMA2      [T b; T b] [K o exp(gamma) | V]       -> W, U
//   MMA4      [T b; L] [W | U]                      -> L W, L U -> Y, Z
//   MMA3      Kbar^T [W | U]                        -> -N, B
// writes the record (Y, N, B, Z bf16) and exp(gamma_c) per key channel; the chain of the
// transition form then runs the recurrence with the per-row decay.
#include <cudaTypedefs.h>

#include "gcl_internal.cuh"
#include "tc_ptx.cuh"
#include "tc_solve.cuh"
#include "transition.cuh"

namespace gcl {
namespace {

using namespace tc;
using namespace tr;

constexpr int kThreads = 256;
constexpr int kGLD = 132;           // gamma row stride (floats): 16-byte rows spread over the banks
// dynamic shared memory, offsets from the 1024-aligned base
constexpr uint32_t kPKQ = 0;        // raw K | Q (TMA): 2 column blocks x [K rows 0..63 | Q rows 0..63]
constexpr uint32_t kPV = 32768;     // raw V (TMA); later the Y boxes and B box (1, 1)
constexpr uint32_t kPTL = 49152;    // [T b; T b; L]: 192 rows of 64 tokens; later Z and B boxes
constexpr uint32_t kPA = 73728;     // fp32 A, L (then T), X; later [W | U]
constexpr uint32_t kPKT = 112640;   // [Kt; Qt]: 128 rows x 128 channels; later K o exp(gamma)
constexpr uint32_t kPKH = kPKT + 32768;    // Khat_1 | Khat_2 | Khat_3: 16, 32, 48 rows x 128
constexpr uint32_t kPG = kPKH + 24576;     // gamma fp32 [64][kGLD]
constexpr uint32_t kEnd = kPG + C * kGLD * 4;
constexpr int kSmem = kEnd + 1024;
static_assert(kPA + kSolveFloats * 4 <= kPKT, "the solve buffers end before the [Kt; Qt] tile");
static_assert(kSolveFloats * 4 >= 4 * 8192, "[W | U] (4 atoms of 8 KiB) reuses the solve buffers");
static_assert(kSmem <= 232448, "shared memory of one CTA");

// Khat_b (b = 1..3) holds rows i < 16 b in two 64-channel column blocks 16 b x 128 bytes apart;
// its GEMM result goes to TMEM columns [kcol(b), kcol(b) + 16 b).
__host__ __device__ constexpr uint32_t khat_off(int b) { return b == 1 ? 0u : b == 2 ? 4096u : 12288u; }
__host__ __device__ constexpr uint32_t kcol(int b) { return b == 1 ? 0u : b == 2 ? 16u : 48u; }

__device__ __forceinline__ void unpack8(uint4 w, float *x) {
    const __nv_bfloat162 *pp = reinterpret_cast<const __nv_bfloat162 *>(&w);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float2 f = __bfloat1622float2(pp[e]);
        x[2 * e] = f.x;
        x[2 * e + 1] = f.y;
    }
}
__device__ __forceinline__ void unpack4(uint2 w, float *x) {
    const __nv_bfloat162 *pp = reinterpret_cast<const __nv_bfloat162 *>(&w);
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const float2 f = __bfloat1622float2(pp[e]);
        x[2 * e] = f.x;
        x[2 * e + 1] = f.y;
    }
}

// Persistent: gridDim.x CTAs (one per SM) walk the items (chunk-head pairs) with stride
// gridDim.x.  The next item's K and Q tiles are requested once MMA3 has consumed the current
// ones, its V tile once the record stores have read their staging buffers, its gates during MMA3.
__global__ void __launch_bounds__(kThreads, 1)
tc_prep_kda_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_rec,
                   PrepTParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    float *sA = reinterpret_cast<float *>(smem + kPA);
    float *sT = sA + C * kSolveLD;            // L (fp32) until the solve writes T here
    float *sX = sT + C * kSolveLD;
    float *sGam = reinterpret_cast<float *>(smem + kPG);
    __shared__ uint64_t bar_kq, bar_v, bar_mma;
    __shared__ uint32_t s_tmem;
    __shared__ int s_err;
    __shared__ float sB[C];
    __shared__ float4 sSeg[8][32];

    // launched as a dependent of the metadata (or any earlier) kernel
    grid_dependency_wait();
    launch_dependents();
    if (status_blocks_cta(p.status)) return;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3, half = warp >> 2;
    const int lrow = quarter * 32 + lane;                 // TMEM lane read by this thread
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const int H = p.H, stride = gridDim.x;
    const uint32_t sbase = smem_u32(smem);

    PrepItem cur, nxt;
    int icur = next_item(p, blockIdx.x, stride, &cur);
    if (icur < 0) return;

    if (tid == 0) {
        mbar_init(&bar_kq, 1);
        mbar_init(&bar_v, 1);
        mbar_init(&bar_mma, 1);
        s_err = 0;
        fence_barrier_init();
    }
    __syncwarp();
    if (warp == 0) {
        tmem_alloc(&s_tmem, 256);
        tmem_relinquish();
    }
    auto load_kq = [&](const PrepItem &it) {
        mbar_arrive_expect_tx(&bar_kq, 32768);
        for (int cb = 0; cb < 2; ++cb) {
            tma_load_3d(smem + kPKQ + cb * 16384, &tm_k, cb * 64, it.h, (int)it.t0, &bar_kq);
            tma_load_3d(smem + kPKQ + cb * 16384 + 8192, &tm_q, cb * 64, it.h, (int)it.t0, &bar_kq);
        }
    };
    auto load_v = [&](const PrepItem &it) {
        mbar_arrive_expect_tx(&bar_v, 16384);
        for (int cb = 0; cb < 2; ++cb) tma_load_3d(smem + kPV + cb * 8192, &tm_v, cb * 64, it.h, (int)it.t0, &bar_v);
    };
    // gates of an item: thread (warp w, lane l) holds g of rows 8 w .. 8 w + 7, channels
    // 4 l .. 4 l + 3 (0 past the end); threads 0..63 also beta of row tid
    auto load_g = [&](const PrepItem &it, float4 *gq, float &bv) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int r = warp * 8 + j;
            gq[j] = r < it.len ? *reinterpret_cast<const float4 *>(p.g + ((it.t0 + r) * H + it.h) * (int64_t)KD + lane * 4)
                               : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        bv = tid < it.len ? __bfloat162float(static_cast<const __nv_bfloat16 *>(p.beta)[(it.t0 + tid) * H + it.h])
                          : 0.f;
    };
    float4 gq[8];
    float b_raw;
    load_g(cur, gq, b_raw);
    if (tid == 0) {
        load_kq(cur);
        load_v(cur);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;

    uint32_t phase = 0, ph_in = 0;
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
    auto box_chunk = [&](uint32_t box, int row, int q) {
        return smem + box + row * 128 + ((q ^ (row & 7)) << 4);
    };
    // 4 or 8 bf16 of the raw tiles: K row r (Q: row C + r), channels c.. (c % 4 == 0)
    auto raw4 = [&](int row, int c) {
        return *reinterpret_cast<const uint2 *>(smem + kPKQ + kmaj16(128, row, c) + (c & 7) * 2);
    };
    auto raw8 = [&](int row, int c) { return reinterpret_cast<uint4 *>(smem + kPKQ + kmaj16(128, row, c)); };
    auto gam8 = [&](int row, int c, float *x) {
        const float4 a = *reinterpret_cast<const float4 *>(sGam + row * kGLD + c);
        const float4 b = *reinterpret_cast<const float4 *>(sGam + row * kGLD + c + 4);
        x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
        x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
    };

    while (icur >= 0) {
        bool item_done = false;
        const int len = cur.len;
        const int unit = icur;
        {   // gamma: inclusive prefix over this thread's 8 rows, then the earlier segments' sums
#pragma unroll
            for (int j = 1; j < 8; ++j) {
                gq[j].x += gq[j - 1].x;
                gq[j].y += gq[j - 1].y;
                gq[j].z += gq[j - 1].z;
                gq[j].w += gq[j - 1].w;
            }
            sSeg[warp][lane] = gq[7];
            if (tid < C) sB[tid] = b_raw;
            __syncthreads();                      // (also: the previous item's buffers are free)
            float4 pre = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int sg = 0; sg < warp; ++sg) {
                const float4 t = sSeg[sg][lane];
                pre.x += t.x; pre.y += t.y; pre.z += t.z; pre.w += t.w;
            }
#pragma unroll
            for (int j = 0; j < 8; ++j)
                *reinterpret_cast<float4 *>(sGam + (warp * 8 + j) * kGLD + lane * 4) =
                    make_float4(gq[j].x + pre.x, gq[j].y + pre.y, gq[j].z + pre.z, gq[j].w + pre.w);
        }
        __syncthreads();
        if (tid < KD)   // per-channel state decay of the chunk (gamma is constant past the end)
            reinterpret_cast<float *>(p.ws + gc_offset(p.nt_max, H, unit))[tid] = __expf(sGam[(C - 1) * kGLD + tid]);
        do {
            const bool landed = mbar_wait(&bar_kq, ph_in, &s_err, 1);
            if (__syncthreads_or(!landed)) break;
            if (len < C) {   // rows past the end: zero K and Q (next sequence or NaN padding)
                const uint4 zero = make_uint4(0, 0, 0, 0);
                for (int t = tid; t < 4 * C * 8; t += kThreads) {
                    const int r = (t >> 3) & 63, blk = t >> 9;       // K0 K1 Q0 Q1
                    if (r >= len)
                        *reinterpret_cast<uint4 *>(smem + kPKQ + (blk & 1) * 16384 + (blk >> 1) * 8192 +
                                                   r * 128 + (t & 7) * 16) = zero;
                }
                __syncthreads();
            }
            // [Kt; Qt] rows 16..63 (block b = r / 16): k_r, q_r times exp(gamma_r - gamma_{16 b})
            for (int t = tid; t < 48 * 16; t += kThreads) {
                const int r = 16 + (t >> 4), c = (t & 15) * 8;
                float gr[8], gb[8], kk[8], qq[8];
                gam8(r, c, gr);
                gam8(r & ~15, c, gb);
                unpack8(*raw8(r, c), kk);
                unpack8(*raw8(C + r, c), qq);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float f = __expf(gr[e] - gb[e]);
                    kk[e] *= f;
                    qq[e] *= f;
                }
                *reinterpret_cast<uint4 *>(smem + kPKT + kmaj16(128, r, c)) = pack8(kk);
                *reinterpret_cast<uint4 *>(smem + kPKT + kmaj16(128, C + r, c)) = pack8(qq);
            }
            // Khat_b rows i < 16 b: k_i times exp(gamma_{16 b} - gamma_i)
            for (int t = tid; t < 96 * 16; t += kThreads) {
                const int row = t >> 4, c = (t & 15) * 8;
                const int b = row < 16 ? 1 : row < 48 ? 2 : 3;
                const int i = row - (b == 1 ? 0 : b == 2 ? 16 : 48);
                float gi[8], gb[8], kk[8];
                gam8(i, c, gi);
                gam8(16 * b, c, gb);
                unpack8(*raw8(i, c), kk);
#pragma unroll
                for (int e = 0; e < 8; ++e) kk[e] *= __expf(gb[e] - gi[e]);
                *reinterpret_cast<uint4 *>(smem + kPKH + khat_off(b) + kmaj16(16 * b, i, c)) = pack8(kk);
            }
            to_async();
            // ---- MMA1: [Kt; Qt] Khat_b^T -> TMEM columns kcol(b) .. (N = 16 b); lanes 0..63 give
            // the K K^T entries of rows in block b, lanes 64..127 the Q K^T entries
            if (tid == 0) {
                const uint64_t a = smem_desc(sbase + kPKT, 16, 1024, kSwizzle128B);
#pragma unroll
                for (int b = 1; b <= 3; ++b) {
                    const uint64_t bd = smem_desc(sbase + kPKH + khat_off(b), 16, 1024, kSwizzle128B);
#pragma unroll
                    for (int s = 0; s < 8; ++s) {
                        const uint64_t oa = (s >> 2) * (16384 >> 4) + (s & 3) * 2;
                        const uint64_t ob = (s >> 2) * ((2048 * b) >> 4) + (s & 3) * 2;
                        mma_bf16(tmem + kcol(b), a + oa, bd + ob, idesc_bf16(128, 16 * b), s > 0);
                    }
                }
                mma_commit(&bar_mma);
            }
            // ---- diagonal blocks (CUDA cores, fp32): 120 strict pairs per block, one thread each
            for (int t = tid; t < 4 * 120; t += kThreads) {
                const int b = t / 120, w = t - b * 120;
                int r = (int)((1.f + sqrtf(1.f + 8.f * (float)w)) * 0.5f);   // w = r (r - 1) / 2 + i
                if (r * (r - 1) / 2 > w) --r;
                if ((r + 1) * r / 2 <= w) ++r;
                const int R = 16 * b + r, I = 16 * b + w - r * (r - 1) / 2;
                const float *gR = sGam + R * kGLD, *gI = sGam + I * kGLD;
                float aa = 0.f, al = 0.f;
#pragma unroll 4
                for (int c = 0; c < KD; c += 4) {
                    const float4 x = *reinterpret_cast<const float4 *>(gR + c);
                    const float4 y = *reinterpret_cast<const float4 *>(gI + c);
                    float kr[4], ki[4], qr[4];
                    unpack4(raw4(R, c), kr);
                    unpack4(raw4(I, c), ki);
                    unpack4(raw4(C + R, c), qr);
                    const float w0 = ki[0] * __expf(x.x - y.x), w1 = ki[1] * __expf(x.y - y.y);
                    const float w2 = ki[2] * __expf(x.z - y.z), w3 = ki[3] * __expf(x.w - y.w);
                    aa = fmaf(kr[0], w0, fmaf(kr[1], w1, fmaf(kr[2], w2, fmaf(kr[3], w3, aa))));
                    al = fmaf(qr[0], w0, fmaf(qr[1], w1, fmaf(qr[2], w2, fmaf(qr[3], w3, al))));
                }
                sA[R * kSolveLD + I] = sB[R] * aa;
                sT[R * kSolveLD + I] = p.scale * al;
            }
            {   // the diagonal of L: scale q_R . k_R (four threads per row, 32 channels each)
                const int R = tid >> 2, c0 = (tid & 3) * 32;
                float d = 0.f;
#pragma unroll
                for (int c = c0; c < c0 + 32; c += 4) {
                    float kr[4], qr[4];
                    unpack4(raw4(R, c), kr);
                    unpack4(raw4(C + R, c), qr);
                    d = fmaf(qr[0], kr[0], fmaf(qr[1], kr[1], fmaf(qr[2], kr[2], fmaf(qr[3], kr[3], d))));
                }
                d += __shfl_xor_sync(0xffffffffu, d, 1);
                d += __shfl_xor_sync(0xffffffffu, d, 2);
                if ((tid & 3) == 0) sT[R * kSolveLD + R] = p.scale * d;
            }
            if (!mma_done(2)) break;
            {   // A (beta_r x) and L (scale x) between blocks: warps of half 0 read columns 0..47
                // (blocks 1, 2), half 1 columns 48..95 (block 3)
                float v[48];
#pragma unroll
                for (int q = 0; q < 3; ++q) tmem_ld16(tmem + lane_off + half * 48 + q * 16, v + q * 16);
                tmem_ld_wait();
                const int r = lrow & 63, b = r >> 4;
                const bool isq = lrow >= C;
                float *dst = (isq ? sT : sA) + r * kSolveLD;
                const float f = isq ? p.scale : sB[r];
                if (half == 0 && b == 1) {
#pragma unroll
                    for (int i = 0; i < 16; i += 4)
                        *reinterpret_cast<float4 *>(dst + i) = make_float4(f * v[i], f * v[i + 1], f * v[i + 2], f * v[i + 3]);
                } else if (half == 0 && b == 2) {
#pragma unroll
                    for (int i = 0; i < 32; i += 4)
                        *reinterpret_cast<float4 *>(dst + i) =
                            make_float4(f * v[16 + i], f * v[17 + i], f * v[18 + i], f * v[19 + i]);
                } else if (half == 1 && b == 3) {
#pragma unroll
                    for (int i = 0; i < 48; i += 4)
                        *reinterpret_cast<float4 *>(dst + i) = make_float4(f * v[i], f * v[i + 1], f * v[i + 2], f * v[i + 3]);
                }
            }
            __syncthreads();
            {   // L -> rows 128.. of [T b; T b; L] (bf16; zero above the diagonal and past the end)
                const int r = tid >> 2;
#pragma unroll
                for (int qq = 0; qq < 2; ++qq) {
                    const int c0 = ((tid & 3) * 2 + qq) * 8;
                    float l8[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) l8[e] = (c0 + e <= r && r < len) ? sT[r * kSolveLD + c0 + e] : 0.f;
                    *reinterpret_cast<uint4 *>(smem + kPTL + kmaj16(192, 2 * C + r, c0)) = pack8(l8);
                }
            }
            __syncthreads();
            solve_unit_lower64<kThreads>(sA, sT, sX);   // T = (I + A)^-1
            {
                const bool vl = mbar_wait(&bar_v, ph_in, &s_err, 6);
                if (__syncthreads_or(!vl)) break;
            }
            if (len < C) {
                const uint4 zero = make_uint4(0, 0, 0, 0);
                for (int t = tid; t < 2 * C * 8; t += kThreads) {
                    const int r = (t >> 3) & 63, cb = t >> 9;
                    if (r >= len) *reinterpret_cast<uint4 *>(smem + kPV + cb * 8192 + r * 128 + (t & 7) * 16) = zero;
                }
            }
            {   // T diag(beta) -> rows 0..63 and 64..127 (bf16, K-major over tokens)
                const int r = tid >> 2;
#pragma unroll
                for (int qq = 0; qq < 2; ++qq) {
                    const int c0 = ((tid & 3) * 2 + qq) * 8;
                    float tb[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) tb[e] = c0 + e <= r ? sT[r * kSolveLD + c0 + e] * sB[c0 + e] : 0.f;
                    const uint4 pk = pack8(tb);
                    *reinterpret_cast<uint4 *>(smem + kPTL + kmaj16(192, r, c0)) = pk;
                    *reinterpret_cast<uint4 *>(smem + kPTL + kmaj16(192, C + r, c0)) = pk;
                }
            }
            // K o exp(gamma) (64 rows, column blocks 8 KiB apart) in place of [Kt; Qt]
            for (int t = tid; t < C * 16; t += kThreads) {
                const int r = t >> 4, c = (t & 15) * 8;
                float gr[8], kk[8];
                gam8(r, c, gr);
                unpack8(*raw8(r, c), kk);
#pragma unroll
                for (int e = 0; e < 8; ++e) kk[e] *= __expf(gr[e]);
                *reinterpret_cast<uint4 *>(smem + kPKT + kmaj16(64, r, c)) = pack8(kk);
            }
            to_async();
            // ---- MMA2: [T b; T b] (K o exp(gamma)) -> cols 0..127 (W in lanes 0..63);
            //            [T b; T b] V -> cols 128..255 (U in lanes 64..127); MN-major B operands
            if (tid == 0) {
                const uint64_t a = smem_desc(sbase + kPTL, 16, 1024, kSwizzle128B);
                const uint64_t bk = smem_desc(sbase + kPKT, 8192, 1024, kSwizzle128B);
                const uint64_t bv = smem_desc(sbase + kPV, 8192, 1024, kSwizzle128B);
                constexpr uint32_t id = idesc_bf16(128, 128, 0, 1);
#pragma unroll
                for (int s = 0; s < 4; ++s) mma_bf16(tmem, a + s * 2, bk + s * 128, id, s > 0);
#pragma unroll
                for (int s = 0; s < 4; ++s) mma_bf16(tmem + 128, a + s * 2, bv + s * 128, id, s > 0);
                mma_commit(&bar_mma);
            }
            if (!mma_done(3)) break;
            {   // [W | U] as one MN-major operand (N = 256: keys then values) in the solve buffers
                const int tok = lrow & 63;
                const int n0 = (lrow < C ? 0 : 128) + half * 64;
                float wu[64];
#pragma unroll
                for (int q = 0; q < 4; ++q) tmem_ld16(tmem + lane_off + n0 + q * 16, wu + q * 16);
                tmem_ld_wait();
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    *reinterpret_cast<uint4 *>(smem + kPA + mnmaj16(8192, tok, n0 + q * 8)) = pack8(wu + q * 8);
                // Kbar = K o exp(gamma_c - gamma), in place of the raw K
                for (int t = tid; t < C * 16; t += kThreads) {
                    const int r = t >> 4, c = (t & 15) * 8;
                    float gr[8], gc[8], kk[8];
                    gam8(r, c, gr);
                    gam8(C - 1, c, gc);
                    uint4 *pk = raw8(r, c);
                    unpack8(*pk, kk);
#pragma unroll
                    for (int e = 0; e < 8; ++e) kk[e] *= __expf(gc[e] - gr[e]);
                    *pk = pack8(kk);
                }
            }
            to_async();
            // ---- MMA4: [T b; L] [W | U] -> lanes 64..127: L W (cols 0..127), L U (cols 128..255)
            if (tid == 0) {
                const uint64_t a = smem_desc(sbase + kPTL + 8192, 16, 1024, kSwizzle128B);
                const uint64_t b = smem_desc(sbase + kPA, 8192, 1024, kSwizzle128B);
                constexpr uint32_t id = idesc_bf16(128, 256, 0, 1);
#pragma unroll
                for (int s = 0; s < 4; ++s) mma_bf16(tmem, a + s * 2, b + s * 128, id, s > 0);
                mma_commit(&bar_mma);
            }
            if (!mma_done(4)) break;
            // the record leaves through shared memory in 64 x 64 boxes: Y 0..63, N 64..191,
            // B 192..319, Z 320..383
            if (lrow >= C) {   // Y = scale (Q o exp(gamma)) - L W and Z = L U, row r, columns half*64..
                const int r = lrow - C;
                const bool live = r < len;
                float x[64];
#pragma unroll
                for (int q = 0; q < 4; ++q) tmem_ld16(tmem + lane_off + half * 64 + q * 16, x + q * 16);
                tmem_ld_wait();
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const int c = half * 64 + q * 8;
                    float qv[8], gr[8], y[8];
                    unpack8(*raw8(C + r, c), qv);
                    gam8(r, c, gr);
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        y[e] = live ? fmaf(p.scale * __expf(gr[e]), qv[e], -x[q * 8 + e]) : 0.f;
                    *reinterpret_cast<uint4 *>(box_chunk(kPV + half * 8192, r, q)) = pack8(y);
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) tmem_ld16(tmem + lane_off + 128 + half * 64 + q * 16, x + q * 16);
                tmem_ld_wait();
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    float z[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) z[e] = live ? x[q * 8 + e] : 0.f;
                    *reinterpret_cast<uint4 *>(box_chunk(kPTL + half * 8192, r, q)) = pack8(z);
                }
            }
            to_async();
            if (tid == 0) {   // Y and Z boxes
                for (int cb = 0; cb < 2; ++cb) {
                    tma_store_3d(&tm_rec, smem + kPV + cb * 8192, cb * 64, 0, unit);
                    tma_store_3d(&tm_rec, smem + kPTL + cb * 8192, cb * 64, 320, unit);
                }
                bulk_commit();
            }
            // ---- MMA3: Kbar^T [W | U] -> cols 0..127: Kbar^T W = -N, cols 128..255: B
            if (tid == 0) {
                const uint64_t a = smem_desc(sbase + kPKQ, 16384, 1024, kSwizzle128B);
                const uint64_t b = smem_desc(sbase + kPA, 8192, 1024, kSwizzle128B);
                constexpr uint32_t id = idesc_bf16(128, 256, 1, 1);
#pragma unroll
                for (int s = 0; s < 4; ++s) mma_bf16(tmem, a + s * 128, b + s * 128, id, s > 0);
                mma_commit(&bar_mma);
            }
            // the next item and its gates, while MMA3 runs
            const int inext = next_item(p, icur + stride, stride, &nxt);
            if (inext >= 0) load_g(nxt, gq, b_raw);
            if (!mma_done(5)) break;
            if (tid == 0) {
                if (inext >= 0) load_kq(nxt);          // K and Q of this item are consumed
                bulk_wait_read();                      // the Y and Z stores have read kPV, kPTL
            }
            __syncthreads();
            {   // key row m = lrow: half 0 -> N boxes in the [W | U] buffer, half 1 -> B boxes
                // (0, 0), (0, 1), (1, 0) in the [..; L] buffer and (1, 1) in the V buffer
                const int m = lrow;
                const float sg = half == 0 ? -1.f : 1.f;
#pragma unroll
                for (int pass = 0; pass < 2; ++pass) {
                    const int bidx = (m >> 6) * 2 + pass;
                    const uint32_t box = half == 0 ? kPA + bidx * 8192 : (bidx < 3 ? kPTL + bidx * 8192 : kPV);
                    float x[64];
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        tmem_ld16(tmem + lane_off + half * 128 + pass * 64 + q * 16, x + q * 16);
                    tmem_ld_wait();
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        float y[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) y[e] = sg * x[q * 8 + e];
                        *reinterpret_cast<uint4 *>(box_chunk(box, m & 63, q)) = pack8(y);
                    }
                }
            }
            fence_async_smem();
            tc_fence_before();
            __syncthreads();
            if (tid == 0) {
                for (int rb = 0; rb < 2; ++rb)
                    for (int cb = 0; cb < 2; ++cb) {
                        const int bidx = rb * 2 + cb;
                        tma_store_3d(&tm_rec, smem + kPA + bidx * 8192, cb * 64, 64 + rb * 64, unit);
                        tma_store_3d(&tm_rec, smem + (bidx < 3 ? kPTL + bidx * 8192 : kPV), cb * 64,
                                     192 + rb * 64, unit);
                    }
                bulk_commit();
                bulk_wait_read();                      // staging buffers are free again
                if (inext >= 0) load_v(nxt);
            }
            tc_fence_after();
            icur = inext;
            cur = nxt;
            ph_in ^= 1;
            item_done = true;
        } while (0);
        if (!item_done) break;                         // a wait gave up (uniformly decided)
    }
    if (tid == 0) bulk_wait_read();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 256);
    if (tid == 0 && s_err != 0) status_set(p.status, GCL_DEV_WAIT_TIMEOUT);
}

}  // namespace

cudaError_t launch_prep_kda(const FwdParams &p, uint8_t *ws, cudaStream_t s) {
    CUtensorMap mq, mk, mv, mrec;
    if (!make_prep_maps(p, ws, &mq, &mk, &mv, &mrec)) return cudaErrorInvalidValue;
    const PrepTParams pp = make_prep_params(p, ws);
    cudaError_t e = cudaFuncSetAttribute(tc_prep_kda_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    const int64_t units = p.nt_max * p.H;
    const int grid = (int)(units < (int64_t)num_sms() ? units : (int64_t)num_sms());
    return launch_dependent(tc_prep_kda_kernel, dim3(grid), dim3(kThreads), kSmem, s, mq, mk, mv, mrec, pp);
}

cudaError_t launch_fwd_tc_kda(const FwdParams &p, int split, cudaStream_t s) {
    uint8_t *ws = static_cast<uint8_t *>(p.workspace);
    const cudaError_t e = launch_prep_kda(p, ws, s);
    if (e != cudaSuccess) return e;
    int n_seg = 0;
    float *seg_ws = nullptr;
    fwd_seg_plan(p, ws, &n_seg, &seg_ws);
    return launch_chain_records(p, ws, split, true, s, n_seg, seg_ws);
}

}  // namespace gcl
