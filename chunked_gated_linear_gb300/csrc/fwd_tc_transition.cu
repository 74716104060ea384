// fwd_tc_transition.cu -- GDN chunk forward in transition form (bf16 or fp16 inputs, d_k =
// d_v = 128, chunk 64), for launches whose serial chain dominates: few (sequence, head)
// units, each split over 4 or 8 value-column slices.  Every MMA operand and record has the
// input type ("bf16" below stands for either; the KDA records are bf16).
//
// HA-NPU paper "Empowering Hybrid Attention Models on NPUs", section 2.1: the Map
// phases are chunk-parallel, only the Reduce is serial; section 5: the
// state-independent GEMMs are grouped and decoupled from the state read.  Here the
// chunk-parallel Map goes one step further and folds everything the state update and
// the output need into per-chunk matrices, so the serial Reduce is one small GEMM per
// chunk.  From E = U - W S, S' = Gamma_c S + Ktil^T E and O = scale diag(Gamma) Q S + L E:
//
//   S' = Gamma_c S + N S + B,          O = Y S + Z,          with
//   N = -Ktil^T W   (128 x 128),       B = Ktil^T U   (128 x V),
//   Y = scale diag(Gamma) Q - L W  (64 x 128),   Z = L U   (64 x V),
//   Ktil = diag(exp(g_c - g)) K,  W = T diag(beta Gamma) K,  U = T diag(beta) V.
//
// The per-chunk affine map (Gamma_c I + N, B) is the chunk-level form of the state
// transition the same paper's Map-Reduce-Map decomposition composes across segments.
// The state stays in fp32; N, B, Y, Z are bf16 MMA operands.
//
// prep_t   one CTA per row of chunk_indices and head, 256 threads, two CTAs per SM:
//            MMA1  [K; Q] K^T                   -> A, L (CUDA cores: decay, mask)
//            solve T = (I + A)^-1               (blocked forward substitution)
//            MMA2  [T bG; T b] K, [T bG; T b] V -> W, U
//            MMA4  [T b; L] [W | U]             -> L W, L U  -> Y, Z
//            MMA3  Ktil^T [W | U]               -> -N, B
//          and writes [Y; N] (192 x 128), B (128 x 128), Z (64 x 128) as bf16 and
//          Gamma_c into one 96 KiB record per chunk and head.
// chain_t  one CTA per (sequence, head, column slice): per chunk the serial step
//          G1 = N S and the output G2 = [Y; .] S, with TMA several chunks ahead.
#include <cudaTypedefs.h>

#include "gcl_internal.cuh"
#include "tc_ptx.cuh"
#include "tc_solve.cuh"
#include "transition.cuh"

namespace gcl {
namespace {

using namespace tc;
using namespace tr;

// ============================================================================ prep_t
constexpr int kPrepThreads = 256;
// dynamic shared memory, offsets from the 1024-aligned base
constexpr uint32_t pKQ = 0;        // [2 col blocks][K rows 0..63 | Q rows 0..63][128 B]  32 KiB
constexpr uint32_t pV = 32768;     // [2 col blocks][64 rows][128 B]                      16 KiB
constexpr uint32_t pTL = 49152;    // [T diag(bG); T diag(b); L], 192 rows of 64 tokens   24 KiB
constexpr uint32_t pA = 73728;     // fp32 A, T [64][kSolveLD], X; later [W | U]
constexpr uint32_t pEnd = pA + kSolveFloats * 4;
constexpr int kPrepTSmem = pEnd + 1024;
static_assert(pEnd - pA >= 4 * 8192, "[W | U] (4 atoms of 8 KiB) reuses the solve buffers");

// Persistent: gridDim.x CTAs (two per SM) walk the items with stride gridDim.x.  The next
// item's K and Q tiles are requested as soon as MMA3 has consumed the current ones, its V tile
// once the output stores have read their staging buffers, and its gates during MMA3.
// T: the input type (bf16, or fp16 for GDN); every MMA operand the kernel forms and every
// record it writes has the same type.
template <typename T>
__global__ void __launch_bounds__(kPrepThreads, 2)
tc_prep_t_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_rec,
                 PrepTParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    float *sA = reinterpret_cast<float *>(smem + pA);
    float *sT = sA + C * kSolveLD;
    float *sX = sT + C * kSolveLD;
    __shared__ uint64_t bar_kq, bar_v, bar_mma;
    __shared__ uint32_t s_tmem;
    __shared__ int s_err;
    __shared__ float sG[C], sB[C], sF[C], sFQ[C], sEG[C], s_carry;

    // launched as a dependent of the metadata (or any earlier) kernel: nothing written by
    // earlier kernels is read before this wait
    grid_dependency_wait();
    // the chain kernel may be scheduled on SMs this grid leaves; it reads the records only
    // after waiting for this grid's completion
    launch_dependents();
    if (status_blocks_cta(p.status)) return;
    const int tid = threadIdx.x, warp = tid >> 5;
    const int quarter = warp & 3, half = warp >> 2;
    const int lrow = quarter * 32 + (tid & 31);           // TMEM lane read by this thread
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
    if (warp == 0) {
        tmem_alloc(&s_tmem, 256);
        tmem_relinquish();
    }
    auto load_kq = [&](const PrepItem &it) {
        mbar_arrive_expect_tx(&bar_kq, 32768);
        for (int cb = 0; cb < 2; ++cb) {
            tma_load_3d(smem + pKQ + cb * 16384, &tm_k, cb * 64, it.h, (int)it.t0, &bar_kq);
            tma_load_3d(smem + pKQ + cb * 16384 + 8192, &tm_q, cb * 64, it.h, (int)it.t0, &bar_kq);
        }
    };
    auto load_v = [&](const PrepItem &it) {
        mbar_arrive_expect_tx(&bar_v, 16384);
        for (int cb = 0; cb < 2; ++cb) tma_load_3d(smem + pV + cb * 8192, &tm_v, cb * 64, it.h, (int)it.t0, &bar_v);
    };
    // gates of an item for threads 0..63 (row tid): raw g and beta (0 past the end)
    auto load_gates = [&](const PrepItem &it, float &gv, float &bv) {
        gv = 0.f;
        bv = 0.f;
        if (tid < it.len) {
            if (GCL_IN_BOUNDS((it.t0 + tid) * H + it.h, p.t_max * H, p.status)) {
                gv = p.g[(it.t0 + tid) * H + it.h];
                bv = Op16<T>::to_float(static_cast<const T *>(p.beta)[(it.t0 + tid) * H + it.h]);
            }
        }
    };
    float g_raw, b_raw;
    load_gates(cur, g_raw, b_raw);
    if (tid == 0) {
        load_kq(cur);
        load_v(cur);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;

    uint32_t phase = 0, ph_in = 0;
    // every thread waits for the tensor-core group just committed; the block then agrees
    // on whether any wait gave up
    auto mma_done = [&](int code) -> bool {
        const bool ok = mbar_wait(&bar_mma, phase, &s_err, code);
        phase ^= 1;
        tc_fence_after();
        return !__syncthreads_or(!ok);
    };
    auto to_async = [&]() {      // shared writes and TMEM reads -> next tensor-core group
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    };
    // 16-byte chunk q of row `row` of a 64 x 64 output box (128-byte swizzle)
    auto box_chunk = [&](uint32_t box, int row, int q) {
        return smem + box + row * 128 + ((q ^ (row & 7)) << 4);
    };
    while (icur >= 0) {
        bool item_done = false;
        const int len = cur.len;
        const int unit = icur;
        float *gGC = reinterpret_cast<float *>(p.ws + gc_offset(p.nt_max, H, unit));
        {   // gamma = inclusive cumsum of g over the chunk (warps 0 and 1), beta
            float x = tid < C ? warp_scan(g_raw) : 0.f;
            if (tid == 31) s_carry = x;
            __syncthreads();                      // (also: the previous item's buffers are free)
            if (tid >= 32 && tid < C) x += s_carry;
            if (tid < C) {
                sG[tid] = x;
                sB[tid] = b_raw;
            }
        }
        __syncthreads();
        // factors and the decay table D[r][c] = exp(g_r - g_c) for c <= r (1 above the
        // diagonal: the exponent is selected, so no lane branches around the exponential) in
        // the T buffer, which the solve only writes later
        if (tid < C) {
            const bool live = tid < len;
            sF[tid] = live ? __expf(sG[C - 1] - sG[tid]) : 0.f;   // row factor of Ktil
            sFQ[tid] = live ? p.scale * __expf(sG[tid]) : 0.f;    // read-out factor
            sEG[tid] = __expf(sG[tid]);                            // Gamma of column tid
        }
        for (int e = tid; e < C * C / 4; e += kPrepThreads) {
            const int r = e >> 4, c = (e & 15) * 4;
            const float gr = sG[r];
            *reinterpret_cast<float4 *>(sT + r * kSolveLD + c) =
                make_float4(__expf(c <= r ? gr - sG[c] : 0.f), __expf(c + 1 <= r ? gr - sG[c + 1] : 0.f),
                            __expf(c + 2 <= r ? gr - sG[c + 2] : 0.f), __expf(c + 3 <= r ? gr - sG[c + 3] : 0.f));
        }
        do {
            const bool landed = mbar_wait(&bar_kq, ph_in, &s_err, 1);
            if (__syncthreads_or(!landed)) break;
            // rows past the end of a partial chunk: zero K and Q (they may hold the next
            // sequence or NaN padding and enter the MMAs raw); V likewise once it lands
            if (len < C) {
                const uint4 zero = make_uint4(0, 0, 0, 0);
                for (int t = tid; t < 4 * C * 8; t += kPrepThreads) {
                    const int r = (t >> 3) & 63, blk = t >> 9;       // K0 K1 Q0 Q1
                    if (r >= len)
                        *reinterpret_cast<uint4 *>(smem + pKQ + (blk & 1) * 16384 + (blk >> 1) * 8192 +
                                                   r * 128 + (t & 7) * 16) = zero;
                }
            }
            to_async();
            // ---- MMA1: [K; Q] K^T -> lanes 0..63: K K^T, lanes 64..127: Q K^T  (N = 64)
            if (tid == 0) {
                const uint64_t d = smem_desc(sbase + pKQ, 16, 1024, kSwizzle128B);
                constexpr uint32_t id = idesc_f16kind(128, 64, 0, 0, Op16<T>::fmt);
#pragma unroll
                for (int s = 0; s < 8; ++s) {
                    const uint64_t o = (s >> 2) * 1024 + (s & 3) * 2;
                    mma_bf16(tmem, d + o, d + o, id, s > 0);
                }
                mma_commit(&bar_mma);
            }
            if (!mma_done(2)) break;
            {   // A (fp32) from lanes 0..63, L (bf16, rows 128.. of [..; L]) from lanes 64..127
                float v[32];
                tmem_ld16(tmem + lane_off + half * 32, v);
                tmem_ld16(tmem + lane_off + half * 32 + 16, v + 16);
                tmem_ld_wait();
                const int r = lrow & 63;
                float dec[32];                                   // D[r][half*32 ..]
#pragma unroll
                for (int i = 0; i < 32; i += 4) {
                    const float4 d4 = *reinterpret_cast<const float4 *>(sT + r * kSolveLD + half * 32 + i);
                    dec[i] = d4.x; dec[i + 1] = d4.y; dec[i + 2] = d4.z; dec[i + 3] = d4.w;
                }
                if (lrow < C) {
                    const float br = sB[r];
#pragma unroll
                    for (int i = 0; i < 32; i += 4) {
                        float a[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int col = half * 32 + i + e;
                            a[e] = (col < r && r < len) ? br * dec[i + e] * v[i + e] : 0.f;
                        }
                        *reinterpret_cast<float4 *>(sA + r * kSolveLD + half * 32 + i) =
                            make_float4(a[0], a[1], a[2], a[3]);
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
                        *reinterpret_cast<uint4 *>(smem + pTL + kmaj16(192, 2 * C + r, half * 32 + q * 8)) =
                            pack8_as<T>(l);
                    }
                }
            }
            __syncthreads();
            solve_unit_lower64<kPrepThreads>(sA, sT, sX);   // T = (I + A)^-1
            {
                const bool vl = mbar_wait(&bar_v, ph_in, &s_err, 6);
                if (__syncthreads_or(!vl)) break;
            }
            if (len < C) {
                const uint4 zero = make_uint4(0, 0, 0, 0);
                for (int t = tid; t < 2 * C * 8; t += kPrepThreads) {
                    const int r = (t >> 3) & 63, cb = t >> 9;
                    if (r >= len) *reinterpret_cast<uint4 *>(smem + pV + cb * 8192 + r * 128 + (t & 7) * 16) = zero;
                }
            }
            // ---- T diag(beta Gamma) -> rows 0..63, T diag(beta) -> rows 64..127 (bf16, K-major)
            {
                const int r = tid >> 2;
#pragma unroll
                for (int qq = 0; qq < 2; ++qq) {
                    const int c0 = ((tid & 3) * 2 + qq) * 8;
                    float tb[8], tg[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        tb[e] = c0 + e <= r ? sT[r * kSolveLD + c0 + e] * sB[c0 + e] : 0.f;
                        tg[e] = tb[e] * sEG[c0 + e];
                    }
                    *reinterpret_cast<uint4 *>(smem + pTL + kmaj16(192, r, c0)) = pack8_as<T>(tg);
                    *reinterpret_cast<uint4 *>(smem + pTL + kmaj16(192, C + r, c0)) = pack8_as<T>(tb);
                }
            }
            to_async();
            // ---- MMA2: [T bG; T b] K -> cols 0..127 (W in lanes 0..63);
            //            [T bG; T b] V -> cols 128..255 (U in lanes 64..127).
            // K and V are MN-major B operands (64-element atoms 16 KiB and 8 KiB apart).
            if (tid == 0) {
                const uint64_t a = smem_desc(sbase + pTL, 16, 1024, kSwizzle128B);
                const uint64_t bk = smem_desc(sbase + pKQ, 16384, 1024, kSwizzle128B);
                const uint64_t bv = smem_desc(sbase + pV, 8192, 1024, kSwizzle128B);
                constexpr uint32_t id = idesc_f16kind(128, 128, 0, 1, Op16<T>::fmt);
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
                    *reinterpret_cast<uint4 *>(smem + pA + mnmaj16(8192, tok, n0 + q * 8)) = pack8_as<T>(wu + q * 8);
                // Ktil = diag(exp(g_c - g)) K, in place (MMA2 has consumed K)
                for (int t = tid; t < 2 * C * 8; t += kPrepThreads) {
                    const int r = (t >> 3) & 63, cb = t >> 9;
                    uint4 *pk = reinterpret_cast<uint4 *>(smem + pKQ + cb * 16384 + r * 128 + (t & 7) * 16);
                    float y[8];
                    unpack8_as<T>(*pk, y);
                    const float f = sF[r];
#pragma unroll
                    for (int e = 0; e < 8; ++e) y[e] *= f;
                    *pk = pack8_as<T>(y);
                }
            }
            to_async();
            // ---- MMA4: [T b; L] [W | U] -> lanes 64..127: L W (cols 0..127), L U (cols 128..255)
            if (tid == 0) {
                const uint64_t a = smem_desc(sbase + pTL + 8192, 16, 1024, kSwizzle128B);
                const uint64_t b = smem_desc(sbase + pA, 8192, 1024, kSwizzle128B);
                constexpr uint32_t id = idesc_f16kind(128, 256, 0, 1, Op16<T>::fmt);
#pragma unroll
                for (int s = 0; s < 4; ++s) mma_bf16(tmem, a + s * 2, b + s * 128, id, s > 0);
                mma_commit(&bar_mma);
            }
            if (!mma_done(4)) break;
            // Outputs leave through shared memory in 64 x 64 boxes (128-byte swizzle) and TMA
            // stores of the record rows: Y 0..63, N 64..191, B 192..319, Z 320..383.
            if (lrow >= C) {   // Y = scale diag(Gamma) Q - L W and Z = L U, row r, columns half*64..
                const int r = lrow - C;
                const float fq = sFQ[r];
                const bool live = r < len;
                float x[64];
#pragma unroll
                for (int q = 0; q < 4; ++q) tmem_ld16(tmem + lane_off + half * 64 + q * 16, x + q * 16);
                tmem_ld_wait();
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const int c = half * 64 + q * 8;
                    float qf[8], y[8];
                    unpack8_as<T>(*reinterpret_cast<const uint4 *>(smem + pKQ + kmaj16(128, C + r, c)), qf);
#pragma unroll
                    for (int e = 0; e < 8; ++e) y[e] = live ? fmaf(fq, qf[e], -x[q * 8 + e]) : 0.f;
                    *reinterpret_cast<uint4 *>(box_chunk(pV + half * 8192, r, q)) = pack8_as<T>(y);
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) tmem_ld16(tmem + lane_off + 128 + half * 64 + q * 16, x + q * 16);
                tmem_ld_wait();
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    float z[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) z[e] = live ? x[q * 8 + e] : 0.f;
                    *reinterpret_cast<uint4 *>(box_chunk(pTL + half * 8192, r, q)) = pack8_as<T>(z);
                }
            }
            if (tid == 0) {
                const float gc = __expf(sG[C - 1]);
                *reinterpret_cast<float4 *>(gGC) = make_float4(gc, 0.f, 0.f, 0.f);
            }
            to_async();
            if (tid == 0) {   // Y and Z boxes
                for (int cb = 0; cb < 2; ++cb) {
                    tma_store_3d(&tm_rec, smem + pV + cb * 8192, cb * 64, 0, unit);
                    tma_store_3d(&tm_rec, smem + pTL + cb * 8192, cb * 64, 320, unit);
                }
                bulk_commit();
            }
            // ---- MMA3: Ktil^T [W | U] -> cols 0..127: Ktil^T W = -N, cols 128..255: B
            if (tid == 0) {
                const uint64_t a = smem_desc(sbase + pKQ, 16384, 1024, kSwizzle128B);
                const uint64_t b = smem_desc(sbase + pA, 8192, 1024, kSwizzle128B);
                constexpr uint32_t id = idesc_f16kind(128, 256, 1, 1, Op16<T>::fmt);
#pragma unroll
                for (int s = 0; s < 4; ++s) mma_bf16(tmem, a + s * 128, b + s * 128, id, s > 0);
                mma_commit(&bar_mma);
            }
            // the next item and its gates, while MMA3 runs
            const int inext = next_item(p, icur + stride, stride, &nxt);
            if (inext >= 0) load_gates(nxt, g_raw, b_raw);
            if (!mma_done(5)) break;
            if (tid == 0) {
                if (inext >= 0) load_kq(nxt);          // K and Q of this item are consumed
                bulk_wait_read();                      // the Y and Z stores have read pV, pTL
            }
            __syncthreads();
            {   // key row m = lrow: half 0 -> N boxes in the [W | U] buffer, half 1 -> B boxes
                // (0, 0), (0, 1), (1, 0) in the [..; L] buffer and (1, 1) in the V buffer
                const int m = lrow;
                const float sg = half == 0 ? -1.f : 1.f;
#pragma unroll
                for (int pass = 0; pass < 2; ++pass) {
                    const int bidx = (m >> 6) * 2 + pass;
                    const uint32_t box = half == 0 ? pA + bidx * 8192 : (bidx < 3 ? pTL + bidx * 8192 : pV);
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
                        *reinterpret_cast<uint4 *>(box_chunk(box, m & 63, q)) = pack8_as<T>(y);
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
                        tma_store_3d(&tm_rec, smem + pA + bidx * 8192, cb * 64, 64 + rb * 64, unit);
                        tma_store_3d(&tm_rec, smem + (bidx < 3 ? pTL + bidx * 8192 : pV), cb * 64,
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

// ============================================================================ chain_t
struct ChainTParams {
    const int32_t *cu, *chunk_offsets, *seq_order;
    const float *h0;
    const uint8_t *ws;
    void *o;                     // [t_max, H, V] of the input type
    float *ht, *h_save;
    int32_t *status;
    int64_t t_max, nt_max;
    int32_t n_max, H;
    // Segment-parallel Reduce (HA-NPU section 4, third tier): a sequence of nch chunks is cut
    // into n_seg segments of ceil(nch / n_seg) chunks, blockIdx.z = sequence slot * n_seg + segment.
    // mode 0: the whole recurrence (n_seg = 1);
    // mode 1: segment summaries over 256 state columns -- columns 0..127 start at the identity and
    //         take no B (they become the segment's transition M), columns 128..255 start at zero
    //         and take B (they become its offset); the end state goes to seg_sum[unit][segment]
    //         as M transposed [128][128] then B transposed [128][128] (the last segment of a
    //         sequence has no summary to give);
    // mode 2: each segment's recurrence from its start state (h0 for segment 0, else
    //         seg_start[unit][segment] as [128][128]); the last segment writes ht.
    int32_t mode, n_seg;
    float *seg_sum;
    const float *seg_start;
};

// Shared memory: NS stages of {[Y; N] (two 64-column blocks of 192 rows, 128-byte
// swizzle), B slice [128][VS], Z slice [64][VS], the Gamma_c slot}, then three bf16 copies of the
// state slice S as MN-major B operands (VS used columns of a 64-element atom): S(n) in
// buffer n % 3, so the copy of S(n+1) overwrites the one G2 read two chunks earlier.
template <int VS, int NS>
struct ChainTLayout {
    static constexpr uint32_t kYN = 49152, kB = VS * 256, kZ = VS * 128, kG = kGBytes;
    static constexpr uint32_t oYN = 0, oB = kYN, oZ = oB + kB, oG = oZ + kZ;
    static constexpr uint32_t kStage = (oG + kG + 1023) / 1024 * 1024;
    static constexpr int kSB = 3;                                // bf16 copies of S
    static constexpr uint32_t oSB = NS * kStage;                 // kSB buffers of 16 KiB
    static constexpr uint32_t total = oSB + kSB * 16384;
    static constexpr uint32_t bytes = total + 1024;              // + alignment slack
    static constexpr uint32_t kTmaBytes = kYN + kB + kZ + kG;
};

constexpr int kComputeThreads = 256;                  // warps 0..7: the state
constexpr int kOutWarps = 2;                          // warps 8, 9: the output rows 0..63
constexpr int kG1Parts = 2;                           // G1 issued from two threads, two accumulators
constexpr int kWarpG1 = 8 + kOutWarps;                // first G1 warp
constexpr int kWarpG2 = kWarpG1 + kG1Parts;
constexpr int kWarpTma = kWarpG2 + 1;
constexpr int kChainThreads = 32 * (kWarpTma + 1);


// Per-(sequence, head, column slice) recurrence, warp-specialised:
//   warps 0..7   the state: thread t owns key row 32 (w & 3) + (t & 31) of the state slice and
//                the column half (w >> 2); S(n+1) = Gamma_c S(n) + B + D1 -> Sb[(n+1) % 3];
//                each warp hands its part over with its own mbarrier arrival;
//   warps 8, 9   the output: token rows 32 (w - 8) + (t & 31); O(n) = D2 + Z;
//   warps 10, 11 (one lane each) G1(n) = N S(n), split over the key dimension into two
//                accumulators (the serial step: it alone sits between S(n) and S(n+1));
//   warp 12      G2(n) = [Y; N_top] S(n) -> D2[n & 1] (the output, off the serial path);
//   warp 13      the TMA loads of chunk n + NS once chunk n's stage is released.
// Every mbarrier waited on by parity is re-armed only after its waiter has passed (barriers
// that a faster party could lap come in sets indexed by chunk: pairs, or four for the hand-off
// of S to G2, which the state warps may run up to three chunks ahead of), so no waiter can
// fall two phases behind.  After a failed (timed-out) wait every further wait returns at once, so
// all loops run to their ends without a uniform break.
// KDA: Gamma_c is a per-key-channel vector (the state row of thread t decays by its own entry).
// T: the records' and the state copies' type (the input type: bf16, or fp16 for GDN).
template <int VS, int NS, bool KDA, typename T>
__global__ void __launch_bounds__(kChainThreads, 1)
tc_chain_t_kernel(const __grid_constant__ CUtensorMap tm_yn, const __grid_constant__ CUtensorMap tm_b,
                  const __grid_constant__ CUtensorMap tm_z, ChainTParams p) {
    using Lay = ChainTLayout<VS, NS>;
    constexpr int HV = VS / 2;                          // columns per state thread
    constexpr int KS = 8 / kG1Parts;                    // K-steps (16 keys) per G1 part
    constexpr uint32_t tD1 = 0, tD2 = kG1Parts * VS;    // D1 parts | D2 (two buffers)
    constexpr uint32_t kCols = (kG1Parts + 2) * VS;
    constexpr uint32_t kTmemCols = kCols <= 32 ? 32 : kCols <= 64 ? 64 : kCols <= 128 ? 128 : 256;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    __shared__ uint64_t bar_tma[NS], bar_free[NS], bar_sb1, bar_sb2[4], bar_g1[kG1Parts], bar_g2[3],
        bar_d2free[2];
    __shared__ uint32_t s_tmem;
    __shared__ int s_err;

    // a segmented launch waits for the grid before it in full (the records, the start states)
    // before any exit, so that its own completion implies theirs
    if (p.mode != 0) grid_dependency_wait();
    if (status_blocks_cta(p.status)) return;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3, half = (warp >> 2) & 1;
    const int row = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const int split = blockIdx.x, h = blockIdx.y;
    const int zs = p.mode == 0 ? (int)blockIdx.z : (int)blockIdx.z / p.n_seg;
    const int seg = p.mode == 0 ? 0 : (int)blockIdx.z % p.n_seg;
    const int n = p.seq_order ? p.seq_order[zs] : zs;
    const int H = p.H, v0 = split * VS;
    // the record columns of this slice: in mode 1 the B columns 128.. of the state are the record's
    const int vr = p.mode == 1 ? (v0 >= VD ? v0 - VD : 0) : v0;
    if (n < 0 || n >= p.n_max) {
        if (tid == 0) status_set(p.status, GCL_DEV_BAD_RANGE);
        return;
    }
    const int64_t bos = p.cu[n], eos = p.cu[n + 1];
    if (bos < 0 || eos < bos || eos > p.t_max) {
        if (tid == 0) status_set(p.status, GCL_DEV_BAD_RANGE);
        return;
    }
    const int nch_seq = (int)((eos - bos + C - 1) / C);
    const int64_t row0 = p.chunk_offsets[n];
    if (nch_seq > 0 && (row0 < 0 || row0 + nch_seq > p.nt_max)) {
        if (tid == 0) status_set(p.status, GCL_DEV_BAD_RANGE);
        return;
    }
    // this CTA's chunks [cb, cb + nch) of the sequence; segments past the end have nothing to do
    // (segment 0 of an empty sequence still passes h0 through to ht in mode 2)
    const int seg_len = p.mode == 0 ? nch_seq : (nch_seq + p.n_seg - 1) / p.n_seg;
    const int cb = seg * seg_len;
    const int nch = max(0, min(seg_len, nch_seq - cb));
    const bool last_seg = cb + nch >= nch_seq;
    if (p.mode == 1 && (nch == 0 || last_seg)) return;
    if (p.mode == 2 && nch == 0 && !(seg == 0 && nch_seq == 0)) return;
    const bool add_b = !(p.mode == 1 && v0 < VD);       // mode 1: the M columns take no B
    const int64_t unit_idx = (int64_t)n * p.H + h;
    const uint32_t sbase = smem_u32(smem);
    const int64_t KV = (int64_t)KD * VD;
    const int64_t state_base = ((int64_t)n * H + h) * KV;

    if (tid == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(&bar_tma[i], 1);
            mbar_init(&bar_free[i], kComputeThreads / 32 + kOutWarps);
        }
        mbar_init(&bar_sb1, kComputeThreads / 32);
        for (int i = 0; i < 4; ++i) mbar_init(&bar_sb2[i], kComputeThreads / 32);
        for (int i = 0; i < 2; ++i) mbar_init(&bar_d2free[i], kOutWarps);
        for (int i = 0; i < 3; ++i) mbar_init(&bar_g2[i], 1);
        for (int i = 0; i < kG1Parts; ++i) mbar_init(&bar_g1[i], 1);
        s_err = 0;
        fence_barrier_init();
    }
    if (warp == kWarpG1) {
        tmem_alloc(&s_tmem, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    constexpr uint32_t idm = idesc_f16kind(128, VS, 0, 1, Op16<T>::fmt);
    auto dS = [&](int ic) {                          // S(ic) as the MN-major B operand
        return smem_desc(sbase + Lay::oSB + (ic % Lay::kSB) * 16384, 8192, 1024, kSwizzle128B);
    };
    auto dYN = [&](int st) {                         // [Y; N] of a stage, K-major
        return smem_desc(sbase + st * Lay::kStage + Lay::oYN, 16, 1024, kSwizzle128B);
    };

    if (warp >= kWarpG1 && warp < kWarpG1 + kG1Parts) {
        // ============================================ G1 part (lane 0)
        const int part = warp - kWarpG1;
        if (lane == 0) {
            for (int ic = 0; ic < nch; ++ic) {
                const int st = ic % NS;
                if (!mbar_wait(&bar_tma[st], (ic / NS) & 1, &s_err, 7)) break;
                if (!mbar_wait(&bar_sb1, ic & 1, &s_err, 8)) break;
                tc_fence_after();
                const uint64_t a = dYN(st) + (8192 >> 4), b = dS(ic);   // N: rows 64..191
#pragma unroll
                for (int j = 0; j < KS; ++j) {
                    const int s = part * KS + j;
                    mma_bf16(tmem + tD1 + part * VS, a + (s >> 2) * (24576 >> 4) + (s & 3) * 2,
                             b + s * 128, idm, j > 0);
                }
                mma_commit(&bar_g1[part]);
            }
        }
    } else if (warp == kWarpG2) {
        // ============================================ G2 (lane 0)
        if (lane == 0) {
            for (int ic = 0; ic < nch; ++ic) {
                const int st = ic % NS;
                if (!mbar_wait(&bar_tma[st], (ic / NS) & 1, &s_err, 9)) break;
                // the state warps may hand over S(ic + 1) and S(ic + 2) before this wait (they
                // only wait for G2 two chunks back), so the hand-off barriers come in fours
                if (!mbar_wait(&bar_sb2[ic % 4], (ic / 4) & 1, &s_err, 10)) break;
                // D2[ic & 1] has been read for chunk ic - 2
                if (ic >= 2 && !mbar_wait(&bar_d2free[ic & 1], ((ic - 2) >> 1) & 1, &s_err, 12)) break;
                tc_fence_after();
                const uint64_t a = dYN(st), b = dS(ic);                // [Y; N_top]: rows 0..127
#pragma unroll
                for (int s = 0; s < 8; ++s)
                    mma_bf16(tmem + tD2 + (ic & 1) * VS, a + (s >> 2) * (24576 >> 4) + (s & 3) * 2,
                             b + s * 128, idm, s > 0);
                mma_commit(&bar_g2[ic % 3]);
            }
        }
    } else if (warp == kWarpTma) {
        // ============================================ TMA producer (lane 0)
        if (lane == 0) {
            auto issue_tma = [&](int ic) {
                const int st = ic % NS;
                const int unit = (int)((row0 + cb + ic) * H + h);
                uint64_t *bar = &bar_tma[st];
                uint8_t *b = smem + st * Lay::kStage;
                mbar_arrive_expect_tx(bar, Lay::kTmaBytes);
                tma_load_3d(b + Lay::oYN, &tm_yn, 0, 0, unit, bar);
                tma_load_3d(b + Lay::oYN + 24576, &tm_yn, 64, 0, unit, bar);
                tma_load_3d(b + Lay::oB, &tm_b, vr, 0, unit, bar);
                tma_load_3d(b + Lay::oZ, &tm_z, vr, 0, unit, bar);
                bulk_load(b + Lay::oG, p.ws + gc_offset(p.nt_max, H, unit), kGBytes, bar);
            };
            grid_dependency_wait();      // the records are complete (launched as a dependent)
            for (int ic = 0; ic < nch; ++ic) {
                if (ic >= NS && !mbar_wait(&bar_free[ic % NS], ((ic - NS) / NS) & 1, &s_err, 11)) break;
                issue_tma(ic);
            }
        }
    } else if (warp >= 8) {
        // ============================================ output (warps 8, 9): O(n) = Y S(n) + Z
        const int orow = (warp - 8) * 32 + lane;               // token row = TMEM lane
        const uint32_t olane = (uint32_t)((warp - 8) * 32) << 16;
        for (int ic = 0; ic < nch; ++ic) {
            const int st = ic % NS;
            const int64_t rem = eos - bos - (int64_t)(cb + ic) * C;
            const int len = (int)(rem < C ? rem : C);
            const int64_t t0 = bos + (int64_t)(cb + ic) * C;
            const uint8_t *stage = smem + st * Lay::kStage;
            mbar_wait(&bar_tma[st], (ic / NS) & 1, &s_err, 5);
            mbar_wait(&bar_g2[ic % 3], (ic / 3) & 1, &s_err, 6);
            tc_fence_after();
            float d2[VS];
#pragma unroll
            for (int j = 0; j < VS; j += 8) tmem_ld8(tmem + olane + tD2 + (ic & 1) * VS + j, d2 + j);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_d2free[ic & 1]);
            if (orow < len && p.o != nullptr &&
                GCL_RANGE_IN_BOUNDS(((t0 + orow) * H + h) * (int64_t)VD + v0,
                                    ((t0 + orow) * H + h) * (int64_t)VD + v0 + VS - 1,
                                    p.t_max * H * (int64_t)VD, p.status)) {
                const uint8_t *zrow = stage + Lay::oZ + orow * (VS * 2);
                T *dst = static_cast<T *>(p.o) + ((t0 + orow) * H + h) * (int64_t)VD + v0;
#pragma unroll
                for (int j = 0; j < VS; j += 8) {
                    float zf[8];
                    unpack8_as<T>(*reinterpret_cast<const uint4 *>(zrow + j * 2), zf);
                    float ov[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) ov[e] = d2[j + e] + zf[e];
                    *reinterpret_cast<uint4 *>(dst + j) = pack8_as<T>(ov);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_free[st]);        // done with Z of stage st
        }
    } else {
        // ============================================ state (warps 0..7)
        const int c0 = half * HV;
        auto st_sb = [&](int buf, const float *x) {       // bf16 copy of this thread's S values
#pragma unroll
            for (int j = 0; j < HV; j += 8)
                *reinterpret_cast<uint4 *>(smem + Lay::oSB + buf * 16384 + mn_sw128(row, c0 + j)) =
                    pack8_as<T>(x + j);
        };
        auto handoff = [&](int ic) {                      // this warp's part of S(ic) is in its buffer
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&bar_sb1);
                mbar_arrive(&bar_sb2[ic % 4]);
            }
        };
        float S[HV];
        if (p.mode == 1) {                                // [I | 0]
#pragma unroll
            for (int j = 0; j < HV; ++j) S[j] = row == v0 + c0 + j ? 1.f : 0.f;
        } else {
            const float *src = seg > 0 ? p.seg_start + (((unit_idx * p.n_seg + seg) * KD + row) * VD + v0 + c0)
                               : (p.h0 && GCL_RANGE_IN_BOUNDS(state_base + (int64_t)row * VD + v0 + c0,
                                                              state_base + (int64_t)row * VD + v0 + c0 + HV - 1,
                                                              (int64_t)p.n_max * H * KV, p.status))
                                   ? p.h0 + state_base + (int64_t)row * VD + v0 + c0
                                   : nullptr;
#pragma unroll
            for (int j = 0; j < HV; ++j) S[j] = src ? src[j] : 0.f;
        }
        st_sb(0, S);
        handoff(0);
        for (int ic = 0; ic < nch; ++ic) {
            const int st = ic % NS;
            const uint8_t *stage = smem + st * Lay::kStage;
            if (p.h_save &&
                GCL_RANGE_IN_BOUNDS(((row0 + cb + ic) * H + h) * KV + (int64_t)row * VD + v0 + c0,
                                    ((row0 + cb + ic) * H + h) * KV + (int64_t)row * VD + v0 + c0 + HV - 1,
                                    p.nt_max * H * KV, p.status)) {
                float *dst = p.h_save + ((row0 + cb + ic) * H + h) * KV + (int64_t)row * VD + v0 + c0;
#pragma unroll
                for (int j = 0; j < HV; j += 4)
                    *reinterpret_cast<float4 *>(dst + j) = make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
            }
            mbar_wait(&bar_tma[st], (ic / NS) & 1, &s_err, 3);
            if (!add_b) {   // Gamma_c S (the transition columns of a segment summary)
                const float gc = reinterpret_cast<const float *>(stage + Lay::oG)[KDA ? row : 0];
#pragma unroll
                for (int j = 0; j < HV; ++j) S[j] *= gc;
            } else {   // Gamma_c S + B while G1 runs
                const float gc = reinterpret_cast<const float *>(stage + Lay::oG)[KDA ? row : 0];
                const uint8_t *brow = stage + Lay::oB + row * (VS * 2) + c0 * 2;
#pragma unroll
                for (int j = 0; j < HV; j += 8) {
                    float bf[8];
                    unpack8_as<T>(*reinterpret_cast<const uint4 *>(brow + j * 2), bf);
#pragma unroll
                    for (int e = 0; e < 8; ++e) S[j + e] = fmaf(gc, S[j + e], bf[e]);
                }
            }
            {   // + N S(n): the G1 parts
                float d1[kG1Parts][HV];
#pragma unroll
                for (int part = 0; part < kG1Parts; ++part) {
                    mbar_wait(&bar_g1[part], ic & 1, &s_err, 4);
                    tc_fence_after();
#pragma unroll
                    for (int j = 0; j < HV; j += 8)
                        tmem_ld8(tmem + lane_off + tD1 + part * VS + c0 + j, d1[part] + j);
                }
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < HV; ++j) {
#pragma unroll
                    for (int part = 0; part < kG1Parts; ++part) S[j] += d1[part][j];
                }
            }
            // Sb[(ic + 1) % 3] was last read by G1 and G2 of chunk ic - 2 (long complete)
            if (ic >= 2) mbar_wait(&bar_g2[(ic - 2) % 3], ((ic - 2) / 3) & 1, &s_err, 13);
            st_sb((ic + 1) % Lay::kSB, S);
            handoff(ic + 1);
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_free[st]);        // done with B of stage st
        }
        if (p.mode == 1 && *reinterpret_cast<volatile int *>(&s_err) == 0) {
            float *blk = p.seg_sum + (unit_idx * p.n_seg + seg) * (2 * KD * VD);
            if (v0 < VD) {                                // M, transposed: [k][row]
#pragma unroll
                for (int j = 0; j < HV; ++j) blk[(int64_t)(v0 + c0 + j) * KD + row] = S[j];
            } else {                                      // B, transposed: [v][row]
#pragma unroll
                for (int j = 0; j < HV; ++j) blk[KD * KD + (int64_t)(v0 - VD + c0 + j) * KD + row] = S[j];
            }
        } else if (p.ht && last_seg && *reinterpret_cast<volatile int *>(&s_err) == 0 &&
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
    if (warp == kWarpG1) tmem_dealloc(tmem, kTmemCols);
    if (tid == 0 && s_err != 0) status_set(p.status, GCL_DEV_WAIT_TIMEOUT);
}

// ============================================================================ segment scan
// The start states of the segments: S(s + 1) = M(s) S(s) + B(s) from S(0) = h0, in fp32, one
// CTA per (kScanSC value columns, head, sequence slot).  A segment summary is M transposed
// ([k][i], 64 KiB) then B transposed ([v][i], 64 KiB).  M(s) and the CTA's kScanSC rows of B(s)
// arrive by bulk copies one segment ahead (two buffers, one mbarrier each).  Warp w adds the
// products of key rows 16 w .. 16 w + 15, lane l owning state rows 4 l .. 4 l + 3 and all
// kScanSC columns (every M value read once, the S row broadcast); thread t < 128 then adds
// the eight warps' partial sums for state row t in warp order.
struct SegScanParams {
    const int32_t *cu;
    const float *h0, *seg_sum;
    float *seg_start;
    int32_t *status;
    int64_t t_max;
    int32_t n_max, H, n_seg;
};
constexpr int kScanSC = 4, kScanWarps = 8, kScanThreads = 32 * kScanWarps, kScanKW = KD / kScanWarps;
struct ScanLayout {
    static constexpr int oMT = 0, oBT = oMT + 2 * KD * KD, oS = oBT + 2 * kScanSC * KD;
    static constexpr int oRed = oS + KD * kScanSC, floats = oRed + kScanWarps * KD * kScanSC;
    static constexpr int bytes = floats * (int)sizeof(float);
    static constexpr uint32_t kTx = (KD * KD + kScanSC * KD) * sizeof(float);
};
static_assert(kScanSC == 4 && KD == 4 * 32 && KD <= kScanThreads, "scan thread mapping");

__global__ void __launch_bounds__(kScanThreads, 1) seg_scan_kernel(SegScanParams p) {
    extern __shared__ __align__(128) float sm_scan[];
    __shared__ uint64_t bar[2];
    __shared__ int s_err;
    float *sS = sm_scan + ScanLayout::oS;                // [KD][kScanSC]
    float *sRed = sm_scan + ScanLayout::oRed;            // [kScanWarps][KD][kScanSC]
    grid_dependency_wait();                              // the segment summaries are complete
    if (status_blocks_cta(p.status)) return;
    const int c0 = blockIdx.x * kScanSC, h = blockIdx.y, n = blockIdx.z;
    const int64_t bos = p.cu[n], eos = p.cu[n + 1];
    if (bos < 0 || eos < bos || eos > p.t_max) return;  // reported by the chain
    const int nch = (int)((eos - bos + C - 1) / C);
    if (nch == 0) return;
    const int seg_len = (nch + p.n_seg - 1) / p.n_seg, nseg = (nch + seg_len - 1) / seg_len;
    if (nseg < 2) return;
    const int64_t unit = (int64_t)n * p.H + h;
    constexpr int64_t kSum = 2 * KD * VD;                // floats per summary
    const float *sum0 = p.seg_sum + unit * p.n_seg * kSum;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int issued[2] = {0, 0};                              // copies issued per buffer (thread 0)
    auto issue = [&](int sg) {                           // M(sg)^T and B(sg)^T rows c0 .. into buffer sg & 1
        const int b = sg & 1;
        const float *src = sum0 + sg * kSum;
        mbar_arrive_expect_tx(&bar[b], ScanLayout::kTx);
        bulk_load(sm_scan + ScanLayout::oMT + b * (KD * KD), src, KD * KD * sizeof(float), &bar[b]);
        bulk_load(sm_scan + ScanLayout::oBT + b * (kScanSC * KD), src + KD * KD + (int64_t)c0 * KD,
                  kScanSC * KD * sizeof(float), &bar[b]);
        ++issued[b];
    };
    if (tid == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        s_err = 0;
        fence_barrier_init();
    }
    if (tid < KD)
        *reinterpret_cast<float4 *>(sS + tid * kScanSC) =
            p.h0 ? *reinterpret_cast<const float4 *>(p.h0 + (unit * KD + tid) * VD + c0)
                 : make_float4(0.f, 0.f, 0.f, 0.f);
    __syncthreads();
    if (tid == 0) issue(0);
    for (int sg = 0; sg + 1 < nseg; ++sg) {
        // buffer (sg + 1) & 1 was last read before the previous step's first barrier
        if (tid == 0 && sg + 2 < nseg) issue(sg + 1);
        mbar_wait(&bar[sg & 1], (sg >> 1) & 1, &s_err, 1);
        const float *mt = sm_scan + ScanLayout::oMT + (sg & 1) * (KD * KD);
        const float *bt = sm_scan + ScanLayout::oBT + (sg & 1) * (kScanSC * KD);
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (tid < KD) v = make_float4(bt[tid], bt[KD + tid], bt[2 * KD + tid], bt[3 * KD + tid]);
        float acc[4][kScanSC];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < kScanSC; ++j) acc[i][j] = 0.f;
#pragma unroll
        for (int kk = 0; kk < kScanKW; ++kk) {
            const int k = warp * kScanKW + kk;
            const float4 a = *reinterpret_cast<const float4 *>(mt + k * KD + 4 * lane);
            const float4 b = *reinterpret_cast<const float4 *>(sS + k * kScanSC);
            const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < kScanSC; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
            *reinterpret_cast<float4 *>(sRed + (warp * KD + 4 * lane + i) * kScanSC) =
                make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
        __syncthreads();                                 // every partial sum is written; S(sg) is read
        if (tid < KD) {
#pragma unroll
            for (int w = 0; w < kScanWarps; ++w) {
                const float4 r = *reinterpret_cast<const float4 *>(sRed + (w * KD + tid) * kScanSC);
                v.x += r.x;
                v.y += r.y;
                v.z += r.z;
                v.w += r.w;
            }
            *reinterpret_cast<float4 *>(sS + tid * kScanSC) = v;
            *reinterpret_cast<float4 *>(p.seg_start + ((unit * p.n_seg + sg + 1) * KD + tid) * VD + c0) = v;
        }
        __syncthreads();                                 // S(sg + 1) is complete; the partial sums are read
    }
    if (tid == 0 && *reinterpret_cast<volatile int *>(&s_err) != 0) {
        // a copy did not arrive in time: wait (bounded) for the last copy into each buffer
        for (int b = 0; b < 2; ++b) {
            if (issued[b] == 0) continue;
            const uint64_t t0 = globaltimer();
            while (!mbar_try_wait(&bar[b], (issued[b] - 1) & 1) && globaltimer() - t0 < kWaitLimitNs) {
            }
        }
        status_set(p.status, GCL_DEV_WAIT_TIMEOUT);
    }
}

template <int VS, int NS, bool KDA, typename T>
cudaError_t launch_chain_t(const CUtensorMap &myn, const uint8_t *ws, const ChainTParams &cp,
                           int n_split, int H, int n_max, cudaStream_t s) {
    using Lay = ChainTLayout<VS, NS>;
    static_assert(Lay::bytes <= 232448, "chain_t shared memory");
    const int64_t units = cp.nt_max * H;
    CUtensorMap mb, mz;
    const cuuint64_t db[3] = {(cuuint64_t)VD, (cuuint64_t)KD, (cuuint64_t)units};
    const cuuint64_t sb[2] = {(cuuint64_t)VD * 2, (cuuint64_t)kUnitBytes};
    const cuuint32_t bb[3] = {(cuuint32_t)VS, (cuuint32_t)KD, 1};
    const cuuint64_t dz[3] = {(cuuint64_t)VD, (cuuint64_t)C, (cuuint64_t)units};
    const cuuint32_t bz[3] = {(cuuint32_t)VS, (cuuint32_t)C, 1};
    if (!make_tensor_map(&mb, ws + kYNBytes, 3, db, sb, bb, CU_TENSOR_MAP_SWIZZLE_NONE, Op16<T>::tma) ||
        !make_tensor_map(&mz, ws + kYNBytes + kBBytes, 3, dz, sb, bz, CU_TENSOR_MAP_SWIZZLE_NONE, Op16<T>::tma))
        return cudaErrorInvalidValue;
    auto kern = tc_chain_t_kernel<VS, NS, KDA, T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)Lay::bytes);
    if (e != cudaSuccess) return e;
    // launched as a programmatic dependent of the prep: its prologue overlaps the prep's tail
    return launch_dependent(kern, dim3(n_split, H, n_max * (cp.mode == 0 ? 1 : cp.n_seg)), dim3(kChainThreads),
                            Lay::bytes, s, myn, mb, mz, cp);
}

}  // namespace

size_t fwd_tc_t_workspace_bytes(int64_t nt_max, int H) {
    return (size_t)nt_max * H * (kUnitBytes + kGBytes);
}

size_t transition_record_bytes(int64_t nt_max, int H) { return fwd_tc_t_workspace_bytes(nt_max, H); }

bool make_prep_maps(const FwdParams &p, uint8_t *ws, CUtensorMap *mq, CUtensorMap *mk, CUtensorMap *mv,
                    CUtensorMap *mrec) {
    const int H = p.H;
    const int64_t units = p.nt_max * H;
    const cuuint64_t dqk[3] = {(cuuint64_t)KD, (cuuint64_t)H, (cuuint64_t)p.t_max};
    const cuuint64_t sqk[2] = {(cuuint64_t)KD * 2, (cuuint64_t)H * KD * 2};
    const cuuint32_t b64[3] = {64, 1, 64};
    const cuuint64_t dv[3] = {(cuuint64_t)VD, (cuuint64_t)H, (cuuint64_t)p.t_max};
    const cuuint64_t sv[2] = {(cuuint64_t)VD * 2, (cuuint64_t)H * VD * 2};
    // the record as 384 rows of 128 bf16, 64 x 64 boxes
    const cuuint64_t drec[3] = {(cuuint64_t)KD, (cuuint64_t)(kUnitBytes / (KD * 2)), (cuuint64_t)units};
    static_assert(kUnitBytes % (KD * 2) == 0, "a record is whole rows");
    const cuuint64_t srec[2] = {(cuuint64_t)KD * 2, (cuuint64_t)kUnitBytes};
    const cuuint32_t brec[3] = {64, 64, 1};
    const CUtensorMapDataType dt = p.dtype == GCL_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                      : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    return make_tensor_map(mq, p.q, 3, dqk, sqk, b64, CU_TENSOR_MAP_SWIZZLE_128B, dt) &&
           make_tensor_map(mk, p.k, 3, dqk, sqk, b64, CU_TENSOR_MAP_SWIZZLE_128B, dt) &&
           make_tensor_map(mv, p.v, 3, dv, sv, b64, CU_TENSOR_MAP_SWIZZLE_128B, dt) &&
           make_tensor_map(mrec, ws, 3, drec, srec, brec, CU_TENSOR_MAP_SWIZZLE_128B, dt);
}

tr::PrepTParams make_prep_params(const FwdParams &p, uint8_t *ws) {
    tr::PrepTParams pp{};
    pp.chunk_indices = p.chunk_indices;
    pp.cu = p.cu_seqlens;
    pp.g = p.g;
    pp.beta = p.beta;
    pp.ws = ws;
    pp.status = p.dev_status;
    pp.t_max = p.t_max;
    pp.nt_max = p.nt_max;
    pp.n_max = p.n_max;
    pp.H = p.H;
    pp.scale = p.scale;
    return pp;
}

template <typename T>
cudaError_t launch_prep_t_as(const FwdParams &p, uint8_t *ws, cudaStream_t s) {
    CUtensorMap mq, mk, mv, mrec;
    if (!make_prep_maps(p, ws, &mq, &mk, &mv, &mrec)) return cudaErrorInvalidValue;
    const PrepTParams pp = make_prep_params(p, ws);
    auto kern = tc_prep_t_kernel<T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kPrepTSmem);
    if (e != cudaSuccess) return e;
    const int64_t units = p.nt_max * p.H;
    const int grid = (int)(units < 2 * (int64_t)num_sms() ? units : 2 * (int64_t)num_sms());
    return launch_dependent(kern, dim3(grid), dim3(kPrepThreads), kPrepTSmem, s, mq, mk, mv, mrec, pp);
}
cudaError_t launch_prep_t(const FwdParams &p, uint8_t *ws, cudaStream_t s) {
    return p.dtype == GCL_F16 ? launch_prep_t_as<__half>(p, ws, s)
                              : launch_prep_t_as<__nv_bfloat16>(p, ws, s);
}

// Segments per sequence: at most one wave of summary CTAs (8 slices of 32 columns per unit),
// the count that minimises the modelled time of summaries + scan + outputs, and only where
// that beats the plain chain.  Chunks per sequence are taken from the capacity
// (nt_max / n_max), so the plan depends on the sizes alone.  Per-chunk and per-step times are
// GB300 measurements of these kernels (ns): summary + output chain per chunk, scan per
// segment, the two extra launches, and the plain chain per chunk.
int fwd_seg_count(int64_t nt_max, int n_max, int H) {
    constexpr int64_t kChainAC = 1830, kScanStep = 1200, kExtra = 8000, kPlain = 700;
    const int64_t units = (int64_t)n_max * H;
    const int64_t p_max = num_sms() / (8 * units);
    if (p_max < 3 || n_max <= 0) return 0;
    const int64_t nc = nt_max / n_max;
    int64_t best = 0, best_t = nc * kPlain;
    for (int64_t P = 3; P <= p_max; ++P) {
        const int64_t t = (nc + P - 1) / P * kChainAC + (P - 1) * kScanStep + kExtra;
        if (t < best_t) {
            best_t = t;
            best = P;
        }
    }
    return (int)best;
}

size_t fwd_seg_workspace_bytes(int64_t nt_max, int n_max, int H) {
    const int P = fwd_seg_count(nt_max, n_max, H);
    return (size_t)n_max * H * P * (size_t)(KD * 2 * VD + KD * VD) * sizeof(float);
}

template <typename T, bool KDA>
cudaError_t launch_chain_records_as(const FwdParams &p, const uint8_t *ws, int split,
                                    cudaStream_t s, int n_seg, float *seg_ws) {
    const int H = p.H;
    const int64_t units = p.nt_max * H;
    CUtensorMap myn;
    const cuuint64_t dyn[3] = {(cuuint64_t)KD, (cuuint64_t)kYNRows, (cuuint64_t)units};
    const cuuint64_t syn[2] = {(cuuint64_t)KD * 2, (cuuint64_t)kUnitBytes};
    const cuuint32_t byn[3] = {64, (cuuint32_t)kYNRows, 1};
    if (!make_tensor_map(&myn, ws, 3, dyn, syn, byn, CU_TENSOR_MAP_SWIZZLE_128B, Op16<T>::tma))
        return cudaErrorInvalidValue;

    ChainTParams cp{};
    cp.cu = p.cu_seqlens;
    cp.chunk_offsets = p.chunk_offsets;
    cp.seq_order = p.seq_order;
    cp.h0 = p.h0;
    cp.ws = ws;
    cp.o = p.o;
    cp.ht = p.ht;
    cp.h_save = p.h_save;
    cp.status = p.dev_status;
    cp.t_max = p.t_max;
    cp.nt_max = p.nt_max;
    cp.n_max = p.n_max;
    cp.H = H;
    cp.n_seg = 1;
    if (n_seg >= 2) {
        // segment summaries (8 slices of 32 over [M | B]), the scan, the segments' outputs
        ChainTParams ca = cp;
        ca.mode = 1;
        ca.n_seg = n_seg;
        ca.o = nullptr;
        ca.ht = nullptr;
        ca.h_save = nullptr;
        ca.seg_sum = seg_ws;
        cudaError_t e = launch_chain_t<32, 2, KDA, T>(myn, ws, ca, 8, H, p.n_max, s);
        if (e != cudaSuccess) return e;
        SegScanParams sp{};
        sp.cu = p.cu_seqlens;
        sp.h0 = p.h0;
        sp.seg_sum = seg_ws;
        sp.seg_start = seg_ws + (size_t)p.n_max * H * n_seg * (KD * 2 * VD);
        sp.status = p.dev_status;
        sp.t_max = p.t_max;
        sp.n_max = p.n_max;
        sp.H = H;
        sp.n_seg = n_seg;
        e = cudaFuncSetAttribute(seg_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, ScanLayout::bytes);
        if (e != cudaSuccess) return e;
        e = launch_dependent(seg_scan_kernel, dim3(VD / kScanSC, H, p.n_max), dim3(kScanThreads),
                             ScanLayout::bytes, s, sp);
        if (e != cudaSuccess) return e;
        cp.mode = 2;
        cp.n_seg = n_seg;
        cp.seg_start = sp.seg_start;
        return launch_chain_t<16, 3, KDA, T>(myn, ws, cp, 8, H, p.n_max, s);
    }
    if (split == 8) return launch_chain_t<16, 3, KDA, T>(myn, ws, cp, split, H, p.n_max, s);
    if (split == 4) return launch_chain_t<32, 2, KDA, T>(myn, ws, cp, split, H, p.n_max, s);
    if (split == 2) return launch_chain_t<64, 2, KDA, T>(myn, ws, cp, split, H, p.n_max, s);
    return cudaErrorInvalidValue;
}

cudaError_t launch_chain_records(const FwdParams &p, const uint8_t *ws, int split, bool kda,
                                 cudaStream_t s, int n_seg, float *seg_ws) {
    if (kda) return launch_chain_records_as<__nv_bfloat16, true>(p, ws, split, s, n_seg, seg_ws);
    if (p.dtype == GCL_F16) return launch_chain_records_as<__half, false>(p, ws, split, s, n_seg, seg_ws);
    return launch_chain_records_as<__nv_bfloat16, false>(p, ws, split, s, n_seg, seg_ws);
}

void fwd_seg_plan(const FwdParams &p, uint8_t *ws, int *n_seg, float **seg_ws) {
    const size_t rec = fwd_tc_t_workspace_bytes(p.nt_max, p.H);
    const size_t need = fwd_seg_workspace_bytes(p.nt_max, p.n_max, p.H);
    *n_seg = 0;
    *seg_ws = nullptr;
    if (need > 0 && p.workspace_bytes >= rec + need) {
        *n_seg = fwd_seg_count(p.nt_max, p.n_max, p.H);
        *seg_ws = reinterpret_cast<float *>(ws + rec);
    }
}

cudaError_t launch_fwd_tc_t(const FwdParams &p, int split, cudaStream_t s) {
    uint8_t *ws = static_cast<uint8_t *>(p.workspace);
    cudaError_t e = launch_prep_t(p, ws, s);
    if (e != cudaSuccess) return e;
    int n_seg = 0;
    float *seg_ws = nullptr;
    fwd_seg_plan(p, ws, &n_seg, &seg_ws);
    return launch_chain_records(p, ws, split, false, s, n_seg, seg_ws);
}

}  // namespace gcl
