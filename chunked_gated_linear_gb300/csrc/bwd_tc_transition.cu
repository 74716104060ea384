// bwd_tc_transition.cu -- the state-gradient sweep of the GDN backward on the tensor cores
// (bf16 inputs, d_k = d_v = 128, chunk 64), from the transition-form records.
//
// FLA RFC "[RFC] Add Graph Capture Support for FLA Prefill and Training Paths on Ascend
// NPUs", section "Step 3": the backward walks the chunks in reverse to carry the state
// gradient.  With the forward of chunk n written as S' = Gamma_c S + N S + B and
// O = Y S + Z (transition.cuh), the gradient w.r.t. the state entering the chunk is
//
//   dS = Gamma_c dS' + N^T dS' + Y^T dO_n,
//
// the transposed recurrence: one small GEMM per chunk on the serial path (N^T dS'), and one
// (Y^T dO_n) that needs no state and is issued ahead.  The sweep saves dS' (the gradient
// w.r.t. the state after every chunk) for the chunk-gradient kernel and writes dh0.
//
// One CTA per (sequence, head, value-column slice): warps 0..7 hold dS' in fp32 registers
// (thread t: key row 32 (w & 3) + (t & 31), column half w >> 2), warp 8 issues the MMAs,
// warp 9 the TMA loads (records and dO tiles, in reverse chunk order, NS stages).
#include <cudaTypedefs.h>

#include "gcl_internal.cuh"
#include "tc_ptx.cuh"
#include "transition.cuh"

namespace gcl {
namespace {

using namespace tc;
using namespace tr;

struct SweepTParams {
    const int32_t *cu, *chunk_offsets;
    const float *dht;
    const uint8_t *ws;          // transition records + Gamma_c slots
    uint8_t *dh;                // dS' per chunk: bf16 tiles of 32 KiB (see below), or
    float *dh_f32;              // (if not null) fp32 [nt_max, H, K, V] for the CUDA-core gradients
    float *dh0;                 // [n_max, H, K, V]
    int32_t *status;
    int64_t t_max, nt_max;
    int32_t n_max, H;
};

// Shared memory per stage: N (rows 64..191 of the record: two 64-column blocks of 128 rows),
// Y (rows 0..63: two blocks of 64 rows), the 64-column dO tile holding this slice, Gamma_c;
// then two bf16 copies of dS' as MN-major B operands.
template <int NS>
struct SweepLayout {
    static constexpr uint32_t kN = 32768, kY = 16384, kDO = 8192, kG = kGBytes;
    static constexpr uint32_t oN = 0, oY = kN, oDO = oY + kY, oG = oDO + kDO;
    static constexpr uint32_t kStage = (oG + kG + 1023) / 1024 * 1024;
    static constexpr uint32_t oDS = NS * kStage;                 // two 16 KiB buffers
    static constexpr uint32_t bytes = oDS + 2 * 16384 + 1024;
    static constexpr uint32_t kTmaBytes = kN + kY + kDO + kG;
};

constexpr int kStateWarps = 8;
constexpr int kSweepThreads = 32 * (kStateWarps + 2);      // + MMA issuer, TMA producer

// Reverse walk: step k handles chunk ic = nch - 1 - k.  Every mbarrier waited on by parity is
// re-armed only after its waiter has passed; a timed-out wait makes every later wait return
// at once, so all loops run to their ends.
// KDA: Gamma_c is a per-key-channel diagonal (dS row m decays by its own entry).
template <int VS, int NS, bool KDA>
__global__ void __launch_bounds__(kSweepThreads, 1)
tc_sweep_t_kernel(const __grid_constant__ CUtensorMap tm_rec128, const __grid_constant__ CUtensorMap tm_rec64,
                  const __grid_constant__ CUtensorMap tm_do, SweepTParams p) {
    using Lay = SweepLayout<NS>;
    constexpr int HV = VS / 2;
    constexpr uint32_t kTmemCols = 2 * VS <= 32 ? 32 : 2 * VS <= 64 ? 64 : 128;   // D x 2
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    __shared__ uint64_t bar_tma[NS], bar_free[NS], bar_ops, bar_ds, bar_g;
    __shared__ uint32_t s_tmem;
    __shared__ int s_err;

    if (status_blocks_cta(p.status)) return;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3, half = (warp >> 2) & 1;
    const int row = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const int split = blockIdx.x, h = blockIdx.y, n = blockIdx.z;
    const int H = p.H, v0 = split * VS;
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

    if (tid == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(&bar_tma[i], 1);
            mbar_init(&bar_free[i], kStateWarps);
        }
        mbar_init(&bar_ops, kStateWarps);
        mbar_init(&bar_ds, kStateWarps);
        mbar_init(&bar_g, 1);
        s_err = 0;
        fence_barrier_init();
    }
    if (warp == kStateWarps) {
        tmem_alloc(&s_tmem, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    auto chunk_of = [&](int k) { return nch - 1 - k; };

    if (warp == kStateWarps) {
        // ============================================ MMA issuer (lane 0)
        if (lane == 0) {
            constexpr uint32_t id = idesc_bf16(128, VS, 1, 1);   // A (N^T, Y^T) and B MN-major
            for (int k = 0; k < nch; ++k) {
                const int st = k % NS;
                const uint32_t sb = sbase + st * Lay::kStage;
                const uint32_t d = tmem + (k & 1) * VS;
                if (!mbar_wait(&bar_tma[st], (k / NS) & 1, &s_err, 7)) break;
                if (!mbar_wait(&bar_ops, k & 1, &s_err, 8)) break;     // dO rows past len zeroed
                tc_fence_after();
                {   // D = Y^T dO: A = Y^T (MN-major: key blocks 8 KiB apart), K = 64 tokens
                    const uint64_t a = smem_desc(sb + Lay::oY, 8192, 1024, kSwizzle128B);
                    const uint64_t b = smem_desc(sb + Lay::oDO + (v0 & 63) * 2, 8192, 1024, kSwizzle128B);
#pragma unroll
                    for (int s = 0; s < 4; ++s) mma_bf16(d, a + s * 128, b + s * 128, id, s > 0);
                }
                if (!mbar_wait(&bar_ds, k & 1, &s_err, 9)) break;      // dS' of this chunk in its buffer
                tc_fence_after();
                {   // D += N^T dS': A = N^T (MN-major: key blocks 16 KiB apart), K = 128 keys
                    const uint64_t a = smem_desc(sb + Lay::oN, 16384, 1024, kSwizzle128B);
                    const uint64_t b = smem_desc(sbase + Lay::oDS + (k & 1) * 16384, 8192, 1024, kSwizzle128B);
#pragma unroll
                    for (int s = 0; s < 8; ++s) mma_bf16(d, a + s * 128, b + s * 128, id, 1);
                }
                mma_commit(&bar_g);
            }
        }
    } else if (warp == kStateWarps + 1) {
        // ============================================ TMA producer (lane 0)
        if (lane == 0) {
            auto issue_tma = [&](int k) {
                const int st = k % NS, ic = chunk_of(k);
                const int unit = (int)((row0 + ic) * H + h);
                const int t0 = (int)(bos + (int64_t)ic * C);
                uint64_t *bar = &bar_tma[st];
                uint8_t *b = smem + st * Lay::kStage;
                mbar_arrive_expect_tx(bar, Lay::kTmaBytes);
                tma_load_3d(b + Lay::oN, &tm_rec128, 0, 64, unit, bar);          // N: rows 64..191
                tma_load_3d(b + Lay::oN + 16384, &tm_rec128, 64, 64, unit, bar);
                tma_load_3d(b + Lay::oY, &tm_rec64, 0, 0, unit, bar);            // Y: rows 0..63
                tma_load_3d(b + Lay::oY + 8192, &tm_rec64, 64, 0, unit, bar);
                tma_load_3d(b + Lay::oDO, &tm_do, v0 & ~63, h, t0, bar);
                bulk_load(b + Lay::oG, p.ws + gc_offset(p.nt_max, H, unit), kGBytes, bar);
            };
            for (int k = 0; k < nch; ++k) {
                if (k >= NS && !mbar_wait(&bar_free[k % NS], ((k - NS) / NS) & 1, &s_err, 11)) break;
                issue_tma(k);
            }
        }
    } else {
        // ============================================ state gradient (warps 0..7)
        const int c0 = half * HV;
        auto put_ds = [&](int buf, const float *x) {      // bf16 copy of this thread's dS' values
#pragma unroll
            for (int j = 0; j < HV; j += 8)
                *reinterpret_cast<uint4 *>(smem + Lay::oDS + buf * 16384 + mn_sw128(row, c0 + j)) = pack8(x + j);
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_ds);
        };
        float dS[HV];
        {
            const float *src = (p.dht && GCL_RANGE_IN_BOUNDS(state_base + (int64_t)row * VD + v0 + c0,
                                                             state_base + (int64_t)row * VD + v0 + c0 + HV - 1,
                                                             (int64_t)p.n_max * H * KV, p.status))
                                   ? p.dht + state_base + (int64_t)row * VD + v0 + c0 : nullptr;
#pragma unroll
            for (int j = 0; j < HV; ++j) dS[j] = src ? src[j] : 0.f;
        }
        if (nch > 0) put_ds(0, dS);
        for (int k = 0; k < nch; ++k) {
            const int st = k % NS, ic = chunk_of(k);
            const int64_t rem = eos - bos - (int64_t)ic * C;
            const int len = (int)(rem < C ? rem : C);
            uint8_t *stage = smem + st * Lay::kStage;
            if (!GCL_IN_BOUNDS((row0 + ic) * H + h, p.nt_max * H, p.status)) {
                // (debug build: a chunk row outside the state-gradient buffer is skipped)
            } else if (p.dh_f32) {   // the gradient w.r.t. the state after chunk ic, fp32 rows
                float *dst = p.dh_f32 + ((row0 + ic) * H + h) * KV + (int64_t)row * VD + v0 + c0;
#pragma unroll
                for (int j = 0; j < HV; j += 4)
                    *reinterpret_cast<float4 *>(dst + j) = make_float4(dS[j], dS[j + 1], dS[j + 2], dS[j + 3]);
            } else {          // or as the tensor-core chunk-gradient kernel's bf16 operand tile:
                              // key rows, two 64-column blocks, 128-byte swizzle
                uint8_t *dst = p.dh + ((row0 + ic) * H + h) * (int64_t)kDsTileBytes;
#pragma unroll
                for (int j = 0; j < HV; j += 8)
                    *reinterpret_cast<uint4 *>(dst + kmaj16(128, row, v0 + c0 + j)) = pack8(dS + j);
            }
            mbar_wait(&bar_tma[st], (k / NS) & 1, &s_err, 3);
            if (len < C) {   // dO rows past the end may hold NaN padding; they enter the MMA raw
                const uint4 zero = make_uint4(0, 0, 0, 0);
                for (int t = tid; t < C * 8; t += kStateWarps * 32) {
                    const int r = t >> 3;
                    if (r >= len) *reinterpret_cast<uint4 *>(stage + Lay::oDO + r * 128 + (t & 7) * 16) = zero;
                }
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_ops);
            const float gc = reinterpret_cast<const float *>(stage + Lay::oG)[KDA ? row : 0];
#pragma unroll
            for (int j = 0; j < HV; ++j) dS[j] *= gc;
            mbar_wait(&bar_g, k & 1, &s_err, 4);
            tc_fence_after();
            {
                float d[HV];
#pragma unroll
                for (int j = 0; j < HV; j += 8) tmem_ld8(tmem + lane_off + (k & 1) * VS + c0 + j, d + j);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < HV; ++j) dS[j] += d[j];
            }
            // buffer (k + 1) & 1 was last read by the MMAs of step k - 1, complete (waited)
            if (k + 1 < nch) put_ds((k + 1) & 1, dS);
            else tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_free[st]);
        }
        if (p.dh0 && *reinterpret_cast<volatile int *>(&s_err) == 0 &&
            GCL_RANGE_IN_BOUNDS(state_base + (int64_t)row * VD + v0 + c0,
                                state_base + (int64_t)row * VD + v0 + c0 + HV - 1,
                                (int64_t)p.n_max * H * KV, p.status)) {
            float *dst = p.dh0 + state_base + (int64_t)row * VD + v0 + c0;
#pragma unroll
            for (int j = 0; j < HV; j += 4)
                *reinterpret_cast<float4 *>(dst + j) = make_float4(dS[j], dS[j + 1], dS[j + 2], dS[j + 3]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kStateWarps) tmem_dealloc(tmem, kTmemCols);
    if (tid == 0 && s_err != 0) status_set(p.status, GCL_DEV_WAIT_TIMEOUT);
}

template <int VS, bool KDA>
cudaError_t launch_sweep(const CUtensorMap &m128, const CUtensorMap &m64, const CUtensorMap &mdo,
                         const SweepTParams &sp, int split, cudaStream_t s) {
    constexpr int NS = 3;
    using Lay = SweepLayout<NS>;
    static_assert(Lay::bytes <= 232448, "sweep shared memory");
    auto kern = tc_sweep_t_kernel<VS, NS, KDA>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Lay::bytes);
    if (e != cudaSuccess) return e;
    kern<<<dim3(split, sp.H, sp.n_max), kSweepThreads, Lay::bytes, s>>>(m128, m64, mdo, sp);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_sweep_t(const BwdParams &p, const uint8_t *ws, bool kda, cudaStream_t s) {
    const int H = p.H;
    const int64_t units = p.nt_max * H;
    CUtensorMap m128, m64, mdo;
    const cuuint64_t drec[3] = {(cuuint64_t)KD, (cuuint64_t)(kUnitBytes / (KD * 2)), (cuuint64_t)units};
    const cuuint64_t srec[2] = {(cuuint64_t)KD * 2, (cuuint64_t)kUnitBytes};
    const cuuint32_t b128[3] = {64, 128, 1}, b64r[3] = {64, 64, 1};
    const cuuint64_t ddo[3] = {(cuuint64_t)VD, (cuuint64_t)H, (cuuint64_t)p.t_max};
    const cuuint64_t sdo[2] = {(cuuint64_t)VD * 2, (cuuint64_t)H * VD * 2};
    const cuuint32_t bdo[3] = {64, 1, 64};
    if (!make_tensor_map(&m128, ws, 3, drec, srec, b128, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tensor_map(&m64, ws, 3, drec, srec, b64r, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tensor_map(&mdo, p.d_o, 3, ddo, sdo, bdo, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    SweepTParams sp{};
    sp.cu = p.cu_seqlens;
    sp.chunk_offsets = p.chunk_offsets;
    sp.dht = p.dht;
    sp.ws = ws;
    sp.dh = reinterpret_cast<uint8_t *>(p.dh);
    sp.dh_f32 = kda ? p.dh : nullptr;           // the KDA chunk gradients read fp32 rows
    sp.dh0 = p.dh0;
    sp.status = p.dev_status;
    sp.t_max = p.t_max;
    sp.nt_max = p.nt_max;
    sp.n_max = p.n_max;
    sp.H = H;
    const int split = fwd_tc_split(p.n_max, H);
    if (kda) {
        switch (VD / split) {
            case 16: return launch_sweep<16, true>(m128, m64, mdo, sp, split, s);
            case 32: return launch_sweep<32, true>(m128, m64, mdo, sp, split, s);
            default: return launch_sweep<64, true>(m128, m64, mdo, sp, split, s);
        }
    }
    switch (VD / split) {
        case 16: return launch_sweep<16, false>(m128, m64, mdo, sp, split, s);
        case 32: return launch_sweep<32, false>(m128, m64, mdo, sp, split, s);
        default: return launch_sweep<64, false>(m128, m64, mdo, sp, split, s);
    }
}

}  // namespace gcl
