// short_conv.cu -- the short causal depthwise convolution before the chunk attention
// (causal_conv1d), forward and backward, varlen, on the CUDA cores.
//
// FLA RFC "[RFC] Add Graph Capture Support for FLA Prefill and Training Paths on Ascend NPUs",
// section "Step 3": dense and varlen inputs, forward and backward, bias, activation and
// residual paths, initial and final states, fixed chunk metadata and state buffers; section
// "API proposal": causal_conv1d takes the same chunk_indices as the chunk attention.  With W
// taps per channel and xx_n(i) the i-th input of sequence n (the initial state for i < 0):
//   y[bos + p] = act(b + sum_j w[:, j] xx_n(p - (W - 1) + j)) + r[bos + p],
//   ht[n, :, k] = xx_n(len - (W - 1) + k)   (k = 0 .. W - 2, oldest first).
// The work list is chunk_indices (64-token chunks) x blocks of channels, so the launch depends
// only on the capacities.  The path is HBM-bound.  Forward: one CTA per (chunk row, block of
// channels), plus one per sequence slot that passes the state through for zero-length
// sequences; a CTA stages its chunk's rows and the W - 1 rows before them (the previous chunk,
// or the initial state) into shared memory with independent 16-byte asynchronous copies, so
// every byte of the chunk is in flight at once, then each thread produces whole output rows of
// 8 channels.  Backward: persistent (a fixed grid of two CTAs per SM walks the chunk rows of
// one block of channels each) and double-buffered: while a CTA computes one chunk from shared
// memory, the rows of its next chunk are already in flight.
//
// Backward (reverse mode of <dy, y> + <dht, ht>): a CTA also stages dy and the W - 1 rows
// after the chunk, forms dpre = dy act'(pre) once in shared memory, then
//   dx[p] = sum_j dpre[p + W - 1 - j] w[:, j] (+ dht for the last W - 1 positions),
//   dh0 from the first chunk of each sequence, and dw, db as partial sums per CTA (each CTA
//   walks its rows in a fixed order for one block of channels) that a second kernel adds over
//   the CTAs in a fixed order (no atomics: reproducible on a given GPU).
#include "gcl_internal.cuh"

namespace gcl {
namespace {

constexpr int C = kChunk;
constexpr int kConvThreads = 256;
constexpr int kChannelsPerThread = 8;                  // one 16-byte vector of bf16
constexpr int kFwdChannels = 256;                      // channels per forward CTA
constexpr int kBwdChannels = 128;                      // channels per backward CTA

struct ConvParams {
    const void *x, *w, *bias, *residual, *h0, *dy;
    void *y, *ht;
    const float *dht;
    float *dx, *dw, *dbias, *dh0, *partial;
    const int32_t *cu, *chunk_indices;
    int32_t *status;
    int64_t t_max, nt_max;
    int32_t n_max, D, act;
    int32_t n_part;                                    // backward: CTAs per block of channels
};

template <typename T>
__device__ __forceinline__ void load8(const T *p, float *v);
template <>
__device__ __forceinline__ void load8<float>(const float *p, float *v) {
    const float4 a = *reinterpret_cast<const float4 *>(p), b = *reinterpret_cast<const float4 *>(p + 4);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
template <>
__device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16 *p, float *v) {
    const uint4 u = *reinterpret_cast<const uint4 *>(p);
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float2 f = __bfloat1622float2(h[e]);
        v[2 * e] = f.x;
        v[2 * e + 1] = f.y;
    }
}
template <typename T>
__device__ __forceinline__ void store8(T *p, const float *v);
template <>
__device__ __forceinline__ void store8<float>(float *p, const float *v) {
    *reinterpret_cast<float4 *>(p) = make_float4(v[0], v[1], v[2], v[3]);
    *reinterpret_cast<float4 *>(p + 4) = make_float4(v[4], v[5], v[6], v[7]);
}
template <>
__device__ __forceinline__ void store8<__nv_bfloat16>(__nv_bfloat16 *p, const float *v) {
    uint4 u;
    __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&u);
#pragma unroll
    for (int e = 0; e < 4; ++e) h[e] = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
    *reinterpret_cast<uint4 *>(p) = u;
}
template <typename T>
__device__ __forceinline__ float ld1(const T *p) { return (float)p[0]; }
template <>
__device__ __forceinline__ float ld1<__nv_bfloat16>(const __nv_bfloat16 *p) { return __bfloat162float(p[0]); }
template <typename T>
__device__ __forceinline__ void st1(T *p, float v) { p[0] = (T)v; }
template <>
__device__ __forceinline__ void st1<__nv_bfloat16>(__nv_bfloat16 *p, float v) { p[0] = __float2bfloat16_rn(v); }

// SiLU and its derivative with the fast reciprocal (a few ulp; the path is bound by memory)
__device__ __forceinline__ float silu(float z) { return __fdividef(z, 1.f + __expf(-z)); }
__device__ __forceinline__ float silu_grad(float z) {
    const float s = __fdividef(1.f, 1.f + __expf(-z));
    return s * (1.f + z * (1.f - s));
}

// The sequence and chunk of work row j; false (nothing to do) for sentinels and invalid rows.
__device__ __forceinline__ bool conv_row(const ConvParams &p, int j, int &n, int &ic, int64_t &bos,
                                         int64_t &eos) {
    n = p.chunk_indices[2 * j];
    if (n < 0) return false;
    ic = p.chunk_indices[2 * j + 1];
    if (n >= p.n_max || ic < 0) {
        if (threadIdx.x == 0) status_set(p.status, GCL_DEV_BAD_RANGE);
        return false;
    }
    bos = p.cu[n];
    eos = p.cu[n + 1];
    if (bos < 0 || eos < bos || eos > p.t_max || bos + (int64_t)ic * C >= eos) {
        if (threadIdx.x == 0) status_set(p.status, GCL_DEV_BAD_RANGE);
        return false;
    }
    return true;
}

// Sequence n, channels [cb * channels, +channels): if the sequence is empty, ht = h0 (or zeros);
// in the backward dh0 = dht (or zeros).
template <typename T, int W>
__device__ __forceinline__ void conv_empty_sequence(const ConvParams &p, int n, int cb, int channels,
                                                    bool backward) {
    const int64_t bos = p.cu[n], eos = p.cu[n + 1];
    if (eos != bos) return;
    for (int e = threadIdx.x; e < channels * (W - 1); e += kConvThreads) {
        const int c = cb * channels + e / (W - 1), k = e % (W - 1);
        if (c >= p.D) continue;
        const int64_t o = ((int64_t)n * p.D + c) * (W - 1) + k;
        if (!backward) {
            if (p.ht) st1(static_cast<T *>(p.ht) + o, p.h0 ? ld1(static_cast<const T *>(p.h0) + o) : 0.f);
        } else if (p.dh0) {
            p.dh0[o] = p.dht ? p.dht[o] : 0.f;
        }
    }
}

// Stage rows [r_lo, r_hi) of the chunk (relative to t0; rows < 0 come from the previous chunk,
// or from the initial state when the chunk is the sequence's first) of `channels` channels
// starting at c_base into tile[(r - r_lo)][channels] in the input type.  Rows of the initial
// state without h0 are zeros.  Channels at or past D are not touched.  The rows of the input
// are asynchronous copies (all in flight at once): conv_stage_wait() before the barrier.
template <typename T, int W>
__device__ __forceinline__ void conv_stage(const ConvParams &p, const T *src, T *tile, int channels, int c_base,
                                           int64_t t0, int ic, int n, int r_lo, int r_hi) {
    const int vec = channels / kChannelsPerThread;          // 16-byte vectors per row (bf16)
    for (int e = threadIdx.x; e < (r_hi - r_lo) * vec; e += kConvThreads) {
        const int rr = e / vec, cv = e % vec, r = r_lo + rr, c = c_base + cv * kChannelsPerThread;
        if (c >= p.D) continue;
        T *dst = tile + (int64_t)rr * channels + cv * kChannelsPerThread;
        if (r >= 0 || ic > 0) {                           // asynchronous 16-byte copies
            const T *s = src + (t0 + r) * p.D + c;
            constexpr int kPer16 = 16 / (int)sizeof(T);  // elements per 16-byte copy
#pragma unroll
            for (int h = 0; h < kChannelsPerThread / kPer16; ++h)
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                                 (uint32_t)__cvta_generic_to_shared(dst + h * kPer16)),
                             "l"(s + h * kPer16)
                             : "memory");
        } else {
#pragma unroll
            for (int q = 0; q < kChannelsPerThread; ++q)
                st1(dst + q, p.h0 ? ld1(static_cast<const T *>(p.h0) + ((int64_t)n * p.D + c + q) * (W - 1) +
                                        (W - 1) + r)
                                  : 0.f);
        }
    }
}

__device__ __forceinline__ void conv_stage_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// all but the most recent group of copies have landed (this thread's; a barrier follows)
__device__ __forceinline__ void conv_stage_wait_prev() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }
__device__ __forceinline__ void conv_stage_wait() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Row j of chunk_indices is a live chunk (live rows come first, then sentinels).
__device__ __forceinline__ bool conv_live(const ConvParams &p, int64_t j) {
    return j < p.nt_max && p.chunk_indices[2 * j] >= 0;
}

template <typename T, int W>
__global__ void __launch_bounds__(kConvThreads, 4)
conv_fwd_kernel(ConvParams p) {
    constexpr int CB = kFwdChannels * 2 / (int)sizeof(T);   // 34 KB tiles for both types
    constexpr int G = CB / kChannelsPerThread, RL = kConvThreads / G;
    __shared__ __align__(16) T tile[(C + W - 1) * CB];
    if (status_blocks_cta(p.status)) return;
    if ((int64_t)blockIdx.x >= p.nt_max) {                 // the sequence slots: zero-length sequences
        const int64_t n = (int64_t)blockIdx.x - p.nt_max;
        if (n < p.n_max) conv_empty_sequence<T, W>(p, (int)n, blockIdx.y, CB, false);
        return;
    }
    int n, ic;
    int64_t bos, eos;
    if (!conv_row(p, blockIdx.x, n, ic, bos, eos)) return;
    const int D = p.D, cb0 = blockIdx.y * CB;
    const int64_t t0 = bos + (int64_t)ic * C;
    const int len = (int)(eos - t0 < C ? eos - t0 : C);
    conv_stage<T, W>(p, static_cast<const T *>(p.x), tile, CB, cb0, t0, ic, n, -(W - 1), len);
    conv_stage_commit();
    conv_stage_wait();
    __syncthreads();
    // thread: 8 channels (vector g) of rows rr, rr + RL, ... (a warp: one row, 512 bytes)
    const int g = threadIdx.x % G, rr = threadIdx.x / G, c0 = cb0 + g * kChannelsPerThread;
    if (c0 < D) {
        float w[W][kChannelsPerThread], b[kChannelsPerThread];
#pragma unroll
        for (int e = 0; e < kChannelsPerThread; ++e) {
#pragma unroll
            for (int j = 0; j < W; ++j) w[j][e] = ld1(static_cast<const T *>(p.w) + (int64_t)(c0 + e) * W + j);
            b[e] = p.bias ? ld1(static_cast<const T *>(p.bias) + c0 + e) : 0.f;
        }
        const T *r = static_cast<const T *>(p.residual);
        T *y = static_cast<T *>(p.y);
        for (int row = rr; row < len; row += RL) {
            float res[kChannelsPerThread];
            if (r) load8(r + (t0 + row) * D + c0, res);
            float a[kChannelsPerThread];
#pragma unroll
            for (int e = 0; e < kChannelsPerThread; ++e) a[e] = b[e];
#pragma unroll
            for (int j = 0; j < W; ++j) {               // tile row row + j holds xx(row - (W - 1) + j)
                float xv[kChannelsPerThread];
                load8(tile + (int64_t)(row + j) * CB + g * kChannelsPerThread, xv);
#pragma unroll
                for (int e = 0; e < kChannelsPerThread; ++e) a[e] = fmaf(w[j][e], xv[e], a[e]);
            }
#pragma unroll
            for (int e = 0; e < kChannelsPerThread; ++e) {
                if (p.act == GCL_ACT_SILU) a[e] = silu(a[e]);
                if (r) a[e] += res[e];
            }
            store8(y + (t0 + row) * D + c0, a);
        }
    }
    if (t0 + len == eos && p.ht) {                        // the last chunk: the final state
        for (int e = threadIdx.x; e < CB * (W - 1); e += kConvThreads) {
            const int c = e / (W - 1), k = e % (W - 1);
            if (cb0 + c < D)                              // tile row len + k: xx(len - (W - 1) + k)
                static_cast<T *>(p.ht)[((int64_t)n * D + cb0 + c) * (W - 1) + k] = tile[(int64_t)(len + k) * CB + c];
        }
    }
}
// Column of channel c in a dpre row: each 8-channel vector is split into two float4 halves
// stored in the two halves of the row.
__device__ __forceinline__ int dp_col(int c, int cb) { return ((c & 4) ? cb / 2 : 0) + ((c >> 3) << 2) + (c & 3); }

// Backward tiles (dynamic shared memory): two buffers of {x rows [-(W - 1), C + W - 1) and dy rows
// [0, C + W - 1) in the input type}, then dpre rows [0, C + W - 1) in fp32, CB channels each.
template <typename T, int W>
struct ConvBwdLayout {
    static constexpr int CB = kBwdChannels * 2 / (int)sizeof(T);
    static constexpr int RX = C + 2 * (W - 1), RQ = C + W - 1;
    static constexpr size_t kX = (size_t)RX * CB * sizeof(T), kDY = (size_t)RQ * CB * sizeof(T);
    static constexpr size_t kBuf = (kX + kDY + 15) / 16 * 16;
    static constexpr size_t oDP = 2 * kBuf;
    static constexpr size_t bytes = oDP + (size_t)RQ * CB * sizeof(float);
    static_assert(kConvThreads % CB == 0 && (size_t)(kConvThreads / CB) * (W + 1) * CB <= (size_t)RQ * CB,
                  "the dpre tile holds the per-group partial sums at the end");
};
constexpr int kBwdCtasPerSm = 2;

template <typename T, int W>
__global__ void __launch_bounds__(kConvThreads, kBwdCtasPerSm)
conv_bwd_kernel(ConvParams p) {
    using Lay = ConvBwdLayout<T, W>;
    constexpr int CB = Lay::CB, G = CB / kChannelsPerThread, RL = kConvThreads / G;
    constexpr int NG = kConvThreads / CB;                 // row groups of the dw, db sums
    extern __shared__ __align__(16) uint8_t smem[];
    float *sdp = reinterpret_cast<float *>(smem + Lay::oDP);
    if (status_blocks_cta(p.status)) return;
    const int D = p.D, cb = blockIdx.y, cb0 = cb * CB, part_idx = blockIdx.x;
    const int64_t step = gridDim.x;
    auto tx = [&](int b) { return reinterpret_cast<T *>(smem + b * Lay::kBuf); };
    auto tdy = [&](int b) { return reinterpret_cast<T *>(smem + b * Lay::kBuf + Lay::kX); };
    // the rows of chunk j with a pre-activation: positions [0, nq) of the chunk
    auto stage = [&](int64_t j, int b) -> bool {
        int n, ic;
        int64_t bos, eos;
        if (!conv_row(p, (int)j, n, ic, bos, eos)) return false;
        const int64_t t0 = bos + (int64_t)ic * C;
        const int L = (int)(eos - bos), P0 = (int)(t0 - bos);
        const int len = L - P0 < C ? L - P0 : C;
        const int nq = (L - P0 < len + W - 1) ? L - P0 : len + W - 1;
        conv_stage<T, W>(p, static_cast<const T *>(p.x), tx(b), CB, cb0, t0, ic, n, -(W - 1), nq);
        conv_stage<T, W>(p, static_cast<const T *>(p.dy), tdy(b), CB, cb0, t0, ic, n, 0, nq);
        return true;
    };
    const int g = threadIdx.x % G, rr = threadIdx.x / G, c0 = cb0 + g * kChannelsPerThread;
    // dpre rows hold a thread's 8 channels as two float4 in the two halves of the row, so the
    // 32-byte vectors of neighbouring lanes do not share banks (dp_col maps a channel)
    auto dp_store = [&](int q, const float *v) {
        float *row = sdp + (int64_t)q * CB;
        *reinterpret_cast<float4 *>(row + g * 4) = make_float4(v[0], v[1], v[2], v[3]);
        *reinterpret_cast<float4 *>(row + CB / 2 + g * 4) = make_float4(v[4], v[5], v[6], v[7]);
    };
    auto dp_load = [&](int q, float *v) {
        const float *row = sdp + (int64_t)q * CB;
        const float4 lo = *reinterpret_cast<const float4 *>(row + g * 4);
        const float4 hi = *reinterpret_cast<const float4 *>(row + CB / 2 + g * 4);
        v[0] = lo.x; v[1] = lo.y; v[2] = lo.z; v[3] = lo.w; v[4] = hi.x; v[5] = hi.y; v[6] = hi.z; v[7] = hi.w;
    };
    float w[W][kChannelsPerThread], b[kChannelsPerThread];
    if (c0 < D) {
#pragma unroll
        for (int e = 0; e < kChannelsPerThread; ++e) {
#pragma unroll
            for (int j = 0; j < W; ++j) w[j][e] = ld1(static_cast<const T *>(p.w) + (int64_t)(c0 + e) * W + j);
            b[e] = p.bias ? ld1(static_cast<const T *>(p.bias) + c0 + e) : 0.f;
        }
    }
    // dw, db partial sums of this CTA: thread (channel cw, row group grp), rows in item order
    const int cw = threadIdx.x % CB, grp = threadIdx.x / CB;
    float acc[W + 1];
#pragma unroll
    for (int j = 0; j <= W; ++j) acc[j] = 0.f;

    int64_t cur = part_idx;
    bool ok_cur = conv_live(p, cur) && stage(cur, 0);
    conv_stage_commit();
    int buf = 0;
    while (conv_live(p, cur)) {
        const int64_t nxt = cur + step;
        const bool ok_nxt = conv_live(p, nxt) && stage(nxt, buf ^ 1);
        conv_stage_commit();
        conv_stage_wait_prev();
        __syncthreads();                                  // the current chunk's rows are in the tiles
        if (ok_cur) {
            const T *sx = tx(buf), *sdy = tdy(buf);
            int n, ic;
            int64_t bos, eos;
            conv_row(p, (int)cur, n, ic, bos, eos);
            const int64_t t0 = bos + (int64_t)ic * C;
            const int L = (int)(eos - bos), P0 = (int)(t0 - bos);
            const int len = L - P0 < C ? L - P0 : C;
            const int nq = (L - P0 < len + W - 1) ? L - P0 : len + W - 1;   // positions with a pre-activation
            if (c0 < D) {
                // dpre at chunk positions q < len + W - 1 (zero past the sequence)
                for (int q = rr; q < len + W - 1; q += RL) {
                    float d[kChannelsPerThread];
                    if (q < nq) {
                        float a[kChannelsPerThread], gy[kChannelsPerThread];
#pragma unroll
                        for (int e = 0; e < kChannelsPerThread; ++e) a[e] = b[e];
#pragma unroll
                        for (int j = 0; j < W; ++j) {   // x tile row q + j holds xx(q - (W - 1) + j)
                            float xv[kChannelsPerThread];
                            load8(sx + (int64_t)(q + j) * CB + g * kChannelsPerThread, xv);
#pragma unroll
                            for (int e = 0; e < kChannelsPerThread; ++e) a[e] = fmaf(w[j][e], xv[e], a[e]);
                        }
                        load8(sdy + (int64_t)q * CB + g * kChannelsPerThread, gy);
#pragma unroll
                        for (int e = 0; e < kChannelsPerThread; ++e)
                            d[e] = p.act == GCL_ACT_SILU ? gy[e] * silu_grad(a[e]) : gy[e];
                    } else {
#pragma unroll
                        for (int e = 0; e < kChannelsPerThread; ++e) d[e] = 0.f;
                    }
                    dp_store(q, d);
                }
            }
            __syncthreads();
            if (c0 < D) {                                 // dx rows of the chunk
                for (int pr = rr; pr < len; pr += RL) {
                    float gx[kChannelsPerThread];
#pragma unroll
                    for (int e = 0; e < kChannelsPerThread; ++e) gx[e] = 0.f;
#pragma unroll
                    for (int j = 0; j < W; ++j) {       // dpre at position pr + W - 1 - j
                        float dv[kChannelsPerThread];
                        dp_load(pr + W - 1 - j, dv);
#pragma unroll
                        for (int e = 0; e < kChannelsPerThread; ++e) gx[e] = fmaf(dv[e], w[j][e], gx[e]);
                    }
                    const int kf = P0 + pr - (L - (W - 1));   // slot of the final state it lands in
                    if (p.dht && kf >= 0) {
#pragma unroll
                        for (int e = 0; e < kChannelsPerThread; ++e)
                            gx[e] += p.dht[((int64_t)n * D + c0 + e) * (W - 1) + kf];
                    }
                    store8(p.dx + (t0 + pr) * D + c0, gx);
                }
            }
            if (ic == 0 && p.dh0) {                       // the initial state: positions -(W - 1) .. -1
                for (int e = threadIdx.x; e < CB * (W - 1); e += kConvThreads) {
                    const int c = e / (W - 1), k = e % (W - 1), pos = k - (W - 1);
                    if (cb0 + c >= D) continue;
                    float a = 0.f;
#pragma unroll
                    for (int j = 0; j < W; ++j) {
                        const int q = pos + W - 1 - j;
                        if (q >= 0 && q < len + W - 1)
                            a = fmaf(sdp[(int64_t)q * CB + dp_col(c, CB)],
                                     ld1(static_cast<const T *>(p.w) + (int64_t)(cb0 + c) * W + j), a);
                    }
                    const int kf = pos - (L - (W - 1));
                    if (p.dht && kf >= 0) a += p.dht[((int64_t)n * D + cb0 + c) * (W - 1) + kf];
                    p.dh0[((int64_t)n * D + cb0 + c) * (W - 1) + k] = a;
                }
            }
            if (cb0 + cw < D) {                           // dw, db of this chunk's tokens
                for (int pr = grp; pr < len; pr += NG) {
                    const float dv = sdp[(int64_t)pr * CB + dp_col(cw, CB)];
#pragma unroll
                    for (int j = 0; j < W; ++j) acc[j] = fmaf(dv, ld1(sx + (int64_t)(pr + j) * CB + cw), acc[j]);
                    acc[W] += dv;
                }
            }
        }
        __syncthreads();                                  // dpre and the tiles are rewritten next
        cur = nxt;
        ok_cur = ok_nxt;
        buf ^= 1;
    }
    conv_stage_wait();
    // this CTA's partial sums: the NG row groups added in group order
    float *red = sdp;
#pragma unroll
    for (int j = 0; j <= W; ++j) red[((int64_t)grp * (W + 1) + j) * CB + cw] = acc[j];
    __syncthreads();
    if (threadIdx.x < CB && cb0 + (int)threadIdx.x < D) {
        float *part = p.partial + (int64_t)part_idx * (W + 1) * D + cb0 + threadIdx.x;
#pragma unroll
        for (int j = 0; j <= W; ++j) {
            float a = 0.f;
            for (int gg = 0; gg < NG; ++gg) a += red[((int64_t)gg * (W + 1) + j) * CB + threadIdx.x];
            part[(int64_t)j * D] = a;
        }
    }
    for (int64_t e = part_idx; e < p.n_max; e += step) conv_empty_sequence<T, W>(p, (int)e, cb, CB, true);
}
// dw[c][j] and db[c]: the backward CTAs' partial sums, 32 channels per CTA (one per lane, so
// every load of a warp is one 128-byte line); warp w takes partials w, w + 16, ..., and the 16
// warp sums are added in warp order.
constexpr int kReduceWarps = 16;

template <int W>
__global__ void __launch_bounds__(kReduceWarps * 32)
conv_reduce_kernel(ConvParams p) {
    __shared__ float red[kReduceWarps][W + 1][32];
    if (status_blocks_cta(p.status)) return;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int c = blockIdx.x * 32 + lane;
    float acc[W + 1];
#pragma unroll
    for (int j = 0; j <= W; ++j) acc[j] = 0.f;
    if (c < p.D) {
        for (int64_t row = warp; row < p.n_part; row += kReduceWarps) {
            const float *part = p.partial + row * (W + 1) * p.D + c;
#pragma unroll
            for (int j = 0; j <= W; ++j) acc[j] += part[(int64_t)j * p.D];
        }
    }
#pragma unroll
    for (int j = 0; j <= W; ++j) red[warp][j][lane] = acc[j];
    __syncthreads();
    if (warp <= W && c < p.D) {                           // warp j adds tap j (j = W: the bias)
        float a = 0.f;
        for (int w = 0; w < kReduceWarps; ++w) a += red[w][warp][lane];
        if (warp < W) p.dw[(int64_t)c * W + warp] = a;
        else if (p.dbias) p.dbias[c] = a;
    }
}

// Backward CTAs per block of channels: one wave of kBwdCtasPerSm per SM, at most one per chunk
// row (the partial-sum buffer holds nt_max rows).
int conv_bwd_parts(int64_t nt_max, int ncb) {
    const int64_t parts = (int64_t)kBwdCtasPerSm * num_sms() / ncb;
    return (int)(parts < 1 ? 1 : parts > nt_max ? nt_max : parts);
}

template <typename T, int W>
cudaError_t launch_conv(const ConvParams &p0, bool backward, cudaStream_t s) {
    ConvParams p = p0;
    cudaError_t e;
    if (!backward) {
        constexpr int CB = kFwdChannels * 2 / (int)sizeof(T);
        const dim3 grid((unsigned)(p.nt_max + p.n_max), (unsigned)((p.D + CB - 1) / CB));
        conv_fwd_kernel<T, W><<<grid, kConvThreads, 0, s>>>(p);
        return cudaGetLastError();
    }
    using Lay = ConvBwdLayout<T, W>;
    auto kern = conv_bwd_kernel<T, W>;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Lay::bytes)) != cudaSuccess)
        return e;
    const int ncb = (p.D + Lay::CB - 1) / Lay::CB;
    p.n_part = conv_bwd_parts(p.nt_max, ncb);
    kern<<<dim3((unsigned)p.n_part, (unsigned)ncb), kConvThreads, Lay::bytes, s>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    conv_reduce_kernel<W><<<(p.D + 31) / 32, kReduceWarps * 32, 0, s>>>(p);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_conv_w(const ConvParams &p, int W, bool backward, cudaStream_t s) {
    switch (W) {
        case 2: return launch_conv<T, 2>(p, backward, s);
        case 3: return launch_conv<T, 3>(p, backward, s);
        default: return launch_conv<T, 4>(p, backward, s);
    }
}

}  // namespace

size_t conv_bwd_workspace_bytes(int64_t nt_max, int D, int W) {
    return (size_t)nt_max * (W + 1) * D * sizeof(float);
}

cudaError_t launch_conv_fwd(const ConvLaunch &a, cudaStream_t s) {
    ConvParams p{};
    p.x = a.x; p.w = a.w; p.bias = a.bias; p.residual = a.residual; p.h0 = a.h0;
    p.y = a.y; p.ht = a.ht;
    p.cu = a.cu_seqlens; p.chunk_indices = a.chunk_indices; p.status = a.dev_status;
    p.t_max = a.t_max; p.nt_max = a.nt_max; p.n_max = a.n_max; p.D = a.D; p.act = a.activation;
    return a.dtype == GCL_BF16 ? launch_conv_w<__nv_bfloat16>(p, a.W, false, s)
                               : launch_conv_w<float>(p, a.W, false, s);
}

cudaError_t launch_conv_bwd(const ConvLaunch &a, cudaStream_t s) {
    ConvParams p{};
    p.x = a.x; p.w = a.w; p.bias = a.bias; p.h0 = a.h0; p.dy = a.dy; p.dht = a.dht;
    p.dx = a.dx; p.dw = a.dw; p.dbias = a.dbias; p.dh0 = a.dh0; p.partial = a.partial;
    p.cu = a.cu_seqlens; p.chunk_indices = a.chunk_indices; p.status = a.dev_status;
    p.t_max = a.t_max; p.nt_max = a.nt_max; p.n_max = a.n_max; p.D = a.D; p.act = a.activation;
    return a.dtype == GCL_BF16 ? launch_conv_w<__nv_bfloat16>(p, a.W, true, s)
                               : launch_conv_w<float>(p, a.W, true, s);
}

}  // namespace gcl
