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
// The work list is chunk_indices (64-token chunks), so the grid depends only on the
// capacities: one CTA per (row, block of 1024 channels); each thread streams 8 channels
// through its chunk with the W - 1 previous inputs in registers.  Extra blocks after the
// chunk rows pass the state through for zero-length sequences.  The path is HBM-bound:
// every input is read once (plus W - 1 halo rows per chunk) and every output written once.
//
// Backward (reverse mode of <dy, y> + <dht, ht>): per chunk, the same walk recomputes the
// pre-activation up to W - 1 positions past the chunk, forms dpre = dy act'(pre), and
//   dx[p] = sum_j dpre[p + W - 1 - j] w[:, j] (+ dht for the last W - 1 positions),
//   dh0 from the first chunk of each sequence, dw and db as per-chunk partial sums that a
//   second kernel adds over the chunks in a fixed order (no atomics: reproducible).
#include "gcl_internal.cuh"

namespace gcl {
namespace {

constexpr int C = kChunk;
constexpr int kConvThreads = 128;
constexpr int kChannelsPerThread = 8;
constexpr int kChannelsPerBlock = kConvThreads * kChannelsPerThread;

struct ConvParams {
    const void *x, *w, *bias, *residual, *h0, *dy;
    void *y, *ht;
    const float *dht;
    float *dx, *dw, *dbias, *dh0, *partial;
    const int32_t *cu, *chunk_indices;
    int32_t *status;
    int64_t t_max, nt_max;
    int32_t n_max, D, act;
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

__device__ __forceinline__ float silu(float z) { return z / (1.f + __expf(-z)); }
__device__ __forceinline__ float silu_grad(float z) {
    const float s = 1.f / (1.f + __expf(-z));
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

// A zero-length sequence n (block index past the chunk rows): ht = h0 (or zeros); in the
// backward dh0 = dht (or zeros).  Returns true if this block was such a block.
template <typename T, int W>
__device__ __forceinline__ bool conv_empty_sequence(const ConvParams &p, bool backward) {
    const int64_t i = (int64_t)blockIdx.x - p.nt_max;
    if (i < 0) return false;
    const int n = (int)i;
    if (n >= p.n_max) return true;
    const int64_t bos = p.cu[n], eos = p.cu[n + 1];
    if (eos != bos) return true;
    const int c0 = (blockIdx.y * kConvThreads + threadIdx.x) * kChannelsPerThread;
    if (c0 >= p.D) return true;
    for (int e = 0; e < kChannelsPerThread; ++e)
        for (int k = 0; k < W - 1; ++k) {
            const int64_t o = ((int64_t)n * p.D + c0 + e) * (W - 1) + k;
            if (!backward) {
                if (p.ht) st1(static_cast<T *>(p.ht) + o, p.h0 ? ld1(static_cast<const T *>(p.h0) + o) : 0.f);
            } else if (p.dh0) {
                p.dh0[o] = p.dht ? p.dht[o] : 0.f;
            }
        }
    return true;
}

template <typename T, int W>
__global__ void __launch_bounds__(kConvThreads)
conv_fwd_kernel(ConvParams p) {
    if (status_blocks(p.status)) return;
    if (conv_empty_sequence<T, W>(p, false)) return;
    int n, ic;
    int64_t bos, eos;
    if (!conv_row(p, blockIdx.x, n, ic, bos, eos)) return;
    const int c0 = (blockIdx.y * kConvThreads + threadIdx.x) * kChannelsPerThread;
    if (c0 >= p.D) return;
    const int D = p.D;
    const int64_t t0 = bos + (int64_t)ic * C;
    const int len = (int)(eos - t0 < C ? eos - t0 : C);
    const T *x = static_cast<const T *>(p.x);
    const T *r = static_cast<const T *>(p.residual);
    T *y = static_cast<T *>(p.y);
    float w[W][kChannelsPerThread], b[kChannelsPerThread], win[W - 1][kChannelsPerThread];
#pragma unroll
    for (int e = 0; e < kChannelsPerThread; ++e) {
#pragma unroll
        for (int j = 0; j < W; ++j) w[j][e] = ld1(static_cast<const T *>(p.w) + (int64_t)(c0 + e) * W + j);
        b[e] = p.bias ? ld1(static_cast<const T *>(p.bias) + c0 + e) : 0.f;
    }
    // the W - 1 inputs before the chunk: the previous rows, or the initial state for chunk 0
#pragma unroll
    for (int k = 0; k < W - 1; ++k) {
        if (ic > 0) {
            load8(x + (t0 - (W - 1) + k) * D + c0, win[k]);
        } else {
#pragma unroll
            for (int e = 0; e < kChannelsPerThread; ++e)
                win[k][e] = p.h0 ? ld1(static_cast<const T *>(p.h0) + ((int64_t)n * D + c0 + e) * (W - 1) + k) : 0.f;
        }
    }
    constexpr int G = 8;                                  // rows loaded ahead
    for (int g0 = 0; g0 < len; g0 += G) {
        float xs[G][kChannelsPerThread], rs[G][kChannelsPerThread];
#pragma unroll
        for (int q = 0; q < G; ++q) {
            if (g0 + q < len) {
                load8(x + (t0 + g0 + q) * D + c0, xs[q]);
                if (r) load8(r + (t0 + g0 + q) * D + c0, rs[q]);
            }
        }
#pragma unroll
        for (int q = 0; q < G; ++q) {
            if (g0 + q < len) {
                float out[kChannelsPerThread];
#pragma unroll
                for (int e = 0; e < kChannelsPerThread; ++e) {
                    float a = b[e];
#pragma unroll
                    for (int j = 0; j < W - 1; ++j) a = fmaf(w[j][e], win[j][e], a);
                    a = fmaf(w[W - 1][e], xs[q][e], a);
                    if (p.act == GCL_ACT_SILU) a = silu(a);
                    out[e] = r ? a + rs[q][e] : a;
                }
                store8(y + (t0 + g0 + q) * D + c0, out);
#pragma unroll
                for (int j = 0; j < W - 2; ++j)
#pragma unroll
                    for (int e = 0; e < kChannelsPerThread; ++e) win[j][e] = win[j + 1][e];
#pragma unroll
                for (int e = 0; e < kChannelsPerThread; ++e) win[W - 2][e] = xs[q][e];
            }
        }
    }
    if (t0 + len == eos && p.ht) {                        // the last chunk: the final state
#pragma unroll
        for (int k = 0; k < W - 1; ++k)
#pragma unroll
            for (int e = 0; e < kChannelsPerThread; ++e)
                st1(static_cast<T *>(p.ht) + ((int64_t)n * D + c0 + e) * (W - 1) + k, win[k][e]);
    }
}

template <typename T, int W>
__global__ void __launch_bounds__(kConvThreads)
conv_bwd_kernel(ConvParams p) {
    if (status_blocks(p.status)) return;
    if (conv_empty_sequence<T, W>(p, true)) return;
    int n, ic;
    int64_t bos, eos;
    if (!conv_row(p, blockIdx.x, n, ic, bos, eos)) return;
    const int c0 = (blockIdx.y * kConvThreads + threadIdx.x) * kChannelsPerThread;
    if (c0 >= p.D) return;
    const int D = p.D;
    const int64_t t0 = bos + (int64_t)ic * C;
    const int L = (int)(eos - bos);                       // sequence length
    const int P0 = (int)(t0 - bos);                       // sequence position of the chunk's row 0
    const int len = L - P0 < C ? L - P0 : C;
    const T *x = static_cast<const T *>(p.x);
    const T *dy = static_cast<const T *>(p.dy);
    float w[W][kChannelsPerThread], b[kChannelsPerThread], win[W - 1][kChannelsPerThread];
    float dpre[W][kChannelsPerThread];                    // dpre at positions q - W + 1 .. q
    float dw[W][kChannelsPerThread], db[kChannelsPerThread];
#pragma unroll
    for (int e = 0; e < kChannelsPerThread; ++e) {
#pragma unroll
        for (int j = 0; j < W; ++j) {
            w[j][e] = ld1(static_cast<const T *>(p.w) + (int64_t)(c0 + e) * W + j);
            dw[j][e] = 0.f;
            dpre[j][e] = 0.f;
        }
        b[e] = p.bias ? ld1(static_cast<const T *>(p.bias) + c0 + e) : 0.f;
        db[e] = 0.f;
    }
#pragma unroll
    for (int k = 0; k < W - 1; ++k) {
        if (ic > 0) {
            load8(x + (t0 - (W - 1) + k) * D + c0, win[k]);
        } else {
#pragma unroll
            for (int e = 0; e < kChannelsPerThread; ++e)
                win[k][e] = p.h0 ? ld1(static_cast<const T *>(p.h0) + ((int64_t)n * D + c0 + e) * (W - 1) + k) : 0.f;
        }
    }
    // walk q = 0 .. len + W - 2: the pre-activation at chunk row q (if it is in the sequence),
    // then the input gradient of chunk row p = q - (W - 1) (the initial state for p < 0, chunk 0)
    for (int q = 0; q < len + W - 1; ++q) {
        float dp[kChannelsPerThread];
        const bool in_seq = P0 + q < L;
        if (in_seq) {
            float xv[kChannelsPerThread], g[kChannelsPerThread];
            load8(x + (t0 + q) * D + c0, xv);
            load8(dy + (t0 + q) * D + c0, g);
#pragma unroll
            for (int e = 0; e < kChannelsPerThread; ++e) {
                float a = b[e];
#pragma unroll
                for (int j = 0; j < W - 1; ++j) a = fmaf(w[j][e], win[j][e], a);
                a = fmaf(w[W - 1][e], xv[e], a);
                dp[e] = p.act == GCL_ACT_SILU ? g[e] * silu_grad(a) : g[e];
                if (q < len) {                            // this chunk's tokens own dw, db
                    db[e] += dp[e];
#pragma unroll
                    for (int j = 0; j < W - 1; ++j) dw[j][e] = fmaf(dp[e], win[j][e], dw[j][e]);
                    dw[W - 1][e] = fmaf(dp[e], xv[e], dw[W - 1][e]);
                }
            }
#pragma unroll
            for (int j = 0; j < W - 2; ++j)
#pragma unroll
                for (int e = 0; e < kChannelsPerThread; ++e) win[j][e] = win[j + 1][e];
#pragma unroll
            for (int e = 0; e < kChannelsPerThread; ++e) win[W - 2][e] = xv[e];
        } else {
#pragma unroll
            for (int e = 0; e < kChannelsPerThread; ++e) dp[e] = 0.f;
        }
#pragma unroll
        for (int j = 0; j < W - 1; ++j)
#pragma unroll
            for (int e = 0; e < kChannelsPerThread; ++e) dpre[j][e] = dpre[j + 1][e];
#pragma unroll
        for (int e = 0; e < kChannelsPerThread; ++e) dpre[W - 1][e] = dp[e];
        // input gradient of row p = q - (W - 1): sum_j dpre(p + W - 1 - j) w_j = sum_j dpre[W-1-j] w_j
        const int pr = q - (W - 1);
        const int P = P0 + pr;                            // its sequence position (< 0: initial state)
        if (pr >= 0 || ic == 0) {
            float gx[kChannelsPerThread];
#pragma unroll
            for (int e = 0; e < kChannelsPerThread; ++e) {
                float a = 0.f;
#pragma unroll
                for (int j = 0; j < W; ++j) a = fmaf(dpre[W - 1 - j][e], w[j][e], a);
                gx[e] = a;
            }
            const int kf = P - (L - (W - 1));             // slot of the final state it lands in
            if (p.dht && kf >= 0 && kf < W - 1) {
#pragma unroll
                for (int e = 0; e < kChannelsPerThread; ++e)
                    gx[e] += p.dht[((int64_t)n * D + c0 + e) * (W - 1) + kf];
            }
            if (pr >= 0) {
                float *dst = p.dx + (t0 + pr) * D + c0;
                *reinterpret_cast<float4 *>(dst) = make_float4(gx[0], gx[1], gx[2], gx[3]);
                *reinterpret_cast<float4 *>(dst + 4) = make_float4(gx[4], gx[5], gx[6], gx[7]);
            } else if (p.dh0) {
#pragma unroll
                for (int e = 0; e < kChannelsPerThread; ++e)
                    p.dh0[((int64_t)n * D + c0 + e) * (W - 1) + (P + (W - 1))] = gx[e];
            }
        }
    }
    // partial sums of this chunk: [row][W + 1][D] (taps, then the bias)
    float *part = p.partial + (int64_t)blockIdx.x * (W + 1) * D + c0;
#pragma unroll
    for (int j = 0; j < W; ++j) store8(part + (int64_t)j * D, dw[j]);
    store8(part + (int64_t)W * D, db);
}

// dw[c][j] and db[c]: the chunk rows' partial sums added in row order (sentinel rows skipped).
template <int W>
__global__ void __launch_bounds__(256)
conv_reduce_kernel(ConvParams p) {
    if (status_blocks(p.status)) return;
    const int c = blockIdx.x * 256 + threadIdx.x;
    if (c >= p.D) return;
    float acc[W + 1];
#pragma unroll
    for (int j = 0; j <= W; ++j) acc[j] = 0.f;
    for (int64_t row = 0; row < p.nt_max; ++row) {
        if (p.chunk_indices[2 * row] < 0) break;          // live rows come first
        const float *part = p.partial + row * (W + 1) * p.D + c;
#pragma unroll
        for (int j = 0; j <= W; ++j) acc[j] += part[(int64_t)j * p.D];
    }
#pragma unroll
    for (int j = 0; j < W; ++j) p.dw[(int64_t)c * W + j] = acc[j];
    if (p.dbias) p.dbias[c] = acc[W];
}

template <typename T, int W>
cudaError_t launch_conv(const ConvParams &p, bool backward, cudaStream_t s) {
    const dim3 grid((unsigned)(p.nt_max + p.n_max), (unsigned)((p.D + kChannelsPerBlock - 1) / kChannelsPerBlock));
    if (!backward) {
        conv_fwd_kernel<T, W><<<grid, kConvThreads, 0, s>>>(p);
        return cudaGetLastError();
    }
    conv_bwd_kernel<T, W><<<grid, kConvThreads, 0, s>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    conv_reduce_kernel<W><<<(p.D + 255) / 256, 256, 0, s>>>(p);
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
