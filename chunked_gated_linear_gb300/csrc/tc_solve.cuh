// tc_solve.cuh -- T = (I + A)^-1 for the 64 x 64 strictly lower triangular A of one chunk,
// in fp32 on the CUDA cores, by blocked forward substitution.
//
// HA-NPU paper "Empowering Hybrid Attention Models on NPUs", section 5: the matrix
// inversion of the WY representation is decoupled from the GEMMs and runs on the vector
// units.  Blocks are 16 x 16:
//   diagonal      T_bb = (I + A_bb)^-1, column by column (forward substitution), one
//                 thread per column with four interleaved partial sums (x[m] = 0 for
//                 m < jj, so the sums need no mask);
//   off-diagonal  T_ij = -T_ii sum_{k=j}^{i-1} A_ik T_kj, by levels i - j = 1, 2, 3; each
//                 thread computes a 1 x 4 strip from float4 shared-memory loads.
// Shared-memory layout: row stride kSolveLD floats (16-byte aligned rows, conflict-free
// for the strip pattern), X scratch [3][16][kSolveLDX].
// T is written on and below the block diagonal (zeros above the diagonal inside the
// diagonal blocks); blocks above the block diagonal are left as they were, so readers
// take T[r][c] only for c <= r.
#pragma once

namespace gcl {

constexpr int kSolveLD = 68;
constexpr int kSolveLDX = 20;
constexpr int kSolveFloats = 2 * 64 * kSolveLD + 3 * 16 * kSolveLDX;   // A, T, X

// Barrier among the solving threads: the whole block (BarId < 0), or threads 0 .. NT-1 on the
// named barrier BarId (the rest of the block does other work meanwhile).
template <int NT, int BarId>
__device__ __forceinline__ void solve_barrier() {
    if constexpr (BarId < 0) {
        __syncthreads();
    } else {
        asm volatile("bar.sync %0, %1;" ::"n"(BarId), "n"(NT) : "memory");
    }
}

// Threads 0 .. NT-1 call it (NT is 128 or 256); with BarId < 0 they are the whole block.
template <int NT, int BarId = -1>
__device__ __forceinline__ void solve_unit_lower64(const float *sA, float *sT, float *sX) {
    static_assert(NT == 128 || NT == 256, "128 or 256 solving threads");
    const int tid = threadIdx.x;
    if (tid < 64) {   // ---- diagonal blocks: thread (block, column jj), four partial sums
        const int o = (tid >> 4) * 16, jj = tid & 15;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) x[r] = (r == jj) ? 1.f : 0.f;
#pragma unroll
        for (int r = 1; r < 16; ++r) {
            float part[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int m = 0; m < r; ++m)
                part[m & 3] = fmaf(sA[(o + r) * kSolveLD + o + m], x[m], part[m & 3]);
            const float sum = (part[0] + part[1]) + (part[2] + part[3]);
            if (r > jj) x[r] = -sum;
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) sT[(o + r) * kSolveLD + o + jj] = x[r];
    }
    solve_barrier<NT, BarId>();
    // ---- off-diagonal blocks.  Strip s of level d: block blk (bi = d + blk, bj = blk),
    // column quad cq, row rr (rows fastest, so 8 consecutive lanes read 8 distinct rows).  The
    // level loop is unrolled, so every dot product has a compile-time length (16 d terms) and
    // its loads are issued ahead of the FMAs; the summation order is the plain one.
#pragma unroll
    for (int d = 1; d < 4; ++d) {
        const int nstrip = (4 - d) * 64;
        for (int s = tid; s < nstrip; s += NT) {
            const int blk = s >> 6, cq = (s >> 4) & 3, rr = s & 15;
            const int bi = d + blk, bj = blk;
            const float *arow = sA + (bi * 16 + rr) * kSolveLD + bj * 16;
            const float *tcol = sT + bj * 16 * kSolveLD + bj * 16 + cq * 4;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int t = 0; t < 4 * d; ++t) {
                const float4 a = *reinterpret_cast<const float4 *>(arow + 4 * t);
                const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float4 tv = *reinterpret_cast<const float4 *>(tcol + (4 * t + e) * kSolveLD);
                    acc.x = fmaf(av[e], tv.x, acc.x);
                    acc.y = fmaf(av[e], tv.y, acc.y);
                    acc.z = fmaf(av[e], tv.z, acc.z);
                    acc.w = fmaf(av[e], tv.w, acc.w);
                }
            }
            *reinterpret_cast<float4 *>(sX + (blk * 16 + rr) * kSolveLDX + cq * 4) = acc;
        }
        solve_barrier<NT, BarId>();
        for (int s = tid; s < nstrip; s += NT) {
            const int blk = s >> 6, cq = (s >> 4) & 3, rr = s & 15;
            const int bi = d + blk, bj = blk;
            const float *trow = sT + (bi * 16 + rr) * kSolveLD + bi * 16;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int m = 0; m < 16; m += 4) {
                const float4 t = *reinterpret_cast<const float4 *>(trow + m);
                const float tv[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float4 xv = *reinterpret_cast<const float4 *>(sX + (blk * 16 + m + e) * kSolveLDX + cq * 4);
                    acc.x = fmaf(tv[e], xv.x, acc.x);
                    acc.y = fmaf(tv[e], xv.y, acc.y);
                    acc.z = fmaf(tv[e], xv.z, acc.z);
                    acc.w = fmaf(tv[e], xv.w, acc.w);
                }
            }
            *reinterpret_cast<float4 *>(sT + (bi * 16 + rr) * kSolveLD + bj * 16 + cq * 4) =
                make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
        }
        solve_barrier<NT, BarId>();
    }
}

}  // namespace gcl
