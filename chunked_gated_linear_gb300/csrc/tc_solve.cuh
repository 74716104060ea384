// tc_solve.cuh -- T = (I + A)^-1 for the 64 x 64 strictly lower triangular A of one chunk,
// in fp32 on the CUDA cores, by blocks of 16 x 16.
//
// HA-NPU paper "Empowering Hybrid Attention Models on NPUs", section 5: the matrix
// inversion of the WY representation is decoupled from the GEMMs and runs on the vector
// units.  With blocks 0..3 of 16 rows, T_ii = (I + A_ii)^-1 and C_ij = T_ii A_ij (i > j),
// expanding T = (I + A)^-1 block by block gives, for every lower block,
//   T_ij = -P_ij T_jj,  P_ij = sum over the block paths i = p_0 > p_1 > ... > p_m = j of
//                              (-1)^(m-1) C_{p_0 p_1} C_{p_1 p_2} ... C_{p_(m-1) p_m},
// which four phases of 16-term products evaluate:
//   diagonal   T_ii by forward substitution, one thread per column, four partial sums;
//   1          C_ij = T_ii A_ij for the six lower blocks;
//   2          P_20 = C_20 - C_21 C_10,  P_31 = C_31 - C_32 C_21,  Q_30 = C_30 - C_31 C_10;
//   3          P_30 = Q_30 - C_32 P_20;
//   4          T_ij = -P_ij T_jj (P_ij = C_ij for i - j = 1).
// Each output strip is 1 x 4 with float4 shared-memory loads; every dot product has 16 terms,
// so the critical path is five short phases (the level-by-level substitution it replaces
// had six phases with dot products up to 48 terms long).
// Shared-memory layout: row stride kSolveLD floats (16-byte aligned rows); X scratch
// [3][16][kSolveLDX] holds P_20, P_31 and P_30.  The C_ij are kept in the upper blocks of A
// (block (j, i) holds C_ij), which therefore does not survive the call.  T is written on and
// below the block diagonal (zeros above the diagonal inside the diagonal blocks); blocks above
// the block diagonal are left as they were, so readers take T[r][c] only for c <= r.
#pragma once

namespace gcl {

constexpr int kSolveLD = 68;
constexpr int kSolveLDX = 20;
constexpr int kSolveFloats = 2 * 64 * kSolveLD + 3 * 16 * kSolveLDX;   // A, T, X

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
__device__ __forceinline__ void solve_unit_lower64(float *sA, float *sT, float *sX) {
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
    // ---- off-diagonal blocks by path products.  A strip is row rr, columns 4 cq .. 4 cq + 3
    // of one 16 x 16 output block; out = sum_m L[rr][m] R[m][4 cq ..] over 16 terms.
    auto strip = [](const float *L, int ldl, const float *R, int ldr, int rr, int cq) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int m = 0; m < 16; m += 4) {
            const float4 a = *reinterpret_cast<const float4 *>(L + rr * ldl + m);
            const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float4 r = *reinterpret_cast<const float4 *>(R + (m + e) * ldr + cq * 4);
                acc.x = fmaf(av[e], r.x, acc.x);
                acc.y = fmaf(av[e], r.y, acc.y);
                acc.z = fmaf(av[e], r.z, acc.z);
                acc.w = fmaf(av[e], r.w, acc.w);
            }
        }
        return acc;
    };
    constexpr int LD = kSolveLD, LX = kSolveLDX;
    // block (i, j) of A / T, and C_ij kept in A's block (j, i)
    auto blkA = [&](int i, int j) { return sA + i * 16 * LD + j * 16; };
    auto blkT = [&](int i, int j) { return sT + i * 16 * LD + j * 16; };
    auto blkC = [&](int i, int j) { return const_cast<float *>(sA) + j * 16 * LD + i * 16; };
    float *X20 = sX, *X31 = sX + 16 * LX, *X30 = sX + 32 * LX;
    // lower block b = 0..5: (1, 0), (2, 0), (3, 0), (2, 1), (3, 1), (3, 2)
    auto low_i = [](int b) { return b < 3 ? b + 1 : (b < 5 ? b - 1 : 3); };
    auto low_j = [](int b) { return b < 3 ? 0 : (b < 5 ? 1 : 2); };
    // phase 1: C_ij = T_ii A_ij
    for (int s = tid; s < 6 * 64; s += NT) {
        const int b = s >> 6, rr = s & 15, cq = (s >> 4) & 3;
        const int i = low_i(b), j = low_j(b);
        const float4 c = strip(blkT(i, i), LD, blkA(i, j), LD, rr, cq);
        *reinterpret_cast<float4 *>(blkC(i, j) + rr * LD + cq * 4) = c;
    }
    solve_barrier<NT, BarId>();
    // phase 2: P_20 = C_20 - C_21 C_10, P_31 = C_31 - C_32 C_21, Q_30 = C_30 - C_31 C_10
    for (int s = tid; s < 3 * 64; s += NT) {
        const int b = s >> 6, rr = s & 15, cq = (s >> 4) & 3;
        // b = 0: (i, k, j) = (2, 1, 0); b = 1: (3, 2, 1); b = 2: (3, 1, 0)
        const int i = b == 0 ? 2 : 3, k = b == 1 ? 2 : 1, j = b == 1 ? 1 : 0;
        const float4 pr = strip(blkC(i, k), LD, blkC(k, j), LD, rr, cq);
        const float4 c = *reinterpret_cast<const float4 *>(blkC(i, j) + rr * LD + cq * 4);
        float *dst = (b == 0 ? X20 : b == 1 ? X31 : X30) + rr * LX + cq * 4;
        *reinterpret_cast<float4 *>(dst) = make_float4(c.x - pr.x, c.y - pr.y, c.z - pr.z, c.w - pr.w);
    }
    solve_barrier<NT, BarId>();
    // phase 3: P_30 = Q_30 - C_32 P_20 (in place)
    for (int s = tid; s < 64; s += NT) {
        const int rr = s & 15, cq = (s >> 4) & 3;
        const float4 pr = strip(blkC(3, 2), LD, X20, LX, rr, cq);
        float4 *dst = reinterpret_cast<float4 *>(X30 + rr * LX + cq * 4);
        const float4 q = *dst;
        *dst = make_float4(q.x - pr.x, q.y - pr.y, q.z - pr.z, q.w - pr.w);
    }
    solve_barrier<NT, BarId>();
    // phase 4: T_ij = -P_ij T_jj
    for (int s = tid; s < 6 * 64; s += NT) {
        const int b = s >> 6, rr = s & 15, cq = (s >> 4) & 3;
        const int i = low_i(b), j = low_j(b);
        const float *P;
        int ldp;
        if (i - j == 1) {
            P = blkC(i, j);
            ldp = LD;
        } else {
            P = (i == 2 ? X20 : j == 1 ? X31 : X30);
            ldp = LX;
        }
        const float4 t = strip(P, ldp, blkT(j, j), LD, rr, cq);
        *reinterpret_cast<float4 *>(blkT(i, j) + rr * LD + cq * 4) = make_float4(-t.x, -t.y, -t.z, -t.w);
    }
    solve_barrier<NT, BarId>();
}

// acc[x][y] += sum over m in [4 mlo, 4 mhi) of L[(r0 + x) ldl + m] R[m ldr + c0 + y]: one TR x 4
// register tile of a block product (float4 loads; each loaded L row segment serves four
// columns and each R row segment TR rows).
template <int TR>
__device__ __forceinline__ void solve_tile(const float *L, int ldl, const float *R, int ldr, int r0,
                                           int c0, int mlo, int mhi, float (&acc)[TR][4]) {
    for (int mb = mlo; mb < mhi; ++mb) {
        float4 l[TR];
#pragma unroll
        for (int x = 0; x < TR; ++x) l[x] = *reinterpret_cast<const float4 *>(L + (r0 + x) * ldl + 4 * mb);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float4 r = *reinterpret_cast<const float4 *>(R + (4 * mb + e) * ldr + c0);
#pragma unroll
            for (int x = 0; x < TR; ++x) {
                const float lv = e == 0 ? l[x].x : e == 1 ? l[x].y : e == 2 ? l[x].z : l[x].w;
                acc[x][0] = fmaf(lv, r.x, acc[x][0]);
                acc[x][1] = fmaf(lv, r.y, acc[x][1]);
                acc[x][2] = fmaf(lv, r.z, acc[x][2]);
                acc[x][3] = fmaf(lv, r.w, acc[x][3]);
            }
        }
    }
}

// T = (I + A)^-1 over two blocks of 32 rows instead (the 2 x 2 block split
// A = [A_00 0; A_10 A_11]: T_ii = (I + A_ii)^-1, T_10 = -T_11 A_10 T_00), in two phases:
//   A  forward substitution down the 32 rows of a diagonal block, one column per thread,
//      four partial sums, for the right-hand sides e_j (the columns of T_00 and T_11) and the
//      columns of A_10 (which gives X = T_11 A_10 without forming a product): three warps;
//   B  T_10 = -X T_00: every thread a TR x 4 register tile (TR = 2 with 128 threads, 1 with
//      256), the sum starting at the tile's first column (T_00 is lower triangular).
// Two block barriers instead of five.  A is only read; X is left in T's block (0, 1), above
// the diagonal.  Alone on an SM it takes about two thirds of the latency of the 16-row scheme;
// inside kernels with several CTAs per SM the 16-row scheme's spread over every thread
// measured as fast or faster, so only the fused forward (solve on four warps beside other
// work) takes this one.
template <int NT, int BarId = -1>
__device__ __forceinline__ void solve_unit_lower64_r32(const float *sA, float *sT) {
    static_assert(NT == 128 || NT == 256, "128 or 256 solving threads");
    constexpr int LD = kSolveLD;
    const int tid = threadIdx.x;
    if (tid < 96) {
        const int grp = tid >> 5, j = tid & 31;       // warp-uniform job
        const float *Ab = grp == 0 ? sA : sA + 32 * LD + 32;
        float x[32];
#pragma unroll
        for (int r = 0; r < 32; ++r) {
            float part[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int m4 = 0; m4 < r; m4 += 4) {
                const float4 a = *reinterpret_cast<const float4 *>(Ab + r * LD + m4);
                part[0] = fmaf(a.x, x[m4], part[0]);
                if (m4 + 1 < r) part[1] = fmaf(a.y, x[m4 + 1], part[1]);
                if (m4 + 2 < r) part[2] = fmaf(a.z, x[m4 + 2], part[2]);
                if (m4 + 3 < r) part[3] = fmaf(a.w, x[m4 + 3], part[3]);
            }
            const float rhs = grp == 2 ? sA[(32 + r) * LD + j] : (r == j ? 1.f : 0.f);
            x[r] = rhs - ((part[0] + part[1]) + (part[2] + part[3]));
        }
        float *dst = grp == 0 ? sT + j : grp == 1 ? sT + 32 * LD + 32 + j : sT + 32 + j;
#pragma unroll
        for (int r = 0; r < 32; ++r) dst[r * LD] = x[r];
    }
    solve_barrier<NT, BarId>();
    constexpr int TR = NT == 128 ? 2 : 1;
    for (int s = tid; s < (32 / TR) * 8; s += NT) {
        const int r0 = (s >> 3) * TR, q = s & 7;
        float acc[TR][4] = {};
        solve_tile<TR>(sT + 32, LD, sT, LD, r0, 4 * q, q, 8, acc);
#pragma unroll
        for (int x = 0; x < TR; ++x)
            *reinterpret_cast<float4 *>(sT + (32 + r0 + x) * LD + 4 * q) =
                make_float4(-acc[x][0], -acc[x][1], -acc[x][2], -acc[x][3]);
    }
    solve_barrier<NT, BarId>();
}

}  // namespace gcl
