/*
 * gcl_oracle.c -- plain fp64 CPU oracle for chunked gated linear attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls
 * this file: only the test suite, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header, table or helper with the
 * CUDA library.
 *
 * What it computes (token by token, in double precision):
 *
 *   GDN, the gated delta rule
 *       S_t = alpha_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T,
 *       o_t = S_t^T (scale * q_t),            alpha_t = exp(g_t), g_t <= 0
 *   KDA, the per-channel gated variant
 *       S_t = (I - beta_t k_t k_t^T) Diag(a_t) S_{t-1} + beta_t k_t v_t^T,
 *       o_t = S_t^T (scale * q_t),            a_t = exp(g_t) in R^{d_k}
 *
 * The HA-NPU paper ("Empowering Hybrid Attention Models on NPUs", section 2.1)
 * names GDN and KDA as fixed-size recurrent states with a strict serial
 * dependency, of which the chunkwise Map-Reduce-Map form is a faster schedule;
 * it does not print the recurrence, so the form above is the published gated
 * delta rule, with Diag(a_t) applied to the key rows before the delta
 * correction for KDA.  The state S is d_k x d_v (section 5 of that paper sizes
 * it at 64 KiB: 128 x 128 fp32).
 *
 * Varlen addressing follows the FLA RFC "[RFC] Add Graph Capture Support for
 * FLA Prefill and Training Paths on Ascend NPUs", section "Core design":
 * sequences are packed along the token axis and delimited by cu_seqlens
 * (length n_seq + 1); chunk metadata is chunk_indices [NT_max, 2] holding
 * (sequence, chunk-in-sequence) with the sentinel [-1, 0] in unused rows,
 * and chunk_offsets [n_seq + 1], where NT_max = ceil(T_max / BT) + N_max - 1.
 *
 * Layouts (row-major, token-major as in the RFC's fixed-shape buffers):
 *   q, k  [T, H, K]       v, o [T, H, V]
 *   g     [T, H] (GDN) or [T, H, K] (KDA)      beta [T, H]
 *   h0,ht [N, H, K, V]    (h0 may be NULL: zero initial state)
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORC_GDN = 0, ORC_KDA = 1 };

/* FLA RFC, "Core design / Fixed-capacity execution": NT_max = ceil(T_max/BT) + N_max - 1. */
int64_t orc_nt_max(int64_t t_max, int64_t n_max, int64_t bt)
{
    return (t_max + bt - 1) / bt + n_max - 1;
}

int orc_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * FLA RFC, "Core design / Device-side metadata": cu_seqlens -> chunk_indices
 * [NT_max, 2] and chunk_offsets [N_max + 1].
 *
 * Row j of chunk_indices is (n, i) for the i-th chunk of sequence n, rows in
 * sequence-major order; rows past the live chunk count hold the sentinel
 * [-1, 0].  chunk_offsets[n] is the number of chunks of all sequences before n
 * (chunk_offsets[n_max] is the live chunk count).
 *
 * Returns 0, or a data error (then every row is the sentinel and every offset
 * is 0):  2 = cu[0] != 0,  1 = cu not non-decreasing,  3 = cu[n_max] > t_max,
 * checked in that order.
 */
int orc_chunk_meta(const int64_t *cu, int64_t n_max, int64_t t_max, int64_t bt,
                   int64_t nt_max, int32_t *chunk_indices, int32_t *chunk_offsets)
{
    int status = 0;
    if (cu[0] != 0) {
        status = 2;
    } else {
        for (int64_t n = 0; n < n_max; ++n)
            if (cu[n + 1] < cu[n]) { status = 1; break; }
        if (status == 0 && cu[n_max] > t_max) status = 3;
    }
    for (int64_t j = 0; j < nt_max; ++j) {
        chunk_indices[2 * j] = -1;
        chunk_indices[2 * j + 1] = 0;
    }
    for (int64_t n = 0; n <= n_max; ++n) chunk_offsets[n] = 0;
    if (status != 0) return status;

    int64_t row = 0;
    for (int64_t n = 0; n < n_max; ++n) {
        chunk_offsets[n] = (int32_t)row;
        int64_t len = cu[n + 1] - cu[n];
        int64_t nc = (len + bt - 1) / bt;
        for (int64_t i = 0; i < nc; ++i) {
            chunk_indices[2 * row] = (int32_t)n;
            chunk_indices[2 * row + 1] = (int32_t)i;
            ++row;
        }
    }
    chunk_offsets[n_max] = (int32_t)row;
    return 0;
}

/* ------------------------------------------------------------------------- */
/* One token of the recurrence.  S (K x V) is updated in place.                */

/* GDN: P = S_{t-1};  w = P^T k;  S_t = alpha (P - beta k w^T) + beta k v^T.   */
static void gdn_token(double *S, int64_t K, int64_t V, const double *k, const double *v,
                      double alpha, double beta, double *w)
{
    for (int64_t j = 0; j < V; ++j) {
        double acc = 0.0;
        for (int64_t c = 0; c < K; ++c) acc += S[c * V + j] * k[c];
        w[j] = acc;
    }
    for (int64_t c = 0; c < K; ++c)
        for (int64_t j = 0; j < V; ++j)
            S[c * V + j] = alpha * (S[c * V + j] - beta * k[c] * w[j]) + beta * k[c] * v[j];
}

/* KDA: D = Diag(a) S_{t-1};  w = D^T k;  S_t = D - beta k w^T + beta k v^T.   */
static void kda_token(double *S, int64_t K, int64_t V, const double *k, const double *v,
                      const double *a, double beta, double *w)
{
    for (int64_t c = 0; c < K; ++c)
        for (int64_t j = 0; j < V; ++j) S[c * V + j] *= a[c];
    for (int64_t j = 0; j < V; ++j) {
        double acc = 0.0;
        for (int64_t c = 0; c < K; ++c) acc += S[c * V + j] * k[c];
        w[j] = acc;
    }
    for (int64_t c = 0; c < K; ++c)
        for (int64_t j = 0; j < V; ++j)
            S[c * V + j] = S[c * V + j] - beta * k[c] * w[j] + beta * k[c] * v[j];
}

/* o_t = S_t^T (scale q_t) */
static void read_out(const double *S, int64_t K, int64_t V, const double *q, double scale,
                     double *o)
{
    for (int64_t j = 0; j < V; ++j) {
        double acc = 0.0;
        for (int64_t c = 0; c < K; ++c) acc += S[c * V + j] * (scale * q[c]);
        o[j] = acc;
    }
}

static void step_forward(int variant, double *S, int64_t K, int64_t V, const double *k,
                         const double *v, const double *g, double beta, double *w, double *a)
{
    if (variant == ORC_GDN) {
        gdn_token(S, K, V, k, v, exp(g[0]), beta, w);
    } else {
        for (int64_t c = 0; c < K; ++c) a[c] = exp(g[c]);
        kda_token(S, K, V, k, v, a, beta, w);
    }
}

/*
 * Forward over a varlen batch.  Units (sequence, head) are independent and run
 * in parallel; inside a unit the tokens run strictly in order.
 *
 * If h_chunk is not NULL it receives, for every chunk i of sequence n, the
 * state before the chunk's first token at row chunk_offsets[n] + i of a
 * [NT, H, K, V] array (chunk size bt); this is what a chunked forward saves for
 * its backward pass (FLA RFC, "Static buffer contract": static intermediate
 * states).
 */
void orc_fwd(int variant, int64_t n_seq, const int64_t *cu, int64_t H, int64_t K, int64_t V,
             double scale, const double *q, const double *k, const double *v, const double *g,
             const double *beta, const double *h0, double *o, double *ht, double *h_chunk,
             int64_t bt, const int32_t *chunk_offsets)
{
    const int64_t gK = (variant == ORC_KDA) ? K : 1;
    const int64_t units = n_seq * H;
#pragma omp parallel
    {
        double *S = (double *)malloc(sizeof(double) * K * V);
        double *w = (double *)malloc(sizeof(double) * V);
        double *a = (double *)malloc(sizeof(double) * K);
#pragma omp for schedule(dynamic, 1)
        for (int64_t u = 0; u < units; ++u) {
            const int64_t n = u / H, h = u % H;
            if (h0) memcpy(S, h0 + (n * H + h) * K * V, sizeof(double) * K * V);
            else memset(S, 0, sizeof(double) * K * V);
            for (int64_t t = cu[n]; t < cu[n + 1]; ++t) {
                const int64_t r = t - cu[n];
                if (h_chunk && r % bt == 0)
                    memcpy(h_chunk + ((chunk_offsets[n] + r / bt) * H + h) * K * V, S,
                           sizeof(double) * K * V);
                step_forward(variant, S, K, V, k + (t * H + h) * K, v + (t * H + h) * V,
                             g + (t * H + h) * gK, beta[t * H + h], w, a);
                read_out(S, K, V, q + (t * H + h) * K, scale, o + (t * H + h) * V);
            }
            if (ht) memcpy(ht + (n * H + h) * K * V, S, sizeof(double) * K * V);
        }
        free(S); free(w); free(a);
    }
}

/*
 * Reverse-mode gradient of   f = <do, o> + <dht, ht>   through the same token
 * loop, for GDN and KDA.  Outputs dq, dk, dv, dg (with respect to the raw log
 * gate g), dbeta and dh0.  dht may be NULL (zero).  h0 may be NULL.
 *
 * The token states are recovered from fp64 checkpoints taken every `ckpt`
 * tokens plus a recompute inside each segment, so memory stays O(ckpt K V).
 *
 * Per token, in reverse, with P = S_{t-1} and dS the gradient w.r.t. S_t:
 *   dS += scale q do^T,  dq = scale S_t do
 *   GDN (w = P^T k):
 *     dv = beta dS^T k,  dbeta = k^T dS (v - alpha w),
 *     dk = beta dS v - alpha beta (dS w + P dS^T k),
 *     dg = alpha <dS, P - beta k w^T>,  dS <- alpha (dS - beta k (k^T dS))
 *   KDA (D = Diag(a) P, w = D^T k):
 *     dv = beta dS^T k,  dbeta = k^T dS (v - w),
 *     dk = beta dS v - beta (dS w + D dS^T k),
 *     dD = dS - beta k (k^T dS),  dg_c = a_c sum_j dD_cj P_cj,  dS <- Diag(a) dD
 */
void orc_bwd(int variant, int64_t n_seq, const int64_t *cu, int64_t H, int64_t K, int64_t V,
             double scale, const double *q, const double *k, const double *v, const double *g,
             const double *beta, const double *h0, const double *d_o, const double *dht,
             double *dq, double *dk, double *dv, double *dg, double *dbeta, double *dh0)
{
    const int64_t gK = (variant == ORC_KDA) ? K : 1;
    const int64_t units = n_seq * H;
    const int64_t ckpt = 64;
#pragma omp parallel
    {
        const int64_t KV = K * V;
        double *S = (double *)malloc(sizeof(double) * KV);
        double *dS = (double *)malloc(sizeof(double) * KV);
        double *dD = (double *)malloc(sizeof(double) * KV);
        double *seg = (double *)malloc(sizeof(double) * KV * (ckpt + 1));
        double *w = (double *)malloc(sizeof(double) * V);
        double *a = (double *)malloc(sizeof(double) * K);
        double *x = (double *)malloc(sizeof(double) * (K > V ? K : V));
        double *y = (double *)malloc(sizeof(double) * (K > V ? K : V));
#pragma omp for schedule(dynamic, 1)
        for (int64_t u = 0; u < units; ++u) {
            const int64_t n = u / H, h = u % H;
            const int64_t bos = cu[n], len = cu[n + 1] - cu[n];
            const int64_t nseg = (len + ckpt - 1) / ckpt;
            double *chk = (double *)malloc(sizeof(double) * KV * (nseg > 0 ? nseg : 1));
            /* forward pass: checkpoints at segment starts */
            if (h0) memcpy(S, h0 + (n * H + h) * KV, sizeof(double) * KV);
            else memset(S, 0, sizeof(double) * KV);
            for (int64_t r = 0; r < len; ++r) {
                const int64_t t = bos + r;
                if (r % ckpt == 0) memcpy(chk + (r / ckpt) * KV, S, sizeof(double) * KV);
                step_forward(variant, S, K, V, k + (t * H + h) * K, v + (t * H + h) * V,
                             g + (t * H + h) * gK, beta[t * H + h], w, a);
            }
            if (dht) memcpy(dS, dht + (n * H + h) * KV, sizeof(double) * KV);
            else memset(dS, 0, sizeof(double) * KV);
            for (int64_t sidx = nseg - 1; sidx >= 0; --sidx) {
                const int64_t r0 = sidx * ckpt;
                const int64_t r1 = (r0 + ckpt < len) ? r0 + ckpt : len;
                /* seg[i] = state before token r0 + i; seg[r1 - r0] = state after the last */
                memcpy(seg, chk + sidx * KV, sizeof(double) * KV);
                for (int64_t r = r0; r < r1; ++r) {
                    const int64_t t = bos + r;
                    double *nxt = seg + (r - r0 + 1) * KV;
                    memcpy(nxt, seg + (r - r0) * KV, sizeof(double) * KV);
                    step_forward(variant, nxt, K, V, k + (t * H + h) * K, v + (t * H + h) * V,
                                 g + (t * H + h) * gK, beta[t * H + h], w, a);
                }
                for (int64_t r = r1 - 1; r >= r0; --r) {
                    const int64_t t = bos + r;
                    const double *P = seg + (r - r0) * KV;
                    const double *St = seg + (r - r0 + 1) * KV;
                    const double *kt = k + (t * H + h) * K, *vt = v + (t * H + h) * V;
                    const double *qt = q + (t * H + h) * K, *dot = d_o + (t * H + h) * V;
                    const double *gt = g + (t * H + h) * gK;
                    const double bt_ = beta[t * H + h];
                    double *dqt = dq + (t * H + h) * K, *dkt = dk + (t * H + h) * K;
                    double *dvt = dv + (t * H + h) * V, *dgt = dg + (t * H + h) * gK;
                    /* output read-out: o_t = S_t^T (scale q_t) */
                    for (int64_t c = 0; c < K; ++c)
                        for (int64_t j = 0; j < V; ++j) dS[c * V + j] += scale * qt[c] * dot[j];
                    for (int64_t c = 0; c < K; ++c) {
                        double acc = 0.0;
                        for (int64_t j = 0; j < V; ++j) acc += St[c * V + j] * dot[j];
                        dqt[c] = scale * acc;
                    }
                    /* D = alpha P (GDN) or Diag(a) P (KDA); w = D^T k */
                    double alpha = 1.0;
                    if (variant == ORC_GDN) alpha = exp(gt[0]);
                    else for (int64_t c = 0; c < K; ++c) a[c] = exp(gt[c]);
                    for (int64_t j = 0; j < V; ++j) {
                        double acc = 0.0;
                        for (int64_t c = 0; c < K; ++c)
                            acc += (variant == ORC_GDN ? 1.0 : a[c]) * P[c * V + j] * kt[c];
                        w[j] = acc;   /* GDN: P^T k;  KDA: (Diag(a) P)^T k */
                    }
                    /* x = dS^T k (length V), y = dS w (length K) */
                    for (int64_t j = 0; j < V; ++j) {
                        double acc = 0.0;
                        for (int64_t c = 0; c < K; ++c) acc += dS[c * V + j] * kt[c];
                        x[j] = acc;
                    }
                    for (int64_t c = 0; c < K; ++c) {
                        double acc = 0.0;
                        for (int64_t j = 0; j < V; ++j) acc += dS[c * V + j] * w[j];
                        y[c] = acc;
                    }
                    for (int64_t j = 0; j < V; ++j) dvt[j] = bt_ * x[j];
                    if (variant == ORC_GDN) {
                        double db = 0.0;
                        for (int64_t j = 0; j < V; ++j) db += x[j] * (vt[j] - alpha * w[j]);
                        dbeta[t * H + h] = db;
                        for (int64_t c = 0; c < K; ++c) {
                            double dsv = 0.0, pdx = 0.0;
                            for (int64_t j = 0; j < V; ++j) {
                                dsv += dS[c * V + j] * vt[j];
                                pdx += P[c * V + j] * x[j];
                            }
                            dkt[c] = bt_ * dsv - alpha * bt_ * (y[c] + pdx);
                        }
                        double da = 0.0;
                        for (int64_t c = 0; c < K; ++c)
                            for (int64_t j = 0; j < V; ++j)
                                da += dS[c * V + j] * (P[c * V + j] - bt_ * kt[c] * w[j]);
                        dgt[0] = alpha * da;
                        for (int64_t c = 0; c < K; ++c)
                            for (int64_t j = 0; j < V; ++j)
                                dS[c * V + j] = alpha * (dS[c * V + j] - bt_ * kt[c] * x[j]);
                    } else {
                        double db = 0.0;
                        for (int64_t j = 0; j < V; ++j) db += x[j] * (vt[j] - w[j]);
                        dbeta[t * H + h] = db;
                        for (int64_t c = 0; c < K; ++c) {
                            double dsv = 0.0, ddx = 0.0;
                            for (int64_t j = 0; j < V; ++j) {
                                dsv += dS[c * V + j] * vt[j];
                                ddx += a[c] * P[c * V + j] * x[j];
                            }
                            dkt[c] = bt_ * dsv - bt_ * (y[c] + ddx);
                        }
                        for (int64_t c = 0; c < K; ++c)
                            for (int64_t j = 0; j < V; ++j)
                                dD[c * V + j] = dS[c * V + j] - bt_ * kt[c] * x[j];
                        for (int64_t c = 0; c < K; ++c) {
                            double acc = 0.0;
                            for (int64_t j = 0; j < V; ++j) acc += dD[c * V + j] * P[c * V + j];
                            dgt[c] = a[c] * acc;
                        }
                        for (int64_t c = 0; c < K; ++c)
                            for (int64_t j = 0; j < V; ++j) dS[c * V + j] = a[c] * dD[c * V + j];
                    }
                }
            }
            memcpy(dh0 + (n * H + h) * KV, dS, sizeof(double) * KV);
            free(chk);
        }
        free(S); free(dS); free(dD); free(seg); free(w); free(a); free(x); free(y);
    }
}
