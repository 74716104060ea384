"""Independent fp64 evaluator of the chunkwise Map-Reduce-Map form.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  It is used to check the
chunk algebra against the token recurrence of ``gcl_oracle.c``; it is written
separately from both that file and the CUDA path, and uses a dense
``numpy.linalg.solve`` for (I + A)^-1 instead of any substitution scheme.

Chunk algebra (HA-NPU paper "Empowering Hybrid Attention Models on NPUs",
section 2.1 Map-Reduce-Map, section 5 chunk-first in-place update and GEMM-first
grouping; FLA RFC step 3 pipeline: gate cumsum -> intra (KK^T, solve) ->
recompute_w_u -> h -> o).  Per chunk of length c with state S at its start,
gamma = inclusive cumsum of the log gates inside the chunk, Gamma = exp(gamma):

  GDN  A[r,i] = beta_r exp(gamma_r - gamma_i) (k_r . k_i)      i < r
       L[r,i] = scale  exp(gamma_r - gamma_i) (q_r . k_i)      i <= r
       T = (I + A)^-1,  W = T diag(beta Gamma) K,  U = T diag(beta) V
       E = U - W S                               (WY order)
         = T diag(beta) (V - diag(Gamma) K S)    (GEMM-first order)
       O = scale diag(Gamma) Q S + L E
       S <- Gamma_c S + (diag(exp(gamma_c - gamma)) K)^T E
  KDA  the decays become per key channel:
       A[r,i] = beta_r sum_d k_rd k_id exp(gamma_rd - gamma_id), likewise L,
       W = T diag(beta) (K * Gamma),  O = scale (Q * Gamma) S + L E,
       S <- Diag(Gamma_c) S + (K * exp(gamma_c - gamma))^T E
"""
from __future__ import annotations

import numpy as np


def _chunk_gdn(Qc, Kc, Vc, gc, bc, S, scale, order):
    c = Kc.shape[0]
    gam = np.cumsum(gc)
    dec = np.exp(gam[:, None] - gam[None, :])
    strict = np.tril(np.ones((c, c)), -1)
    incl = np.tril(np.ones((c, c)))
    A = strict * (bc[:, None] * dec * (Kc @ Kc.T))
    L = incl * (scale * dec * (Qc @ Kc.T))
    Tm = np.linalg.solve(np.eye(c) + A, np.eye(c))
    Gam = np.exp(gam)
    if order == "wy":
        W = Tm @ ((bc * Gam)[:, None] * Kc)
        U = Tm @ (bc[:, None] * Vc)
        E = U - W @ S
    else:
        E = Tm @ (bc[:, None] * (Vc - Gam[:, None] * (Kc @ S)))
    O = scale * Gam[:, None] * (Qc @ S) + L @ E
    gC = gam[-1]
    Kt = np.exp(gC - gam)[:, None] * Kc
    S_new = np.exp(gC) * S + Kt.T @ E
    return O, S_new


def _chunk_kda(Qc, Kc, Vc, gc, bc, S, scale, order):
    c = Kc.shape[0]
    gam = np.cumsum(gc, axis=0)                       # [c, K]
    dec = np.exp(gam[:, None, :] - gam[None, :, :])   # [r, i, K]
    strict = np.tril(np.ones((c, c)), -1)
    incl = np.tril(np.ones((c, c)))
    with np.errstate(over="ignore", invalid="ignore"):
        A = np.einsum("rd,id,rid->ri", Kc, Kc, dec)
        L = np.einsum("rd,id,rid->ri", Qc, Kc, dec)
    A = np.where(strict > 0, bc[:, None] * A, 0.0)
    L = np.where(incl > 0, scale * L, 0.0)
    Tm = np.linalg.solve(np.eye(c) + A, np.eye(c))
    Gam = np.exp(gam)
    if order == "wy":
        W = Tm @ (bc[:, None] * (Kc * Gam))
        U = Tm @ (bc[:, None] * Vc)
        E = U - W @ S
    else:
        E = Tm @ (bc[:, None] * (Vc - (Kc * Gam) @ S))
    O = scale * (Qc * Gam) @ S + L @ E
    gC = gam[-1]
    Kt = Kc * np.exp(gC[None, :] - gam)
    S_new = np.exp(gC)[:, None] * S + Kt.T @ E
    return O, S_new


def chunk_fwd(variant, q, k, v, g, beta, h0, cu_seqlens, scale, bt, order="wy"):
    """Chunked forward over a varlen batch.  variant 0 = GDN, 1 = KDA.

    Returns (o [T,H,V], ht [N,H,K,V]) in float64.  ``order`` selects the WY form
    ("wy") or the GEMM-first form ("gemm_first") of E."""
    q, k, v, g, beta = (np.asarray(x, dtype=np.float64) for x in (q, k, v, g, beta))
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    T, H, K = q.shape
    V = v.shape[2]
    N = cu.shape[0] - 1
    o = np.zeros((T, H, V))
    ht = np.zeros((N, H, K, V))
    step = _chunk_kda if variant == 1 else _chunk_gdn
    for n in range(N):
        for h in range(H):
            S = np.zeros((K, V)) if h0 is None else np.array(h0[n, h], dtype=np.float64)
            for t0 in range(int(cu[n]), int(cu[n + 1]), bt):
                t1 = min(t0 + bt, int(cu[n + 1]))
                O, S = step(q[t0:t1, h], k[t0:t1, h], v[t0:t1, h], g[t0:t1, h],
                            beta[t0:t1, h], S, scale, order)
                o[t0:t1, h] = O
            ht[n, h] = S
    return o, ht
