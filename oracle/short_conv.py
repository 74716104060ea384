"""fp64 oracle of the short (causal, depthwise) convolution that precedes the chunk attention.

TEST INFRASTRUCTURE ONLY, like the rest of this package: the CUDA library never imports it.

FLA RFC "[RFC] Add Graph Capture Support for FLA Prefill and Training Paths on Ascend NPUs",
section "Step 3": the short convolution covers dense and varlen inputs, forward and backward,
bias, activation and residual paths, initial and final states.  The pages print no formula;
the reading taken is the causal depthwise convolution of width W over the tokens of each
sequence (the section "Step 4" places it between the projection and the chunk attention):

    xx_n(i) = x[bos_n + i]              for 0 <= i < len_n
            = h0[n, :, W - 1 + i]       for -(W - 1) <= i < 0   (zeros without h0)
    pre[bos_n + p] = b + sum_j w[:, j] * xx_n(p - (W - 1) + j)        (j = 0 .. W - 1)
    y = act(pre) + r                    (act: identity or silu(z) = z / (1 + exp(-z)))
    ht[n, :, k] = xx_n(len_n - (W - 1) + k)                          (k = 0 .. W - 2)

Layouts: x, r, y [T, D] token-major; w [D, W]; b [D]; h0, ht [N, D, W - 1] (oldest first).
The backward is reverse mode of <dy, y> + <dht, ht>: dx, dw, db, dh0 (the residual's
gradient is dy itself).
"""
from __future__ import annotations

import numpy as np


def _silu(z):
    return z / (1.0 + np.exp(-z))


def _silu_grad(z):
    s = 1.0 / (1.0 + np.exp(-z))
    return s * (1.0 + z * (1.0 - s))


def _window(x, h0, n, bos, length, W, D):
    """xx_n(i) for i = -(W - 1) .. length - 1 as rows of an array (row i + W - 1)."""
    xx = np.zeros((length + W - 1, D))
    if h0 is not None:
        xx[:W - 1] = np.asarray(h0[n], dtype=np.float64).T
    xx[W - 1:] = x[bos:bos + length]
    return xx


def conv_fwd(x, w, b, r, h0, cu_seqlens, activation=None):
    """y [T, D] and ht [N, D, W - 1]; token rows outside every sequence stay zero."""
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    T, D = x.shape
    W = w.shape[1]
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    N = len(cu) - 1
    y = np.zeros((T, D))
    ht = np.zeros((N, D, W - 1))
    for n in range(N):
        bos, eos = int(cu[n]), int(cu[n + 1])
        length = eos - bos
        xx = _window(x, h0, n, bos, length, W, D)
        for p in range(length):
            pre = np.zeros(D) if b is None else np.asarray(b, dtype=np.float64).copy()
            for j in range(W):
                pre += w[:, j] * xx[p + j]           # xx_n(p - (W - 1) + j) is row p + j
            out = _silu(pre) if activation == "silu" else pre
            if r is not None:
                out = out + np.asarray(r[bos + p], dtype=np.float64)
            y[bos + p] = out
        for k in range(W - 1):
            ht[n, :, k] = xx[length + k]             # xx_n(len - (W - 1) + k)
    return y, ht


def conv_bwd(x, w, b, h0, cu_seqlens, dy, dht=None, activation=None):
    """dx [T, D], dw [D, W], db [D], dh0 [N, D, W - 1] of <dy, y> + <dht, ht>."""
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    dy = np.asarray(dy, dtype=np.float64)
    T, D = x.shape
    W = w.shape[1]
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    N = len(cu) - 1
    dx = np.zeros((T, D))
    dw = np.zeros((D, W))
    db = np.zeros(D)
    dh0 = np.zeros((N, D, W - 1))
    for n in range(N):
        bos, eos = int(cu[n]), int(cu[n + 1])
        length = eos - bos
        xx = _window(x, h0, n, bos, length, W, D)
        dxx = np.zeros_like(xx)
        for p in range(length):
            pre = np.zeros(D) if b is None else np.asarray(b, dtype=np.float64).copy()
            for j in range(W):
                pre += w[:, j] * xx[p + j]
            g = dy[bos + p] * (_silu_grad(pre) if activation == "silu" else 1.0)
            db += g
            for j in range(W):
                dw[:, j] += g * xx[p + j]
                dxx[p + j] += g * w[:, j]
        if dht is not None:
            for k in range(W - 1):
                dxx[length + k] += np.asarray(dht[n, :, k], dtype=np.float64)
        dx[bos:eos] = dxx[W - 1:]
        dh0[n] = dxx[:W - 1].T
    return dx, dw, db, dh0
