"""Seeded synthetic inputs for chunked gated linear attention.

This module holds no arithmetic of the method itself: it only draws the
random inputs (numpy ``Generator(PCG64(seed))`` in fp32), rounds them to bf16
where a workload says so, and lays them out in the token-major buffers of the
FLA RFC "[RFC] Add Graph Capture Support for FLA Prefill and Training Paths on
Ascend NPUs" (section "Core design": fixed-capacity buffers of T_max tokens and
N_max + 1 cu_seqlens entries).  The same arrays feed the CPU oracle and the
CUDA library, so both see identical rounded values.

Input recipe (one draw per tensor, in this order):
  q, k   ~ N(0, 1), then L2-normalised over d_k
  v      ~ N(0, 1)
  beta   = sigmoid(N(0, 1))                  per token and head
  g      = -softplus(N(0, 1))                per token and head (GDN) or per key channel (KDA)
  h0     ~ N(0, 0.1^2) fp32, or zeros
  do     ~ N(0, 1), dht ~ N(0, 0.1^2)        (backward workloads)
bf16 tensors (q, k, v, beta, do) are rounded to nearest-even after drawing;
g, h0 and dht stay fp32.  Rows of the fixed-capacity buffers past the last
live token are filled with NaN so that any read of them shows up.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

GDN, KDA = 0, 1


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to the nearest bf16 (ties to even); NaN stays NaN.

    Returns float32 values that are exactly representable in bf16."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000).astype(np.uint32)
    out = r.view(np.float32).copy()
    nan = np.isnan(x)
    out[nan] = np.float32("nan")
    return out


def f16_round(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to the nearest fp16 (numpy's IEEE conversion, ties to even).

    Returns float32 values that are exactly representable in fp16."""
    return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).astype(np.float32)


def round_to(x: np.ndarray, dtype: str) -> np.ndarray:
    """Inputs of a workload of element type dtype ("f32", "bf16" or "f16") as float32."""
    if dtype == "bf16":
        return bf16_round(x)
    if dtype == "f16":
        return f16_round(x)
    return np.ascontiguousarray(x, dtype=np.float32)


@dataclass
class Workload:
    """A named synthetic workload.  Sizes follow the method's own notation."""
    name: str
    variant: int                 # GDN or KDA
    dtype: str                   # "f32" or "bf16": type of q, k, v, beta (and o)
    H: int
    K: int
    V: int
    lengths: list                # live sequence lengths (may contain zeros)
    n_max: int                   # cu_seqlens capacity - 1
    t_max: int                   # token capacity
    bt: int = 64
    h0: bool = True
    backward: bool = False
    seed: int = 0
    extra: dict = field(default_factory=dict)

    @property
    def total_tokens(self) -> int:
        return int(sum(self.lengths))

    @property
    def scale(self) -> float:
        return float(self.K) ** -0.5


def dense(name, variant, dtype, B, T, H, K, V, h0=True, backward=False, seed=0, bt=64):
    """B equal-length sequences of T tokens (a dense batch is varlen with equal lengths)."""
    return Workload(name, variant, dtype, H, K, V, [T] * B, B, B * T, bt, h0, backward, seed)


def varlen(name, variant, dtype, lengths, n_max, t_max, H, K, V, h0=True, backward=False,
           seed=0, bt=64):
    return Workload(name, variant, dtype, H, K, V, list(lengths), n_max, t_max, bt, h0,
                    backward, seed)


def random_lengths(n: int, lo: int, hi: int, seed: int) -> list:
    """n lengths uniform in [lo, hi] from a seeded PCG64 stream."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return [int(x) for x in rng.integers(lo, hi + 1, size=n)]


# The five standard workloads.  Index = seed.
def standard_workloads():
    return [
        dense("gdn_fwd_fp32_T256_H2_d64", GDN, "f32", 1, 256, 2, 64, 64, h0=False, seed=0),
        dense("gdn_fwd_bf16_T4096_H16_d128", GDN, "bf16", 1, 4096, 16, 128, 128, seed=1),
        dense("kda_fwd_bf16_T2048_H10_d128", KDA, "bf16", 1, 2048, 10, 128, 128, seed=2),
        varlen("gdn_varlen_bf16_N32_Nmax64_Tmax65536_H16_d128", GDN, "bf16",
               random_lengths(32, 1, 2048, 30), 64, 65536, 16, 128, 128, seed=3),
        dense("gdn_fwdbwd_bf16_B4_T8192_H16_d128", GDN, "bf16", 4, 8192, 16, 128, 128,
              backward=True, seed=4),
        # beyond the five configurations above: the KDA backward, at the KDA forward's sizes
        dense("kda_fwdbwd_bf16_T2048_H10_d128", KDA, "bf16", 1, 2048, 10, 128, 128,
              backward=True, seed=5),
        # the extreme tail: one long sequence of one head (one unit for 152 SMs), the case
        # the chunk-head-chunk mapping of the third scheduling tier serves
        dense("gdn_fwd_bf16_T65536_H1_d128", GDN, "bf16", 1, 65536, 1, 128, 128, seed=6),
        dense("kda_fwd_bf16_T65536_H1_d128", KDA, "bf16", 1, 65536, 1, 128, 128, seed=7),
        # the RFC test matrix's variants at the headline sizes: fp16 inputs, chunk size 32
        dense("gdn_fwd_f16_T4096_H16_d128", GDN, "f16", 1, 4096, 16, 128, 128, seed=8),
        dense("gdn_fwd_bf16_bt32_T4096_H16_d128", GDN, "bf16", 1, 4096, 16, 128, 128, seed=9,
              bt=32),
    ]


def workload_by_name(name: str) -> Workload:
    for w in standard_workloads():
        if w.name == name:
            return w
    raise KeyError(name)


def cu_seqlens_of(w: Workload) -> np.ndarray:
    """cu_seqlens of shape [n_max + 1]; slots past the live sequences are zero-length."""
    lens = list(w.lengths) + [0] * (w.n_max - len(w.lengths))
    cu = np.zeros(w.n_max + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lens)
    return cu


def make_inputs(w: Workload, seed: int | None = None, pad_value: float = float("nan")):
    """Draw the inputs of workload ``w``.

    Returns a dict of float32 numpy arrays (bf16- or fp16-representable where w.dtype is
    bf16 or f16) in fixed-capacity layout: q, k [T_max,H,K]; v [T_max,H,V]; beta [T_max,H];
    g [T_max,H] or [T_max,H,K]; h0 [N_max,H,K,V] or None; cu_seqlens int32
    [N_max+1]; and, for backward workloads, do [T_max,H,V] and dht [N_max,H,K,V]."""
    seed = w.seed if seed is None else seed
    rng = np.random.Generator(np.random.PCG64(seed))
    T, Tm, H, K, V = w.total_tokens, w.t_max, w.H, w.K, w.V
    assert T <= Tm

    def pad(a):
        out = np.full((Tm,) + a.shape[1:], pad_value, dtype=np.float32)
        out[:T] = a
        return out

    def rnd(a):
        return round_to(a, w.dtype)

    q = rng.standard_normal((T, H, K), dtype=np.float32)
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k = rng.standard_normal((T, H, K), dtype=np.float32)
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, V), dtype=np.float32)
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, H), dtype=np.float32)))
    gshape = (T, H, K) if w.variant == KDA else (T, H)
    g = -np.logaddexp(0.0, rng.standard_normal(gshape, dtype=np.float32)).astype(np.float32)
    out = dict(q=pad(rnd(q)), k=pad(rnd(k)), v=pad(rnd(v)), beta=pad(rnd(beta)),
               g=pad(g.astype(np.float32)), cu_seqlens=cu_seqlens_of(w))
    out["h0"] = ((0.1 * rng.standard_normal((w.n_max, H, K, V), dtype=np.float32))
                 if w.h0 else None)
    if w.backward:
        out["do"] = pad(rnd(rng.standard_normal((T, H, V), dtype=np.float32)))
        out["dht"] = 0.1 * rng.standard_normal((w.n_max, H, K, V), dtype=np.float32)
    return out


def layout_seeds(w: Workload):
    """Seeds of the replay layouts of a varlen workload: capture layout, then three replays."""
    return [w.seed * 10, w.seed * 10 + 1, w.seed * 10 + 2, w.seed * 10 + 3]


def varlen_layout(w: Workload, layout_seed: int) -> Workload:
    """A fresh varlen layout with the same capacities: same sequence count, new lengths."""
    n = len(w.lengths)
    hi = w.extra.get("max_len", 2048)
    lens = random_lengths(n, 1, hi, layout_seed)
    return varlen(w.name, w.variant, w.dtype, lens, w.n_max, w.t_max, w.H, w.K, w.V, w.h0,
                  w.backward, seed=layout_seed, bt=w.bt)


def make_conv_inputs(lengths, n_max: int, t_max: int, D: int, W: int, dtype: str, seed: int,
                     h0: bool = True, bias: bool = True, residual: bool = False,
                     pad_value: float = float("nan")):
    """Inputs of the short convolution over the sequences ``lengths`` (n_max slots, t_max
    token capacity): x [t_max, D] ~ N(0, 1); weight [D, W] ~ N(0, 1/W); bias [D] ~ N(0, 0.1^2);
    residual [t_max, D] ~ N(0, 1); h0 [n_max, D, W - 1] ~ N(0, 1) (the inputs before each
    sequence); dy [t_max, D] ~ N(0, 1); dht [n_max, D, W - 1] ~ N(0, 0.1^2) fp32.  Everything
    but dht is rounded to bf16 when dtype is bf16; padding rows hold ``pad_value``."""
    rng = np.random.Generator(np.random.PCG64(seed))
    lens = list(lengths) + [0] * (n_max - len(lengths))
    cu = np.zeros(n_max + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lens)
    T = int(cu[-1])
    assert T <= t_max

    def rnd(a):
        return bf16_round(a) if dtype == "bf16" else a.astype(np.float32)

    def pad(a):
        out = np.full((t_max,) + a.shape[1:], pad_value, dtype=np.float32)
        out[:T] = a
        return out

    out = dict(cu_seqlens=cu)
    out["x"] = pad(rnd(rng.standard_normal((T, D), dtype=np.float32)))
    out["weight"] = rnd(rng.standard_normal((D, W), dtype=np.float32) / np.sqrt(W))
    out["bias"] = rnd(0.1 * rng.standard_normal(D, dtype=np.float32)) if bias else None
    out["residual"] = pad(rnd(rng.standard_normal((T, D), dtype=np.float32))) if residual else None
    out["h0"] = rnd(rng.standard_normal((n_max, D, W - 1), dtype=np.float32)) if h0 else None
    out["dy"] = pad(rnd(rng.standard_normal((T, D), dtype=np.float32)))
    out["dht"] = (0.1 * rng.standard_normal((n_max, D, W - 1), dtype=np.float32)).astype(np.float32)
    return out


def conv_workloads():
    """Short-convolution workloads (forward + backward per step): the dense batch of the
    forward+backward attention workload, D = 2048 channels (16 heads x 128), W = 4 taps, SiLU,
    bias and initial states."""
    return [dict(name="conv_fwdbwd_bf16_B4_T8192_D2048_W4", B=4, T=8192, D=2048, W=4,
                 dtype="bf16", act="silu", seed=40)]


def conv_workload_by_name(name: str):
    for c in conv_workloads():
        if c["name"] == name:
            return c
    raise KeyError(name)
