"""fp64 CPU oracle for chunked gated linear attention (GDN and KDA).

TEST INFRASTRUCTURE ONLY.  The CUDA library never imports, loads or calls
anything in this package; only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg do.  It shares no code with the CUDA path.

Two independent implementations live here:

* ``gcl_oracle.c`` (wrapped below): the token-by-token recurrence in double
  precision -- the definition of what the method computes -- plus the chunk
  metadata built by plain loops and the reverse-mode backward.
* ``chunk_form.py``: a separate fp64 evaluator of the chunkwise
  (Map-Reduce-Map) form, used only to cross-check the chunk algebra.
* ``short_conv.py``: the short causal depthwise convolution that precedes the
  chunk attention, forward and reverse mode (numpy, fp64).

Every function takes numpy arrays in the token-major layouts of the FLA RFC
"[RFC] Add Graph Capture Support for FLA Prefill and Training Paths on Ascend
NPUs" (section "Core design"): q, k [T, H, K]; v [T, H, V]; g [T, H] for GDN
or [T, H, K] for KDA; beta [T, H]; states [N, H, K, V]; packed sequences
delimited by cu_seqlens [N + 1].
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gcl_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None

GDN, KDA = 0, 1

from .short_conv import conv_bwd, conv_fwd  # noqa: E402,F401  (the short convolution)


def build(force: bool = False) -> str:
    """Compile the C oracle into ``oracle/liboracle.so`` (gcc, OpenMP, no fast-math)."""
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def bind(lib):
    """Declare the C signatures on a loaded oracle library (also used on test mutants)."""
    i64 = ctypes.c_int64
    vp = ctypes.c_void_p
    lib.orc_nt_max.restype = i64
    lib.orc_nt_max.argtypes = [i64, i64, i64]
    lib.orc_num_threads.restype = ctypes.c_int
    lib.orc_chunk_meta.restype = ctypes.c_int
    lib.orc_chunk_meta.argtypes = [vp, i64, i64, i64, i64, vp, vp]
    lib.orc_fwd.restype = None
    lib.orc_fwd.argtypes = ([ctypes.c_int, i64, vp, i64, i64, i64, ctypes.c_double]
                            + [vp] * 9 + [i64, vp])
    lib.orc_bwd.restype = None
    lib.orc_bwd.argtypes = [ctypes.c_int, i64, vp, i64, i64, i64, ctypes.c_double] + [vp] * 14
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = bind(ctypes.CDLL(build()))
    return _lib


def _f64(x):
    return None if x is None else np.ascontiguousarray(x, dtype=np.float64)


def _ptr(x):
    return None if x is None else x.ctypes.data


def num_threads() -> int:
    """OpenMP threads the oracle uses (all host cores unless OMP_NUM_THREADS says otherwise)."""
    return int(_load().orc_num_threads())


def nt_max(t_max: int, n_max: int, bt: int) -> int:
    """NT_max = ceil(T_max / BT) + N_max - 1 (FLA RFC, "Fixed-capacity execution")."""
    return int(_load().orc_nt_max(t_max, n_max, bt))


def chunk_meta(cu_seqlens, t_max: int, bt: int):
    """Plain-loop chunk metadata (FLA RFC, "Device-side metadata").

    Returns (status, chunk_indices int32 [NT_max, 2], chunk_offsets int32 [N_max + 1]).
    status: 0 ok; 2 cu[0] != 0; 1 decreasing cu_seqlens; 3 cu[N_max] > T_max.
    """
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int64)
    n_max = cu.shape[0] - 1
    ntm = nt_max(t_max, n_max, bt)
    idx = np.empty((ntm, 2), dtype=np.int32)
    off = np.empty((n_max + 1,), dtype=np.int32)
    st = _load().orc_chunk_meta(_ptr(cu), n_max, t_max, bt, ntm, _ptr(idx), _ptr(off))
    return int(st), idx, off


def _dims(variant, q, v, g, cu):
    T, H, K = q.shape
    V = v.shape[2]
    if variant == KDA:
        assert g.shape == (T, H, K), "KDA gate is per channel: [T, H, K]"
    else:
        assert g.shape == (T, H), "GDN gate is per head: [T, H]"
    return T, H, K, V, cu.shape[0] - 1


def fwd(variant, q, k, v, g, beta, h0, cu_seqlens, scale, bt=None, chunk_offsets=None,
        nt_rows=None):
    """Token recurrence forward.  Returns (o [T,H,V], ht [N,H,K,V]) in float64, plus
    h_chunk [nt_rows,H,K,V] (state before each chunk of size ``bt``) when ``bt`` is given."""
    q, k, v, g, beta, h0 = map(_f64, (q, k, v, g, beta, h0))
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int64)
    T, H, K, V, N = _dims(variant, q, v, g, cu)
    o = np.zeros((T, H, V))
    ht = np.zeros((N, H, K, V))
    h_chunk = None
    off = None
    if bt is not None:
        off = np.ascontiguousarray(chunk_offsets, dtype=np.int32)
        h_chunk = np.zeros((nt_rows, H, K, V))
    _load().orc_fwd(variant, N, _ptr(cu), H, K, V, float(scale), _ptr(q), _ptr(k), _ptr(v),
                    _ptr(g), _ptr(beta), _ptr(h0), _ptr(o), _ptr(ht), _ptr(h_chunk),
                    int(bt or 1), _ptr(off))
    if bt is not None:
        return o, ht, h_chunk
    return o, ht


def bwd(variant, q, k, v, g, beta, h0, d_o, dht, cu_seqlens, scale):
    """Reverse-mode gradients of <do, o> + <dht, ht>.

    Returns dict with dq, dk [T,H,K]; dv [T,H,V]; dg (shape of g); dbeta [T,H]; dh0 [N,H,K,V].
    Token rows outside every sequence are left at zero."""
    q, k, v, g, beta, h0, d_o, dht = map(_f64, (q, k, v, g, beta, h0, d_o, dht))
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int64)
    T, H, K, V, N = _dims(variant, q, v, g, cu)
    out = dict(dq=np.zeros((T, H, K)), dk=np.zeros((T, H, K)), dv=np.zeros((T, H, V)),
               dg=np.zeros(g.shape), dbeta=np.zeros((T, H)), dh0=np.zeros((N, H, K, V)))
    _load().orc_bwd(variant, N, _ptr(cu), H, K, V, float(scale), _ptr(q), _ptr(k), _ptr(v),
                    _ptr(g), _ptr(beta), _ptr(h0), _ptr(d_o), _ptr(dht), _ptr(out["dq"]),
                    _ptr(out["dk"]), _ptr(out["dv"]), _ptr(out["dg"]), _ptr(out["dbeta"]),
                    _ptr(out["dh0"]))
    return out


def gdn_fwd(*a, **kw):
    return fwd(GDN, *a, **kw)


def kda_fwd(*a, **kw):
    return fwd(KDA, *a, **kw)


def gdn_bwd(*a, **kw):
    return bwd(GDN, *a, **kw)


def kda_bwd(*a, **kw):
    return bwd(KDA, *a, **kw)
