"""Python binding of libgcl, the GB300 chunked gated linear attention library.

Argument marshalling only: every entry point forwards torch tensors' device
pointers and the current CUDA stream to the C ABI declared in
``include/gcl.h``; all computation happens in the library's CUDA kernels.  The
library must have been built (``python -m chunked_gated_linear_gb300._build``
or ``__graft_entry__.build()``); importing this package fails loudly otherwise,
and there is no other implementation to fall back on.

The library sees raw pointers only, so before each launch the binding checks what a
pointer cannot carry: every tensor is a contiguous CUDA tensor on the call's device, of the
dtype and at least the size ``include/gcl.h`` gives it.  A host tensor or a too-small buffer
would otherwise be read or written out of bounds on the device.
"""
from __future__ import annotations

import ctypes
import inspect
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libgcl.so")
# the bounds-checking debug build (GCL_DEBUG_BOUNDS), for tests: load_library(DEBUG_LIB_PATH)
DEBUG_LIB_PATH = os.path.join(PKG, "libgcl_debug.so")

GCL_F32, GCL_BF16, GCL_F16 = 0, 1, 2
DEV_STATUS = {0: "ok", 1: "cu_seqlens decreasing", 2: "cu_seqlens[0] != 0",
              3: "cu_seqlens[N_max] > T_max", 4: "invalid sequence range"}
CHUNK = 64


class GclError(RuntimeError):
    def __init__(self, fn, status, msg):
        super().__init__(f"{fn} failed with status {status}: {msg}")
        self.status = status


class FwdArgs(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("g", ctypes.c_void_p), ("beta", ctypes.c_void_p), ("h0", ctypes.c_void_p),
                ("cu_seqlens", ctypes.c_void_p), ("chunk_indices", ctypes.c_void_p),
                ("chunk_offsets", ctypes.c_void_p),
                ("seq_order", ctypes.c_void_p), ("o", ctypes.c_void_p), ("ht", ctypes.c_void_p),
                ("h_save", ctypes.c_void_p), ("dev_status", ctypes.c_void_p),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
                ("t_max", ctypes.c_int64), ("n_max", ctypes.c_int32), ("H", ctypes.c_int32),
                ("K", ctypes.c_int32), ("V", ctypes.c_int32), ("bt", ctypes.c_int32),
                ("scale", ctypes.c_float), ("dtype", ctypes.c_int32)]


class BwdArgs(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("g", ctypes.c_void_p), ("beta", ctypes.c_void_p), ("h0", ctypes.c_void_p),
                ("d_o", ctypes.c_void_p), ("dht", ctypes.c_void_p),
                ("cu_seqlens", ctypes.c_void_p), ("chunk_indices", ctypes.c_void_p),
                ("chunk_offsets", ctypes.c_void_p), ("h_save", ctypes.c_void_p),
                ("dq", ctypes.c_void_p), ("dk", ctypes.c_void_p), ("dv", ctypes.c_void_p),
                ("dg", ctypes.c_void_p), ("dbeta", ctypes.c_void_p), ("dh0", ctypes.c_void_p),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
                ("dev_status", ctypes.c_void_p), ("t_max", ctypes.c_int64),
                ("n_max", ctypes.c_int32), ("H", ctypes.c_int32), ("K", ctypes.c_int32),
                ("V", ctypes.c_int32), ("bt", ctypes.c_int32), ("scale", ctypes.c_float),
                ("dtype", ctypes.c_int32), ("fwd_workspace", ctypes.c_void_p),
                ("fwd_workspace_bytes", ctypes.c_size_t)]


class ConvArgs(ctypes.Structure):
    _fields_ = [("x", ctypes.c_void_p), ("weight", ctypes.c_void_p), ("bias", ctypes.c_void_p),
                ("residual", ctypes.c_void_p), ("h0", ctypes.c_void_p), ("y", ctypes.c_void_p),
                ("ht", ctypes.c_void_p), ("dy", ctypes.c_void_p), ("dht", ctypes.c_void_p),
                ("dx", ctypes.c_void_p), ("dweight", ctypes.c_void_p), ("dbias", ctypes.c_void_p),
                ("dh0", ctypes.c_void_p), ("cu_seqlens", ctypes.c_void_p),
                ("chunk_indices", ctypes.c_void_p), ("dev_status", ctypes.c_void_p),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
                ("t_max", ctypes.c_int64), ("n_max", ctypes.c_int32), ("D", ctypes.c_int32),
                ("W", ctypes.c_int32), ("bt", ctypes.c_int32), ("activation", ctypes.c_int32),
                ("dtype", ctypes.c_int32)]


def load_library(path: str = LIB_PATH):
    """Load libgcl.so and declare its C signatures."""
    if not os.path.exists(path):
        raise ImportError(f"libgcl.so not built at {path}; run chunked_gated_linear_gb300._build")
    lib = ctypes.CDLL(path)
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    lib.gcl_last_error.restype = ctypes.c_char_p
    lib.gcl_status_string.restype = ctypes.c_char_p
    lib.gcl_status_string.argtypes = [i32]
    lib.gcl_nt_max.restype = i64
    lib.gcl_nt_max.argtypes = [i64, i64, i32]
    lib.gcl_fwd_chain_segments.restype = i32
    lib.gcl_fwd_chain_segments.argtypes = [i64, i32, i32, i32]
    lib.gcl_selftest_wait_timeout.restype = ctypes.c_int
    lib.gcl_selftest_wait_timeout.argtypes = [vp, vp]
    lib.chunk_meta_build.restype = ctypes.c_int
    lib.chunk_meta_build.argtypes = [vp, i32, i64, i32, i64, vp, vp, vp, vp, vp]
    lib.chunk_meta_build_i64.restype = ctypes.c_int
    lib.chunk_meta_build_i64.argtypes = [vp, i32, i64, i32, i64, vp, vp, vp, vp, vp, vp]
    for fn in ("gdn_chunk_fwd", "kda_chunk_fwd"):
        getattr(lib, fn).restype = ctypes.c_int
        getattr(lib, fn).argtypes = [ctypes.POINTER(FwdArgs), vp]
    lib.gdn_chunk_fwd_noalloc.restype = ctypes.c_int
    lib.gdn_chunk_fwd_noalloc.argtypes = [ctypes.POINTER(FwdArgs), vp]
    lib.gcl_noalloc_scratch_bytes.restype = ctypes.c_size_t
    lib.gcl_noalloc_scratch_bytes.argtypes = []
    for fn in ("gcl_fwd_workspace_bytes", "gcl_fwd_workspace_min_bytes", "gcl_kda_fwd_workspace_bytes"):
        getattr(lib, fn).restype = ctypes.c_size_t
        getattr(lib, fn).argtypes = [ctypes.POINTER(FwdArgs)]
    for fn in ("gcl_fwd_plan", "gcl_kda_fwd_plan"):
        getattr(lib, fn).restype = i32
        getattr(lib, fn).argtypes = [ctypes.POINTER(FwdArgs)]
    for fn in ("gdn_chunk_bwd", "kda_chunk_bwd"):
        getattr(lib, fn).restype = ctypes.c_int
        getattr(lib, fn).argtypes = [ctypes.POINTER(BwdArgs), vp]
    for fn in ("gcl_bwd_workspace_bytes", "gcl_kda_bwd_workspace_bytes"):
        getattr(lib, fn).restype = ctypes.c_size_t
        getattr(lib, fn).argtypes = [ctypes.POINTER(BwdArgs)]
    for fn in ("causal_conv1d_fwd", "causal_conv1d_bwd"):
        getattr(lib, fn).restype = ctypes.c_int
        getattr(lib, fn).argtypes = [ctypes.POINTER(ConvArgs), vp]
    lib.gcl_causal_conv1d_bwd_workspace_bytes.restype = ctypes.c_size_t
    lib.gcl_causal_conv1d_bwd_workspace_bytes.argtypes = [ctypes.POINTER(ConvArgs)]
    return lib


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = load_library()
    return _lib


def _p(t):
    """Device pointer of a tensor (or None)."""
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to libgcl must be contiguous")
    return t.data_ptr()


def _stream(stream):
    if stream is not None:
        return ctypes.c_void_p(stream if isinstance(stream, int) else stream.cuda_stream)
    import torch
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _check(fn, st):
    if st != 0:
        raise GclError(fn, st, lib().gcl_last_error().decode())


def _dtype_of(t):
    import torch
    if t.dtype == torch.float32:
        return GCL_F32
    if t.dtype == torch.bfloat16:
        return GCL_BF16
    if t.dtype == torch.float16:
        return GCL_F16
    raise ValueError(f"unsupported dtype {t.dtype}")


class _Layout:
    """Checks one call's tensors against their layouts in include/gcl.h: a CUDA tensor on the
    call's device (when require_cuda), contiguous, of the given dtype(s), with the given
    trailing dimensions and at least the given number of rows."""

    def __init__(self, fn: str, require_cuda: bool = True):
        self.fn, self.require_cuda, self.device = fn, require_cuda, None

    def __call__(self, name, t, dtypes=None, shape=None):
        if t is None:
            return
        if self.require_cuda:
            dev = t.get_device()                         # -1 for a host tensor
            if dev < 0:
                raise ValueError(f"{self.fn}: {name} must be a CUDA tensor (got {t.device})")
            if self.device is None:
                self.device = dev
            elif dev != self.device:
                raise ValueError(f"{self.fn}: {name} is on cuda:{dev}, other tensors on "
                                 f"cuda:{self.device}")
        if not t.is_contiguous():
            raise ValueError(f"{self.fn}: {name} must be contiguous")
        if dtypes is not None:
            dtypes = dtypes if isinstance(dtypes, tuple) else (dtypes,)
            if t.dtype not in dtypes:
                raise ValueError(f"{self.fn}: {name} has dtype {t.dtype}, expected "
                                 + " or ".join(str(d) for d in dtypes))
        if shape is not None:
            got = t.shape
            if len(got) != len(shape) or tuple(got[1:]) != tuple(shape[1:]) or got[0] < shape[0]:
                raise ValueError(f"{self.fn}: {name} has shape {tuple(got)}, expected "
                                 f"{tuple(shape)} (more rows are allowed)")


_SIGNATURES = {}


def _named(builder, args, kw):
    """The arguments of a call of `builder` (fwd_args, bwd_args, conv_args) by name."""
    sig = _SIGNATURES.get(builder)
    if sig is None:
        sig = _SIGNATURES[builder] = inspect.signature(builder)
    b = sig.bind(*args, **kw)
    b.apply_defaults()
    return b.arguments


def validate_fwd(fn, a, kda, require_cuda=True):
    """Layouts of a forward call's tensors (a: fwd_args' arguments by name)."""
    import torch
    L = _Layout(fn, require_cuda)
    q, cu = a["q"], a["cu_seqlens"]
    T, H, K = q.shape
    V = a["v"].shape[-1]
    N = cu.shape[0] - 1
    ntm = nt_max(T, N, a["bt"])
    dt, f32, i32 = q.dtype, torch.float32, torch.int32
    for name, shp in (("q", (T, H, K)), ("k", (T, H, K)), ("v", (T, H, V)), ("beta", (T, H)),
                      ("o", (T, H, V))):
        L(name, a[name], dt, shp)
    L("g", a["g"], f32, (T, H, K) if kda else (T, H))
    L("cu_seqlens", cu, i32, (N + 1,))
    for name in ("h0", "ht"):
        L(name, a[name], f32, (N, H, K, V))
    L("h_save", a["h_save"], f32, (ntm, H, K, V))
    L("chunk_indices", a["chunk_indices"], i32, (ntm, 2))
    L("chunk_offsets", a["chunk_offsets"], i32, (N + 1,))
    L("seq_order", a["seq_order"], i32, (N,))
    L("dev_status", a["dev_status"], i32, (1,))
    L("workspace", a["workspace"])


def validate_bwd(fn, a, kda, require_cuda=True):
    """Layouts of a backward call's tensors (a: bwd_args' arguments by name)."""
    import torch
    L = _Layout(fn, require_cuda)
    q, cu = a["q"], a["cu_seqlens"]
    T, H, K = q.shape
    V = a["v"].shape[-1]
    N = cu.shape[0] - 1
    ntm = nt_max(T, N, a["bt"])
    dt, f32, i32 = q.dtype, torch.float32, torch.int32
    gshape = (T, H, K) if kda else (T, H)
    for name, shp in (("q", (T, H, K)), ("k", (T, H, K)), ("v", (T, H, V)), ("beta", (T, H)),
                      ("d_o", (T, H, V))):
        L(name, a[name], dt, shp)
    for name, shp in (("g", gshape), ("dg", gshape), ("dq", (T, H, K)), ("dk", (T, H, K)),
                      ("dv", (T, H, V)), ("dbeta", (T, H)), ("h0", (N, H, K, V)),
                      ("dht", (N, H, K, V)), ("dh0", (N, H, K, V)), ("h_save", (ntm, H, K, V))):
        L(name, a[name], f32, shp)
    L("cu_seqlens", cu, i32, (N + 1,))
    L("chunk_indices", a["chunk_indices"], i32, (ntm, 2))
    L("chunk_offsets", a["chunk_offsets"], i32, (N + 1,))
    L("dev_status", a["dev_status"], i32, (1,))
    L("workspace", a["workspace"])
    L("fwd_workspace", a["fwd_workspace"])


def validate_conv(fn, a, require_cuda=True):
    """Layouts of a causal_conv1d call's tensors (a: conv_args' arguments by name)."""
    import torch
    L = _Layout(fn, require_cuda)
    x, w, cu = a["x"], a["weight"], a["cu_seqlens"]
    T, D = x.shape
    W = w.shape[1]
    N = cu.shape[0] - 1
    dt, f32, i32 = x.dtype, torch.float32, torch.int32
    for name, shp in (("x", (T, D)), ("weight", (D, W)), ("bias", (D,)), ("residual", (T, D)),
                      ("h0", (N, D, W - 1)), ("y", (T, D)), ("ht", (N, D, W - 1)),
                      ("dy", (T, D))):
        L(name, a[name], dt, shp)
    for name, shp in (("dht", (N, D, W - 1)), ("dx", (T, D)), ("dweight", (D, W)),
                      ("dbias", (D,)), ("dh0", (N, D, W - 1))):
        L(name, a[name], f32, shp)
    L("cu_seqlens", cu, i32, (N + 1,))
    L("chunk_indices", a["chunk_indices"], i32, (nt_max(T, N, a["bt"]), 2))
    L("dev_status", a["dev_status"], i32, (1,))
    L("workspace", a["workspace"])


def nt_max(t_max: int, n_max: int, bt: int = CHUNK) -> int:
    return int(lib().gcl_nt_max(t_max, n_max, bt))


def selftest_wait_timeout(dev_status, stream=None):
    """One CTA waits on an mbarrier nothing arrives at; after the time limit dev_status holds
    GCL_DEV_WAIT_TIMEOUT (the bounded-wait path of every tensor-core kernel)."""
    import torch
    _Layout("gcl_selftest_wait_timeout")("dev_status", dev_status, torch.int32, (1,))
    _check("gcl_selftest_wait_timeout", lib().gcl_selftest_wait_timeout(_p(dev_status), _stream(stream)))


def fwd_chain_segments(t_max: int, n_max: int, H: int, bt: int = CHUNK) -> int:
    """Segments per sequence of the fastest tensor-core forward plan (0: the plain chain)."""
    return int(lib().gcl_fwd_chain_segments(t_max, n_max, H, bt))


def chunk_meta_build(cu_seqlens, t_max, chunk_indices, chunk_offsets, dev_status,
                     seq_order=None, bt: int = CHUNK, stream=None, cu_seqlens32=None):
    """Chunk metadata from cu_seqlens (int32, or int64 with an int32 copy written to
    cu_seqlens32 for the compute calls)."""
    import torch
    n_max = cu_seqlens.shape[0] - 1
    L = _Layout("chunk_meta_build")
    L("cu_seqlens", cu_seqlens, (torch.int32, torch.int64), (n_max + 1,))
    L("chunk_indices", chunk_indices, torch.int32, (chunk_indices.shape[0], 2))
    L("chunk_offsets", chunk_offsets, torch.int32, (n_max + 1,))
    L("seq_order", seq_order, torch.int32, (n_max,))
    L("dev_status", dev_status, torch.int32, (1,))
    L("cu_seqlens32", cu_seqlens32, torch.int32, (n_max + 1,))
    if cu_seqlens.element_size() == 8:
        if cu_seqlens32 is None:
            raise ValueError("an int64 cu_seqlens needs cu_seqlens32 (int32 [n_max + 1]) for its copy")
        _check("chunk_meta_build_i64",
               lib().chunk_meta_build_i64(_p(cu_seqlens), n_max, t_max, bt, chunk_indices.shape[0],
                                          _p(cu_seqlens32), _p(chunk_indices), _p(chunk_offsets),
                                          _p(seq_order), _p(dev_status), _stream(stream)))
        return
    _check("chunk_meta_build",
           lib().chunk_meta_build(_p(cu_seqlens), n_max, t_max, bt, chunk_indices.shape[0],
                                  _p(chunk_indices), _p(chunk_offsets), _p(seq_order),
                                  _p(dev_status), _stream(stream)))


def _nbytes(t):
    return 0 if t is None else t.numel() * t.element_size()


def fwd_args(q, k, v, g, beta, cu_seqlens, o, h0=None, ht=None, h_save=None,
             chunk_indices=None, chunk_offsets=None, seq_order=None, dev_status=None,
             workspace=None, scale=None, bt=CHUNK):
    T, H, K = q.shape
    V = v.shape[-1]
    a = FwdArgs(q=_p(q), k=_p(k), v=_p(v), g=_p(g), beta=_p(beta), h0=_p(h0),
                cu_seqlens=_p(cu_seqlens), chunk_indices=_p(chunk_indices),
                chunk_offsets=_p(chunk_offsets), seq_order=_p(seq_order), o=_p(o), ht=_p(ht),
                h_save=_p(h_save), dev_status=_p(dev_status), workspace=_p(workspace),
                workspace_bytes=_nbytes(workspace), t_max=T, n_max=cu_seqlens.shape[0] - 1,
                H=H, K=K, V=V, bt=bt, scale=float(K ** -0.5 if scale is None else scale),
                dtype=_dtype_of(q))
    return a


def fwd_workspace_bytes(*args, **kw) -> int:
    """Workspace of the fastest launch plan for these sizes."""
    a = fwd_args(*args, **kw)
    return int(lib().gcl_fwd_workspace_bytes(ctypes.byref(a)))


def fwd_workspace_min_bytes(*args, **kw) -> int:
    """Least workspace the forward accepts (it then runs the W-form plan; 0 where the fused
    plan runs)."""
    a = fwd_args(*args, **kw)
    return int(lib().gcl_fwd_workspace_min_bytes(ctypes.byref(a)))


def kda_fwd_workspace_bytes(*args, **kw) -> int:
    """Workspace kda_chunk_fwd needs (its one tensor-core plan; 0 on the CUDA-core path)."""
    a = fwd_args(*args, **kw)
    return int(lib().gcl_kda_fwd_workspace_bytes(ctypes.byref(a)))


PLANS = {0: "cuda_cores", 1: "fused", 2: "w_form", 3: "transition", 4: "segmented",
         5: "cuda_cores_split"}


def fwd_plan(*args, kda=False, **kw) -> str:
    """Name of the launch plan the forward runs with these arguments (workspace included):
    cuda_cores, fused, w_form, transition or segmented (include/gcl.h, gcl_fwd_plan)."""
    a = fwd_args(*args, **kw)
    code = int((lib().gcl_kda_fwd_plan if kda else lib().gcl_fwd_plan)(ctypes.byref(a)))
    if code < 0:
        raise GclError("gcl_fwd_plan", code, lib().gcl_last_error().decode())
    return PLANS[code]


def gdn_chunk_fwd(*args, stream=None, **kw):
    validate_fwd("gdn_chunk_fwd", _named(fwd_args, args, kw), kda=False)
    a = fwd_args(*args, **kw)
    _check("gdn_chunk_fwd", lib().gdn_chunk_fwd(ctypes.byref(a), _stream(stream)))


def gdn_chunk_fwd_noalloc(*args, stream=None, **kw):
    """gdn_chunk_fwd without a workspace argument: the library's static scratch is used
    (for callers that cannot allocate device memory; see include/gcl.h)."""
    kw.pop("workspace", None)
    validate_fwd("gdn_chunk_fwd_noalloc", _named(fwd_args, args, kw), kda=False)
    a = fwd_args(*args, **kw)
    _check("gdn_chunk_fwd_noalloc", lib().gdn_chunk_fwd_noalloc(ctypes.byref(a), _stream(stream)))


def noalloc_scratch_bytes() -> int:
    return int(lib().gcl_noalloc_scratch_bytes())


def kda_chunk_fwd(*args, stream=None, **kw):
    validate_fwd("kda_chunk_fwd", _named(fwd_args, args, kw), kda=True)
    a = fwd_args(*args, **kw)
    _check("kda_chunk_fwd", lib().kda_chunk_fwd(ctypes.byref(a), _stream(stream)))


def bwd_args(q, k, v, g, beta, d_o, cu_seqlens, chunk_indices, chunk_offsets, dq, dk, dv, dg,
             dbeta, h0=None, dht=None, dh0=None, h_save=None, workspace=None,
             dev_status=None, scale=None, bt=CHUNK, fwd_workspace=None):
    T, H, K = q.shape
    V = v.shape[-1]
    return BwdArgs(q=_p(q), k=_p(k), v=_p(v), g=_p(g), beta=_p(beta), h0=_p(h0), d_o=_p(d_o),
                   dht=_p(dht), cu_seqlens=_p(cu_seqlens), chunk_indices=_p(chunk_indices),
                   chunk_offsets=_p(chunk_offsets), h_save=_p(h_save), dq=_p(dq), dk=_p(dk),
                   dv=_p(dv), dg=_p(dg), dbeta=_p(dbeta), dh0=_p(dh0),
                   workspace=_p(workspace), workspace_bytes=_nbytes(workspace),
                   dev_status=_p(dev_status), t_max=T, n_max=cu_seqlens.shape[0] - 1, H=H, K=K,
                   V=V, bt=bt, scale=float(K ** -0.5 if scale is None else scale),
                   dtype=_dtype_of(q), fwd_workspace=_p(fwd_workspace),
                   fwd_workspace_bytes=_nbytes(fwd_workspace))


def bwd_workspace_bytes(*args, **kw) -> int:
    a = bwd_args(*args, **kw)
    return int(lib().gcl_bwd_workspace_bytes(ctypes.byref(a)))


def gdn_chunk_bwd(*args, stream=None, **kw):
    validate_bwd("gdn_chunk_bwd", _named(bwd_args, args, kw), kda=False)
    a = bwd_args(*args, **kw)
    _check("gdn_chunk_bwd", lib().gdn_chunk_bwd(ctypes.byref(a), _stream(stream)))


def kda_bwd_workspace_bytes(*args, **kw) -> int:
    a = bwd_args(*args, **kw)
    return int(lib().gcl_kda_bwd_workspace_bytes(ctypes.byref(a)))


def kda_chunk_bwd(*args, stream=None, **kw):
    """The KDA backward; dg has the shape of g, [T, H, K]."""
    validate_bwd("kda_chunk_bwd", _named(bwd_args, args, kw), kda=True)
    a = bwd_args(*args, **kw)
    _check("kda_chunk_bwd", lib().kda_chunk_bwd(ctypes.byref(a), _stream(stream)))


# ---------------------------------------------------------------- causal_conv1d
ACTIVATIONS = {None: 0, "silu": 1}


def conv_args(x, weight, cu_seqlens, chunk_indices, bias=None, residual=None, h0=None, y=None,
              ht=None, dy=None, dht=None, dx=None, dweight=None, dbias=None, dh0=None,
              workspace=None, dev_status=None, activation=None, bt=CHUNK):
    """gcl_conv_args for x [T, D], weight [D, W]; see include/gcl.h (causal_conv1d)."""
    T, D = x.shape
    return ConvArgs(x=_p(x), weight=_p(weight), bias=_p(bias), residual=_p(residual), h0=_p(h0),
                    y=_p(y), ht=_p(ht), dy=_p(dy), dht=_p(dht), dx=_p(dx), dweight=_p(dweight),
                    dbias=_p(dbias), dh0=_p(dh0), cu_seqlens=_p(cu_seqlens),
                    chunk_indices=_p(chunk_indices), dev_status=_p(dev_status),
                    workspace=_p(workspace), workspace_bytes=_nbytes(workspace), t_max=T,
                    n_max=cu_seqlens.shape[0] - 1, D=D, W=weight.shape[1], bt=bt,
                    activation=ACTIVATIONS[activation], dtype=_dtype_of(x))


def causal_conv1d_fwd(*args, stream=None, **kw):
    validate_conv("causal_conv1d_fwd", _named(conv_args, args, kw))
    a = conv_args(*args, **kw)
    _check("causal_conv1d_fwd", lib().causal_conv1d_fwd(ctypes.byref(a), _stream(stream)))


def causal_conv1d_bwd_workspace_bytes(*args, **kw) -> int:
    a = conv_args(*args, **kw)
    return int(lib().gcl_causal_conv1d_bwd_workspace_bytes(ctypes.byref(a)))


def causal_conv1d_bwd(*args, stream=None, **kw):
    validate_conv("causal_conv1d_bwd", _named(conv_args, args, kw))
    a = conv_args(*args, **kw)
    _check("causal_conv1d_bwd", lib().causal_conv1d_bwd(ctypes.byref(a), _stream(stream)))
