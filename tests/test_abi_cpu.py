"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every function include/gcl.h declares, and rejects bad arguments before it
touches the device."""
import ctypes
import os
import re

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from chunked_gated_linear_gb300 import _build
    _build.build()
    import chunked_gated_linear_gb300 as gcl
    return gcl.load_library()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "gcl.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*([a-z_0-9]+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_four_entry_points():
    names = declared_functions()
    for fn in ("chunk_meta_build", "gdn_chunk_fwd", "kda_chunk_fwd", "gdn_chunk_bwd"):
        assert fn in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_nt_max_matches_oracle(lib):
    for t in (1, 63, 64, 65, 4096, 65536):
        for n in (1, 2, 64):
            for bt in (16, 32, 64):
                assert lib.gcl_nt_max(t, n, bt) == oracle.nt_max(t, n, bt)
    assert lib.gcl_nt_max(0, 1, 64) == -1


def test_host_errors_before_any_launch(lib):
    import chunked_gated_linear_gb300 as gcl
    INVALID, UNSUPPORTED, CAPACITY = 1, 2, 3
    # NULL args struct
    assert lib.gdn_chunk_fwd(None, None) == INVALID
    assert lib.kda_chunk_fwd(None, None) == INVALID
    assert lib.gdn_chunk_bwd(None, None) == INVALID
    # missing required pointers
    a = gcl.FwdArgs(t_max=128, n_max=1, H=1, K=128, V=128, bt=64, scale=1.0, dtype=1)
    assert lib.gdn_chunk_fwd(ctypes.byref(a), None) == INVALID
    assert b"required" in lib.gcl_last_error()
    fake = 1 << 20   # a 16-byte aligned non-null value; never dereferenced on these paths
    full = dict(q=fake, k=fake, v=fake, g=fake, beta=fake, cu_seqlens=fake, o=fake, t_max=128,
                n_max=1, H=1, K=128, V=128, bt=64, scale=1.0, dtype=1)
    for bad, code in ((dict(bt=16), UNSUPPORTED), (dict(K=96), UNSUPPORTED),
                      (dict(V=256), UNSUPPORTED), (dict(dtype=7), UNSUPPORTED),
                      (dict(t_max=0), INVALID), (dict(n_max=0), INVALID),
                      (dict(q=fake + 4), INVALID), (dict(h_save=fake), INVALID)):
        args = gcl.FwdArgs(**{**full, **bad})
        assert lib.gdn_chunk_fwd(ctypes.byref(args), None) == code, bad
        assert lib.kda_chunk_fwd(ctypes.byref(args), None) == code, bad
        assert lib.gcl_last_error() != b""
    # chunk_meta_build: nt_max must match, pointers required
    assert lib.chunk_meta_build(fake, 4, 256, 64, 7, fake, fake, None, None, None) == INVALID
    assert lib.chunk_meta_build(fake, 4, 256, 64, 8, fake, fake, None, fake, None) == INVALID
    assert b"nt_max" in lib.gcl_last_error()
    # the int64 variant also needs the int32 copy
    assert lib.chunk_meta_build_i64(fake, 4, 256, 64, 8, None, fake, fake, None, fake, None) == INVALID
    assert b"cu_seqlens32" in lib.gcl_last_error()
    assert lib.chunk_meta_build_i64(fake, 4, 256, 64, 9, fake, fake, fake, None, fake, None) == INVALID
    # backward: workspace capacity is checked on the host
    b = gcl.BwdArgs(q=fake, k=fake, v=fake, g=fake, beta=fake, d_o=fake, cu_seqlens=fake,
                    chunk_indices=fake, chunk_offsets=fake, dq=fake, dk=fake, dv=fake, dg=fake,
                    dbeta=fake, workspace=fake, workspace_bytes=16, t_max=128, n_max=1, H=1,
                    K=128, V=128, bt=64, scale=1.0, dtype=1)
    need = lib.gcl_bwd_workspace_bytes(ctypes.byref(b))
    assert need >= 2 * 4 * 2 * 128 * 128            # dh and recomputed h for NT_max = 2 chunks
    assert lib.gdn_chunk_bwd(ctypes.byref(b), None) == CAPACITY
    b.h_save = fake
    assert lib.gcl_bwd_workspace_bytes(ctypes.byref(b)) < need


def test_status_strings(lib):
    assert lib.gcl_status_string(0) == b"GCL_OK"
    assert lib.gcl_status_string(3) == b"GCL_ERR_CAPACITY"


def test_plan_rules_from_sizes_alone(lib):
    """Host-side plan rules (no device access): a training forward (h_save) asks for the
    transition records even with many units; handing its workspace to the backward shrinks
    the backward's; one long sequence of one head is cut into segments, many units are not."""
    import chunked_gated_linear_gb300 as gcl
    fake = 1 << 20
    base = dict(q=fake, k=fake, v=fake, g=fake, beta=fake, cu_seqlens=fake, o=fake,
                t_max=8192 * 4, n_max=4, H=16, K=128, V=128, bt=64, scale=1.0, dtype=1)
    infer = gcl.FwdArgs(**base)
    train = gcl.FwdArgs(**base, h_save=fake, chunk_offsets=fake)
    w_inf = lib.gcl_fwd_workspace_bytes(ctypes.byref(infer))
    w_tr = lib.gcl_fwd_workspace_bytes(ctypes.byref(train))
    assert w_tr > w_inf                                  # transition records (96.5 KiB per chunk-head)
    assert w_inf == lib.gcl_fwd_workspace_min_bytes(ctypes.byref(infer))   # W form
    b = dict(q=fake, k=fake, v=fake, g=fake, beta=fake, d_o=fake, cu_seqlens=fake,
             chunk_indices=fake, chunk_offsets=fake, dq=fake, dk=fake, dv=fake, dg=fake,
             dbeta=fake, h_save=fake, t_max=8192 * 4, n_max=4, H=16, K=128, V=128, bt=64,
             scale=1.0, dtype=1)
    own = lib.gcl_bwd_workspace_bytes(ctypes.byref(gcl.BwdArgs(**b)))
    reuse = lib.gcl_bwd_workspace_bytes(ctypes.byref(gcl.BwdArgs(**b, fwd_workspace=fake,
                                                                 fwd_workspace_bytes=w_tr)))
    small = lib.gcl_bwd_workspace_bytes(ctypes.byref(gcl.BwdArgs(**b, fwd_workspace=fake,
                                                                 fwd_workspace_bytes=w_inf)))
    assert reuse < own and small == own                  # a W-form forward has no records to give
    assert lib.gcl_fwd_chain_segments(65536, 1, 1, 64) >= 3
    assert lib.gcl_fwd_chain_segments(4096, 1, 16, 64) == 0
    assert lib.gcl_fwd_chain_segments(65536, 1, 1, 32) == 0


def test_cuda_core_plans_from_sizes_alone(lib):
    """The CUDA-core sizes: no workspace at the minimum (one kernel); the fastest workspace holds
    the split plan's records, (3 BT (K + 4) + BT (BT + 4) + K + BT V) fp32 per chunk row and
    head (rows of W, Q', K', L padded by 4 floats), for K = V only; the split plan runs only
    with that workspace and the chunk metadata."""
    import chunked_gated_linear_gb300 as gcl
    fake = 1 << 20
    nt = lambda t, n, bt: lib.gcl_nt_max(t, n, bt)
    for K, bt, dtype in ((64, 64, 0), (128, 64, 0), (128, 32, 1), (64, 32, 2)):
        base = dict(q=fake, k=fake, v=fake, g=fake, beta=fake, cu_seqlens=fake, o=fake,
                    t_max=4096, n_max=3, H=2, K=K, V=K, bt=bt, scale=1.0, dtype=dtype,
                    chunk_indices=fake, chunk_offsets=fake)
        a = gcl.FwdArgs(**base)
        rec = 4 * nt(4096, 3, bt) * 2 * (3 * bt * (K + 4) + bt * (bt + 4) + K + bt * K)
        fastest = lib.gcl_fwd_workspace_bytes(ctypes.byref(a))
        assert lib.gcl_fwd_workspace_min_bytes(ctypes.byref(a)) == 0
        assert rec <= fastest <= rec + 1024, (K, bt, dtype)           # + alignment slack
        assert lib.gcl_fwd_plan(ctypes.byref(a)) == 0                  # no workspace: one kernel
        w = gcl.FwdArgs(**base, workspace=fake, workspace_bytes=fastest)
        assert lib.gcl_fwd_plan(ctypes.byref(w)) == 5                  # GCL_PLAN_CUDA_CORES_SPLIT
        assert lib.gcl_kda_fwd_plan(ctypes.byref(w)) == 5
        short = gcl.FwdArgs(**base, workspace=fake, workspace_bytes=rec - 16)
        assert lib.gcl_fwd_plan(ctypes.byref(short)) == 0
        nometa = gcl.FwdArgs(**{**base, "chunk_indices": None}, workspace=fake, workspace_bytes=fastest)
        assert lib.gcl_fwd_plan(ctypes.byref(nometa)) == 0
    mixed = gcl.FwdArgs(q=fake, k=fake, v=fake, g=fake, beta=fake, cu_seqlens=fake, o=fake,
                        t_max=4096, n_max=3, H=2, K=64, V=128, bt=64, scale=1.0, dtype=0)
    assert lib.gcl_fwd_workspace_bytes(ctypes.byref(mixed)) == 0       # K != V: one kernel


def test_host_errors_other_entry_points(lib):
    """The KDA backward, the short convolution, the no-allocation forward and the wait
    self-test reject bad arguments on the host, before anything is enqueued."""
    import chunked_gated_linear_gb300 as gcl
    INVALID, UNSUPPORTED, CAPACITY = 1, 2, 3
    fake = 1 << 20
    # kda_chunk_bwd: same checks as the GDN backward
    assert lib.kda_chunk_bwd(None, None) == INVALID
    b = dict(q=fake, k=fake, v=fake, g=fake, beta=fake, d_o=fake, cu_seqlens=fake,
             chunk_indices=fake, chunk_offsets=fake, dq=fake, dk=fake, dv=fake, dg=fake,
             dbeta=fake, workspace=fake, workspace_bytes=16, t_max=128, n_max=1, H=1, K=128,
             V=128, bt=64, scale=1.0, dtype=1)
    assert lib.kda_chunk_bwd(ctypes.byref(gcl.BwdArgs(**b)), None) == CAPACITY
    assert b"workspace" in lib.gcl_last_error()
    assert lib.kda_chunk_bwd(ctypes.byref(gcl.BwdArgs(**{**b, "d_o": None})), None) == INVALID
    assert lib.kda_chunk_bwd(ctypes.byref(gcl.BwdArgs(**{**b, "K": 96})), None) == UNSUPPORTED
    need = lib.gcl_kda_bwd_workspace_bytes(ctypes.byref(gcl.BwdArgs(**b)))
    assert need > 0
    ok = {**b, "workspace_bytes": need}
    assert lib.kda_chunk_bwd(ctypes.byref(gcl.BwdArgs(**{**ok, "dq": fake + 4})), None) == INVALID
    assert b"aligned" in lib.gcl_last_error()
    # causal_conv1d: forward and backward argument checks
    assert lib.causal_conv1d_fwd(None, None) == INVALID
    assert lib.causal_conv1d_bwd(None, None) == INVALID
    c = dict(x=fake, weight=fake, y=fake, cu_seqlens=fake, chunk_indices=fake, t_max=256,
             n_max=2, D=64, W=4, bt=64, activation=0, dtype=1)
    for bad, code in ((dict(W=1), UNSUPPORTED), (dict(W=5), UNSUPPORTED), (dict(D=12), UNSUPPORTED),
                      (dict(dtype=7), UNSUPPORTED), (dict(bt=32), UNSUPPORTED),
                      (dict(activation=9), UNSUPPORTED), (dict(t_max=0), INVALID),
                      (dict(y=None), INVALID), (dict(x=fake + 8), INVALID)):
        assert lib.causal_conv1d_fwd(ctypes.byref(gcl.ConvArgs(**{**c, **bad})), None) == code, bad
        assert lib.gcl_last_error() != b""
    cb = {**c, "y": None, "dy": fake, "dx": fake, "dweight": fake}
    assert lib.causal_conv1d_bwd(ctypes.byref(gcl.ConvArgs(**{**cb, "dx": None})), None) == INVALID
    assert lib.causal_conv1d_bwd(ctypes.byref(gcl.ConvArgs(**cb)), None) == CAPACITY
    assert lib.gcl_causal_conv1d_bwd_workspace_bytes(ctypes.byref(gcl.ConvArgs(**cb))) > 0
    assert lib.gcl_causal_conv1d_bwd_workspace_bytes(ctypes.byref(gcl.ConvArgs(**{**cb, "W": 7}))) == 0
    # the no-allocation forward: sizes whose scratch exceeds the static array are rejected
    assert lib.gdn_chunk_fwd_noalloc(None, None) == INVALID
    # (few sequence-head units: the plans with per-chunk scratch; many units run the fused
    # plan, which needs none)
    big = gcl.FwdArgs(q=fake, k=fake, v=fake, g=fake, beta=fake, cu_seqlens=fake, o=fake,
                      t_max=1 << 22, n_max=2, H=16, K=128, V=128, bt=64, scale=1.0, dtype=1)
    assert lib.gcl_fwd_workspace_min_bytes(ctypes.byref(big)) > lib.gcl_noalloc_scratch_bytes()
    assert lib.gcl_fwd_plan(ctypes.byref(big)) == 2                 # GCL_PLAN_W_FORM
    many = gcl.FwdArgs(q=fake, k=fake, v=fake, g=fake, beta=fake, cu_seqlens=fake, o=fake,
                       t_max=1 << 16, n_max=64, H=16, K=128, V=128, bt=64, scale=1.0, dtype=1)
    assert lib.gcl_fwd_plan(ctypes.byref(many)) == 1                # GCL_PLAN_FUSED
    assert lib.gcl_fwd_workspace_bytes(ctypes.byref(many)) == 0
    assert lib.gcl_fwd_workspace_min_bytes(ctypes.byref(many)) == 0
    assert lib.gcl_kda_fwd_plan(ctypes.byref(many)) == 3            # KDA: transition form
    assert lib.gcl_fwd_plan(ctypes.byref(gcl.FwdArgs(**{**{f: getattr(many, f) for f, _ in gcl.FwdArgs._fields_}, "dtype": 0}))) == 0
    assert lib.gcl_fwd_plan(None) == -1
    assert lib.gdn_chunk_fwd_noalloc(ctypes.byref(big), None) == CAPACITY
    assert b"scratch" in lib.gcl_last_error()
    # the wait self-test needs a status word
    assert lib.gcl_selftest_wait_timeout(None, None) == INVALID


def test_plain_c_caller(lib, tmp_path):
    """A C99 program that includes include/gcl.h and links libgcl.so builds with gcc and its
    host-side ABI checks pass (the header is C, not C++; no GPU is touched)."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not available")
    libdir = os.path.join(ROOT, "chunked_gated_linear_gb300")
    exe = str(tmp_path / "abi_host_check")
    subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                    "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "c", "abi_host_check.c"),
                    "-L", libdir, "-lgcl", "-Wl,-rpath," + libdir, "-o", exe], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert "c abi ok" in r.stdout
