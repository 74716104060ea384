"""The binding's layout checks (no GPU): valid calls of every shape family pass; a tensor of
the wrong dtype, too few rows or wrong trailing dimensions is rejected before the library
sees its pointer; host tensors are rejected by every launching entry point."""
import pytest

torch = pytest.importorskip("torch")
import chunked_gated_linear_gb300 as gcl  # noqa: E402

F32, BF16, F16, I32 = torch.float32, torch.bfloat16, torch.float16, torch.int32


def fwd_call(kda=False, dt=BF16, T=300, N=3, H=2, K=128, V=64, bt=64, h_save=True):
    ntm = gcl.nt_max(T, N, bt)
    e = lambda *s, d=F32: torch.zeros(s, dtype=d)
    return dict(q=e(T, H, K, d=dt), k=e(T, H, K, d=dt), v=e(T, H, V, d=dt),
                g=e(T, H, K) if kda else e(T, H), beta=e(T, H, d=dt),
                cu_seqlens=e(N + 1, d=I32), o=e(T, H, V, d=dt), h0=e(N, H, K, V),
                ht=e(N, H, K, V), h_save=e(ntm, H, K, V) if h_save else None,
                chunk_indices=e(ntm, 2, d=I32), chunk_offsets=e(N + 1, d=I32),
                seq_order=e(N, d=I32), dev_status=e(1, d=I32), workspace=e(64, d=torch.uint8),
                scale=None, bt=bt)


def bwd_call(kda=False, dt=BF16, T=300, N=3, H=2, K=64, V=64, bt=64):
    ntm = gcl.nt_max(T, N, bt)
    e = lambda *s, d=F32: torch.zeros(s, dtype=d)
    gs = (T, H, K) if kda else (T, H)
    return dict(q=e(T, H, K, d=dt), k=e(T, H, K, d=dt), v=e(T, H, V, d=dt), g=e(*gs),
                beta=e(T, H, d=dt), d_o=e(T, H, V, d=dt), cu_seqlens=e(N + 1, d=I32),
                chunk_indices=e(ntm, 2, d=I32), chunk_offsets=e(N + 1, d=I32),
                dq=e(T, H, K), dk=e(T, H, K), dv=e(T, H, V), dg=e(*gs), dbeta=e(T, H),
                h0=e(N, H, K, V), dht=e(N, H, K, V), dh0=e(N, H, K, V), h_save=e(ntm, H, K, V),
                workspace=e(64, d=torch.uint8), dev_status=e(1, d=I32), scale=None, bt=bt,
                fwd_workspace=None)


def conv_call(dt=BF16, T=200, N=2, D=64, W=4):
    ntm = gcl.nt_max(T, N, 64)
    e = lambda *s, d=F32: torch.zeros(s, dtype=d)
    return dict(x=e(T, D, d=dt), weight=e(D, W, d=dt), cu_seqlens=e(N + 1, d=I32),
                chunk_indices=e(ntm, 2, d=I32), bias=e(D, d=dt), residual=e(T, D, d=dt),
                h0=e(N, D, W - 1, d=dt), y=e(T, D, d=dt), ht=e(N, D, W - 1, d=dt),
                dy=e(T, D, d=dt), dht=e(N, D, W - 1), dx=e(T, D), dweight=e(D, W), dbias=e(D),
                dh0=e(N, D, W - 1), workspace=e(64, d=torch.uint8), dev_status=e(1, d=I32),
                activation=None, bt=64)


@pytest.mark.parametrize("kda", [False, True], ids=["gdn", "kda"])
@pytest.mark.parametrize("dt", [F32, BF16, F16], ids=["f32", "bf16", "f16"])
@pytest.mark.parametrize("bt", [32, 64])
def test_valid_calls_pass(kda, dt, bt):
    gcl.validate_fwd("fwd", fwd_call(kda, dt, bt=bt), kda, require_cuda=False)
    gcl.validate_fwd("fwd", fwd_call(kda, dt, bt=bt, h_save=False), kda, require_cuda=False)
    gcl.validate_bwd("bwd", bwd_call(kda, dt, bt=bt), kda, require_cuda=False)
    if dt != F16:
        gcl.validate_conv("conv", conv_call(dt), require_cuda=False)


def test_optional_tensors_may_be_absent_and_buffers_may_be_larger():
    a = fwd_call()
    for name in ("o", "h0", "ht", "h_save", "chunk_indices", "seq_order", "dev_status", "workspace"):
        a[name] = None
    a["q"] = torch.zeros(300, 2, 128, dtype=BF16)
    gcl.validate_fwd("fwd", a, False, require_cuda=False)
    b = fwd_call()
    b["h_save"] = torch.zeros(b["h_save"].shape[0] + 5, 2, 128, 64)   # extra rows are fine
    b["v"] = torch.zeros(400, 2, 64, dtype=BF16)
    gcl.validate_fwd("fwd", b, False, require_cuda=False)


@pytest.mark.parametrize("name,bad", [
    ("k", torch.zeros(300, 2, 128, dtype=F32)),            # dtype differs from q
    ("v", torch.zeros(299, 2, 64, dtype=BF16)),            # too few token rows
    ("beta", torch.zeros(300, 3, dtype=BF16)),             # wrong head count
    ("g", torch.zeros(300, 2, dtype=BF16)),                # the gate is fp32
    ("cu_seqlens", torch.zeros(4, dtype=torch.int64)),     # compute calls take int32
    ("h0", torch.zeros(3, 2, 128, 32)),                    # wrong V
    ("h_save", torch.zeros(2, 2, 128, 64)),                # fewer rows than nt_max
    ("chunk_indices", torch.zeros(20, 3, dtype=I32)),      # [nt_max, 2]
    ("seq_order", torch.zeros(2, dtype=I32)),              # [n_max]
    ("o", torch.zeros(300, 2, 64, dtype=F32)),             # o has the input dtype
    ("o", torch.zeros(64, 2, 300, dtype=BF16).permute(2, 1, 0)),   # not contiguous
])
def test_forward_rejects(name, bad):
    a = fwd_call()
    a[name] = bad
    with pytest.raises(ValueError, match=name):
        gcl.validate_fwd("gdn_chunk_fwd", a, False, require_cuda=False)


def test_kda_gate_is_per_channel():
    a = fwd_call(kda=True)
    a["g"] = torch.zeros(300, 2)
    with pytest.raises(ValueError, match="g has shape"):
        gcl.validate_fwd("kda_chunk_fwd", a, True, require_cuda=False)
    b = bwd_call(kda=True)
    b["dg"] = torch.zeros(300, 2)
    with pytest.raises(ValueError, match="dg has shape"):
        gcl.validate_bwd("kda_chunk_bwd", b, True, require_cuda=False)


@pytest.mark.parametrize("name,bad", [
    ("dq", torch.zeros(300, 2, 64, dtype=BF16)),           # gradients are fp32
    ("d_o", torch.zeros(300, 2, 64, dtype=F32)),           # d_o has the input dtype
    ("dbeta", torch.zeros(100, 2)),
    ("dh0", torch.zeros(2, 2, 64, 64)),
])
def test_backward_rejects(name, bad):
    b = bwd_call()
    b[name] = bad
    with pytest.raises(ValueError, match=name):
        gcl.validate_bwd("gdn_chunk_bwd", b, False, require_cuda=False)


@pytest.mark.parametrize("name,bad", [
    ("weight", torch.zeros(64, 4)),                        # weight has the input dtype
    ("h0", torch.zeros(2, 64, 4, dtype=BF16)),             # [n_max, D, W - 1]
    ("dweight", torch.zeros(64, 4, dtype=BF16)),           # gradients are fp32
    ("y", torch.zeros(100, 64, dtype=BF16)),
    ("chunk_indices", torch.zeros(3, 2, dtype=I32)),
])
def test_conv_rejects(name, bad):
    c = conv_call()
    c[name] = bad
    with pytest.raises(ValueError, match=name):
        gcl.validate_conv("causal_conv1d_fwd", c, require_cuda=False)


def test_launchers_reject_host_tensors_before_the_library_call():
    a = fwd_call()
    args = [a.pop(n) for n in ("q", "k", "v", "g", "beta", "cu_seqlens", "o")]
    for fn in (gcl.gdn_chunk_fwd, gcl.kda_chunk_fwd, gcl.gdn_chunk_fwd_noalloc):
        with pytest.raises(ValueError, match="CUDA tensor"):
            fn(*args, **a)
    b = bwd_call()
    bargs = [b.pop(n) for n in ("q", "k", "v", "g", "beta", "d_o", "cu_seqlens", "chunk_indices",
                                "chunk_offsets", "dq", "dk", "dv", "dg", "dbeta")]
    for fn in (gcl.gdn_chunk_bwd, gcl.kda_chunk_bwd):
        with pytest.raises(ValueError, match="CUDA tensor"):
            fn(*bargs, **b)
    c = conv_call()
    cargs = [c.pop(n) for n in ("x", "weight", "cu_seqlens", "chunk_indices")]
    for fn in (gcl.causal_conv1d_fwd, gcl.causal_conv1d_bwd):
        with pytest.raises(ValueError, match="CUDA tensor"):
            fn(*cargs, **c)
    m = fwd_call()
    with pytest.raises(ValueError, match="CUDA tensor"):
        gcl.chunk_meta_build(m["cu_seqlens"], 300, m["chunk_indices"], m["chunk_offsets"],
                             m["dev_status"], seq_order=m["seq_order"])
    with pytest.raises(ValueError, match="CUDA tensor"):
        gcl.selftest_wait_timeout(m["dev_status"])
