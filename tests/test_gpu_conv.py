"""causal_conv1d (the short convolution before the chunk attention) against the fp64 oracle,
through the C ABI: forward and backward, fp32 and bf16, W = 2..4, bias / SiLU / residual /
initial-state combinations, ragged and empty sequences, two channel blocks with a ragged
tail, reproducibility and graph capture."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
import oracle  # noqa: E402
import chunked_gated_linear_gb300 as gcl  # noqa: E402
from chunked_gated_linear_gb300 import synth  # noqa: E402
from gpu_util import CANARY, DEV, TOL, Meta, relF  # noqa: E402


def _dev(a, dtype):
    if a is None:
        return None
    t = torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    return t.to(torch.bfloat16) if dtype == "bf16" else t


def run_conv(x, dtype, t_max, n_max, act, backward=True, meta=None):
    """Metadata, forward and (optionally) backward on device copies of the inputs x."""
    td = torch.bfloat16 if dtype == "bf16" else torch.float32
    D, W = x["weight"].shape
    d = {k: _dev(v, dtype) for k, v in x.items() if k not in ("cu_seqlens", "dht")}
    d["cu_seqlens"] = torch.from_numpy(x["cu_seqlens"]).to(DEV)
    d["dht"] = torch.from_numpy(x["dht"]).to(DEV)
    if meta is None:
        meta = Meta(t_max, n_max)
        meta.build(d["cu_seqlens"])
    f32 = dict(dtype=torch.float32, device=DEV)
    out = dict(y=torch.full((t_max, D), CANARY, dtype=td, device=DEV),
               ht=torch.full((n_max, D, W - 1), CANARY, dtype=td, device=DEV))
    common = (d["x"], d["weight"], d["cu_seqlens"], meta.idx)
    kw = dict(bias=d.get("bias"), h0=d.get("h0"), dev_status=meta.status, activation=act)
    gcl.causal_conv1d_fwd(*common, residual=d.get("residual"), y=out["y"], ht=out["ht"], **kw)
    if backward:
        out.update(dx=torch.full((t_max, D), CANARY, **f32), dw=torch.zeros((D, W), **f32),
                   db=torch.zeros(D, **f32), dh0=torch.zeros((n_max, D, W - 1), **f32))
        bkw = dict(dy=d["dy"], dht=d["dht"], dx=out["dx"], dweight=out["dw"],
                   dbias=out["db"] if x.get("bias") is not None else None, dh0=out["dh0"], **kw)
        ws = torch.empty(max(gcl.causal_conv1d_bwd_workspace_bytes(*common, **bkw), 16),
                         dtype=torch.uint8, device=DEV)
        gcl.causal_conv1d_bwd(*common, workspace=ws, **bkw)
    torch.cuda.synchronize()
    assert int(meta.status.item()) == 0
    return {k: v.float().cpu().numpy() for k, v in out.items()}, meta


def check_conv(x, got, act, dtype, backward=True, label=""):
    cu = x["cu_seqlens"]
    live = int(cu[-1])
    h0 = x["h0"]
    y, ht = oracle.conv_fwd(x["x"], x["weight"], x["bias"], x["residual"], h0, cu, activation=act)
    tol = TOL[dtype]
    assert relF(got["y"][:live], y[:live]) <= tol, (label, "y", relF(got["y"][:live], y[:live]))
    assert relF(got["ht"], ht) <= tol, (label, "ht")
    assert (got["y"][live:] == np.float32(CANARY)).all(), (label, "padding rows of y written")
    if not backward:
        return
    dx, dw, db, dh0 = oracle.conv_bwd(x["x"], x["weight"], x["bias"], h0, cu, x["dy"], x["dht"],
                                      activation=act)
    # the gradients are fp32 sums over the same (rounded) inputs: the fp32 bar for both dtypes
    for key, a, b in (("dx", got["dx"][:live], dx[:live]), ("dw", got["dw"], dw),
                      ("dh0", got["dh0"], dh0 if h0 is not None else got["dh0"] * 0)):
        if key == "dh0" and h0 is None:
            continue
        e = relF(a, b)
        assert e <= TOL["f32"], (label, key, e)
    if x["bias"] is not None:
        assert relF(got["db"], db) <= TOL["f32"], (label, "db")
    assert (got["dx"][live:] == np.float32(CANARY)).all(), (label, "padding rows of dx written")


LENS = [1, 63, 0, 64, 65, 200, 2, 0]
CASES = [(dt, W, act, bias, res, h0)
         for dt in ("f32", "bf16") for W in (2, 3, 4) for act in (None, "silu")
         for (bias, res, h0) in ((True, True, True), (False, False, False))]


@pytest.mark.parametrize("dtype,W,act,bias,res,h0", CASES,
                         ids=[f"{c[0]}-W{c[1]}-{c[2] or 'lin'}-{'brh' if c[3] else 'bare'}"
                              for c in CASES])
def test_varlen_parity(dtype, W, act, bias, res, h0):
    """Ragged and empty sequences over two channel blocks with a ragged tail (D = 1040)."""
    x = synth.make_conv_inputs(LENS, len(LENS), sum(LENS) + 29, 1040, W, dtype, seed=7 + W,
                               h0=h0, bias=bias, residual=res)
    got, _ = run_conv(x, dtype, sum(LENS) + 29, len(LENS), act)
    check_conv(x, got, act, dtype, label=f"{dtype} W={W} {act}")


def test_empty_and_single_token_sequences():
    """Every sequence empty: ht = h0 and dh0 = dht, y untouched; then one token."""
    x = synth.make_conv_inputs([0, 0, 0], 3, 64, 64, 4, "bf16", seed=3)
    got, _ = run_conv(x, "bf16", 64, 3, "silu")
    np.testing.assert_array_equal(got["ht"], x["h0"])
    np.testing.assert_array_equal(got["dh0"], x["dht"])
    assert (got["y"] == np.float32(CANARY)).all()
    x = synth.make_conv_inputs([1], 2, 8, 16, 4, "f32", seed=4)
    got, _ = run_conv(x, "f32", 8, 2, None)
    check_conv(x, got, None, "f32", label="T=1")


def test_long_sequences_cross_many_chunks():
    """Chunk boundaries inside a sequence take their halo from the previous chunk."""
    lens = [1000, 333, 64 * 5]
    x = synth.make_conv_inputs(lens, 3, sum(lens), 256, 4, "bf16", seed=5, residual=True)
    got, _ = run_conv(x, "bf16", sum(lens), 3, "silu")
    check_conv(x, got, "silu", "bf16", label="long")


def test_backward_is_reproducible():
    x = synth.make_conv_inputs([300, 77, 5], 3, 400, 2048, 4, "bf16", seed=6)
    a, meta = run_conv(x, "bf16", 400, 3, "silu")
    b, _ = run_conv(x, "bf16", 400, 3, "silu", meta=meta)
    for key in ("y", "ht", "dx", "dw", "db", "dh0"):
        np.testing.assert_array_equal(a[key], b[key], err_msg=key)


def test_full_size_sampled_channels():
    """The bench workload (4 sequences of 8192 tokens, D = 2048, W = 4, bf16, SiLU, bias,
    initial states): every token of 16 sampled channels against the oracle."""
    B, T, D, W = 4, 8192, 2048, 4
    x = synth.make_conv_inputs([T] * B, B, B * T, D, W, "bf16", seed=8)
    got, _ = run_conv(x, "bf16", B * T, B, "silu")
    ch = np.arange(0, D, D // 16) + 3
    sub = dict(x=x["x"][:, ch], weight=x["weight"][ch], bias=x["bias"][ch], residual=None,
               h0=x["h0"][:, ch], dy=x["dy"][:, ch], dht=x["dht"][:, ch], cu_seqlens=x["cu_seqlens"])
    sub_got = dict(y=got["y"][:, ch], ht=got["ht"][:, ch], dx=got["dx"][:, ch], dw=got["dw"][ch],
                   db=got["db"][ch], dh0=got["dh0"][:, ch])
    check_conv(sub, sub_got, "silu", "bf16", label="full size")


def test_capture_once_replay():
    """Forward + backward captured in a CUDA graph, replayed for new inputs copied in place:
    bit-identical to eager calls on the same buffers."""
    lens = [130, 7, 0, 64]
    t_max, n_max, D, W = 256, 4, 512, 3
    x0 = synth.make_conv_inputs(lens, n_max, t_max, D, W, "bf16", seed=20)
    td = torch.bfloat16
    dev = {k: _dev(v, "bf16") for k, v in x0.items() if k not in ("cu_seqlens", "dht")}
    dev["cu_seqlens"] = torch.from_numpy(x0["cu_seqlens"]).to(DEV)
    dev["dht"] = torch.from_numpy(x0["dht"]).to(DEV)
    meta = Meta(t_max, n_max)
    f32 = dict(dtype=torch.float32, device=DEV)
    y = torch.zeros((t_max, D), dtype=td, device=DEV)
    ht = torch.zeros((n_max, D, W - 1), dtype=td, device=DEV)
    dx, dw = torch.zeros((t_max, D), **f32), torch.zeros((D, W), **f32)
    db, dh0 = torch.zeros(D, **f32), torch.zeros((n_max, D, W - 1), **f32)
    common = (dev["x"], dev["weight"], dev["cu_seqlens"], meta.idx)
    kw = dict(bias=dev["bias"], h0=dev["h0"], dev_status=meta.status, activation="silu")
    bkw = dict(dy=dev["dy"], dht=dev["dht"], dx=dx, dweight=dw, dbias=db, dh0=dh0, **kw)
    ws = torch.empty(gcl.causal_conv1d_bwd_workspace_bytes(*common, **bkw), dtype=torch.uint8,
                     device=DEV)

    def step(stream=None):
        meta.build(dev["cu_seqlens"], stream=stream)
        gcl.causal_conv1d_fwd(*common, y=y, ht=ht, stream=stream, **kw)
        gcl.causal_conv1d_bwd(*common, workspace=ws, stream=stream, **bkw)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step(stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for seed in (21, 22):
        xn = synth.make_conv_inputs(lens, n_max, t_max, D, W, "bf16", seed=seed)
        for k in ("x", "weight", "bias", "h0", "dy"):
            dev[k].copy_(_dev(xn[k], "bf16"))
        dev["dht"].copy_(torch.from_numpy(xn["dht"]))
        g.replay()
        torch.cuda.synchronize()
        res = {k: t.clone() for k, t in dict(y=y, ht=ht, dx=dx, dw=dw, db=db, dh0=dh0).items()}
        got = {k: v.float().cpu().numpy() for k, v in res.items()}
        got["y"][int(x0["cu_seqlens"][-1]):] = np.float32(CANARY)   # (y was zero-filled)
        got["dx"][int(x0["cu_seqlens"][-1]):] = np.float32(CANARY)
        xn["residual"] = None
        check_conv(xn, got, "silu", "bf16", label=f"replay {seed}")
        step()
        torch.cuda.synchronize()
        for k, t in dict(y=y, ht=ht, dx=dx, dw=dw, db=db, dh0=dh0).items():
            assert torch.equal(t, res[k]), k
