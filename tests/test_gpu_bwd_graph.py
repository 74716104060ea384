"""Forward + backward under CUDA graph capture (the training path of the RFC's graph
work): chunk_meta_build, the forward with saved chunk states and the backward are captured
once on static buffers, then replayed for fresh inputs copied in place.  Each replay must
equal an eager call on the same buffers bit for bit and the oracle within the bf16 bar; the
backward either forms its own chunk records or reads the forward's (fwd_workspace)."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
import oracle  # noqa: E402
import chunked_gated_linear_gb300 as gcl  # noqa: E402
from chunked_gated_linear_gb300 import synth  # noqa: E402
from gpu_util import DEV, TOL, Meta, relF, tdtype, to_device  # noqa: E402

GRADS = ("dq", "dk", "dv", "dg", "dbeta", "dh0")


@pytest.mark.parametrize("variant", [synth.GDN, synth.KDA], ids=["gdn", "kda"])
@pytest.mark.parametrize("reuse", [False, True], ids=["own-records", "forward-records"])
def test_fwd_bwd_capture_once_replay(variant, reuse):
    lens = [300, 1, 0, 129]
    w = synth.varlen("graph-bwd", variant, "bf16", lens, 4, 512, 4, 128, 128, backward=True,
                     seed=31)
    kda = variant == synth.KDA
    static = to_device(w, synth.make_inputs(w))
    meta = Meta(w.t_max, w.n_max)
    T, H, K, V = w.t_max, w.H, w.K, w.V
    f32 = dict(dtype=torch.float32, device=DEV)
    o = torch.zeros((T, H, V), dtype=tdtype(w), device=DEV)
    ht = torch.zeros((w.n_max, H, K, V), **f32)
    hs = torch.zeros((meta.nt_max, H, K, V), **f32)
    out = dict(dq=torch.zeros((T, H, K), **f32), dk=torch.zeros((T, H, K), **f32),
               dv=torch.zeros((T, H, V), **f32),
               dg=torch.zeros((T, H, K) if kda else (T, H), **f32),
               dbeta=torch.zeros((T, H), **f32), dh0=torch.zeros((w.n_max, H, K, V), **f32))
    fargs = (static["q"], static["k"], static["v"], static["g"], static["beta"],
             static["cu_seqlens"], o)
    fkw = dict(h0=static["h0"], ht=ht, h_save=hs, chunk_indices=meta.idx,
               chunk_offsets=meta.off, seq_order=meta.order, dev_status=meta.status,
               scale=w.scale)
    fws = torch.empty(max((gcl.kda_fwd_workspace_bytes if kda else gcl.fwd_workspace_bytes)(
        *fargs, **fkw), 16), dtype=torch.uint8, device=DEV)
    bargs = (static["q"], static["k"], static["v"], static["g"], static["beta"], static["do"],
             static["cu_seqlens"], meta.idx, meta.off, out["dq"], out["dk"], out["dv"],
             out["dg"], out["dbeta"])
    bkw = dict(h0=static["h0"], dht=static["dht"], dh0=out["dh0"], h_save=hs,
               dev_status=meta.status, scale=w.scale, fwd_workspace=fws if reuse else None)
    bws = torch.empty((gcl.kda_bwd_workspace_bytes if kda else gcl.bwd_workspace_bytes)(
        *bargs, **bkw), dtype=torch.uint8, device=DEV)
    fwd = gcl.kda_chunk_fwd if kda else gcl.gdn_chunk_fwd
    bwd = gcl.kda_chunk_bwd if kda else gcl.gdn_chunk_bwd

    def step(stream=None):
        meta.build(static["cu_seqlens"], stream=stream)
        fwd(*fargs, workspace=fws, stream=stream, **fkw)
        bwd(*bargs, workspace=bws, stream=stream, **bkw)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step(stream=s)                            # warm-up before capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for seed in (32, 33):
        x = synth.make_inputs(w, seed=seed)
        new = to_device(w, x)
        for name in ("q", "k", "v", "g", "beta", "h0", "do", "dht", "cu_seqlens"):
            static[name].copy_(new[name])
        for t in out.values():
            t.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert int(meta.status.item()) == 0
        got = {k_: v_.clone() for k_, v_ in out.items()}
        ref = oracle.bwd(variant, x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"], x["do"],
                         x["dht"], x["cu_seqlens"], w.scale)
        live = w.total_tokens
        for key in GRADS:
            a = got[key].cpu().numpy()
            b = ref[key]
            e = relF(a, b) if key == "dh0" else relF(a[:live], b[:live])
            assert e <= TOL["bf16"], f"replay seed {seed} {key}: {e:.3e}"
        for t in out.values():
            t.zero_()
        step()                                    # eager on the same buffers
        torch.cuda.synchronize()
        for key in GRADS:
            assert torch.equal(out[key], got[key]), key
