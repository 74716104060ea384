"""Varlen GDN prefill with fixed capacity under CUDA graph capture: capture once
(N_max=64, T_max=65536, H=16, d=128, bf16), then replay three fresh seeded
layouts updated in place with copy_, each checked against the oracle and
against an eager call on the same buffers (bit-identical)."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
from chunked_gated_linear_gb300 import synth  # noqa: E402
import chunked_gated_linear_gb300 as gcl  # noqa: E402
from gpu_util import CANARY, DEV, Meta, check_fwd, tdtype, to_device  # noqa: E402


def test_capture_once_replay_three_layouts():
    base = synth.standard_workloads()[3]
    seeds = synth.layout_seeds(base)
    w0 = synth.varlen_layout(base, seeds[0])
    static = to_device(w0, synth.make_inputs(w0))
    meta = Meta(base.t_max, base.n_max)
    o = torch.full((base.t_max, base.H, base.V), CANARY, dtype=tdtype(base), device=DEV)
    ht = torch.zeros((base.n_max, base.H, base.K, base.V), dtype=torch.float32, device=DEV)

    args = (static["q"], static["k"], static["v"], static["g"], static["beta"],
            static["cu_seqlens"], o)
    kw = dict(h0=static["h0"], ht=ht, chunk_indices=meta.idx, chunk_offsets=meta.off,
              seq_order=meta.order, dev_status=meta.status, scale=base.scale)
    ws = torch.empty(max(gcl.fwd_workspace_bytes(*args, **kw), 16), dtype=torch.uint8,
                     device=DEV)

    def step(stream=None):
        meta.build(static["cu_seqlens"], stream=stream)
        gcl.gdn_chunk_fwd(*args, workspace=ws, stream=stream, **kw)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step(stream=s)                          # warm-up before capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for seed in seeds[1:]:
        w = synth.varlen_layout(base, seed)
        x = synth.make_inputs(w)                # NaN in every padding row
        new = to_device(w, x)
        for name in ("q", "k", "v", "g", "beta", "h0", "cu_seqlens"):
            static[name].copy_(new[name])
        o.fill_(CANARY)
        g.replay()
        torch.cuda.synchronize()
        e_o, e_h = check_fwd(w, x, dict(o=o, ht=ht, meta=meta), label=f"replay seed {seed}")
        print(f"seed {seed}: T={w.total_tokens} live chunks {int(meta.off[-1])} / "
              f"{meta.nt_max}: o {e_o:.2e} ht {e_h:.2e}")
        o_graph, ht_graph = o.clone(), ht.clone()
        o.fill_(CANARY)
        step()                                  # eager on the same buffers
        torch.cuda.synchronize()
        assert torch.equal(o, o_graph) and torch.equal(ht, ht_graph)
