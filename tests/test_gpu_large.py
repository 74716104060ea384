"""Maximum sizes: a varlen batch whose last sequence starts past 2^31 elements of q, k, v and o
(one 2^20-token sequence of 16 heads ahead of it), so every token offset of that sequence
needs 64-bit arithmetic.  Both tensor-core plans run over the whole batch; the oracle checks
the outputs and final state of the far sequence and the first 256 outputs of the long one
(they depend only on its first 256 tokens and its initial state)."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
import oracle  # noqa: E402
from chunked_gated_linear_gb300 import synth  # noqa: E402
from gpu_util import CANARY, DEV, TOL, Meta, relF  # noqa: E402
import chunked_gated_linear_gb300 as gcl  # noqa: E402

H, K, V = 16, 128, 128
LONG = 1 << 20                  # tokens of sequence 0: LONG * H * K = 2^31 elements
TILE = 256                      # sequence 0 is its first TILE tokens repeated
FAR = 300                       # tokens of sequence 1, all past element 2^31
PAD = 20


def _inputs():
    """Host inputs of the small batch [TILE, FAR] and device inputs of the large batch
    [LONG, FAR] built from them (sequence 0 = the TILE-token block repeated)."""
    small = synth.varlen("large-small", synth.GDN, "bf16", [TILE, FAR], 2, TILE + FAR + PAD,
                         H, K, V, seed=81)
    x = synth.make_inputs(small)
    t_max = LONG + FAR + PAD
    d = {}
    for name, dt in (("q", torch.bfloat16), ("k", torch.bfloat16), ("v", torch.bfloat16),
                     ("beta", torch.bfloat16), ("g", torch.float32)):
        a = torch.from_numpy(x[name]).to(DEV).to(dt)
        big = torch.empty((t_max,) + tuple(a.shape[1:]), dtype=dt, device=DEV)
        big[:LONG].view((LONG // TILE, TILE) + tuple(a.shape[1:])).copy_(
            a[:TILE].unsqueeze(0).expand((LONG // TILE, TILE) + tuple(a.shape[1:])))
        big[LONG:].copy_(a[TILE:])                 # sequence 1, then the NaN padding
        d[name] = big
    d["h0"] = torch.from_numpy(x["h0"]).to(DEV)
    d["cu_seqlens"] = torch.tensor([0, LONG, LONG + FAR], dtype=torch.int32, device=DEV)
    return small, x, d, t_max


@pytest.mark.parametrize("plan", ["fastest", "min"], ids=["transition", "wform"])
def test_last_sequence_past_2_31_elements(plan):
    small, x, d, t_max = _inputs()
    assert LONG * H * K >= 1 << 31
    meta = Meta(t_max, 2)
    meta.build(d["cu_seqlens"])
    o = torch.full((t_max, H, V), CANARY, dtype=torch.bfloat16, device=DEV)
    ht = torch.full((2, H, K, V), CANARY, dtype=torch.float32, device=DEV)
    args = (d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], o)
    kw = dict(h0=d["h0"], ht=ht, chunk_indices=meta.idx, chunk_offsets=meta.off,
              seq_order=meta.order, dev_status=meta.status, scale=small.scale)
    nb = (gcl.fwd_workspace_bytes if plan == "fastest" else gcl.fwd_workspace_min_bytes)(*args, **kw)
    ws = torch.empty(max(nb, 16), dtype=torch.uint8, device=DEV)
    gcl.gdn_chunk_fwd(*args, workspace=ws, **kw)
    torch.cuda.synchronize()
    assert int(meta.status.item()) == 0
    o_ref, ht_ref = oracle.fwd(synth.GDN, x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"],
                               x["cu_seqlens"], small.scale)
    far = o[LONG:LONG + FAR].float().cpu().numpy()
    assert relF(far, o_ref[TILE:TILE + FAR]) <= TOL["bf16"]
    assert relF(ht[1].cpu().numpy(), ht_ref[1]) <= TOL["bf16"]
    assert relF(o[:TILE].float().cpu().numpy(), o_ref[:TILE]) <= TOL["bf16"]
    assert torch.isfinite(ht[0]).all()
    assert (o[LONG + FAR:].float() == CANARY).all()     # padding rows untouched
    del args, kw, o, ht, ws, d
    torch.cuda.empty_cache()
