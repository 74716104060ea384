"""The segmented chain (few long sequences: segment summaries, the scan of the segments' start
states, the segments' outputs) against the fp64 oracle and against the plain chain, GDN and KDA
bf16 d = 128, through the C ABI: one 64K-token sequence, ragged and empty sequences over several
heads, sequences shorter than the segment count, and graph replay over changing lengths."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
import oracle  # noqa: E402
import chunked_gated_linear_gb300 as gcl  # noqa: E402
from chunked_gated_linear_gb300 import synth  # noqa: E402
from gpu_util import CANARY, DEV, TOL, Meta, check_fwd, relF, run_fwd, tdtype, to_device  # noqa: E402

SEG_UNIT_BYTES = 192 * 1024          # segment buffers per sequence slot, head and segment


def segments(w):
    return gcl.fwd_chain_segments(w.t_max, w.n_max, w.H, w.bt)


def run_plain(w, d):
    """The same forward with the workspace of the plain chain (the records, no segment buffers)."""
    fn = gcl.kda_chunk_fwd if w.variant == synth.KDA else gcl.gdn_chunk_fwd
    meta = Meta(w.t_max, w.n_max, w.bt)
    meta.build(d["cu_seqlens"])
    o = torch.full((w.t_max, w.H, w.V), CANARY, dtype=tdtype(w), device=DEV)
    ht = torch.full((w.n_max, w.H, w.K, w.V), CANARY, dtype=torch.float32, device=DEV)
    args = (d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], o)
    kw = dict(h0=d.get("h0"), ht=ht, chunk_indices=meta.idx, chunk_offsets=meta.off,
              seq_order=meta.order, dev_status=meta.status, scale=w.scale, bt=w.bt)
    q = gcl.kda_fwd_workspace_bytes if w.variant == synth.KDA else gcl.fwd_workspace_bytes
    nb = q(*args, **kw) - w.n_max * w.H * segments(w) * SEG_UNIT_BYTES
    ws = torch.full((nb,), 0xFF, dtype=torch.uint8, device=DEV)
    fn(*args, workspace=ws, **kw)
    return dict(o=o, ht=ht, meta=meta)


def check_saved_states(w, x, out):
    meta = out["meta"]
    off = meta.off.cpu().numpy()
    _, _, hc = oracle.fwd(w.variant, x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"],
                          x["cu_seqlens"], w.scale, bt=64, chunk_offsets=off, nt_rows=meta.nt_max)
    live = int(off[-1])
    hs = out["h_save"].cpu().numpy()
    assert relF(hs[:live], hc[:live]) <= TOL["bf16"]
    assert (hs[live:] == np.float32(CANARY)).all(), "rows past the live chunks were written"


@pytest.mark.parametrize("variant", [synth.GDN, synth.KDA], ids=["gdn", "kda"])
def test_long_single_sequence(variant):
    """One 64K-token sequence of one head (1024 chunks) cut into segments: o, ht and every
    chunk's start state against the oracle, and o, ht against the plain chain."""
    name = ("kda" if variant == synth.KDA else "gdn") + "_fwd_bf16_T65536_H1_d128"
    w = synth.workload_by_name(name)
    assert segments(w) >= 3
    x = synth.make_inputs(w)
    d = to_device(w, x)
    out = run_fwd(w, d, h_save=True)
    e_o, e_h = check_fwd(w, x, out, label=name)
    check_saved_states(w, x, out)
    plain = run_plain(w, d)
    e_po, e_ph = check_fwd(w, x, plain, label=name + " plain")
    o_seg = out["o"].float().cpu().numpy()
    o_pl = plain["o"].float().cpu().numpy()
    assert relF(o_seg, o_pl) <= TOL["bf16"]
    print(f"{name}: {segments(w)} segments: o {e_o:.2e} ht {e_h:.2e}; plain o {e_po:.2e} ht {e_ph:.2e}")


@pytest.mark.parametrize("variant", [synth.GDN, synth.KDA], ids=["gdn", "kda"])
@pytest.mark.parametrize("use_order", [True, False], ids=["ordered", "slot-order"])
@pytest.mark.parametrize("lens,H", [([12000, 0, 130], 1), ([130, 12000], 2)],
                         ids=["empty-slot-H1", "H2"])
def test_ragged_and_empty_sequences(variant, use_order, lens, H):
    """A long and a short sequence (and an empty slot) in a 12800-token capacity, over one or
    two heads: 3 or 4 units, so 6 or 4 segments per sequence; the short sequence (3 chunks)
    has fewer chunks than segments."""
    w = synth.varlen("seg-ragged", variant, "bf16", lens, len(lens), 12800, H, 128, 128, seed=31)
    assert segments(w) >= 3
    x = synth.make_inputs(w)
    out = run_fwd(w, to_device(w, x), h_save=True, use_order=use_order)
    check_fwd(w, x, out, label=f"ragged {lens}")
    check_saved_states(w, x, out)
    for n, L in enumerate(lens):
        if L == 0:
            np.testing.assert_array_equal(out["ht"].cpu().numpy()[n], x["h0"][n])


@pytest.mark.parametrize("T", [30, 100, 1221, 4000])
@pytest.mark.parametrize("h0", [True, False], ids=["h0", "zero-h0"])
def test_short_sequences_in_a_long_capacity(T, h0):
    """One sequence of 1, 2, 20 and 63 chunks in an 8192-token capacity, whose plan cuts each
    sequence into P segments (16 on 152 SMs) of ceil(chunks / P) chunks: one segment, two
    single-chunk segments, ten of two chunks, and so on."""
    w = synth.varlen("seg-short", synth.GDN, "bf16", [T], 1, 8192, 1, 128, 128, h0=h0, seed=32)
    assert segments(w) >= 3
    x = synth.make_inputs(w)
    out = run_fwd(w, to_device(w, x), h_save=True)
    check_fwd(w, x, out, label=f"T={T}")
    check_saved_states(w, x, out)


def test_graph_replay_over_changing_lengths():
    """Captured once at capacity (two slots, 8192 tokens, one head), replayed for layouts of
    different lengths copied in place: each against the oracle and bit-identical to an eager
    call on the same buffers."""
    t_max, n_max, H = 8192, 2, 1
    layouts = [[8000, 100], [3000, 4000], [64, 0], [0, 8192]]
    base = synth.varlen("seg-graph", synth.KDA, "bf16", layouts[0], n_max, t_max, H, 128, 128,
                        seed=33)
    assert segments(base) >= 3
    static = to_device(base, synth.make_inputs(base))
    meta = Meta(t_max, n_max)
    o = torch.full((t_max, H, 128), CANARY, dtype=torch.bfloat16, device=DEV)
    ht = torch.zeros((n_max, H, 128, 128), dtype=torch.float32, device=DEV)
    args = (static["q"], static["k"], static["v"], static["g"], static["beta"],
            static["cu_seqlens"], o)
    kw = dict(h0=static["h0"], ht=ht, chunk_indices=meta.idx, chunk_offsets=meta.off,
              seq_order=meta.order, dev_status=meta.status, scale=base.scale)
    ws = torch.empty(gcl.kda_fwd_workspace_bytes(*args, **kw), dtype=torch.uint8, device=DEV)

    def step(stream=None):
        meta.build(static["cu_seqlens"], stream=stream)
        gcl.kda_chunk_fwd(*args, workspace=ws, stream=stream, **kw)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step(stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for i, lens in enumerate(layouts[1:]):
        w = synth.varlen("seg-graph", synth.KDA, "bf16", lens, n_max, t_max, H, 128, 128,
                         seed=34 + i)
        x = synth.make_inputs(w)
        new = to_device(w, x)
        for name in ("q", "k", "v", "g", "beta", "h0", "cu_seqlens"):
            static[name].copy_(new[name])
        o.fill_(CANARY)
        g.replay()
        torch.cuda.synchronize()
        check_fwd(w, x, dict(o=o, ht=ht, meta=meta), label=f"replay {lens}")
        o_graph, ht_graph = o.clone(), ht.clone()
        o.fill_(CANARY)
        step()
        torch.cuda.synchronize()
        assert torch.equal(o, o_graph) and torch.equal(ht, ht_graph)
