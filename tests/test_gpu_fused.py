"""The fused tensor-core forward (one CTA per (sequence, head), every intermediate on chip)
against the fp64 oracle: ragged and empty sequences, NaN padding, with and without h0, saved
chunk states, the degenerate gate and beta regimes, and sampled units at full size."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
import oracle  # noqa: E402
import chunked_gated_linear_gb300 as gcl  # noqa: E402
from chunked_gated_linear_gb300 import synth  # noqa: E402
from gpu_util import CANARY, TOL, Meta, check_fwd, run_fwd, to_device  # noqa: E402
from parity import check as parity_check  # noqa: E402

LENS = [1, 63, 0, 64, 65, 200, 130, 0]
HF = 20                                       # 8 slots x 20 heads = 160 units >= SMs: the fused plan


def _plan(w, d, meta, h_save=None, workspace=None):
    o = torch.empty((w.t_max, w.H, w.V), dtype=torch.bfloat16, device=d["q"].device)
    return gcl.fwd_plan(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], o,
                        h0=d.get("h0"), h_save=h_save, chunk_indices=meta.idx,
                        chunk_offsets=meta.off, workspace=workspace, scale=w.scale)


@pytest.mark.parametrize("h0", [True, False], ids=["h0", "no-h0"])
def test_fused_ragged(h0):
    w = synth.varlen("fused", synth.GDN, "bf16", LENS, 8, sum(LENS) + 40, HF, 128, 128, h0=h0,
                     seed=31)
    x = synth.make_inputs(w)
    d = to_device(w, x)
    a = run_fwd(w, d)
    assert _plan(w, d, a["meta"]) == "fused"
    assert a["ws"].numel() == 16                    # the fused plan asks for no workspace
    check_fwd(w, x, a, label=f"fused h0={h0}")
    b = run_fwd(w, d)
    c = run_fwd(w, d, use_order=False)
    torch.cuda.synchronize()
    for key in ("o", "ht"):                         # run to run and order independent, bitwise
        assert torch.equal(a[key], b[key]) and torch.equal(a[key], c[key]), key


def test_fused_saved_chunk_states():
    """A forward with h_save and less workspace than the transition records runs the fused
    plan; every saved chunk state against the oracle's, unused rows untouched."""
    w = synth.varlen("fused-hs", synth.GDN, "bf16", LENS, 8, sum(LENS) + 40, HF, 128, 128, seed=32)
    x = synth.make_inputs(w)
    d = to_device(w, x)
    out = run_fwd(w, d, h_save=True, plan="min")
    assert _plan(w, d, out["meta"], h_save=out["h_save"], workspace=out["ws"]) == "fused"
    check_fwd(w, x, out, label="fused h_save")
    meta = out["meta"]
    off = meta.off.cpu().numpy()
    _, _, hc = oracle.fwd(synth.GDN, x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"],
                          x["cu_seqlens"], w.scale, bt=64, chunk_offsets=off, nt_rows=meta.nt_max)
    live = int(off[-1])
    hs = out["h_save"].cpu().numpy()
    parity_check("h_save", hs[:live], hc[:live], TOL["bf16"])
    assert (hs[live:] == np.float32(CANARY)).all()


@pytest.mark.parametrize("regime", ["beta0", "nodecay", "strong", "mixed"])
def test_fused_degenerate_gates_and_beta(regime):
    """beta = 0 (A = 0, T = I: the state only decays), g = 0, log gates 20x the generator's
    (chunk decay far below fp32's range) and a mix of strong and zero gates."""
    w = synth.varlen("fused-gates", synth.GDN, "bf16", LENS, 8, sum(LENS) + 40, HF, 128, 128,
                     seed=33)
    x = synth.make_inputs(w)
    T = w.total_tokens
    rng = np.random.default_rng(34)
    if regime == "beta0":
        x["beta"][:T] = 0.0
    elif regime == "nodecay":
        x["g"][:T] = 0.0
    elif regime == "strong":
        x["g"][:T] *= 20.0
    else:
        g = x["g"][:T]
        g[rng.random(g.shape) < 0.2] *= 40.0
        g[rng.random(g.shape) < 0.3] = 0.0
        x["g"][:T] = g
    check_fwd(w, x, run_fwd(w, to_device(w, x)), label=f"fused {regime}")


def test_fused_dense_full_size_sampled_units():
    """B = 10, T = 8192, H = 16 (160 units of 128 chunks), inference forward: the fused plan;
    sampled units (first and last sequence and head among them) against the oracle at the
    global, per-unit and per-row bars."""
    w = synth.dense("fused-dense", synth.GDN, "bf16", 10, 8192, 16, 128, 128, seed=35)
    x = synth.make_inputs(w)
    d = to_device(w, x)
    out = run_fwd(w, d)
    torch.cuda.synchronize()
    assert int(out["meta"].status.item()) == 0
    assert _plan(w, d, out["meta"]) == "fused"
    o = out["o"].float().cpu().numpy()
    ht = out["ht"].cpu().numpy()
    T = 8192
    cu1 = np.array([0, T], dtype=np.int64)
    for (b, h) in ((0, 0), (0, 15), (3, 5), (6, 10), (9, 0), (9, 15)):
        s, e = b * T, (b + 1) * T
        sl = {m: x[m][s:e, h:h + 1] for m in ("q", "k", "v", "g", "beta")}
        o_ref, ht_ref = oracle.fwd(synth.GDN, sl["q"], sl["k"], sl["v"], sl["g"], sl["beta"],
                                   x["h0"][b:b + 1, h:h + 1], [0, T], w.scale)
        parity_check(f"unit ({b},{h}) o", o[s:e, h:h + 1], o_ref, TOL["bf16"], cu=cu1)
        parity_check(f"unit ({b},{h}) ht", ht[b:b + 1, h:h + 1], ht_ref, TOL["bf16"])


def test_fused_matches_split_plans_closely():
    """The same inputs through the fused plan (160 units) and, head by head, through the
    split plans (one head per call: 8 units): both within the bar of the oracle and of each
    other."""
    w = synth.varlen("fused-vs", synth.GDN, "bf16", LENS, 8, sum(LENS) + 40, HF, 128, 128, seed=36)
    x = synth.make_inputs(w)
    d = to_device(w, x)
    fused = run_fwd(w, d)
    torch.cuda.synchronize()
    T = w.total_tokens
    o_f = fused["o"].float().cpu().numpy()[:T]
    for h in (0, HF - 1):
        w1 = synth.varlen("one-head", synth.GDN, "bf16", LENS, 8, sum(LENS) + 40, 1, 128, 128,
                          seed=36)
        x1 = {k: (v[:, h:h + 1] if k in ("q", "k", "v", "g", "beta") else v) for k, v in x.items()}
        x1["h0"] = x["h0"][:, h:h + 1]
        d1 = to_device(w1, x1)
        meta1 = Meta(w1.t_max, w1.n_max)
        meta1.build(d1["cu_seqlens"])
        assert _plan(w1, d1, meta1) != "fused"
        one = run_fwd(w1, d1, meta=meta1)
        check_fwd(w1, x1, one, label=f"split head {h}")
        o1 = one["o"].float().cpu().numpy()[:T]
        parity_check(f"fused vs split head {h}", o_f[:, h:h + 1], o1, 2 * TOL["bf16"],
                     cu=np.asarray(x["cu_seqlens"], dtype=np.int64))
