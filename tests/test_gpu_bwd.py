"""GDN backward parity against the fp64 reverse-mode oracle."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
import oracle  # noqa: E402
import chunked_gated_linear_gb300 as gcl  # noqa: E402
from chunked_gated_linear_gb300 import synth  # noqa: E402
from gpu_util import DEV, TOL, Meta, check_fwd, relF, run_fwd, to_device  # noqa: E402
from parity import check as parity_check  # noqa: E402

GRADS = ("dq", "dk", "dv", "dg", "dbeta", "dh0")


def run_bwd(w, d, meta, h_save=None, with_dht=True, fwd_ws=None):
    T, H, K, V = w.t_max, w.H, w.K, w.V
    f32 = dict(dtype=torch.float32, device=DEV)
    kda = w.variant == synth.KDA
    out = dict(dq=torch.zeros((T, H, K), **f32), dk=torch.zeros((T, H, K), **f32),
               dv=torch.zeros((T, H, V), **f32),
               dg=torch.zeros((T, H, K) if kda else (T, H), **f32),
               dbeta=torch.zeros((T, H), **f32), dh0=torch.zeros((w.n_max, H, K, V), **f32))
    args = (d["q"], d["k"], d["v"], d["g"], d["beta"], d["do"], d["cu_seqlens"], meta.idx,
            meta.off, out["dq"], out["dk"], out["dv"], out["dg"], out["dbeta"])
    kw = dict(h0=d.get("h0"), dht=d["dht"] if with_dht else None, dh0=out["dh0"],
              h_save=h_save, dev_status=meta.status, scale=w.scale, bt=w.bt, fwd_workspace=fwd_ws)
    nbytes = (gcl.kda_bwd_workspace_bytes if kda else gcl.bwd_workspace_bytes)(*args, **kw)
    ws = torch.full((nbytes,), 0xFF, dtype=torch.uint8, device=DEV)      # stale contents
    (gcl.kda_chunk_bwd if kda else gcl.gdn_chunk_bwd)(*args, workspace=ws, **kw)
    torch.cuda.synchronize()
    assert int(meta.status.item()) == 0
    return {k_: v_.cpu().numpy() for k_, v_ in out.items()}


def oracle_bwd(w, x, with_dht=True):
    return oracle.bwd(w.variant, x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"], x["do"],
                      x["dht"] if with_dht else None, x["cu_seqlens"], w.scale)


def compare(w, got, ref, tol):
    """Every gradient at the global, per-unit and per-row bars (tests/parity.py)."""
    T = w.total_tokens
    cu = np.asarray(synth.cu_seqlens_of(w), dtype=np.int64)
    for key in GRADS:
        if key == "dh0":
            parity_check(key, got[key], ref[key], tol)
        else:
            parity_check(key, got[key][:T], ref[key][:T], tol, cu=cu)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("KV", [(64, 64), (128, 128)])
@pytest.mark.parametrize("saved", [True, False])
def test_small_varlen(dtype, KV, saved):
    K, V = KV
    lens = [1, 63, 0, 64, 65, 150]
    w = synth.varlen("bwd", synth.GDN, dtype, lens, 7, sum(lens) + 20, 2, K, V, backward=True,
                     seed=11)
    x = synth.make_inputs(w)
    d = to_device(w, x)
    fw = run_fwd(w, d, h_save=saved)
    got = run_bwd(w, d, fw["meta"], h_save=fw["h_save"])
    compare(w, got, oracle_bwd(w, x), TOL[dtype])


def test_no_dht_no_h0():
    w = synth.varlen("bwd0", synth.GDN, "bf16", [130, 7], 2, 200, 2, 128, 128, h0=False,
                     backward=True, seed=12)
    x = synth.make_inputs(w)
    d = to_device(w, x)
    meta = Meta(w.t_max, w.n_max)
    meta.build(d["cu_seqlens"])
    got = run_bwd(w, d, meta, with_dht=False)
    compare(w, got, oracle_bwd(w, x, with_dht=False), TOL["bf16"])


def test_fwd_bwd_full_size_sampled_units():
    """B=4, T=8192, H=16, d=128, bf16: forward + backward on the GPU at full size; the oracle
    recomputes sampled (sequence, head) units one by one (eight of the 64, including the last
    sequence and the last head), and o, ht and every gradient of those units are compared at
    the global, per-unit and per-row bars."""
    w = synth.standard_workloads()[4]
    x = synth.make_inputs(w)
    d = to_device(w, x)
    fw = run_fwd(w, d, h_save=True)
    torch.cuda.synchronize()
    assert int(fw["meta"].status.item()) == 0
    o = fw["o"].float().cpu().numpy()
    ht = fw["ht"].cpu().numpy()
    got = run_bwd(w, d, fw["meta"], h_save=fw["h_save"])
    T = w.lengths[0]
    cu1 = np.array([0, T], dtype=np.int64)
    units = ((0, 0), (0, 15), (1, 3), (1, 9), (2, 7), (2, 12), (3, 0), (3, 15))
    for (b, h) in units:
        s, e = b * T, (b + 1) * T
        sl = {m: x[m][s:e, h:h + 1] for m in ("q", "k", "v", "g", "beta", "do")}
        h0 = x["h0"][b:b + 1, h:h + 1]
        o_ref, ht_ref = oracle.fwd(synth.GDN, sl["q"], sl["k"], sl["v"], sl["g"], sl["beta"], h0,
                                   [0, T], w.scale)
        parity_check(f"unit ({b},{h}) o", o[s:e, h:h + 1], o_ref, TOL["bf16"], cu=cu1)
        parity_check(f"unit ({b},{h}) ht", ht[b:b + 1, h:h + 1], ht_ref, TOL["bf16"])
        ref = oracle.bwd(synth.GDN, sl["q"], sl["k"], sl["v"], sl["g"], sl["beta"], h0,
                         sl["do"], x["dht"][b:b + 1, h:h + 1], [0, T], w.scale)
        for key in ("dq", "dk", "dv", "dg", "dbeta"):
            parity_check(f"unit ({b},{h}) {key}", got[key][s:e, h:h + 1], ref[key], TOL["bf16"],
                         cu=cu1)
        parity_check(f"unit ({b},{h}) dh0", got["dh0"][b:b + 1, h:h + 1], ref["dh0"], TOL["bf16"])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("KV", [(64, 64), (128, 128)])
@pytest.mark.parametrize("saved", [True, False])
def test_kda_small_varlen(dtype, KV, saved):
    """kda_chunk_bwd: every gradient (dg per key channel) against the oracle's reverse mode,
    ragged lengths, with saved chunk states or recomputing them."""
    K, V = KV
    lens = [1, 63, 0, 64, 65, 150]
    w = synth.varlen("kda-bwd", synth.KDA, dtype, lens, 7, sum(lens) + 20, 2, K, V, backward=True,
                     seed=13)
    x = synth.make_inputs(w)
    d = to_device(w, x)
    fw = run_fwd(w, d, h_save=saved)
    got = run_bwd(w, d, fw["meta"], h_save=fw["h_save"])
    compare(w, got, oracle_bwd(w, x), TOL[dtype])


def test_kda_no_dht_no_h0_strong_gates():
    """KDA backward without dht and h0, with per-channel log gates down to -40 per token."""
    w = synth.varlen("kda-bwd0", synth.KDA, "bf16", [130, 7], 2, 200, 2, 128, 128, h0=False,
                     backward=True, seed=14)
    x = synth.make_inputs(w)
    g = x["g"].copy()
    g[np.random.default_rng(3).random(g.shape) < 0.1] *= 20.0
    x["g"] = g.astype(np.float32)
    d = to_device(w, x)
    meta = Meta(w.t_max, w.n_max)
    meta.build(d["cu_seqlens"])
    got = run_bwd(w, d, meta, with_dht=False)
    compare(w, got, oracle_bwd(w, x, with_dht=False), TOL["bf16"])


@pytest.mark.parametrize("variant", [synth.GDN, synth.KDA], ids=["gdn", "kda"])
@pytest.mark.parametrize("H", [2, 8], ids=["few-units", "many-units"])
def test_backward_reuses_forward_records(variant, H):
    """A training forward (h_save) runs the transition plan; handing its workspace to the
    backward skips the recompute of the chunk records: gradients bitwise equal to the backward
    that recomputes them, and within the bar of the oracle.  H = 8 over 8 sequence slots gives
    64 units (two value slices per head), H = 2 gives 16 (eight slices)."""
    lens = [1, 63, 0, 64, 65, 200, 130, 77]
    w = synth.varlen("reuse", variant, "bf16", lens, 8, sum(lens) + 40, H, 128, 128,
                     backward=True, seed=81)
    x = synth.make_inputs(w)
    d = to_device(w, x)
    fw = run_fwd(w, d, h_save=True)
    check_fwd(w, x, fw, label="training forward")
    a = run_bwd(w, d, fw["meta"], h_save=fw["h_save"], fwd_ws=fw["ws"])
    b = run_bwd(w, d, fw["meta"], h_save=fw["h_save"])
    for key in GRADS:
        np.testing.assert_array_equal(a[key], b[key], err_msg=key)
    compare(w, a, oracle_bwd(w, x), TOL["bf16"])
