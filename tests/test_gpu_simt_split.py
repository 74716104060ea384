"""The CUDA-core forward's two plans against the fp64 oracle: the split plan (chunk prep over
every chunk at once, then the chain over value-column slices, half-width slices when the grid
would not fill the GPU; taken when the workspace holds its records) and the single kernel (no
workspace).  fp32 inputs at the 1e-5 bar, GDN and KDA,
d = 64 and 128, chunk 32 and 64, ragged and empty sequences, saved chunk states, and the
small fp32 configuration (one 256-token sequence, 2 heads, d = 64, h0 = 0)."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
import oracle  # noqa: E402
import chunked_gated_linear_gb300 as gcl  # noqa: E402
from chunked_gated_linear_gb300 import synth  # noqa: E402
from gpu_util import CANARY, DEV, TOL, Meta, check_fwd, relF, tdtype, to_device  # noqa: E402

LENS = [1, 63, 0, 64, 65, 200, 130, 0]


def _run(w, d, split, h_save=True):
    meta = Meta(w.t_max, w.n_max, w.bt)
    meta.build(d["cu_seqlens"])
    o = torch.full((w.t_max, w.H, w.V), CANARY, dtype=tdtype(w), device=DEV)
    ht = torch.full((w.n_max, w.H, w.K, w.V), CANARY, dtype=torch.float32, device=DEV)
    hs = torch.full((meta.nt_max, w.H, w.K, w.V), CANARY, dtype=torch.float32, device=DEV) if h_save else None
    kda = w.variant == synth.KDA
    args = (d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], o)
    kw = dict(h0=d.get("h0"), ht=ht, h_save=hs, chunk_indices=meta.idx, chunk_offsets=meta.off,
              seq_order=meta.order, dev_status=meta.status, scale=w.scale, bt=w.bt)
    nb = (gcl.kda_fwd_workspace_bytes if kda else gcl.fwd_workspace_bytes)(*args, **kw) if split else 0
    ws = torch.full((max(nb, 16),), 0xFF, dtype=torch.uint8, device=DEV)    # stale contents
    plan = gcl.fwd_plan(*args, workspace=ws, kda=kda, **kw)
    assert plan == ("cuda_cores_split" if split else "cuda_cores"), plan
    (gcl.kda_chunk_fwd if kda else gcl.gdn_chunk_fwd)(*args, workspace=ws, **kw)
    return dict(o=o, ht=ht, h_save=hs, meta=meta, ws=ws)


def _check_states(w, x, out):
    meta = out["meta"]
    off = meta.off.cpu().numpy()
    _, _, hc = oracle.fwd(w.variant, x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"],
                          x["cu_seqlens"], w.scale, bt=w.bt, chunk_offsets=off, nt_rows=meta.nt_max)
    live = int(off[-1])
    hs = out["h_save"].cpu().numpy()
    assert relF(hs[:live], hc[:live]) <= TOL["f32"]
    assert (hs[live:] == np.float32(CANARY)).all()


@pytest.mark.parametrize("variant", [synth.GDN, synth.KDA], ids=["gdn", "kda"])
@pytest.mark.parametrize("d", [64, 128], ids=["d64", "d128"])
@pytest.mark.parametrize("bt", [64, 32], ids=["bt64", "bt32"])
def test_split_plan_fp32(variant, d, bt):
    w = synth.varlen("simt-split", variant, "f32", LENS, len(LENS), sum(LENS) + 24, 3, d, d,
                     seed=71, bt=bt)
    x = synth.make_inputs(w)
    dv = to_device(w, x)
    a = _run(w, dv, split=True)
    check_fwd(w, x, a, label=f"split {variant} d{d} bt{bt}")
    _check_states(w, x, a)
    b = _run(w, dv, split=False)
    check_fwd(w, x, b, label=f"single {variant} d{d} bt{bt}")
    torch.cuda.synchronize()
    T = w.total_tokens
    # the two plans round differently, both far inside the bar of each other
    assert relF(a["o"][:T].cpu().numpy(), b["o"][:T].cpu().numpy()) <= 1e-5
    assert relF(a["ht"].cpu().numpy(), b["ht"].cpu().numpy()) <= 1e-5


@pytest.mark.parametrize("d", [64, 128], ids=["d64", "d128"])
@pytest.mark.parametrize("bt", [64, 32], ids=["bt64", "bt32"])
def test_split_plan_full_width_slices(d, bt):
    """Enough (slot, head) units that the chain's CTAs fill the SMs at the full slice width
    (16 value columns at d = 64, 32 at d = 128); the smaller grids above take half-width
    slices.  fp32 GDN at the 1e-5 bar, ragged and empty sequences."""
    lens = [1, 63, 0, 64, 65, 200, 130, 0, 97, 31, 128, 5]
    w = synth.varlen("simt-split-wide", synth.GDN, "f32", lens, len(lens), sum(lens) + 40, 4, d, d,
                     seed=74, bt=bt)
    assert len(lens) * 4 * 4 >= 152      # n_max x H x (V / slice) at the full slice width
    x = synth.make_inputs(w)
    dv = to_device(w, x)
    a = _run(w, dv, split=True)
    check_fwd(w, x, a, label=f"split wide d{d} bt{bt}")
    _check_states(w, x, a)


def test_split_plan_run_to_run_and_reduced_precision_inputs():
    """bf16 inputs at d = 64 (CUDA cores, fp32 arithmetic): the split plan within the bf16
    bar; two calls bitwise equal."""
    w = synth.varlen("simt-split-bf16", synth.GDN, "bf16", LENS, len(LENS), sum(LENS) + 24, 2, 64,
                     64, seed=72)
    x = synth.make_inputs(w)
    dv = to_device(w, x)
    a = _run(w, dv, split=True)
    b = _run(w, dv, split=True)
    check_fwd(w, x, a, label="split bf16")
    torch.cuda.synchronize()
    assert torch.equal(a["o"], b["o"]) and torch.equal(a["ht"], b["ht"])


def test_small_fp32_configuration():
    """One 256-token sequence, 2 heads, d = 64, h0 = 0, chunk 64: both plans at 1e-5."""
    w = synth.dense("small-fp32", synth.GDN, "f32", 1, 256, 2, 64, 64, h0=False, seed=73)
    x = synth.make_inputs(w)
    dv = to_device(w, x)
    for split in (True, False):
        out = _run(w, dv, split=split, h_save=False)
        check_fwd(w, x, out, label=f"small split={split}")
