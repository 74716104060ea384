"""The RFC test matrix's variants against the fp64 oracle, through the C ABI: fp16 inputs (the
GDN forward at d = 128 on the tensor cores, everything else on the CUDA cores in fp32) and chunk
size BT = 32 (CUDA cores), forward and backward, GDN and KDA, ragged and empty sequences, saved
chunk states."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
import oracle  # noqa: E402
from chunked_gated_linear_gb300 import synth  # noqa: E402
from gpu_util import CANARY, TOL, check_fwd, relF, run_fwd, to_device  # noqa: E402
from test_gpu_bwd import GRADS, oracle_bwd, run_bwd  # noqa: E402

LENS = [1, 31, 0, 32, 33, 64, 65, 150]
VARIANTS = [(synth.GDN, "gdn"), (synth.KDA, "kda")]


def _w(variant, dtype, KV, bt, backward=False, seed=60):
    K, V = KV
    return synth.varlen("variant", variant, dtype, LENS, len(LENS), sum(LENS) + 20, 2, K, V,
                        backward=backward, seed=seed, bt=bt)


def _check_states(w, x, out, tol=TOL["f32"]):
    meta = out["meta"]
    off = meta.off.cpu().numpy()
    _, _, hc = oracle.fwd(w.variant, x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"],
                          x["cu_seqlens"], w.scale, bt=w.bt, chunk_offsets=off,
                          nt_rows=meta.nt_max)
    live = int(off[-1])
    hs = out["h_save"].cpu().numpy()
    assert relF(hs[:live], hc[:live]) <= tol
    assert (hs[live:] == np.float32(CANARY)).all()


def _compare_grads(w, got, ref, tol):
    T = w.total_tokens
    for key in GRADS:
        a, b = (got[key], ref[key]) if key == "dh0" else (got[key][:T], ref[key][:T])
        e = relF(a, b)
        assert e <= tol, f"{key}: rel-Frobenius {e:.3e} > {tol}"


@pytest.mark.parametrize("variant,vname", VARIANTS, ids=[v[1] for v in VARIANTS])
@pytest.mark.parametrize("KV", [(64, 64), (128, 128)], ids=["d64", "d128"])
def test_fp16_forward_and_backward(variant, vname, KV):
    """fp16 q, k, v, beta, dO.  On the CUDA cores (fp32 arithmetic): o within the fp16 output
    rounding, ht, the saved chunk states and every gradient within the fp32 bar.  GDN at
    d = 128 runs the forward on the tensor cores with every MMA operand in fp16: every output
    within the fp16 bar (TOL["f16"], about twice fp16's unit roundoff), and the gradients,
    computed from those saved states, likewise."""
    w = _w(variant, "f16", KV, 64, backward=True)
    x = synth.make_inputs(w)
    d = to_device(w, x)
    assert d["q"].dtype == torch.float16
    tc = variant == synth.GDN and KV == (128, 128)
    tol = TOL["f16"] if tc else TOL["f32"]
    out = run_fwd(w, d, h_save=True)
    e_o, e_h = check_fwd(w, x, out, label=f"{vname} f16", tol=TOL["f16"])
    assert e_h <= tol, e_h
    _check_states(w, x, out, tol)
    got = run_bwd(w, d, out["meta"], h_save=out["h_save"])
    _compare_grads(w, got, oracle_bwd(w, x), tol)


F16_TC = [("transition-split8", 1, 4096, 16), ("segmented", 1, 16384, 1), ("fused", 10, 1024, 16)]


@pytest.mark.parametrize("label,B,T,H", F16_TC, ids=[c[0] for c in F16_TC])
def test_fp16_tensor_core_plans(label, B, T, H):
    """GDN with fp16 inputs on the tensor cores in each plan it takes: the transition form at
    the 4,096-token, 16-head size (eight value slices per head), the segmented transition form
    (one 16,384-token head) and the fused plan (160 units); o and ht within the fp16 bar at the
    global, per-unit and per-row levels."""
    import chunked_gated_linear_gb300 as gcl
    w = synth.dense("f16-tc", synth.GDN, "f16", B, T, H, 128, 128, seed=64)
    x = synth.make_inputs(w)
    d = to_device(w, x)
    out = run_fwd(w, d)
    plan = gcl.fwd_plan(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], out["o"],
                        h0=d["h0"], chunk_indices=out["meta"].idx, chunk_offsets=out["meta"].off,
                        workspace=out["ws"], scale=w.scale)
    assert plan == label.split("-")[0], plan
    check_fwd(w, x, out, label=f"f16 {label}", tol=TOL["f16"])


@pytest.mark.parametrize("variant,vname", VARIANTS, ids=[v[1] for v in VARIANTS])
@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_chunk32_forward_and_backward(variant, vname, dtype):
    """BT = 32: metadata, forward (o, ht, a saved state per 32-token chunk) and backward
    (from saved and from recomputed states) against the oracle."""
    w = _w(variant, dtype, (128, 128), 32, backward=True, seed=61)
    x = synth.make_inputs(w)
    d = to_device(w, x)
    out = run_fwd(w, d, h_save=True)
    assert out["meta"].nt_max == (w.t_max + 31) // 32 + w.n_max - 1
    check_fwd(w, x, out, label=f"{vname} {dtype} bt32")
    _check_states(w, x, out)
    ref = oracle_bwd(w, x)
    tol = TOL["f32"] if dtype != "bf16" else TOL["bf16"]
    _compare_grads(w, run_bwd(w, d, out["meta"], h_save=out["h_save"]), ref, tol)
    _compare_grads(w, run_bwd(w, d, out["meta"], h_save=None), ref, tol)


@pytest.mark.parametrize("variant,vname", VARIANTS, ids=[v[1] for v in VARIANTS])
def test_chunk32_equals_chunk64(variant, vname):
    """The chunked form is exact for any chunk size: fp32 results at BT = 32 and BT = 64
    agree to fp32 rounding, and the BT = 32 chunk states are every other BT = 64 one."""
    w32 = _w(variant, "f32", (64, 64), 32, seed=62)
    w64 = _w(variant, "f32", (64, 64), 64, seed=62)
    x = synth.make_inputs(w32)
    a = run_fwd(w32, to_device(w32, x), h_save=True)
    b = run_fwd(w64, to_device(w64, x), h_save=True)
    T = w32.total_tokens
    assert relF(a["o"].cpu().numpy()[:T], b["o"].cpu().numpy()[:T]) <= TOL["f32"]
    assert relF(a["ht"].cpu().numpy(), b["ht"].cpu().numpy()) <= TOL["f32"]
    off32, off64 = a["meta"].off.cpu().numpy(), b["meta"].off.cpu().numpy()
    hs32, hs64 = a["h_save"].cpu().numpy(), b["h_save"].cpu().numpy()
    for n in range(len(LENS)):
        n64 = off64[n + 1] - off64[n]
        for i in range(n64):   # the state before 64-chunk i is the state before 32-chunk 2i
            assert relF(hs32[off32[n] + 2 * i], hs64[off64[n] + i]) <= TOL["f32"]
