"""Repetition: the tensor-core forwards, run back to back many times on one status word, never
give up a bounded wait (a give-up would set GCL_DEV_WAIT_TIMEOUT and cost the wait's time
limit), and every run returns the same outputs.  Catches barrier-phase races that a single
call rarely shows."""
import time

import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
from chunked_gated_linear_gb300 import synth  # noqa: E402
from gpu_util import Meta, run_fwd, to_device  # noqa: E402

CASES = [("gdn_fwd_bf16_T4096_H16_d128", 400), ("kda_fwd_bf16_T2048_H10_d128", 600),
         ("gdn_fwd_bf16_T65536_H1_d128", 100)]


@pytest.mark.parametrize("name,reps", CASES, ids=[c[0] for c in CASES])
def test_repeated_forwards_never_time_out(name, reps):
    w = synth.workload_by_name(name)
    x = synth.make_inputs(w)
    d = to_device(w, x)
    meta = Meta(w.t_max, w.n_max, w.bt)
    meta.build(d["cu_seqlens"])
    ref = run_fwd(w, d, meta=meta)
    torch.cuda.synchronize()
    assert int(meta.status.item()) == 0
    o_ref, ht_ref = ref["o"].clone(), ref["ht"].clone()
    ws = ref["ws"]
    import chunked_gated_linear_gb300 as gcl
    fn = gcl.kda_chunk_fwd if w.variant == synth.KDA else gcl.gdn_chunk_fwd
    args = (d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], ref["o"])
    kw = dict(h0=d.get("h0"), ht=ref["ht"], chunk_indices=meta.idx, chunk_offsets=meta.off,
              seq_order=meta.order, dev_status=meta.status, scale=w.scale, bt=w.bt, workspace=ws)
    t0 = time.perf_counter()
    for _ in range(reps):
        fn(*args, **kw)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert int(meta.status.item()) == 0, "a bounded wait gave up"
    assert elapsed < 0.15, f"{reps} forwards took {elapsed:.3f} s (a wait limit is 0.2 s)"
    assert torch.equal(ref["o"], o_ref) and torch.equal(ref["ht"], ht_ref)


@pytest.mark.parametrize("variant", [synth.GDN, synth.KDA], ids=["gdn", "kda"])
def test_repeated_backwards_never_time_out(variant):
    """The backward's tensor-core kernels (state-gradient sweep; GDN's chunk gradients) run
    back to back on one status word: no bounded wait gives up, results repeat bitwise."""
    from test_gpu_bwd import run_bwd
    w = synth.dense("stress-bwd", variant, "bf16", 2, 4096, 8, 128, 128, backward=True, seed=91)
    x = synth.make_inputs(w)
    d = to_device(w, x)
    fw = run_fwd(w, d, h_save=True)
    first = run_bwd(w, d, fw["meta"], h_save=fw["h_save"], fwd_ws=fw["ws"])
    t0 = time.perf_counter()
    for _ in range(20):
        again = run_bwd(w, d, fw["meta"], h_save=fw["h_save"], fwd_ws=fw["ws"])
    elapsed = time.perf_counter() - t0
    assert int(fw["meta"].status.item()) == 0, "a bounded wait gave up"
    assert elapsed < 2.0, f"20 backwards took {elapsed:.3f} s"
    for key in first:
        assert (first[key] == again[key]).all(), key
