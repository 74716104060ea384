"""The bounds-checking debug build (libgcl_debug.so, GCL_DEBUG_BOUNDS) on the small and
ragged shapes: every plan and kernel family runs with each checked index tested against its
buffer; the status word must stay 0 (no index fell outside) and the results must match the
oracle as in the release build."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
import chunked_gated_linear_gb300 as gcl  # noqa: E402
from chunked_gated_linear_gb300 import synth  # noqa: E402
from gpu_util import TOL, check_fwd, run_fwd, to_device  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def debug_library():
    """Route every call of this module through the debug build, then restore the release one."""
    import os
    if not os.path.exists(gcl.DEBUG_LIB_PATH):
        pytest.fail("libgcl_debug.so not built (__graft_entry__.build() builds it)")
    saved = gcl._lib
    gcl._lib = gcl.load_library(gcl.DEBUG_LIB_PATH)
    yield
    gcl._lib = saved


SHAPES = {"T<=8": [1, 5, 8], "T=65": [65], "ragged": [1, 63, 0, 64, 65, 200], "empty": [0, 0]}


@pytest.mark.parametrize("shape", list(SHAPES), ids=list(SHAPES))
@pytest.mark.parametrize("case", ["gdn-bf16-fastest", "gdn-bf16-wform", "gdn-bf16-fused",
                                  "kda-bf16", "gdn-f32-d64", "kda-f32-d64"])
def test_forward_in_bounds(case, shape):
    lens = SHAPES[shape]
    variant = synth.KDA if case.startswith("kda") else synth.GDN
    dtype = "f32" if "f32" in case else "bf16"
    K = 64 if "d64" in case else 128
    H = 20 if case.endswith("fused") else 2                  # 20 heads x slots >= SMs: fused
    n_max = 8 if case.endswith("fused") else len(lens)
    w = synth.varlen("dbg", variant, dtype, lens, n_max, max(sum(lens), 1) + 24, H, K, K, seed=61)
    x = synth.make_inputs(w)
    out = run_fwd(w, to_device(w, x), h_save=True,
                  plan="min" if case.endswith(("wform", "fused")) else "fastest")
    check_fwd(w, x, out, label=f"debug {case} {shape}")      # asserts status 0 first


def test_segmented_forward_in_bounds():
    """One 16,384-token sequence of one head: the segment-parallel chain (summaries, scan,
    outputs)."""
    w = synth.dense("dbg-seg", synth.GDN, "bf16", 1, 16384, 1, 128, 128, seed=62)
    assert gcl.fwd_chain_segments(w.t_max, w.n_max, w.H) > 0
    x = synth.make_inputs(w)
    check_fwd(w, x, run_fwd(w, to_device(w, x)), label="debug segmented")


@pytest.mark.parametrize("case", ["gdn-bf16", "kda-bf16", "gdn-f32-d64"])
@pytest.mark.parametrize("saved", [True, False], ids=["saved", "recomputed"])
def test_backward_in_bounds(case, saved):
    from test_gpu_bwd import compare, oracle_bwd, run_bwd
    lens = [1, 63, 0, 64, 65, 150]
    variant = synth.KDA if case.startswith("kda") else synth.GDN
    dtype = "f32" if "f32" in case else "bf16"
    K = 64 if "d64" in case else 128
    w = synth.varlen("dbg-bwd", variant, dtype, lens, 7, sum(lens) + 20, 2, K, K,
                     backward=True, seed=63)
    x = synth.make_inputs(w)
    d = to_device(w, x)
    fw = run_fwd(w, d, h_save=saved)
    got = run_bwd(w, d, fw["meta"], h_save=fw["h_save"])     # asserts status 0
    compare(w, got, oracle_bwd(w, x), TOL[dtype])
    assert np.isfinite(got["dq"][:w.total_tokens]).all()
