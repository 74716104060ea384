"""gdn_chunk_fwd_noalloc: the forward for callers that cannot allocate device memory.

It must give bitwise the same results as gdn_chunk_fwd with a caller workspace that selects
the same plan, call after call (the static scratch keeps the previous call's contents), in
each of the plans its scratch can hold (W form, transition form, segmented transition form),
and refuse sizes whose minimum scratch does not fit.  This file is collected last so that a run stopping at the first
failure has already run every other test."""
import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
import chunked_gated_linear_gb300 as gcl  # noqa: E402
from chunked_gated_linear_gb300 import synth  # noqa: E402
from gpu_util import CANARY, DEV, Meta, check_fwd, tdtype, to_device  # noqa: E402


def _outputs(w):
    o = torch.full((w.t_max, w.H, w.V), CANARY, dtype=tdtype(w), device=DEV)
    ht = torch.full((w.n_max, w.H, w.K, w.V), CANARY, dtype=torch.float32, device=DEV)
    return o, ht


# (label, B, T, H, whether the fastest plan's scratch fits the static array): the W form
# (4,096 tokens x 16 heads: its transition records would need 96 MiB), the transition form
# (1,024 x 16: 24 MiB of records) and the segmented transition form (one 16,384-token head:
# 24 MiB of records and the segment buffers after them).
PLANS = [("wform", 1, 4096, 16, False), ("transition", 1, 1024, 16, True),
         ("segmented", 1, 16384, 1, True)]


@pytest.mark.parametrize("label,B,T,H,fastest_fits", PLANS, ids=[p[0] for p in PLANS])
def test_noalloc_matches_workspace_entry_point_on_consecutive_calls(label, B, T, H, fastest_fits):
    """Two calls in a row with different inputs: each bitwise equal to gdn_chunk_fwd given a
    caller workspace that selects the same plan (the static scratch keeps the previous call's
    contents, which must not matter), and within the bf16 bar of the oracle."""
    w = synth.dense("noalloc-" + label, synth.GDN, "bf16", B, T, H, 128, 128, seed=77)
    nt = w.total_tokens
    for call, seed in enumerate((77, 78)):
        x = synth.make_inputs(w, seed=seed)
        d = to_device(w, x)
        meta = Meta(w.t_max, w.n_max)
        meta.build(d["cu_seqlens"])
        args = (d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"])
        kw = dict(h0=d["h0"], chunk_indices=meta.idx, chunk_offsets=meta.off,
                  seq_order=meta.order, dev_status=meta.status, scale=w.scale)
        o_ref, ht_ref = _outputs(w)
        need_min = gcl.fwd_workspace_min_bytes(*args, o_ref, ht=ht_ref, **kw)
        need_fast = gcl.fwd_workspace_bytes(*args, o_ref, ht=ht_ref, **kw)
        cap = gcl.noalloc_scratch_bytes()
        assert 0 < need_min <= cap
        assert (need_fast <= cap) == fastest_fits
        # the plan the static scratch selects: the fastest one whose scratch fits
        ws = torch.empty(need_fast if fastest_fits else need_min, dtype=torch.uint8, device=DEV)
        gcl.gdn_chunk_fwd(*args, o_ref, ht=ht_ref, workspace=ws, **kw)
        o_na, ht_na = _outputs(w)
        gcl.gdn_chunk_fwd_noalloc(*args, o_na, ht=ht_na, **kw)
        torch.cuda.synchronize()
        assert int(meta.status.item()) == 0
        assert torch.equal(o_na, o_ref), (label, call, "o differs from gdn_chunk_fwd")
        assert torch.equal(ht_na, ht_ref), (label, call, "ht differs from gdn_chunk_fwd")
        if call == 0:
            check_fwd(w, x, dict(o=o_na, ht=ht_na, meta=meta), label="noalloc " + label)
        else:
            assert np.isfinite(o_na.float().cpu().numpy()[:nt]).all()


def test_noalloc_rejects_sizes_beyond_its_scratch():
    # one 65,536-token sequence of 16 heads: 16 units run the plans with per-chunk scratch,
    # the least of which (W form) needs 400 MiB
    w = synth.dense("noalloc-big", synth.GDN, "bf16", 1, 65536, 16, 128, 128, seed=79)
    x = synth.make_inputs(w)
    d = to_device(w, x)
    meta = Meta(w.t_max, w.n_max)
    o, ht = _outputs(w)
    a = gcl.fwd_args(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], o, ht=ht,
                     chunk_indices=meta.idx, chunk_offsets=meta.off, dev_status=meta.status,
                     scale=w.scale)
    assert gcl.lib().gcl_fwd_workspace_min_bytes(ctypes.byref(a)) > gcl.noalloc_scratch_bytes()
    st = gcl.lib().gdn_chunk_fwd_noalloc(ctypes.byref(a), None)
    assert st == 3                                   # GCL_ERR_CAPACITY, nothing enqueued
    assert b"static scratch" in gcl.lib().gcl_last_error()
