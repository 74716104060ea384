"""gdn_chunk_fwd_noalloc: the forward for callers that cannot allocate device memory.

It must give the same results as gdn_chunk_fwd with a caller workspace, call after
call (the static scratch keeps the previous call's contents), fall back to the W-form
plan when the transition form's records do not fit its scratch, and refuse sizes whose
minimum scratch does not fit.  This file is collected last so that a run stopping at the first
failure has already run every other test."""
import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
import chunked_gated_linear_gb300 as gcl  # noqa: E402
from chunked_gated_linear_gb300 import synth  # noqa: E402
from gpu_util import CANARY, DEV, TOL, Meta, relF, tdtype, to_device  # noqa: E402


def _outputs(w):
    o = torch.full((w.t_max, w.H, w.V), CANARY, dtype=tdtype(w), device=DEV)
    ht = torch.full((w.n_max, w.H, w.K, w.V), CANARY, dtype=torch.float32, device=DEV)
    return o, ht


def test_noalloc_matches_workspace_entry_point_on_consecutive_calls():
    w = synth.dense("noalloc", synth.GDN, "bf16", 1, 4096, 16, 128, 128, seed=77)
    T = w.total_tokens
    for call, seed in enumerate((77, 78)):           # two calls in a row, different inputs
        x = synth.make_inputs(w, seed=seed)
        d = to_device(w, x)
        meta = Meta(w.t_max, w.n_max)
        meta.build(d["cu_seqlens"])
        args = (d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"])
        kw = dict(h0=d["h0"], chunk_indices=meta.idx, chunk_offsets=meta.off,
                  seq_order=meta.order, dev_status=meta.status, scale=w.scale)
        o_ref, ht_ref = _outputs(w)
        need = gcl.fwd_workspace_min_bytes(*args, o_ref, ht=ht_ref, **kw)
        assert 0 < need <= gcl.noalloc_scratch_bytes()
        assert gcl.fwd_workspace_bytes(*args, o_ref, ht=ht_ref, **kw) > gcl.noalloc_scratch_bytes()
        ws = torch.empty(need, dtype=torch.uint8, device=DEV)
        gcl.gdn_chunk_fwd(*args, o_ref, ht=ht_ref, workspace=ws, **kw)
        o_na, ht_na = _outputs(w)
        gcl.gdn_chunk_fwd_noalloc(*args, o_na, ht=ht_na, **kw)
        torch.cuda.synchronize()
        assert int(meta.status.item()) == 0
        e_o = relF(o_na.float().cpu().numpy()[:T], o_ref.float().cpu().numpy()[:T])
        e_h = relF(ht_na.cpu().numpy(), ht_ref.cpu().numpy())
        assert e_o <= TOL["bf16"] and e_h <= TOL["bf16"], (call, e_o, e_h)
        assert np.isfinite(o_na.float().cpu().numpy()[:T]).all()


def test_noalloc_rejects_sizes_beyond_its_scratch():
    w = synth.standard_workloads()[3]                # N_max=64, T_max=65536, H=16: ~408 MiB
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
