"""Helpers for the GPU parity tests: move synthetic inputs to the device, call the
library through its C ABI, and compare against the fp64 oracle."""
from __future__ import annotations

import numpy as np
import torch

import chunked_gated_linear_gb300 as gcl
import oracle
from chunked_gated_linear_gb300 import synth

DEV = "cuda:0"
CANARY = 1536.0          # exact in bf16; written into output padding, must survive every call
# rel-Frobenius bounds: fp32 inputs; bf16 inputs; fp16 inputs (on the CUDA cores, fp32
# arithmetic: o is rounded to fp16 once, at most 2^-11 relative per element, so 1e-3, while ht
# and the fp32 gradients keep the fp32 bar; on the tensor cores every MMA operand is rounded to
# fp16 (unit roundoff 2^-11 = 4.9e-4): the bf16 path's errors, 0.75 and 0.6 of bf16's unit
# roundoff 2^-8 for o and ht, put fp16's near 3.7e-4 and 2.9e-4, so 1e-3 for every output)
TOL = {"f32": 1e-5, "bf16": 5e-3, "f16": 1e-3}


from parity import check as parity_check  # noqa: E402  (global, per-unit and per-row bars)
from parity import relF  # noqa: E402,F401


def tdtype(w):
    return {"bf16": torch.bfloat16, "f16": torch.float16}.get(w.dtype, torch.float32)


def to_device(w, x):
    """Device tensors for the library: q, k, v, beta, do in the workload dtype; g, h0, dht fp32."""
    dt = tdtype(w)
    d = {}
    for name in ("q", "k", "v", "beta", "do"):
        if name in x and x[name] is not None:
            d[name] = torch.from_numpy(x[name]).to(DEV).to(dt).contiguous()
    for name in ("g", "h0", "dht"):
        if name in x and x[name] is not None:
            d[name] = torch.from_numpy(x[name]).to(DEV).contiguous()
    d["cu_seqlens"] = torch.from_numpy(x["cu_seqlens"].astype(np.int32)).to(DEV)
    return d


class Meta:
    """Static metadata buffers of one capacity (T_max, N_max, BT)."""

    def __init__(self, t_max, n_max, bt=64):
        self.t_max, self.n_max, self.bt = t_max, n_max, bt
        self.nt_max = gcl.nt_max(t_max, n_max, bt)
        self.idx = torch.full((self.nt_max, 2), 77, dtype=torch.int32, device=DEV)
        self.off = torch.full((n_max + 1,), 77, dtype=torch.int32, device=DEV)
        self.order = torch.full((n_max,), 77, dtype=torch.int32, device=DEV)
        self.status = torch.full((1,), 77, dtype=torch.int32, device=DEV)

    def build(self, cu_dev, stream=None, cu_seqlens32=None):
        gcl.chunk_meta_build(cu_dev, self.t_max, self.idx, self.off, self.status,
                             seq_order=self.order, bt=self.bt, stream=stream,
                             cu_seqlens32=cu_seqlens32)


def run_fwd(w, d, meta=None, h_save=False, o_fill=CANARY, use_order=True, plan="fastest"):
    """Run chunk_meta_build + the forward for workload w on device inputs d.

    plan "fastest" hands the forward the workspace of its fastest launch plan, "min" the
    least it accepts (the W-form plan of the tensor-core path).
    Returns dict of device outputs: o, ht, h_save (if asked), plus meta."""
    if meta is None:
        meta = Meta(w.t_max, w.n_max, w.bt)
        meta.build(d["cu_seqlens"])
    o = torch.full((w.t_max, w.H, w.V), o_fill, dtype=tdtype(w), device=DEV)
    ht = torch.full((w.n_max, w.H, w.K, w.V), o_fill, dtype=torch.float32, device=DEV)
    hs = None
    if h_save:
        hs = torch.full((meta.nt_max, w.H, w.K, w.V), o_fill, dtype=torch.float32, device=DEV)
    fn = gcl.kda_chunk_fwd if w.variant == synth.KDA else gcl.gdn_chunk_fwd
    args = (d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], o)
    kw = dict(h0=d.get("h0"), ht=ht, h_save=hs, chunk_indices=meta.idx, chunk_offsets=meta.off,
              seq_order=meta.order if use_order else None, dev_status=meta.status,
              scale=w.scale, bt=w.bt)
    if w.variant == synth.KDA:
        nb = gcl.kda_fwd_workspace_bytes(*args, **kw)
    else:
        nb = (gcl.fwd_workspace_bytes if plan == "fastest" else gcl.fwd_workspace_min_bytes)(*args, **kw)
    ws = torch.full((max(nb, 16),), 0xFF, dtype=torch.uint8, device=DEV)   # stale contents
    fn(*args, workspace=ws, **kw)
    return dict(o=o, ht=ht, h_save=hs, meta=meta, ws=ws)


def oracle_fwd(w, x):
    return oracle.fwd(w.variant, x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"],
                      x["cu_seqlens"], w.scale)


def check_fwd(w, x, out, tol=None, label=""):
    """Compare device outputs against the oracle (global, per-unit and per-row bars of
    tests/parity.py); check padding canaries."""
    tol = TOL[w.dtype] if tol is None else tol
    torch.cuda.synchronize()
    assert int(out["meta"].status.item()) == 0, "device status " + str(out["meta"].status.item())
    o_ref, ht_ref = oracle_fwd(w, x)
    T = w.total_tokens
    o = out["o"].float().cpu().numpy()
    ht = out["ht"].cpu().numpy()
    assert np.isfinite(o[:T]).all(), label + " non-finite o"
    cu = np.asarray(x["cu_seqlens"], dtype=np.int64)
    e_o = parity_check(label + " o", o[:T], o_ref[:T], tol, cu=cu)[0]
    e_h = parity_check(label + " ht", ht, ht_ref, tol)[0]
    if T < w.t_max:
        pad = o[T:]
        assert (pad == np.float32(CANARY)).all(), label + " output padding was written"
    return e_o, e_h
