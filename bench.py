#!/usr/bin/env python
"""GDN/KDA chunk prefill throughput on GB300: tokens/s and fraction of roofline.

One step = the whole hot path over one batch: chunk_meta_build (device
metadata from cu_seqlens) followed by the chunk forward (and, for the
forward+backward workload, the backward).  Inputs are seeded synthetic data
already resident in HBM.  Several input sets are rotated so that the bytes one
step touches were evicted from L2 by the steps in between (total footprint
> 3x L2); no explicit flush is needed.

The headline workload is the varlen prefill (32 sequences of 1..2048 tokens in
a capacity of 64 slots and 65,536 tokens, 16 heads, d = 128): each input set is
one of the workload's seeded layouts, every set's step is captured once in a
CUDA graph, and the timed steps replay the graphs in rotation (graph replay,
fixed grids).  Beside it: the same steps launched directly, and
graph-update-replay (the next layout's live rows copied into the captured
buffers, then a replay), each with p50 and p95.  The other standard
configurations follow under per_config, each with its own roofline.

Prints ONE JSON line (rank 0).  Under torchrun (N > 1) every rank runs an
independent replica of the workload (weak scaling: the (sequence, head) units
are independent, there is no exchange step), timings are max-reduced.

--impl reference times the fp64 CPU oracle instead (rank 0 only) on a bounded
sample of the same workload.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from chunked_gated_linear_gb300 import synth  # noqa: E402

DEFAULT_WORKLOAD = "gdn_varlen_bf16_N32_Nmax64_Tmax65536_H16_d128"
# the other standard configurations measured in the same run, one line each under per_config
PER_CONFIG = ("gdn_fwd_fp32_T256_H2_d64", "gdn_fwd_bf16_T4096_H16_d128", "kda_fwd_bf16_T2048_H10_d128",
              "gdn_fwdbwd_bf16_B4_T8192_H16_d128")
L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="gcl", choices=["gcl", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    choices=[w.name for w in synth.standard_workloads()] +
                            [c["name"] for c in synth.conv_workloads()])
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="measure only the headline workload")
    ap.add_argument("--batch", type=int, default=0,
                    help="profiling aid: run a dense workload with this many sequences instead "
                         "of its own count (a smaller case for ncu); never for a bench line")
    return ap.parse_args()


# ----------------------------------------------------------------------------- accounting
def bytes_per_step(w) -> int:
    """Algorithmic HBM bytes of one forward launch: every input read once, o written once,
    h0 read and ht written once per (sequence, head)."""
    b = 4 if w.dtype == "f32" else 2
    th = w.total_tokens * w.H
    per_th = (2 * w.K + 2 * w.V + 1) * b + 4 * (w.K if w.variant == synth.KDA else 1)
    units = w.n_max * w.H          # ht is written for every sequence slot (ht = h0 if empty)
    state = w.K * w.V * 4 * ((1 if w.h0 else 0) + 1) * units
    return th * per_th + state


def flops_per_step(w) -> float:
    """Tensor-core FLOPs of one forward launch (chunk size 64, per token-head):
    KK^T and QK^T (2 x 2CK), W (2CK), U and L.E (2 x 2CV), WS, QS and the state update
    (3 x 2KV), solve (2C^2/3)."""
    C = 64
    per = 6 * C * w.K + 4 * C * w.V + 6 * w.K * w.V + 2 * C * C / 3
    return per * w.total_tokens * w.H


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


FALLBACK_BF16_TFLOPS = 1900.0
# fp32 FMA roof of the CUDA-core kernels: 152 SMs x 128 FP32 lanes x 2 FLOP x 2.07 GHz
FP32_ALU_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12


def bf16_peak():
    """Dense bf16 tensor-core peak (burst: the forward is timed alone, a fraction of a ms per
    launch), measured or the fallback."""
    try:
        d = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
        return float(d["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback"


def tensor_path(w) -> bool:
    """The workload's forward runs on the tensor cores: bf16 inputs (GDN and KDA), or fp16
    inputs for GDN, at d_k = d_v = 128 and chunk 64 (fp16 and bf16 share one tensor-core rate)."""
    typed = w.dtype == "bf16" or (w.dtype == "f16" and w.variant == synth.GDN)
    return typed and w.K == 128 and w.V == 128 and w.bt == 64


def roofline(w, kernel_ms, traffic=None, kind="forward"):
    """The slower of the algorithmic bytes at the measured HBM bandwidth and the algorithmic
    FLOPs at the compute peak of the path (bf16 tensor cores, or the fp32 FMA roof of the
    CUDA-core kernels) sets the roofline time; frac = that time / the measured kernel time."""
    hbm, hbm_kind = peaks()
    ab, fl = bytes_per_step(w), flops_per_step(w)
    if tensor_path(w):
        cpeak, ckind, cbound = *bf16_peak(), "tensor"
    else:
        cpeak, ckind, cbound = FP32_ALU_TFLOPS, "derived (152 SMs x 128 FP32 lanes x 2 x 2.07 GHz)", "alu"
    t_hbm = ab / (hbm * 1e9)
    t_cmp = fl / (cpeak * 1e12)
    sec = kernel_ms * 1e-3
    if t_cmp > t_hbm:
        bound, achieved, peak, unit, pkind = cbound, fl / sec / 1e12, cpeak, "TFLOP/s", ckind
    else:
        bound, achieved, peak, unit, pkind = "hbm", ab / sec / 1e9, hbm, "GB/s", hbm_kind
    return {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
            "frac": achieved / peak, "traffic": traffic, "kernel": kind, "kernel_ms": kernel_ms,
            "algorithmic_bytes_per_launch": ab, "algorithmic_flops_per_launch": fl,
            "hbm_time_ms": t_hbm * 1e3, "compute_time_ms": t_cmp * 1e3, "peak_source": pkind}


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the platform)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.processor() or platform.machine()


def traffic_record(workload: str):
    """DRAM bytes per forward call of `workload` from the committed ncu summary
    (profiles/traffic.txt, one [workload] section each), if it was taken on the current
    kernel sources (checked by hash over the listed files), else None."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    sections, cur = {}, None
    for line in open(path):
        line = line.strip()
        if line.startswith("[") and line.endswith("]"):
            cur = sections.setdefault(line[1:-1], {})
        elif cur is not None and ":" in line and not line.startswith("#"):
            k, v = line.split(":", 1)
            cur[k.strip()] = v.strip()
    kv = sections.get(workload)
    if not kv or not kv.get("kernel_sources"):
        return None
    h = hashlib.sha256()
    for src in kv["kernel_sources"].split():
        f = os.path.join(ROOT, src)
        if not os.path.exists(f):
            return None
        h.update(open(f, "rb").read())
    if h.hexdigest()[:16] != kv.get("kernel_sources_sha256_16"):
        return None
    try:
        return float(kv["dram_bytes_per_launch_scaled"])
    except (KeyError, ValueError):
        return None


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.samples = []
        self.proc = None
        self.marks = [None, None]
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(gpu_index), "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [s.strip() for s in line.split(",")]))

    def start(self):
        self.marks[0] = time.time()

    def stop(self):
        self.marks[1] = time.time()

    def summary(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        t0, t1 = self.marks
        inside = [s for (t, s) in self.samples if t0 <= t <= t1 + 0.1]
        if not inside:   # region shorter than the sampling period: nearest samples
            inside = [s for (t, s) in sorted(self.samples, key=lambda ts: abs(ts[0] - t1))[:2]]
        if not inside:
            return None
        sm = [float(s[1]) for s in inside if s[1].replace(".", "").isdigit()]
        mx = [float(s[2]) for s in inside if s[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in inside for i in range(4)
                          if len(s) > 5 + i and s[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(inside)}


# ----------------------------------------------------------------------------- GPU arm
class Runner:
    """Static device buffers for one input set plus prebuilt C-ABI argument structs."""

    def __init__(self, gcl, w, x, dev):
        import torch
        self.gcl, self.w = gcl, w
        dt = {"bf16": torch.bfloat16, "f16": torch.float16}.get(w.dtype, torch.float32)
        self.t = {}
        for n in ("q", "k", "v", "beta", "do"):
            if x.get(n) is not None:
                self.t[n] = torch.from_numpy(x[n]).to(dev).to(dt).contiguous()
        for n in ("g", "h0", "dht"):
            if x.get(n) is not None:
                self.t[n] = torch.from_numpy(x[n]).to(dev).contiguous()
        self.t["cu"] = torch.from_numpy(x["cu_seqlens"]).to(dev)
        ntm = gcl.nt_max(w.t_max, w.n_max, w.bt)
        i32 = dict(dtype=torch.int32, device=dev)
        self.t["idx"] = torch.empty((ntm, 2), **i32)
        self.t["off"] = torch.empty((w.n_max + 1,), **i32)
        self.t["order"] = torch.empty((w.n_max,), **i32)
        self.t["status"] = torch.zeros((1,), **i32)
        self.t["o"] = torch.empty((w.t_max, w.H, w.V), dtype=dt, device=dev)
        self.t["ht"] = torch.empty((w.n_max, w.H, w.K, w.V), dtype=torch.float32, device=dev)
        if w.backward:
            self.t["hs"] = torch.empty((ntm, w.H, w.K, w.V), dtype=torch.float32, device=dev)
            f32 = dict(dtype=torch.float32, device=dev)
            for n, shp in (("dq", (w.t_max, w.H, w.K)), ("dk", (w.t_max, w.H, w.K)),
                           ("dv", (w.t_max, w.H, w.V)), ("dg", tuple(x["g"].shape)),
                           ("dbeta", (w.t_max, w.H)), ("dh0", (w.n_max, w.H, w.K, w.V))):
                self.t[n] = torch.empty(shp, **f32)
        t = self.t
        self.meta_args = (t["cu"].data_ptr(), w.n_max, w.t_max, w.bt, ntm, t["idx"].data_ptr(),
                          t["off"].data_ptr(), t["order"].data_ptr(), t["status"].data_ptr())
        fargs = (t["q"], t["k"], t["v"], t["g"], t["beta"], t["cu"], t["o"])
        fkw = dict(h0=t.get("h0"), ht=t["ht"], h_save=t.get("hs"), chunk_indices=t["idx"],
                   chunk_offsets=t["off"], seq_order=t["order"], dev_status=t["status"],
                   scale=w.scale, bt=w.bt)
        wsq = gcl.kda_fwd_workspace_bytes if w.variant == synth.KDA else gcl.fwd_workspace_bytes
        t["fws"] = torch.empty(max(wsq(*fargs, **fkw), 16), dtype=torch.uint8, device=dev)
        self.fwd_args = gcl.fwd_args(*fargs, workspace=t["fws"], **fkw)
        self.fwd = gcl.lib().kda_chunk_fwd if w.variant == synth.KDA else gcl.lib().gdn_chunk_fwd
        if w.backward:
            args = (t["q"], t["k"], t["v"], t["g"], t["beta"], t["do"], t["cu"], t["idx"],
                    t["off"], t["dq"], t["dk"], t["dv"], t["dg"], t["dbeta"])
            kw = dict(h0=t.get("h0"), dht=t.get("dht"), dh0=t["dh0"], h_save=t["hs"],
                      dev_status=t["status"], scale=w.scale, bt=w.bt, fwd_workspace=t["fws"])
            nb = (gcl.kda_bwd_workspace_bytes if w.variant == synth.KDA else gcl.bwd_workspace_bytes)(*args, **kw)
            t["ws"] = torch.empty(nb, dtype=torch.uint8, device=dev)
            self.bwd_args = gcl.bwd_args(*args, workspace=t["ws"], **kw)

    def footprint(self) -> int:
        return sum(v.numel() * v.element_size() for v in self.t.values())

    def meta(self, s):
        st = self.gcl.lib().chunk_meta_build(*self.meta_args, s)
        if st:
            raise RuntimeError(self.gcl.lib().gcl_last_error().decode())

    def forward(self, s):
        st = self.fwd(ctypes.byref(self.fwd_args), s)
        if st:
            raise RuntimeError(self.gcl.lib().gcl_last_error().decode())

    def backward(self, s):
        bwd = self.gcl.lib().kda_chunk_bwd if self.w.variant == synth.KDA else self.gcl.lib().gdn_chunk_bwd
        st = bwd(ctypes.byref(self.bwd_args), s)
        if st:
            raise RuntimeError(self.gcl.lib().gcl_last_error().decode())


def reduce_max(values, dist, device):
    """Element-wise maximum over the ranks of a list of timings (the slowest replica sets the
    job's time); identity without a process group."""
    import torch
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    if dist is not None:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t]


def job_throughput(tokens_per_rank: int, world: int, ms_per_step: float) -> float:
    """Whole-job tokens/s: every rank processes its own replica (weak scaling), the step time
    is the slowest rank's."""
    return tokens_per_rank * world / (ms_per_step * 1e-3)


def fwd_plan_of(w) -> str:
    """The forward's launch plan for w's sizes with the workspace the bench gives it (the
    fastest plan's), from the library's host-side plan query (no GPU needed)."""
    import ctypes as ct
    import chunked_gated_linear_gb300 as gcl
    fake = 1 << 20                      # an aligned stand-in address: only sizes are read
    a = gcl.FwdArgs(q=fake, k=fake, v=fake, g=fake, beta=fake, cu_seqlens=fake, o=fake,
                    ht=fake, h_save=fake if w.backward else None, chunk_indices=fake,
                    chunk_offsets=fake, t_max=w.t_max, n_max=w.n_max, H=w.H, K=w.K, V=w.V,
                    bt=w.bt, scale=w.scale, dtype={"bf16": 1, "f16": 2}.get(w.dtype, 0))
    kda = w.variant == synth.KDA
    lib = gcl.lib()
    a.workspace_bytes = (lib.gcl_kda_fwd_workspace_bytes if kda else lib.gcl_fwd_workspace_bytes)(ct.byref(a))
    if a.workspace_bytes:
        a.workspace = fake
    code = (lib.gcl_kda_fwd_plan if kda else lib.gcl_fwd_plan)(ct.byref(a))
    return gcl.PLANS[int(code)]


def launches_per_step(w) -> int:
    """Library kernels per step: chunk_meta_build, the forward (the fused plan and the CUDA-core
    kernel: one launch; the W-form, transition and CUDA-core split plans: the chunk prep and the
    chain; the
    segmented plan: prep, segment summaries, scan and segment outputs) and the backward (GDN on
    the tensor cores: state-gradient sweep from the forward's records and two chunk-gradient
    kernels; otherwise the sweep and one chunk-gradient kernel)."""
    plan = fwd_plan_of(w)
    fwd = {"cuda_cores": 1, "cuda_cores_split": 2, "fused": 1, "w_form": 2, "transition": 2,
           "segmented": 4}[plan]
    tc_bwd = tensor_path(w) and w.variant == synth.GDN and w.dtype == "bf16"
    return 1 + fwd + ((3 if tc_bwd else 2) if w.backward else 0)


def pct(values, q):
    v = sorted(values)
    return v[min(len(v) - 1, max(0, int(round(q / 100.0 * (len(v) - 1)))))]


def input_sets(w, rank, dev, gcl, min_sets=2):
    """Input sets for the timed steps: the varlen workload's seeded layouts (capture layout and
    three replay layouts), else fresh seeds of the same shape; as many as keep the rotation
    above 3x L2."""
    if len(set(w.lengths)) > 1 or w.n_max > len(w.lengths):
        layouts = [synth.varlen_layout(w, s) for s in synth.layout_seeds(w)]
    else:
        layouts = [w]
    sets = []
    i = 0
    while True:
        wl = layouts[i % len(layouts)]
        seed = wl.seed + 1000 * rank + (i // len(layouts)) * 7919
        sets.append(Runner(gcl, wl, synth.make_inputs(wl, seed=seed), dev))
        i += 1
        if i >= max(min_sets, len(layouts)) and i * sets[0].footprint() > 3 * L2_BYTES:
            return sets


def per_set_means(times, n_sets):
    """Mean of the times of the steps that ran each input set (step i ran set i mod n_sets);
    None for a set that no step reached (fewer steps than sets)."""
    return [float(np.mean(times[j::n_sets])) if j < len(times) else None for j in range(n_sets)]


def measure(gcl, w, args, rank, world, dist, dev, steps, warmup, graphs=True):
    """Time one workload: direct launches (per-step and forward-kernel CUDA events, L2-cold by
    rotation), then, with graphs, the same steps captured once per input set and replayed in
    rotation (the headline), and graph-update-replay.  Returns the timings and the sets."""
    import torch
    sets = input_sets(w, rank, dev, gcl)
    n = len(sets)
    stream = torch.cuda.current_stream()
    s = ctypes.c_void_p(stream.cuda_stream)

    def step(r, ev=None, sp=None):
        sp = s if sp is None else sp
        r.meta(sp)
        if ev is not None:
            ev[0].record(stream)
        r.forward(sp)
        if ev is not None:
            ev[1].record(stream)
        if r.w.backward:
            r.backward(sp)

    for i in range(warmup):
        step(sets[i % n])
    torch.cuda.synchronize()
    for r in sets:
        assert int(r.t["status"].item()) == 0
    ev = lambda: torch.cuda.Event(enable_timing=True)
    out = {"sets": n}
    # ---- direct launches
    e_s, e_e = [ev() for _ in range(steps)], [ev() for _ in range(steps)]
    e_k = [(ev(), ev()) for _ in range(steps)]
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    for i in range(steps):
        e_s[i].record(stream)
        step(sets[i % n], e_k[i])
        e_e[i].record(stream)
    torch.cuda.synchronize()
    direct = [a.elapsed_time(b) for a, b in zip(e_s, e_e)]
    kern = [a.elapsed_time(b) for a, b in e_k]
    tok = [sets[i % n].w.total_tokens for i in range(steps)]
    out["direct"] = {"region_ms": e_s[0].elapsed_time(e_e[-1]), "p50_ms": pct(direct, 50),
                     "p95_ms": pct(direct, 95), "tokens": sum(tok)}
    # the forward kernels' time per set (its algorithmic bytes differ by layout)
    out["kernel_ms_per_set"] = per_set_means(kern, n)
    out["kernel_ms"] = float(np.mean(kern))
    if not graphs:
        return out, sets, step
    # ---- graph replay: one capture per input set, replayed in rotation
    cap = torch.cuda.Stream()
    cap.wait_stream(stream)
    gs = []
    for r in sets:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            step(r, sp=ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        gs.append(g)
    torch.cuda.synchronize()
    for i in range(3 * n):
        gs[i % n].replay()
    torch.cuda.synchronize()
    e_s, e_e = [ev() for _ in range(steps)], [ev() for _ in range(steps)]
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    for i in range(steps):
        e_s[i].record(stream)
        gs[i % n].replay()
        e_e[i].record(stream)
    torch.cuda.synchronize()
    rep = [a.elapsed_time(b) for a, b in zip(e_s, e_e)]
    out["graph"] = {"region_ms": e_s[0].elapsed_time(e_e[-1]), "p50_ms": pct(rep, 50),
                    "p95_ms": pct(rep, 95), "tokens": sum(tok)}
    # ---- graph-update-replay: the next set's live rows copied into set 0's captured buffers
    names = [k for k in ("q", "k", "v", "g", "beta", "do") if k in sets[0].t]
    small = [k for k in ("cu", "h0", "dht") if k in sets[0].t]
    reps = min(steps, 200)
    e_s, e_e = [ev() for _ in range(reps)], [ev() for _ in range(reps)]
    for i in range(reps):
        src = sets[1 + i % (n - 1)] if n > 1 else sets[0]
        live = src.w.total_tokens
        e_s[i].record(stream)
        for k in names:
            sets[0].t[k][:live].copy_(src.t[k][:live])
        for k in small:
            sets[0].t[k].copy_(src.t[k])
        gs[0].replay()
        e_e[i].record(stream)
    torch.cuda.synchronize()
    upd = [a.elapsed_time(b) for a, b in zip(e_s, e_e)]
    out["graph_update_replay"] = {"p50_ms": pct(upd, 50), "p95_ms": pct(upd, 95), "reps": reps,
                                  "copies": "live rows of " + ", ".join(names) + "; " + ", ".join(small)}
    for r in sets:
        assert int(r.t["status"].item()) == 0
    return out, sets, step


def resolve_workload(args):
    """The named workload, or (--batch) the same dense workload with another sequence count."""
    w = synth.workload_by_name(args.workload)
    if args.batch:
        if len(set(w.lengths)) != 1 or w.n_max != len(w.lengths):
            raise SystemExit("--batch applies to dense workloads only")
        w = synth.dense(f"{w.name}@batch{args.batch}", w.variant, w.dtype, args.batch,
                        w.lengths[0], w.H, w.K, w.V, h0=w.h0, backward=w.backward, seed=w.seed,
                        bt=w.bt)
    return w


def run_gpu(args, rank, world, dist):
    import torch
    import chunked_gated_linear_gb300 as gcl

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    w = resolve_workload(args)
    clocks = ClockSampler(local)
    time.sleep(0.3)
    clocks.start()
    t_wall = time.perf_counter()
    m, sets, step = measure(gcl, w, args, rank, world, dist, dev, args.steps, args.warmup)
    wall = time.perf_counter() - t_wall
    clocks.stop()
    K = args.steps
    # the headline: graph replay of the captured steps, max over ranks
    tot = reduce_max([m["graph"]["region_ms"], m["direct"]["region_ms"], m["kernel_ms"]], dist, dev)
    ms_step, ms_direct, ms_kern = tot[0] / K, tot[1] / K, tot[2]
    tokens = m["graph"]["tokens"] / K                       # per step, averaged over layouts
    value = tokens * world / (ms_step * 1e-3)
    n = m["sets"]
    # roofline of the forward kernels: each set's algorithmic bytes over its kernel time
    fw = [r.w for r in sets]
    rl = [roofline(x, km, kind=fwd_plan_of(x)) for x, km in zip(fw, m["kernel_ms_per_set"])
          if km is not None]
    roof = roofline_mean(rl, ms_kern, traffic_record(w.name))
    util = [int(r.t["off"][-1].item()) / gcl.nt_max(x.t_max, x.n_max, x.bt) for r, x in zip(sets, fw)]
    e2e = run_e2e(gcl, sets[:2], torch.cuda.current_stream(),
                  ctypes.c_void_p(torch.cuda.current_stream().cuda_stream), args.e2e_steps, world,
                  dist)
    clk = clocks.summary()
    per = {}
    if not args.no_per_config and world == 1:
        for name in PER_CONFIG:
            if name == w.name:
                continue
            wc = synth.workload_by_name(name)
            mc, sc, _ = measure(gcl, wc, args, rank, world, dist, dev, max(50, min(K, 300)),
                                max(args.warmup, 3), graphs=False)
            km = mc["kernel_ms"]
            per[name] = {"ms_per_step": mc["direct"]["region_ms"] / max(50, min(K, 300)),
                         "p50_ms": mc["direct"]["p50_ms"], "p95_ms": mc["direct"]["p95_ms"],
                         "tokens_per_step": wc.total_tokens,
                         "value": wc.total_tokens / (mc["direct"]["region_ms"] / max(50, min(K, 300)) * 1e-3),
                         "unit": "tokens/s", "plan": fwd_plan_of(wc),
                         "roofline": roofline(wc, km, traffic_record(name), kind=fwd_plan_of(wc))}
            del sc
            torch.cuda.empty_cache()
    if rank != 0:
        return None
    line = {
        "metric": "GDN/KDA chunk prefill tokens/s on 1 GB300 and % of roofline (HBM/TC)",
        "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic (seeded PCG64; q,k L2-normalised N(0,1), v N(0,1), "
                "beta=sigmoid(N), g=-softplus(N), h0 N(0,0.1^2); varlen layouts from seeded "
                "uniform lengths)",
        "config": {"workload": w.name, "tokens_per_step": tokens, "heads": w.H,
                   "d_k": w.K, "d_v": w.V, "chunk": w.bt, "n_max": w.n_max,
                   "t_max": w.t_max, "parallelism": f"replicas x{world}", "plan": fwd_plan_of(w),
                   "timing": "CUDA-graph replay of each input set's captured step, in rotation",
                   "l2": f"rotating {n} input sets ({n * sets[0].footprint() / 2**20:.0f} MiB, "
                         f"> 3x L2); no flush",
                   "host_wall_s": wall},
        "roofline": roof,
        "e2e": e2e,
        "timing": {"graph_replay": m["graph"], "direct": m["direct"],
                   "graph_update_replay": m["graph_update_replay"],
                   "direct_ms_per_step": ms_direct,
                   "chunk_utilisation": float(np.mean(util)),
                   "chunk_utilisation_per_layout": util,
                   "tokens_per_layout": [x.total_tokens for x in fw]},
        "per_config": per,
        "gpu_launches": K * launches_per_step(w),
        "clocks": clk,
    }
    return line


def roofline_mean(rl, kernel_ms, traffic):
    """One roofline object for rotating sets: algorithmic bytes and FLOPs averaged over the
    sets, against the mean forward-kernel time."""
    n = len(rl)
    r0 = dict(rl[0])
    ab = sum(r["algorithmic_bytes_per_launch"] for r in rl) / n
    fl = sum(r["algorithmic_flops_per_launch"] for r in rl) / n
    t_hbm = sum(r["hbm_time_ms"] for r in rl) / n
    t_cmp = sum(r["compute_time_ms"] for r in rl) / n
    if r0["bound"] == "hbm":
        achieved = ab / (kernel_ms * 1e-3) / 1e9
    else:
        achieved = fl / (kernel_ms * 1e-3) / 1e12
    r0.update(achieved=achieved, frac=achieved / r0["peak"], traffic=traffic, kernel_ms=kernel_ms,
              algorithmic_bytes_per_launch=ab, algorithmic_flops_per_launch=fl,
              hbm_time_ms=t_hbm, compute_time_ms=t_cmp)
    return r0


def run_e2e(gcl, runners, stream, s, steps, world, dist):
    """Same metric through the public C-ABI calls with pinned host buffers: per step the H2D
    copy of the live rows of every token input (and cu_seqlens, h0), meta + forward (+ backward),
    and the D2H copy of the live rows of o and of ht.  Steps are pipelined over two device input
    sets and three streams: step i+1's inputs are copied in and step i-1's results copied out
    while step i's kernels run; a set's buffers are rewritten only after its previous step's
    kernels and result copies are done.  The timed region runs from the first timed step's H2D
    to the last timed step's D2H (every copy of every timed step inside it)."""
    import torch
    sets = []
    for r in runners:
        w = r.w
        live = w.total_tokens
        names = [n for n in ("q", "k", "v", "g", "beta", "do") if n in r.t]
        small = [n for n in ("h0", "dht", "cu") if n in r.t]
        host = {n: torch.empty_like(r.t[n][:live], device="cpu").pin_memory() for n in names}
        host.update({n: torch.empty_like(r.t[n], device="cpu").pin_memory() for n in small})
        for n in names:
            host[n].copy_(r.t[n][:live])
        for n in small:
            host[n].copy_(r.t[n])
        out_h = {"o": torch.empty_like(r.t["o"][:live], device="cpu").pin_memory(),
                 "ht": torch.empty_like(r.t["ht"], device="cpu").pin_memory()}
        sets.append((r, live, names, small, host, out_h))
    h2d = [sum(x[4][n].numel() * x[4][n].element_size() for n in x[4]) for x in sets]
    d2h = [sum(x[5][n].numel() * x[5][n].element_size() for n in x[5]) for x in sets]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event(enable_timing=True)
    warm = 3
    total = warm + steps
    e_in, e_comp, e_out = [ev() for _ in range(total)], [ev() for _ in range(total)], [ev() for _ in range(total)]
    e_start = ev()
    R = len(sets)
    torch.cuda.synchronize()
    tokens = 0
    for i in range(total):
        r, live, names, small, host, out_h = sets[i % R]
        if i >= R:          # this set's buffers: its previous step's kernels and copies are done
            s_in.wait_event(e_comp[i - R])
            s_in.wait_event(e_out[i - R])
        if i == warm:
            e_start.record(s_in)
        with torch.cuda.stream(s_in):
            for n in names:
                r.t[n][:live].copy_(host[n], non_blocking=True)
            for n in small:
                r.t[n].copy_(host[n], non_blocking=True)
        e_in[i].record(s_in)
        stream.wait_event(e_in[i])
        r.meta(s)
        r.forward(s)
        if r.w.backward:
            r.backward(s)
        e_comp[i].record(stream)
        s_out.wait_event(e_comp[i])
        with torch.cuda.stream(s_out):
            out_h["o"].copy_(r.t["o"][:live], non_blocking=True)
            out_h["ht"].copy_(r.t["ht"], non_blocking=True)
        e_out[i].record(s_out)
        if i >= warm:
            tokens += live
    torch.cuda.synchronize()
    per = [e_in[i - 1].elapsed_time(e_in[i]) for i in range(warm + 1, total)] or [0.0]
    region = e_start.elapsed_time(e_out[total - 1])
    ms = reduce_max([region / steps], dist, sets[0][0].t["q"].device)[0]
    return {"value": (tokens / steps) * world / (ms * 1e-3), "unit": "tokens/s",
            "h2d_bytes_per_step": int(np.mean(h2d)), "d2h_bytes_per_step": int(np.mean(d2h)),
            "ms_per_step": ms, "p50_ms": pct(per, 50), "p95_ms": pct(per, 95),
            "pipeline": f"{R} input sets, H2D / kernels / D2H on three streams"}


# ----------------------------------------------------------------------------- CPU oracle
def oracle_sample(w, x, heads, tokens, seqs=None):
    """The oracle on the first `tokens` tokens of every sequence (of the first `seqs`
    sequences, if given) and the first `heads` heads; returns (seconds, token-heads
    processed)."""
    import oracle
    cu = x["cu_seqlens"].astype(np.int64)
    nseq = len(cu) - 1 if seqs is None else min(seqs, len(cu) - 1)
    rows = []
    new_cu = [0]
    for n in range(nseq):
        s, e = int(cu[n]), int(min(cu[n + 1], cu[n] + tokens))
        rows.append(np.arange(s, e))
        new_cu.append(new_cu[-1] + (e - s))
    rows = np.concatenate(rows) if rows else np.zeros(0, dtype=np.int64)
    sl = {n: x[n][rows][:, :heads] for n in ("q", "k", "v", "g", "beta")}
    h0 = None if x["h0"] is None else x["h0"][:nseq, :heads]
    t0 = time.perf_counter()
    oracle.fwd(w.variant, sl["q"], sl["k"], sl["v"], sl["g"], sl["beta"], h0, new_cu, w.scale)
    return time.perf_counter() - t0, len(rows) * heads


def cpu_baseline(w, x, budget_s=12.0):
    import oracle
    heads = w.H
    dt, th = oracle_sample(w, x, heads, 64)          # calibration
    rate = th / max(dt, 1e-6)
    tokens = int(min(max(64, budget_s * rate / max(heads * len(w.lengths), 1)),
                     max(w.lengths)))
    dt, th = oracle_sample(w, x, heads, tokens)
    # the whole workload takes less than the budget: run it again until the budget is spent
    reps = 1
    while dt < 0.8 * budget_s and reps < 500:
        d2, t2 = oracle_sample(w, x, heads, tokens)
        dt += d2
        th += t2
        reps += 1
    line = {"value": th / w.H / dt, "unit": "tokens/s",
            "cores": min(oracle.num_threads(), heads * len(w.lengths)), "kind": "oracle",
            "cpu_model": cpu_model(), "host_threads": os.cpu_count(),
            "sample": f"fp64 token recurrence, first {tokens} tokens of every sequence, all "
                      f"{heads} heads, {reps} run(s) ({th} token-heads, {dt:.1f} s)"}
    # the same oracle on one (sequence, head) unit: one host thread, about 3 s
    if w.lengths and w.lengths[0] > 0:
        d1, t1 = oracle_sample(w, x, 1, 64, seqs=1)
        tok1 = int(min(max(64, 3.0 * t1 / max(d1, 1e-6)), w.lengths[0]))
        d1, t1 = oracle_sample(w, x, 1, tok1, seqs=1)
        reps1 = 1
        while d1 < 2.4 and reps1 < 500:
            d2, t2 = oracle_sample(w, x, 1, tok1, seqs=1)
            d1 += d2
            t1 += t2
            reps1 += 1
        line["single_thread"] = {
            "value": t1 / w.H / d1, "unit": "tokens/s", "cores": 1,
            "sample": f"first {tok1} tokens of sequence 0, head 0, {reps1} run(s) "
                      f"({t1} token-heads, {d1:.1f} s), per token of all {w.H} heads"}
    return line


def run_reference(args):
    import oracle
    oracle.build()
    w = synth.workload_by_name(args.workload)
    x = synth.make_inputs(w)
    heads = max(1, min(w.H, oracle.num_threads()))      # one (sequence, head) unit per host thread
    dt, th = oracle_sample(w, x, heads, 64)
    per_th = dt / max(th, 1)
    budget = 120.0 / max(args.steps + args.warmup, 1)    # whole run within ~2 minutes
    tokens = int(min(max(1, budget / per_th / max(len(w.lengths), 1)), max(w.lengths)))
    for _ in range(args.warmup):
        oracle_sample(w, x, heads, tokens)
    times = []
    th = 0
    for _ in range(args.steps):
        dt, th = oracle_sample(w, x, heads, tokens)
        times.append(dt)
    sec = float(np.mean(times))
    value = th / sec / w.H               # token-heads/s over H: tokens/s of the full workload
    sample = (f"fp64 token recurrence on host cores, per step the first {tokens} tokens of "
              f"every sequence for {heads} of {w.H} heads, scaled to all heads")
    return {
        "impl": "reference",
        "metric": "GDN/KDA chunk prefill tokens/s on 1 GB300 and % of roofline (HBM/TC)",
        "value": value, "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "tokens_per_step": w.total_tokens, "heads": w.H},
        "cpu_baseline": {"value": value, "unit": "tokens/s",
                         "cores": min(oracle.num_threads(), heads * len(w.lengths)),
                         "kind": "oracle", "sample": sample, "cpu_model": cpu_model()},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


# ----------------------------------------------------------------------------- causal_conv1d
CONV_METRIC = "causal_conv1d fwd+bwd tokens/s on 1 GB300 and % of HBM roofline"


def conv_bytes(c):
    """Algorithmic HBM bytes of one forward and one backward call: forward reads x and writes
    y (and h0 -> ht); backward reads x and dy, writes dx (fp32) and dw, db, dh0."""
    b = 2 if c["dtype"] == "bf16" else 4
    T, D, W, N = c["B"] * c["T"], c["D"], c["W"], c["B"]
    state = N * D * (W - 1)
    fwd = T * D * 2 * b + D * (W + 1) * b + 2 * state * b
    bwd = T * D * (2 * b + 4) + D * (W + 1) * (b + 4) + state * (b + 4 + 4)
    return fwd, bwd


def run_conv_gpu(args, rank, world, dist):
    import torch
    import chunked_gated_linear_gb300 as gcl

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    c = synth.conv_workload_by_name(args.workload)
    B, T, D, W = c["B"], c["T"], c["D"], c["W"]
    tm = B * T
    x = synth.make_conv_inputs([T] * B, B, tm, D, W, c["dtype"], seed=c["seed"] + 1000 * rank)
    td = torch.bfloat16 if c["dtype"] == "bf16" else torch.float32
    t = {k: torch.from_numpy(v).to(dev).to(td) for k, v in x.items()
         if v is not None and k not in ("cu_seqlens", "dht")}
    t["cu"] = torch.from_numpy(x["cu_seqlens"]).to(dev)
    t["dht"] = torch.from_numpy(x["dht"]).to(dev)
    ntm = gcl.nt_max(tm, B, 64)
    i32 = dict(dtype=torch.int32, device=dev)
    f32 = dict(dtype=torch.float32, device=dev)
    t.update(idx=torch.empty((ntm, 2), **i32), off=torch.empty((B + 1,), **i32),
             status=torch.zeros((1,), **i32), y=torch.empty((tm, D), dtype=td, device=dev),
             ht=torch.empty((B, D, W - 1), dtype=td, device=dev), dx=torch.empty((tm, D), **f32),
             dw=torch.empty((D, W), **f32), db=torch.empty((D,), **f32),
             dh0=torch.empty((B, D, W - 1), **f32))
    common = (t["x"], t["weight"], t["cu"], t["idx"])
    kw = dict(bias=t.get("bias"), h0=t.get("h0"), dev_status=t["status"], activation=c["act"])
    fa = gcl.conv_args(*common, y=t["y"], ht=t["ht"], **kw)
    bkw = dict(dy=t["dy"], dht=t["dht"], dx=t["dx"], dweight=t["dw"], dbias=t["db"], dh0=t["dh0"], **kw)
    t["ws"] = torch.empty(gcl.causal_conv1d_bwd_workspace_bytes(*common, **bkw), dtype=torch.uint8,
                          device=dev)
    ba = gcl.conv_args(*common, workspace=t["ws"], **bkw)
    lib = gcl.lib()
    meta_args = (t["cu"].data_ptr(), B, tm, 64, ntm, t["idx"].data_ptr(), t["off"].data_ptr(),
                 None, t["status"].data_ptr())
    stream = torch.cuda.current_stream()
    s = ctypes.c_void_p(stream.cuda_stream)

    def step(ev=None):
        if lib.chunk_meta_build(*meta_args, s) != 0:
            raise RuntimeError(gcl.lib().gcl_last_error().decode())
        if ev is not None:
            ev[0].record(stream)
        if lib.causal_conv1d_fwd(ctypes.byref(fa), s) != 0:
            raise RuntimeError(gcl.lib().gcl_last_error().decode())
        if ev is not None:
            ev[1].record(stream)
        if lib.causal_conv1d_bwd(ctypes.byref(ba), s) != 0:
            raise RuntimeError(gcl.lib().gcl_last_error().decode())
        if ev is not None:
            ev[2].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert int(t["status"].item()) == 0
    clocks = ClockSampler(local)
    time.sleep(0.3)
    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    for i in range(K):
        ev[i][0].record(stream)
        step(ev[i][1:])
        ev[i][3].record(stream)
    torch.cuda.synchronize()
    clocks.stop()
    if dist is not None:
        dist.barrier()
    tot = reduce_max([ev[0][0].elapsed_time(ev[-1][3]), sum(e[1].elapsed_time(e[2]) for e in ev),
                      sum(e[2].elapsed_time(e[3]) for e in ev)], dist, dev)
    ms_step, ms_fwd, ms_bwd = (v / K for v in tot)   # step: the whole bracketed region
    e2e = conv_e2e(torch, lib, t, x, fa, ba, step, stream, args.e2e_steps, world, dist, tm)
    clk = clocks.summary()
    if rank != 0:
        return None
    peak, peak_kind = peaks()
    fb, bb = conv_bytes(c)
    return {
        "metric": CONV_METRIC, "value": job_throughput(tm, world, ms_step), "unit": "tokens/s",
        "n_gpus": world, "steps": K, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": c["dtype"],
        "data": "synthetic (seeded PCG64; x, dy N(0,1), weight N(0,1/W), bias N(0,0.1^2), "
                "h0 N(0,1), dht N(0,0.1^2))",
        "config": {"workload": c["name"], "tokens_per_step": tm, "channels": D, "taps": W,
                   "activation": c["act"], "parallelism": f"replicas x{world}",
                   "l2": f"inputs {2 * tm * D * (2 if c['dtype'] == 'bf16' else 4) / 2**20:.0f} MiB "
                         f"per step (> L2); no flush"},
        "roofline": {"bound": "hbm", "achieved": bb / (ms_bwd * 1e-3) / 1e9, "peak": peak,
                     "unit": "GB/s", "frac": bb / (ms_bwd * 1e-3) / 1e9 / peak,
                     "traffic": traffic_record(c["name"]), "kernel": "causal_conv1d_bwd",
                     "kernel_ms": ms_bwd, "algorithmic_bytes_per_launch": bb, "peak_source": peak_kind},
        "roofline_fwd": {"bound": "hbm", "achieved": fb / (ms_fwd * 1e-3) / 1e9, "peak": peak,
                         "unit": "GB/s", "frac": fb / (ms_fwd * 1e-3) / 1e9 / peak,
                         "kernel": "causal_conv1d_fwd", "kernel_ms": ms_fwd,
                         "algorithmic_bytes_per_launch": fb},
        "e2e": e2e,
        "gpu_launches": K * 4,
        "clocks": clk,
    }


def conv_e2e(torch, lib, t, x, fa, ba, step, stream, steps, world, dist, tm):
    """The conv step through the C ABI with pinned host buffers: H2D of x, dy (and the small
    weight, bias, h0, dht, cu_seqlens) each step, D2H of y and dx."""
    names = [n for n in ("x", "weight", "bias", "h0", "dy", "dht", "cu") if n in t]
    host = {n: torch.empty_like(t[n], device="cpu").pin_memory() for n in names}
    for n in names:
        host[n].copy_(t[n])
    out_h = {n: torch.empty_like(t[n], device="cpu").pin_memory() for n in ("y", "dx")}
    h2d = sum(host[n].numel() * host[n].element_size() for n in names)
    d2h = sum(out_h[n].numel() * out_h[n].element_size() for n in out_h)
    times = []
    for i in range(steps + 3):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for n in names:
            t[n].copy_(host[n], non_blocking=True)
        step()
        for n in out_h:
            out_h[n].copy_(t[n], non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        if i >= 3:
            times.append(e0.elapsed_time(e1))
    ms = reduce_max([float(np.mean(times))], dist, t["x"].device)[0]
    return {"value": job_throughput(tm, world, ms), "unit": "tokens/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms}


def conv_oracle_sample(c, x, tokens):
    """The conv oracle (forward and backward) on the first `tokens` tokens of every sequence;
    returns (seconds, tokens processed)."""
    import oracle
    cu = x["cu_seqlens"].astype(np.int64)
    rows, new_cu = [], [0]
    for n in range(len(cu) - 1):
        st, en = int(cu[n]), int(min(cu[n + 1], cu[n] + tokens))
        rows.append(np.arange(st, en))
        new_cu.append(new_cu[-1] + (en - st))
    rows = np.concatenate(rows)
    xs, dys = x["x"][rows], x["dy"][rows]
    t0 = time.perf_counter()
    oracle.conv_fwd(xs, x["weight"], x["bias"], None, x["h0"], new_cu, activation=c["act"])
    oracle.conv_bwd(xs, x["weight"], x["bias"], x["h0"], new_cu, dys, x["dht"], activation=c["act"])
    return time.perf_counter() - t0, len(rows)


def conv_cpu_baseline(c, budget_s=12.0):
    x = synth.make_conv_inputs([c["T"]] * c["B"], c["B"], c["B"] * c["T"], c["D"], c["W"],
                               c["dtype"], seed=c["seed"])
    dt, n = conv_oracle_sample(c, x, 16)                  # calibration
    tokens = int(min(max(16, budget_s * n / max(dt, 1e-6) / c["B"]), c["T"]))
    dt, n = conv_oracle_sample(c, x, tokens)
    reps = 1
    while dt < 0.8 * budget_s and reps < 50:             # the whole workload fits: repeat it
        d2, n2 = conv_oracle_sample(c, x, tokens)
        dt, n, reps = dt + d2, n + n2, reps + 1
    return {"value": n / dt, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"fp64 numpy forward + backward, first {tokens} tokens of every sequence, "
                      f"all {c['D']} channels, {reps} run(s) ({n} tokens, {dt:.1f} s)"}


def run_conv_reference(args):
    c = synth.conv_workload_by_name(args.workload)
    x = synth.make_conv_inputs([c["T"]] * c["B"], c["B"], c["B"] * c["T"], c["D"], c["W"],
                               c["dtype"], seed=c["seed"])
    dt, n = conv_oracle_sample(c, x, 16)
    budget = 120.0 / max(args.steps + args.warmup, 1)
    tokens = int(min(max(1, budget * n / max(dt, 1e-6) / c["B"]), c["T"]))
    for _ in range(args.warmup):
        conv_oracle_sample(c, x, tokens)
    times = []
    for _ in range(args.steps):
        dt, n = conv_oracle_sample(c, x, tokens)
        times.append(dt)
    sec = float(np.mean(times))
    value = n / sec
    sample = (f"fp64 numpy forward + backward on one host core, per step the first {tokens} "
              f"tokens of every sequence, all {c['D']} channels")
    return {
        "impl": "reference", "metric": CONV_METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": c["name"], "tokens_per_step": c["B"] * c["T"]},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    conv = args.workload in [c["name"] for c in synth.conv_workloads()]
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_conv_reference(args) if conv else run_reference(args)), flush=True)
        return
    dist = None
    if world > 1:
        import torch
        import torch.distributed as dist_
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist_.init_process_group("nccl")
        dist = dist_
    line = run_conv_gpu(args, rank, world, dist) if conv else run_gpu(args, rank, world, dist)
    if rank == 0:
        if world > 1:
            line["cpu_baseline"] = None      # the oracle is timed at one GPU only
        elif not args.no_cpu_baseline:
            if conv:
                line["cpu_baseline"] = conv_cpu_baseline(synth.conv_workload_by_name(args.workload))
            else:
                w = resolve_workload(args)
                line["cpu_baseline"] = cpu_baseline(w, synth.make_inputs(w))
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
