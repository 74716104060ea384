"""bench.py's host arithmetic on CPU: the algorithmic bytes and FLOPs per step behind the
roofline fraction, the peak lookup, and the traffic record that is reported only while the
kernel sources it was measured on are unchanged."""
import hashlib
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from chunked_gated_linear_gb300 import synth  # noqa: E402


def test_algorithmic_bytes_per_token_head():
    """Per token and head: q, k, v read and o written once, beta and the gate read once
    (GDN bf16 1,030 B; KDA adds the per-channel fp32 gate: 1,538 B; fp32 K = V = 64: 1,032 B),
    plus h0 read and ht written once per (sequence, head) state of K x V fp32."""
    for w, per in ((synth.dense("a", synth.GDN, "bf16", 1, 4096, 16, 128, 128, h0=False), 1030),
                   (synth.dense("b", synth.KDA, "bf16", 1, 2048, 10, 128, 128, h0=False), 1538),
                   (synth.dense("c", synth.GDN, "f32", 1, 256, 2, 64, 64, h0=False), 1032)):
        state = w.K * w.V * 4 * w.n_max * w.H                 # ht only (no h0)
        assert bench.bytes_per_step(w) == w.total_tokens * w.H * per + state
    w = synth.dense("d", synth.GDN, "bf16", 1, 4096, 16, 128, 128)      # with h0
    assert bench.bytes_per_step(w) == 4096 * 16 * 1030 + 2 * 128 * 128 * 4 * 16
    assert bench.bytes_per_step(w) == 69_599_232        # the bench line's figure


def test_tensor_flops_per_token_head():
    """6CK + 4CV + 6KV + 2C^2/3 with C = 64, K = V = 128: about 183 kFLOP per token and head."""
    w = synth.dense("a", synth.GDN, "bf16", 1, 4096, 16, 128, 128)
    per = bench.flops_per_step(w) / (4096 * 16)
    assert per == pytest.approx(6 * 64 * 128 + 4 * 64 * 128 + 6 * 128 * 128 + 2 * 64 * 64 / 3)
    assert 182_000 < per < 184_000


def test_peaks_measured_or_fallback(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.peaks() == (bench.FALLBACK_HBM_GBS, "fallback")
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 6681.8}))
    assert bench.peaks() == (6681.8, "measured")


def test_traffic_record_follows_the_source_hash(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_record("wl") is None                     # no record file
    src = tmp_path / "k.cu"
    src.write_bytes(b"__global__ void k() {}\n")
    digest = hashlib.sha256(src.read_bytes()).hexdigest()[:16]
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.txt").write_text(
        "# comment: ignored\n\n[wl]\nkernel_sources: k.cu\n"
        f"kernel_sources_sha256_16: {digest}\nprep_dram_bytes: 1\n"
        "dram_bytes_per_launch_scaled: 12345\n\n[other]\nkernel_sources: missing.cu\n"
        "kernel_sources_sha256_16: 0\ndram_bytes_per_launch_scaled: 7\n")
    assert bench.traffic_record("wl") == 12345.0
    assert bench.traffic_record("other") is None                  # its source is missing
    assert bench.traffic_record("absent") is None
    src.write_bytes(b"__global__ void k() { /* changed */ }\n")
    assert bench.traffic_record("wl") is None                     # stale once the kernel changes


def test_roofline_takes_the_slower_roof(tmp_path, monkeypatch):
    """The roofline time is the slower of the algorithmic bytes at the HBM peak and the
    algorithmic FLOPs at the path's compute peak: the bf16 GDN forward is HBM-bound (about
    178 FLOP per byte against a ridge near 290), the fp32 CUDA-core K = V = 64 forward is bound
    by the fp32 FMA roof; frac is achieved over peak of the binding roof either way."""
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 6681.8, "bf16_tflops": 1956.7}))
    ws = {w.name: w for w in synth.standard_workloads()}
    w1 = ws["gdn_fwd_bf16_T4096_H16_d128"]
    r = bench.roofline(w1, 0.1)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] == 6681.8
    assert r["frac"] == pytest.approx(69_599_232 / 1e-4 / 1e9 / 6681.8)
    assert r["compute_time_ms"] < r["hbm_time_ms"]
    w0 = ws["gdn_fwd_fp32_T256_H2_d64"]
    r0 = bench.roofline(w0, 0.01)
    assert r0["bound"] == "alu" and r0["unit"] == "TFLOP/s"
    assert r0["frac"] == pytest.approx(bench.flops_per_step(w0) / 1e-5 / 1e12 / bench.FP32_ALU_TFLOPS)
    assert r0["compute_time_ms"] > r0["hbm_time_ms"]


def test_cpu_model_is_a_name():
    name = bench.cpu_model()
    assert isinstance(name, str) and name


def test_committed_traffic_records_are_current():
    """Every section of the committed ncu traffic summary was taken on the kernel sources now in
    the tree (its hash matches), and the bench line's workloads -- the headline and the
    per-configuration entries -- each have one; a kernel edited without a new capture fails
    here instead of silently reporting traffic: null."""
    import re
    text = open(os.path.join(ROOT, "profiles", "traffic.txt")).read()
    names = re.findall(r"^\[([^\]]+)\]$", text, flags=re.M)
    assert names
    stale = [n for n in names if bench.traffic_record(n) is None]
    assert not stale, f"traffic records taken on other kernel sources: {stale}"
    wanted = {synth.standard_workloads()[3].name, *bench.PER_CONFIG}
    assert wanted <= set(names), wanted - set(names)


def test_per_set_means_rotation_and_unreached_sets():
    """Step i runs input set i mod n: each set's mean is over its own steps, and a set that no
    timed step reached (fewer steps than sets, the small workloads' long rotations) has None,
    so the roofline averages only over sets that were timed."""
    assert bench.per_set_means([1.0, 2.0, 3.0, 5.0], 2) == [2.0, 3.5]
    assert bench.per_set_means([1.0, 2.0], 4) == [1.0, 2.0, None, None]
    assert bench.per_set_means([], 1) == [None]
