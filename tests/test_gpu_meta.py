"""chunk_meta_build on the GPU: bit-exact against the oracle's plain loops."""
import json
import os

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
import oracle  # noqa: E402
from gpu_util import DEV, Meta  # noqa: E402

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def expected_order(cu):
    lens = np.diff(np.asarray(cu, dtype=np.int64))
    return np.argsort(-lens, kind="stable").astype(np.int32)


def run(cu, t_max, bt=64, meta=None):
    meta = meta or Meta(t_max, len(cu) - 1, bt)
    cu_d = torch.tensor(cu, dtype=torch.int32, device=DEV)
    meta.build(cu_d)
    torch.cuda.synchronize()
    return meta


def check(meta, cu, t_max, bt):
    st, idx, off = oracle.chunk_meta(cu, t_max, bt)
    assert int(meta.status.item()) == st
    np.testing.assert_array_equal(meta.idx.cpu().numpy(), idx)
    np.testing.assert_array_equal(meta.off.cpu().numpy(), off)
    order = meta.order.cpu().numpy()
    if st == 0:
        np.testing.assert_array_equal(order, expected_order(cu))
    else:
        np.testing.assert_array_equal(order, np.arange(len(cu) - 1))


def test_golden_cases():
    d = json.load(open(os.path.join(GOLDEN, "chunk_meta_examples.json")))
    for c in d["cases"]:
        m = run(c["cu_seqlens"], c["t_max"], c["bt"])
        assert int(m.status.item()) == c["status"], c["note"]
        assert m.idx.cpu().tolist() == c["chunk_indices"], c["note"]
        assert m.off.cpu().tolist() == c["chunk_offsets"], c["note"]
        check(m, c["cu_seqlens"], c["t_max"], c["bt"])


def test_random_layouts_bit_exact():
    rng = np.random.default_rng(1)
    for trial in range(150):
        n_max = int(rng.choice([1, 2, 7, 64, 1000, 1500, 3000]))
        bt = int(rng.choice([16, 32, 64]))
        n_live = int(rng.integers(0, n_max + 1))
        lens = np.zeros(n_max, dtype=np.int64)
        lens[:n_live] = rng.integers(0, 300, size=n_live)
        lens[rng.random(n_max) < 0.2] = 0
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
        t_max = int(max(cu[-1], 1) + rng.integers(0, 200))
        m = run(cu.tolist(), t_max, bt)
        check(m, cu.tolist(), t_max, bt)


def test_invalid_layouts_give_status_and_sentinels():
    for cu, t_max, code in (([0, 50, 40, 60], 128, 1), ([3, 50, 60], 128, 2),
                            ([0, 100, 300], 256, 3), ([1, 0, 5], 8, 2)):
        m = run(cu, t_max)
        check(m, cu, t_max, 64)
        assert int(m.status.item()) == code


def test_graph_capture_and_replay_new_layouts():
    """Capture once, then change cu_seqlens in place and replay (no re-capture)."""
    t_max, n_max = 65536, 64
    meta = Meta(t_max, n_max)
    cu_static = torch.zeros(n_max + 1, dtype=torch.int32, device=DEV)
    layouts = []
    rng = np.random.default_rng(2)
    for _ in range(4):
        lens = np.zeros(n_max, dtype=np.int64)
        lens[:32] = rng.integers(1, 2049, size=32)
        layouts.append(np.concatenate([[0], np.cumsum(lens)]).astype(np.int32))
    cu_static.copy_(torch.from_numpy(layouts[0]).to(DEV))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        meta.build(cu_static, stream=s)       # warm-up outside the graph
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        meta.build(cu_static)
    for cu in layouts[1:] + layouts[:1]:
        cu_static.copy_(torch.from_numpy(cu).to(DEV))
        g.replay()
        torch.cuda.synchronize()
        check(meta, cu.tolist(), t_max, 64)


def run64(cu, t_max, bt=64):
    """chunk_meta_build_i64 on an int64 cu_seqlens: the metadata and the int32 copy."""
    meta = Meta(t_max, len(cu) - 1, bt)
    cu_d = torch.tensor(cu, dtype=torch.int64, device=DEV)
    cu32 = torch.full((len(cu),), 77, dtype=torch.int32, device=DEV)
    meta.build(cu_d, cu_seqlens32=cu32)
    torch.cuda.synchronize()
    return meta, cu32.cpu().numpy()


def test_int64_cu_seqlens_bit_exact():
    """int64 offsets give the same metadata as int32 ones, and an exact int32 copy."""
    rng = np.random.default_rng(2)
    for trial in range(60):
        n_max = int(rng.choice([1, 3, 64, 1500]))
        bt = int(rng.choice([32, 64]))
        lens = rng.integers(0, 400, size=n_max)
        lens[rng.random(n_max) < 0.25] = 0
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
        t_max = int(max(cu[-1], 1) + rng.integers(0, 100))
        m, cu32 = run64(cu.tolist(), t_max, bt)
        check(m, cu.tolist(), t_max, bt)
        np.testing.assert_array_equal(cu32, cu.astype(np.int32))


def test_int64_cu_seqlens_out_of_int32_range():
    """Entries past 2^31 (or negative) are caught by the int64 checks; the copy is zeroed."""
    big = 1 << 33
    for cu, code in (([0, big, 10], 1), ([0, 5, big], 3), ([0, 7, -3, 9], 1), ([big, big + 1], 2),
                     ([0, (1 << 32) + 5], 3)):
        m, cu32 = run64(cu, 1 << 20)
        assert int(m.status.item()) == code, cu
        assert (cu32 == 0).all(), cu
        assert (m.idx.cpu().numpy()[:, 0] == -1).all()


def test_int64_cu_seqlens_forward_and_graph_replay():
    """The forward on the int32 copy written by chunk_meta_build_i64 matches the oracle; captured
    once with the int64 metadata call inside the graph, replayed for a new layout."""
    from chunked_gated_linear_gb300 import synth
    import chunked_gated_linear_gb300 as gcl
    from gpu_util import CANARY, check_fwd, to_device
    t_max, n_max, H = 1024, 4, 2
    lay = [[300, 0, 511, 77], [64, 700, 1, 200]]
    w0 = synth.varlen("i64", synth.GDN, "bf16", lay[0], n_max, t_max, H, 128, 128, seed=51)
    static = to_device(w0, synth.make_inputs(w0))
    cu64 = static["cu_seqlens"].to(torch.int64)
    cu32 = torch.zeros(n_max + 1, dtype=torch.int32, device=DEV)
    meta = Meta(t_max, n_max)
    o = torch.full((t_max, H, 128), CANARY, dtype=torch.bfloat16, device=DEV)
    ht = torch.zeros((n_max, H, 128, 128), dtype=torch.float32, device=DEV)
    args = (static["q"], static["k"], static["v"], static["g"], static["beta"], cu32, o)
    kw = dict(h0=static["h0"], ht=ht, chunk_indices=meta.idx, chunk_offsets=meta.off,
              seq_order=meta.order, dev_status=meta.status, scale=w0.scale)
    ws = torch.empty(gcl.fwd_workspace_bytes(*args, **kw), dtype=torch.uint8, device=DEV)

    def step(stream=None):
        meta.build(cu64, stream=stream, cu_seqlens32=cu32)
        gcl.gdn_chunk_fwd(*args, workspace=ws, stream=stream, **kw)

    step()
    torch.cuda.synchronize()
    x0 = synth.make_inputs(w0)
    check_fwd(w0, x0, dict(o=o, ht=ht, meta=meta), label="int64 eager")
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step(stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        step()
    w1 = synth.varlen("i64", synth.GDN, "bf16", lay[1], n_max, t_max, H, 128, 128, seed=52)
    x1 = synth.make_inputs(w1)
    new = to_device(w1, x1)
    for name in ("q", "k", "v", "g", "beta", "h0"):
        static[name].copy_(new[name])
    cu64.copy_(new["cu_seqlens"].to(torch.int64))
    o.fill_(CANARY)
    g.replay()
    torch.cuda.synchronize()
    check_fwd(w1, x1, dict(o=o, ht=ht, meta=meta), label="int64 replay")
    np.testing.assert_array_equal(cu32.cpu().numpy(), x1["cu_seqlens"])
