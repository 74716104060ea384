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
