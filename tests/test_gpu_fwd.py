"""Forward parity (GDN and KDA) against the fp64 oracle, through the C ABI."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
import oracle  # noqa: E402
from chunked_gated_linear_gb300 import synth  # noqa: E402
from gpu_util import CANARY, DEV, Meta, TOL, check_fwd, relF, run_fwd, to_device  # noqa: E402

STD = synth.standard_workloads()


@pytest.mark.parametrize("idx,plan", [(0, "fastest"), (1, "fastest"), (1, "min"), (2, "fastest")],
                         ids=[STD[0].name, STD[1].name + "-transition", STD[1].name + "-wform",
                              STD[2].name])
def test_standard_workload_full_size(idx, plan):
    """The 4096-token, 16-head GDN workload runs both tensor-core plans: the transition
    form (its fastest plan, 8 column slices per head) and the W form (least workspace)."""
    w = STD[idx]
    x = synth.make_inputs(w)
    out = run_fwd(w, to_device(w, x), plan=plan)
    e_o, e_h = check_fwd(w, x, out, label=w.name)
    print(f"{w.name} ({plan}): o {e_o:.2e} ht {e_h:.2e}")


@pytest.mark.parametrize("H", [3, 1], ids=["split4", "split8"])
@pytest.mark.parametrize("plan", ["fastest", "min"], ids=["transition", "wform"])
def test_gdn_bf16_plans_ragged(plan, H):
    """Both tensor-core plans on ragged lengths (1, 63, 64, 65, 200, empty), with h0 and
    saved chunk states, at column splits 4 (H=3: 24 units) and 8 (H=1: 8 units)."""
    lens = [1, 63, 0, 64, 65, 200, 130, 0]
    w = synth.varlen("plans", synth.GDN, "bf16", lens, 8, sum(lens) + 40, H, 128, 128, seed=15)
    x = synth.make_inputs(w)
    out = run_fwd(w, to_device(w, x), h_save=True, plan=plan)
    check_fwd(w, x, out, label=f"plans {plan}")
    meta = out["meta"]
    off = meta.off.cpu().numpy()
    _, _, hc = oracle.fwd(synth.GDN, x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"],
                          x["cu_seqlens"], w.scale, bt=64, chunk_offsets=off, nt_rows=meta.nt_max)
    live = int(off[-1])
    hs = out["h_save"].cpu().numpy()
    assert relF(hs[:live], hc[:live]) <= TOL["bf16"]
    assert (hs[live:] == np.float32(CANARY)).all()


CASES = []
for variant in (synth.GDN, synth.KDA):
    for dtype in ("f32", "bf16"):
        for KV in ((64, 64), (128, 128), (64, 128), (128, 64)):
            CASES.append((variant, dtype, KV))


@pytest.mark.parametrize("variant,dtype,KV", CASES,
                         ids=[f"{'kda' if c[0] else 'gdn'}-{c[1]}-K{c[2][0]}V{c[2][1]}" for c in CASES])
def test_varlen_ragged_shapes(variant, dtype, KV):
    """Lengths 1, 63, 64, 65, 200, zero-length in the middle and at the tail, slack in T_max."""
    K, V = KV
    lens = [1, 63, 0, 64, 65, 200]
    w = synth.varlen("ragged", variant, dtype, lens, 8, sum(lens) + 37, 3, K, V, seed=5)
    x = synth.make_inputs(w)
    out = run_fwd(w, to_device(w, x), h_save=True)
    check_fwd(w, x, out, label="ragged")
    # saved chunk states
    meta = out["meta"]
    off = meta.off.cpu().numpy()
    _, _, hc = oracle.fwd(variant, x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"],
                          x["cu_seqlens"], w.scale, bt=64, chunk_offsets=off,
                          nt_rows=meta.nt_max)
    live = int(off[-1])
    hs = out["h_save"].cpu().numpy()
    assert relF(hs[:live], hc[:live]) <= TOL[dtype]
    assert (hs[live:] == np.float32(CANARY)).all()      # unused rows untouched


@pytest.mark.parametrize("variant", [synth.GDN, synth.KDA])
def test_zero_initial_state_and_dense_batch(variant):
    w = synth.dense("dense", variant, "bf16", 3, 300, 2, 128, 128, h0=False, seed=9)
    x = synth.make_inputs(w)
    check_fwd(w, x, run_fwd(w, to_device(w, x)), label="dense h0=None")


def test_single_token_and_empty_batch():
    w = synth.varlen("one", synth.GDN, "bf16", [1], 2, 64, 2, 128, 128, seed=4)
    x = synth.make_inputs(w)
    check_fwd(w, x, run_fwd(w, to_device(w, x)), label="T=1")
    # every sequence empty: ht = h0, o untouched
    w = synth.varlen("empty", synth.GDN, "bf16", [0, 0], 2, 64, 2, 128, 128, seed=4)
    x = synth.make_inputs(w)
    out = run_fwd(w, to_device(w, x))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(out["ht"].cpu().numpy(), x["h0"])
    assert (out["o"].float().cpu().numpy() == np.float32(CANARY)).all()


def test_deterministic_and_order_independent():
    w = synth.varlen("det", synth.GDN, "bf16", [300, 5, 700, 64], 6, 1200, 4, 128, 128, seed=6)
    x = synth.make_inputs(w)
    d = to_device(w, x)
    a = run_fwd(w, d)
    b = run_fwd(w, d)
    c = run_fwd(w, d, use_order=False)
    torch.cuda.synchronize()
    for key in ("o", "ht"):
        assert torch.equal(a[key], b[key]) and torch.equal(a[key], c[key]), key


def test_invalid_cu_seqlens_do_nothing():
    w = synth.varlen("bad", synth.GDN, "bf16", [100, 50], 2, 256, 2, 128, 128, seed=7)
    x = synth.make_inputs(w)
    d = to_device(w, x)
    d["cu_seqlens"] = torch.tensor([0, 100, 60], dtype=torch.int32, device=DEV)   # decreasing
    out = run_fwd(w, d)
    torch.cuda.synchronize()
    assert int(out["meta"].status.item()) == 1
    assert (out["o"].float().cpu().numpy() == np.float32(CANARY)).all()
    assert (out["ht"].cpu().numpy() == np.float32(CANARY)).all()


@pytest.mark.parametrize("H", [2, 4, 6], ids=["split8", "split4", "split2"])
def test_kda_tensor_core_column_splits(H):
    """KDA bf16 d=128 at 8, 4 and 2 value-column slices per head (16, 32 and 48
    sequence-head units), ragged lengths, h0 and saved chunk states."""
    lens = [1, 63, 0, 64, 65, 200, 130, 0]
    w = synth.varlen("kda-split", synth.KDA, "bf16", lens, 8, sum(lens) + 40, H, 128, 128, seed=21)
    x = synth.make_inputs(w)
    out = run_fwd(w, to_device(w, x), h_save=True)
    check_fwd(w, x, out, label=f"kda H={H}")
    meta = out["meta"]
    off = meta.off.cpu().numpy()
    _, _, hc = oracle.fwd(synth.KDA, x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"],
                          x["cu_seqlens"], w.scale, bt=64, chunk_offsets=off, nt_rows=meta.nt_max)
    live = int(off[-1])
    assert relF(out["h_save"].cpu().numpy()[:live], hc[:live]) <= TOL["bf16"]


@pytest.mark.parametrize("regime", ["strong", "none", "mixed"])
def test_kda_gate_extremes(regime):
    """Per-channel gates far outside the generator's range: strong decay (log gates down to
    -80 per token, so the decay over a 16-token block underflows fp32 when factored through
    one reference), no decay (g = 0) and a mix of both across channels and tokens."""
    lens = [300, 77]
    w = synth.varlen("kda-gates", synth.KDA, "bf16", lens, 2, 400, 2, 128, 128, seed=23)
    x = synth.make_inputs(w)
    g = x["g"].copy()
    rng = np.random.default_rng(5)
    if regime == "strong":
        g *= 20.0
    elif regime == "none":
        g[:] = 0.0
    else:
        g[rng.random(g.shape) < 0.1] *= 40.0       # scattered strong gates
        g[:, :, :32] = 0.0                          # and undecayed channels
    x["g"] = g.astype(np.float32)
    check_fwd(w, x, run_fwd(w, to_device(w, x)), label=f"kda gates {regime}")


@pytest.mark.parametrize("plan", ["fastest", "min"], ids=["transition", "wform"])
@pytest.mark.parametrize("regime", ["beta0", "nodecay", "strong", "mixed"])
def test_gdn_degenerate_gates_and_beta(regime, plan):
    """GDN on the tensor cores in the method's degenerate regimes: beta = 0 (no delta rule:
    the state only decays, A = 0 and T = I), g = 0 (no decay), log gates 20x the generator's
    (decay over a chunk far below fp32's range) and a mix of strong and zero gates."""
    lens = [300, 77, 0, 130]
    w = synth.varlen("gdn-gates", synth.GDN, "bf16", lens, 4, 540, 2, 128, 128, seed=25)
    x = synth.make_inputs(w)
    T = w.total_tokens
    rng = np.random.default_rng(26)
    if regime == "beta0":
        x["beta"][:T] = 0.0
    elif regime == "nodecay":
        x["g"][:T] = 0.0
    elif regime == "strong":
        x["g"][:T] *= 20.0
    else:
        g = x["g"][:T]
        g[rng.random(g.shape) < 0.2] *= 40.0
        g[rng.random(g.shape) < 0.3] = 0.0
        x["g"][:T] = g
    check_fwd(w, x, run_fwd(w, to_device(w, x), plan=plan), label=f"gdn {regime} {plan}")


def test_many_short_sequences():
    """1,000 sequence slots of 0..100 tokens (a fifth of them empty), two heads: the longest-
    first order over many slots, many zero-length sequences passing h0 through."""
    rng = np.random.default_rng(27)
    lens = [int(v) for v in rng.integers(0, 101, size=1000)]
    for i in rng.choice(1000, size=200, replace=False):
        lens[i] = 0
    for variant in (synth.GDN, synth.KDA):
        w = synth.varlen("many", variant, "bf16", lens, 1000, sum(lens) + 64, 2, 128, 128, seed=28)
        x = synth.make_inputs(w)
        out = run_fwd(w, to_device(w, x))
        check_fwd(w, x, out, label=f"many short ({'kda' if variant else 'gdn'})")
        ht = out["ht"].cpu().numpy()
        for n, L in enumerate(lens):
            if L == 0:
                np.testing.assert_array_equal(ht[n], x["h0"][n])
