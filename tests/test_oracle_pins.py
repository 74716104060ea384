"""Pins of the fp64 oracle against facts that do not come from the oracle itself.

Each test ties the oracle to a hand-worked example, a closed form, an
invariant of the recurrence, a brute-force evaluation, or finite differences.
They run on the CPU only.
"""
import itertools
import json
import os

import numpy as np
import pytest

import oracle
from oracle import chunk_form
from chunked_gated_linear_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
GDN, KDA = 0, 1


def rel(a, b):
    return float(np.linalg.norm(np.asarray(a) - np.asarray(b)) / max(np.linalg.norm(b), 1e-300))


def rand_case(variant, T, H=2, K=8, V=6, seed=0, h0=True):
    w = synth.dense("t", variant, "f32", 1, T, H, K, V, h0=h0)
    x = synth.make_inputs(w, seed=seed)
    return w, x


def run_fwd(variant, x, scale, **kw):
    return oracle.fwd(variant, x["q"], x["k"], x["v"], x["g"], x["beta"], x.get("h0"),
                      x["cu_seqlens"], scale, **kw)


# --------------------------------------------------------------------------- hand examples
@pytest.mark.parametrize("fname", ["gdn_hand_T2_K2_V2.json", "kda_hand_T2_K2_V2.json"])
def test_hand_worked_example(fname):
    d = json.load(open(os.path.join(GOLDEN, fname)))
    variant = GDN if d["variant"] == "gdn" else KDA
    q = np.array(d["q"])[:, None, :]
    k = np.array(d["k"])[:, None, :]
    v = np.array(d["v"])[:, None, :]
    beta = np.array(d["beta"])[:, None]
    if variant == GDN:
        g = np.log(np.array(d["alpha"]))[:, None]
    else:
        g = np.log(np.array(d["a"]))[:, None, :]
    h0 = np.array(d["h0"])[None, None]
    o, ht = oracle.fwd(variant, q, k, v, g, beta, h0, [0, 2], d["scale"])
    np.testing.assert_allclose(o[:, 0], d["o"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(ht[0, 0], d["ht"], rtol=0, atol=1e-12)


def test_chunk_meta_golden():
    d = json.load(open(os.path.join(GOLDEN, "chunk_meta_examples.json")))
    for c in d["cases"]:
        assert oracle.nt_max(c["t_max"], len(c["cu_seqlens"]) - 1, c["bt"]) == c["nt_max"]
        st, idx, off = oracle.chunk_meta(c["cu_seqlens"], c["t_max"], c["bt"])
        assert st == c["status"], c["note"]
        assert idx.tolist() == c["chunk_indices"], c["note"]
        assert off.tolist() == c["chunk_offsets"], c["note"]


# --------------------------------------------------------------------------- I1 closed form
@pytest.mark.parametrize("variant", [GDN, KDA])
def test_I1_beta_zero_is_pure_decay(variant):
    w, x = rand_case(variant, T=37, K=8, V=5, seed=11)
    x["beta"][:] = 0.0
    o, ht = run_fwd(variant, x, 0.7)
    h0 = x["h0"][0].astype(np.float64)            # [H, K, V]
    g = x["g"][:37].astype(np.float64)
    cum = np.cumsum(g, axis=0)                     # [T, H] or [T, H, K]
    for h in range(w.H):
        for t in range(37):
            if variant == GDN:
                want = 0.7 * np.exp(cum[t, h]) * h0[h].T @ x["q"][t, h]
            else:
                want = 0.7 * h0[h].T @ (np.exp(cum[t, h]) * x["q"][t, h])
            np.testing.assert_allclose(o[t, h], want, rtol=1e-12, atol=1e-14)
        want_ht = (np.exp(cum[-1, h]) * h0[h] if variant == GDN
                   else np.exp(cum[-1, h])[:, None] * h0[h])
        np.testing.assert_allclose(ht[0, h], want_ht, rtol=1e-12, atol=1e-14)


# --------------------------------------------------------------------------- I2 delta rule
@pytest.mark.parametrize("variant", [GDN, KDA])
def test_I2_unit_beta_recovers_value(variant):
    """beta=1, |k|=1, q=k, scale=1: S_t^T k_t = v_t whatever the gate and the state."""
    w, x = rand_case(variant, T=50, K=8, V=7, seed=12)
    x = {n: (a.astype(np.float64) if isinstance(a, np.ndarray) and a.dtype == np.float32 else a)
         for n, a in x.items()}
    x["k"] /= np.linalg.norm(x["k"], axis=-1, keepdims=True)      # unit norm in fp64
    x["beta"][:] = 1.0
    x["q"] = x["k"].copy()
    o, _ = run_fwd(variant, x, 1.0)
    np.testing.assert_allclose(o[:50], x["v"][:50], rtol=0, atol=1e-12)


def test_I2_orthonormal_keys_no_decay():
    """g=0, beta=1, orthonormal keys (T <= K): every written value is read back."""
    rng = np.random.default_rng(3)
    K, V, T = 8, 5, 8
    Qm, _ = np.linalg.qr(rng.standard_normal((K, K)))
    k = Qm.T[:T][:, None, :]
    v = rng.standard_normal((T, 1, V))
    g = np.zeros((T, 1))
    beta = np.ones((T, 1))
    h0 = rng.standard_normal((1, 1, K, V))
    for variant in (GDN, KDA):
        gg = g if variant == GDN else np.zeros((T, 1, K))
        _, ht = oracle.fwd(variant, k, k, v, gg, beta, h0, [0, T], 1.0)
        for t in range(T):
            np.testing.assert_allclose(ht[0, 0].T @ k[t, 0], v[t, 0], atol=1e-12)


# --------------------------------------------------------------------------- I3 brute force
@pytest.mark.parametrize("variant", [GDN, KDA])
@pytest.mark.parametrize("T", [1, 2, 5, 8])
def test_I3_brute_force_transition_products(variant, T):
    """S_T = sum_t (prod_{j>t} M_j) beta_t k_t v_t^T + (prod_j M_j) h0 with explicit K x K
    transition matrices M_j = alpha_j (I - beta_j k_j k_j^T) (GDN) or
    (I - beta_j k_j k_j^T) Diag(a_j) (KDA); o_t from S_t."""
    w, x = rand_case(variant, T=T, H=1, K=5, V=4, seed=20 + T)
    o, ht = run_fwd(variant, x, 0.9)
    K = 5
    q, k, v = (x[n][:, 0].astype(np.float64) for n in ("q", "k", "v"))
    beta = x["beta"][:, 0].astype(np.float64)
    g = x["g"][:, 0].astype(np.float64)
    h0 = x["h0"][0, 0].astype(np.float64)
    M = []
    for j in range(T):
        proj = np.eye(K) - beta[j] * np.outer(k[j], k[j])
        M.append(np.exp(g[j]) * proj if variant == GDN else proj @ np.diag(np.exp(g[j])))
    for t_end in range(T):
        S = np.zeros((K, 4))
        prod_all = np.eye(K)
        for j in range(t_end + 1):
            prod_all = M[j] @ prod_all
        S += prod_all @ h0
        for t in range(t_end + 1):
            P = np.eye(K)
            for j in range(t + 1, t_end + 1):
                P = M[j] @ P
            S += P @ (beta[t] * np.outer(k[t], v[t]))
        np.testing.assert_allclose(o[t_end, 0], 0.9 * S.T @ q[t_end], rtol=1e-11, atol=1e-13)
        if t_end == T - 1:
            np.testing.assert_allclose(ht[0, 0], S, rtol=1e-11, atol=1e-13)


# --------------------------------------------------------------------------- I4 chunk form
@pytest.mark.parametrize("variant", [GDN, KDA])
@pytest.mark.parametrize("T", [1, 63, 64, 65, 200])
def test_I4_chunk_form_equals_recurrence(variant, T):
    w, x = rand_case(variant, T=T, H=2, K=16, V=12, seed=40 + T)
    o, ht = run_fwd(variant, x, w.scale)
    for bt in (1, 16, 64):
        oc, htc = chunk_form.chunk_fwd(variant, x["q"], x["k"], x["v"], x["g"], x["beta"],
                                       x["h0"], x["cu_seqlens"], w.scale, bt)
        assert rel(oc[:T], o[:T]) <= 1e-12
        assert rel(htc, ht) <= 1e-12


# --------------------------------------------------------------------------- I5 KDA -> GDN
def test_I5_kda_with_equal_channel_gates_is_gdn():
    w, x = rand_case(GDN, T=90, H=3, K=8, V=6, seed=5)
    o1, ht1 = run_fwd(GDN, x, 0.4)
    xk = dict(x)
    xk["g"] = np.repeat(x["g"][:, :, None], 8, axis=2)
    o2, ht2 = run_fwd(KDA, xk, 0.4)
    np.testing.assert_allclose(o2, o1, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(ht2, ht1, rtol=1e-12, atol=1e-14)


# --------------------------------------------------------------------------- I6 state passing
@pytest.mark.parametrize("variant", [GDN, KDA])
def test_I6_split_and_chain(variant):
    w, x = rand_case(variant, T=150, H=2, K=8, V=6, seed=6)
    o, ht = run_fwd(variant, x, 0.5)
    t1 = 61
    a = {n: x[n][:t1] for n in ("q", "k", "v", "g", "beta")}
    b = {n: x[n][t1:150] for n in ("q", "k", "v", "g", "beta")}
    oa, hta = oracle.fwd(variant, a["q"], a["k"], a["v"], a["g"], a["beta"], x["h0"], [0, t1], 0.5)
    ob, htb = oracle.fwd(variant, b["q"], b["k"], b["v"], b["g"], b["beta"], hta,
                         [0, 150 - t1], 0.5)
    np.testing.assert_allclose(np.concatenate([oa, ob]), o[:150], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(htb, ht, rtol=1e-12, atol=1e-14)


# --------------------------------------------------------------------------- I7 varlen
@pytest.mark.parametrize("variant", [GDN, KDA])
def test_I7_varlen_equals_independent_runs_and_padding_is_not_read(variant):
    lens = [70, 0, 1, 129, 0]
    w = synth.varlen("t", variant, "f32", lens, 6, 260, 2, 8, 6)
    x = synth.make_inputs(w, seed=7)           # rows >= 200 are NaN
    o, ht = run_fwd(variant, x, 0.3)
    T = w.total_tokens
    assert np.isfinite(o[:T]).all() and np.isfinite(ht).all()
    cu = x["cu_seqlens"]
    for n in range(6):
        s, e = int(cu[n]), int(cu[n + 1])
        sl = {m: x[m][s:e] for m in ("q", "k", "v", "g", "beta")}
        on, htn = oracle.fwd(variant, sl["q"], sl["k"], sl["v"], sl["g"], sl["beta"],
                             x["h0"][n:n + 1], [0, e - s], 0.3)
        np.testing.assert_allclose(o[s:e], on, rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(ht[n], htn[0], rtol=1e-13, atol=1e-15)
        if e == s:       # a zero-length sequence passes its state through
            np.testing.assert_array_equal(ht[n], x["h0"][n])


# --------------------------------------------------------------------------- I8 NT_max bound
def test_I8_nt_max_bound_brute_force():
    for bt, t_max, n_max in itertools.product((2, 3, 4), range(1, 13), range(1, 5)):
        ntm = oracle.nt_max(t_max, n_max, bt)
        best = 0
        # all compositions of at most t_max tokens into n_max ordered lengths
        for lens in itertools.product(range(t_max + 1), repeat=n_max):
            if sum(lens) > t_max:
                continue
            nt = sum((L + bt - 1) // bt for L in lens)
            assert nt <= ntm, (bt, t_max, n_max, lens)
            best = max(best, nt)
        # n_max - 1 one-token sequences plus one long one reach the bound whenever the long
        # one still needs ceil(t_max / bt) chunks
        if t_max >= n_max and -(-(t_max - n_max + 1) // bt) == -(-t_max // bt):
            assert best == ntm, (bt, t_max, n_max, best, ntm)


def test_chunk_meta_matches_token_enumeration():
    """Live rows are exactly the distinct (sequence, token_offset // BT) pairs, in token order."""
    rng = np.random.default_rng(8)
    for trial in range(200):
        n_max = int(rng.integers(1, 9))
        bt = int(rng.choice([16, 32, 64]))
        lens = rng.integers(0, 150, size=n_max)
        lens[rng.random(n_max) < 0.3] = 0
        cu = np.concatenate([[0], np.cumsum(lens)])
        t_max = int(cu[-1] + rng.integers(0, 100))
        st, idx, off = oracle.chunk_meta(cu, t_max, bt)
        assert st == 0
        seen = []
        for n in range(n_max):
            for t in range(int(cu[n]), int(cu[n + 1])):
                p = (n, (t - int(cu[n])) // bt)
                if not seen or seen[-1] != p:
                    seen.append(p)
        live = len(seen)
        assert idx[:live].tolist() == [list(p) for p in seen]
        assert (idx[live:] == [-1, 0]).all()
        for n in range(n_max):
            first = [j for j, p in enumerate(seen) if p[0] == n]
            if first:
                assert off[n] == first[0]
        assert off[n_max] == live


# --------------------------------------------------------------------------- I9 backward
def _f_and_grads(variant, x, scale, d_o, dht):
    o, ht = run_fwd(variant, x, scale)
    f = float(np.sum(d_o * o) + np.sum(dht * ht))
    gr = oracle.bwd(variant, x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"], d_o, dht,
                    x["cu_seqlens"], scale)
    return f, gr


@pytest.mark.parametrize("variant", [GDN, KDA])
@pytest.mark.parametrize("KV", [(16, 16), (128, 128)])
def test_I9_backward_finite_differences(variant, KV):
    K, V = KV
    T = 16
    w, x = rand_case(variant, T=T, H=1, K=K, V=V, seed=90 + K)
    x = {n: (a.astype(np.float64) if isinstance(a, np.ndarray) and a.dtype == np.float32 else a)
         for n, a in x.items()}
    rng = np.random.default_rng(91)
    d_o = rng.standard_normal((T, 1, V))
    dht = 0.1 * rng.standard_normal((1, 1, K, V))
    scale = K ** -0.5
    f0, gr = _f_and_grads(variant, x, scale, d_o, dht)
    eps = 1e-6
    names = {"q": "dq", "k": "dk", "v": "dv", "g": "dg", "beta": "dbeta", "h0": "dh0"}
    for name, gname in names.items():
        d = rng.standard_normal(x[name].shape)
        xp = dict(x); xp[name] = x[name] + eps * d
        xm = dict(x); xm[name] = x[name] - eps * d
        fp = float(np.sum(d_o * run_fwd(variant, xp, scale)[0]) +
                   np.sum(dht * run_fwd(variant, xp, scale)[1]))
        fm = float(np.sum(d_o * run_fwd(variant, xm, scale)[0]) +
                   np.sum(dht * run_fwd(variant, xm, scale)[1]))
        fd = (fp - fm) / (2 * eps)
        an = float(np.sum(gr[gname] * d))
        assert abs(fd - an) <= 1e-7 * max(1.0, abs(an)), (name, fd, an)


@pytest.mark.parametrize("variant", [GDN, KDA])
def test_I9_exact_adjoint_of_linear_arguments(variant):
    """o and ht are jointly linear in (v, h0), so f = <dv, v> + <dh0, h0> exactly."""
    w, x = rand_case(variant, T=100, H=2, K=8, V=6, seed=95)
    rng = np.random.default_rng(96)
    d_o = rng.standard_normal((100, 2, 6))
    dht = rng.standard_normal((1, 2, 8, 6))
    f, gr = _f_and_grads(variant, x, 0.35, d_o, dht)
    lin = float(np.sum(gr["dv"] * x["v"]) + np.sum(gr["dh0"] * x["h0"]))
    assert abs(f - lin) <= 1e-11 * max(1.0, abs(f))


def test_backward_chunk_boundaries_and_varlen():
    """Checkpoint segments (64 tokens) and sequence boundaries do not change gradients:
    a varlen batch equals per-sequence runs."""
    lens = [130, 0, 64, 3]
    w = synth.varlen("t", GDN, "f32", lens, 4, 200, 2, 8, 6)
    x = synth.make_inputs(w, seed=97)
    rng = np.random.default_rng(98)
    d_o = rng.standard_normal((200, 2, 6))
    dht = rng.standard_normal((4, 2, 8, 6))
    gr = oracle.bwd(GDN, x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"], d_o, dht,
                    x["cu_seqlens"], 0.5)
    cu = x["cu_seqlens"]
    for n in range(4):
        s, e = int(cu[n]), int(cu[n + 1])
        gn = oracle.bwd(GDN, *(x[m][s:e] for m in ("q", "k", "v", "g", "beta")),
                        x["h0"][n:n + 1], d_o[s:e], dht[n:n + 1], [0, e - s], 0.5)
        for key in ("dq", "dk", "dv", "dg", "dbeta"):
            np.testing.assert_allclose(gr[key][s:e], gn[key], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(gr["dh0"][n], gn["dh0"][0], rtol=1e-12, atol=1e-14)


# --------------------------------------------------------------------------- I10 masking
@pytest.mark.parametrize("variant", [GDN, KDA])
def test_I10_masked_rows_leave_state_unchanged(variant):
    w, x = rand_case(variant, T=40, H=2, K=8, V=6, seed=10)
    _, ht = run_fwd(variant, x, 0.5)
    y = {n: x[n][:40] for n in ("q", "k", "v", "g", "beta")}
    pad = 24
    z = {}
    for n, a in y.items():
        extra = np.random.default_rng(1).standard_normal((pad,) + a.shape[1:])
        if n in ("k", "g", "beta"):
            extra[:] = 0.0
        z[n] = np.concatenate([a, extra])
    _, ht2 = oracle.fwd(variant, z["q"], z["k"], z["v"], z["g"], z["beta"], x["h0"],
                        [0, 40 + pad], 0.5)
    np.testing.assert_allclose(ht2, ht, rtol=1e-13, atol=1e-15)


# --------------------------------------------------------------------------- I11 GEMM-first
@pytest.mark.parametrize("variant", [GDN, KDA])
def test_I11_gemm_first_order_equals_wy_order(variant):
    w, x = rand_case(variant, T=150, H=2, K=16, V=8, seed=12)
    a = chunk_form.chunk_fwd(variant, x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"],
                             x["cu_seqlens"], w.scale, 64, order="wy")
    b = chunk_form.chunk_fwd(variant, x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"],
                             x["cu_seqlens"], w.scale, 64, order="gemm_first")
    assert rel(b[0], a[0]) <= 1e-12 and rel(b[1], a[1]) <= 1e-12


# --------------------------------------------------------------------------- I12 columns
@pytest.mark.parametrize("variant", [GDN, KDA])
def test_I12_value_columns_are_independent(variant):
    w, x = rand_case(variant, T=80, H=2, K=8, V=9, seed=13)
    o, ht = run_fwd(variant, x, 0.5)
    perm = np.random.default_rng(0).permutation(9)
    xp = dict(x)
    xp["v"] = x["v"][:, :, perm]
    xp["h0"] = x["h0"][..., perm]
    op, htp = run_fwd(variant, xp, 0.5)
    np.testing.assert_allclose(op, o[:, :, perm], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(htp, ht[..., perm], rtol=1e-13, atol=1e-15)
    # one column alone gives the same column
    xs = dict(x)
    xs["v"] = x["v"][:, :, 4:5]
    xs["h0"] = x["h0"][..., 4:5]
    os_, hts = run_fwd(variant, xs, 0.5)
    np.testing.assert_allclose(os_[:, :, 0], o[:, :, 4], rtol=1e-13, atol=1e-15)


# --------------------------------------------------------------------------- saved chunk states
def test_saved_chunk_states_equal_prefix_runs():
    """h_chunk[chunk_offsets[n] + i] is the state after the first i*bt tokens of sequence n,
    i.e. the final state of a run over that prefix alone."""
    lens = [130, 0, 64, 5]
    w = synth.varlen("t", GDN, "f32", lens, 4, 220, 2, 8, 6)
    x = synth.make_inputs(w, seed=99)
    st, idx, off = oracle.chunk_meta(x["cu_seqlens"], 220, 64)
    o, ht, hc = oracle.fwd(GDN, x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"],
                           x["cu_seqlens"], 0.5, bt=64, chunk_offsets=off,
                           nt_rows=idx.shape[0])
    cu = x["cu_seqlens"]
    for j in range(int(off[-1])):
        n, i = idx[j]
        s = int(cu[n])
        e = s + 64 * int(i)
        _, htp = oracle.fwd(GDN, *(x[m][s:e] for m in ("q", "k", "v", "g", "beta")),
                            x["h0"][n:n + 1], [0, e - s], 0.5)
        np.testing.assert_allclose(hc[j], htp[0], rtol=1e-13, atol=1e-15)


def test_chunk_states_at_bt32_are_every_other_bt64_state():
    """The state before 64-token chunk i of a sequence is the state before 32-token chunk 2i:
    both are the token recurrence's state after the same prefix."""
    lens = [130, 0, 64, 5, 97]
    w = synth.varlen("t", GDN, "f32", lens, 5, 300, 2, 8, 6)
    x = synth.make_inputs(w, seed=98)
    hc = {}
    offs = {}
    for bt in (32, 64):
        st, idx, off = oracle.chunk_meta(x["cu_seqlens"], 300, bt)
        _, _, hc[bt] = oracle.fwd(GDN, x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"],
                                  x["cu_seqlens"], 0.5, bt=bt, chunk_offsets=off,
                                  nt_rows=idx.shape[0])
        offs[bt] = off
    for n in range(len(lens)):
        for i in range(int(offs[64][n + 1] - offs[64][n])):
            np.testing.assert_array_equal(hc[32][offs[32][n] + 2 * i], hc[64][offs[64][n] + i])
