"""Pins of the short-convolution oracle (CPU): closed forms, a library special case, state
chaining, varlen independence and the reverse mode by finite differences and the adjoint
identity."""
import numpy as np
import pytest

from oracle.short_conv import conv_bwd, conv_fwd

RNG = np.random.default_rng(1234)


def _case(T=23, D=5, W=4, lens=(9, 0, 1, 13), h0=True):
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    x = RNG.standard_normal((T, D))
    x[cu[-1]:] = np.nan                                     # padding rows are never read
    w = RNG.standard_normal((D, W))
    b = RNG.standard_normal(D)
    h = RNG.standard_normal((len(lens), D, W - 1)) if h0 else None
    return x, w, b, h, cu


@pytest.mark.parametrize("W", [2, 3, 4])
def test_identity_kernel(W):
    """Only the newest tap: y = x and ht = the last W-1 inputs (initial state for short ones)."""
    x, w, _, h, cu = _case(W=W)
    w[:] = 0.0
    w[:, W - 1] = 1.0
    y, ht = conv_fwd(x, w, None, None, h, cu)
    live = cu[-1]
    assert np.array_equal(y[:live], x[:live])
    for n in range(len(cu) - 1):
        ext = np.concatenate([h[n].T, x[cu[n]:cu[n + 1]]])
        assert np.array_equal(ht[n], ext[-(W - 1):].T)


@pytest.mark.parametrize("W", [2, 4])
def test_delay_kernel_reads_initial_state(W):
    """Only the oldest tap: y at position p is the input W-1 steps back, the initial state
    for p < W-1."""
    x, w, _, h, cu = _case(W=W)
    w[:] = 0.0
    w[:, 0] = 1.0
    y, _ = conv_fwd(x, w, None, None, h, cu)
    for n in range(len(cu) - 1):
        for p in range(cu[n + 1] - cu[n]):
            want = x[cu[n] + p - (W - 1)] if p >= W - 1 else h[n, :, p]
            assert np.array_equal(y[cu[n] + p], want)


def test_single_sequence_is_numpy_convolve():
    """No initial state: each channel is numpy's full convolution with the reversed taps,
    truncated to the sequence, plus the bias."""
    T, D, W = 40, 6, 4
    x = RNG.standard_normal((T, D))
    w = RNG.standard_normal((D, W))
    b = RNG.standard_normal(D)
    y, _ = conv_fwd(x, w, b, None, None, [0, T])
    for d in range(D):
        ref = np.convolve(x[:, d], w[d, ::-1])[:T] + b[d]
        np.testing.assert_allclose(y[:, d], ref, rtol=1e-13, atol=1e-13)


def test_silu_and_residual():
    x, w, b, h, cu = _case()
    r = RNG.standard_normal(x.shape)
    lin, _ = conv_fwd(x, w, b, None, h, cu)
    act, _ = conv_fwd(x, w, b, None, h, cu, activation="silu")
    res, _ = conv_fwd(x, w, b, r, h, cu, activation="silu")
    live = cu[-1]
    sig = 0.5 * (1.0 + np.tanh(0.5 * lin[:live]))          # logistic function, another form
    np.testing.assert_allclose(act[:live], lin[:live] * sig, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(res[:live] - act[:live], r[:live], rtol=1e-13, atol=1e-14)


@pytest.mark.parametrize("split", [1, 2, 3, 7])
def test_split_and_chain(split):
    """Running the first part, then the rest from its final state, equals one run."""
    W, D, L = 4, 5, 11
    x = RNG.standard_normal((L, D))
    w = RNG.standard_normal((D, W))
    b = RNG.standard_normal(D)
    h = RNG.standard_normal((1, D, W - 1))
    y, ht = conv_fwd(x, w, b, None, h, [0, L], activation="silu")
    y1, h1 = conv_fwd(x[:split], w, b, None, h, [0, split], activation="silu")
    y2, h2 = conv_fwd(x[split:], w, b, None, h1, [0, L - split], activation="silu")
    np.testing.assert_allclose(np.concatenate([y1, y2]), y, rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(h2, ht, rtol=0, atol=0)


def test_varlen_is_per_sequence_and_never_reads_padding():
    x, w, b, h, cu = _case()
    y, ht = conv_fwd(x, w, b, None, h, cu, activation="silu")
    assert np.isfinite(y).all()
    for n in range(len(cu) - 1):
        s, e = cu[n], cu[n + 1]
        yn, hn = conv_fwd(x[s:e], w, b, None, h[n:n + 1], [0, e - s], activation="silu")
        np.testing.assert_array_equal(y[s:e], yn)
        np.testing.assert_array_equal(ht[n], hn[0])
    assert (y[cu[-1]:] == 0).all()


def _loss(x, w, b, h, cu, dy, dht, act):
    y, ht = conv_fwd(x, w, b, None, h, cu, activation=act)
    live = cu[-1]
    return float(np.sum(dy[:live] * y[:live]) + np.sum(dht * ht))


@pytest.mark.parametrize("act", [None, "silu"])
def test_backward_finite_differences(act):
    x, w, b, h, cu = _case(T=19, D=3, W=4, lens=(6, 1, 0, 9))
    live = cu[-1]
    x[live:] = 0.0
    dy = RNG.standard_normal(x.shape)
    dht = RNG.standard_normal(h.shape)
    dx, dw, db, dh0 = conv_bwd(x, w, b, h, cu, dy, dht, activation=act)
    eps = 1e-6
    for name, arr, grad in (("x", x, dx), ("w", w, dw), ("b", b, db), ("h", h, dh0)):
        for _ in range(3):
            u = RNG.standard_normal(arr.shape)
            if name == "x":
                u[live:] = 0.0
            args = dict(x=x, w=w, b=b, h=h)
            args[name] = arr + eps * u
            fp = _loss(args["x"], args["w"], args["b"], args["h"], cu, dy, dht, act)
            args[name] = arr - eps * u
            fm = _loss(args["x"], args["w"], args["b"], args["h"], cu, dy, dht, act)
            fd = (fp - fm) / (2 * eps)
            an = float(np.sum(grad * u))
            assert abs(fd - an) <= 1e-7 * max(1.0, abs(an)), (name, fd, an)


def test_backward_adjoint_identity_linear():
    """Without bias and activation y and ht are linear in (x, h0), so
    <dy, y> + <dht, ht> = <dx, x> + <dh0, h0> exactly (up to rounding)."""
    x, w, _, h, cu = _case(T=30, D=4, W=3, lens=(12, 2, 0, 15))
    live = cu[-1]
    x[live:] = 0.0
    dy = RNG.standard_normal(x.shape)
    dht = RNG.standard_normal(h.shape)
    y, ht = conv_fwd(x, w, None, None, h, cu)
    dx, _, _, dh0 = conv_bwd(x, w, None, h, cu, dy, dht)
    lhs = np.sum(dy[:live] * y[:live]) + np.sum(dht * ht)
    rhs = np.sum(dx[:live] * x[:live]) + np.sum(dh0 * h)
    assert abs(lhs - rhs) <= 1e-12 * abs(lhs)


def test_zero_length_sequence_passes_state_through():
    x, w, b, h, cu = _case(lens=(0, 5))
    _, ht = conv_fwd(x, w, b, None, h, cu)
    np.testing.assert_array_equal(ht[0], h[0])


MUTANTS = [
    ("tap order", "pre += w[:, j] * xx[p + j]", "pre += w[:, j] * xx[p + W - 1 - j]"),
    ("state order", "xx[:W - 1] = np.asarray(h0[n], dtype=np.float64).T",
     "xx[:W - 1] = np.asarray(h0[n], dtype=np.float64)[:, ::-1].T"),
    ("final state shift", "ht[n, :, k] = xx[length + k]", "ht[n, :, k] = xx[length + k - 1]"),
    ("silu derivative", "return s * (1.0 + z * (1.0 - s))", "return s"),
    ("dht sign", "dxx[length + k] += np.asarray", "dxx[length + k] -= np.asarray"),
    ("bias gradient", "db += g", "db += dy[bos + p]"),
]


@pytest.mark.parametrize("label,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistakes(label, old, new):
    """Each plausible mistake, planted in a private copy of the oracle, fails a pin."""
    import oracle.short_conv as sc
    src = open(sc.__file__).read()
    assert src.count(old) >= 1, label
    ns = {"__name__": "mutant"}
    exec(compile(src.replace(old, new), "mutant", "exec"), ns)
    pins = [test_identity_kernel, test_delay_kernel_reads_initial_state,
            test_single_sequence_is_numpy_convolve, test_silu_and_residual, test_split_and_chain,
            test_varlen_is_per_sequence_and_never_reads_padding, test_backward_finite_differences,
            test_backward_adjoint_identity_linear, test_zero_length_sequence_passes_state_through]
    g = globals()
    saved = g["conv_fwd"], g["conv_bwd"]
    g["conv_fwd"], g["conv_bwd"] = ns["conv_fwd"], ns["conv_bwd"]
    caught = False
    try:
        for pin in pins:
            args = {"test_identity_kernel": [(4,)], "test_delay_kernel_reads_initial_state": [(4,)],
                    "test_split_and_chain": [(2,)], "test_backward_finite_differences": [(None,), ("silu",)]}
            for a in args.get(pin.__name__, [()]):
                try:
                    pin(*a)
                except AssertionError:
                    caught = True
    finally:
        g["conv_fwd"], g["conv_bwd"] = saved
    assert caught, f"no pin fails for the planted mistake: {label}"
