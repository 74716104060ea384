"""The oracle's pins must catch plausible mistakes.

Each case plants one mistake (a dropped term, a wrong sign, a wrong index, a
wrong order of steps) in a private copy of the C oracle, builds it, binds it in
place of the real one and runs the pins of ``test_oracle_pins.py``: at least
one pin must fail.  CPU only; the real oracle is untouched.
"""
import ctypes
import os
import subprocess

import pytest

import oracle
import test_oracle_pins as pins

MUTANTS = [
    ("GDN decay also applied to the new k v^T term",
     "S[c * V + j] = alpha * (S[c * V + j] - beta * k[c] * w[j]) + beta * k[c] * v[j];",
     "S[c * V + j] = alpha * (S[c * V + j] - beta * k[c] * w[j] + beta * k[c] * v[j]);"),
    ("GDN delta correction with the wrong sign",
     "S[c * V + j] = alpha * (S[c * V + j] - beta * k[c] * w[j]) + beta * k[c] * v[j];",
     "S[c * V + j] = alpha * (S[c * V + j] + beta * k[c] * w[j]) + beta * k[c] * v[j];"),
    ("KDA gate applied to value columns instead of key rows",
     "for (int64_t j = 0; j < V; ++j) S[c * V + j] *= a[c];",
     "for (int64_t j = 0; j < V; ++j) S[c * V + j] *= a[j < K ? j : 0];"),
    ("KDA delta correction dropped",
     "S[c * V + j] = S[c * V + j] - beta * k[c] * w[j] + beta * k[c] * v[j];",
     "S[c * V + j] = S[c * V + j] + beta * k[c] * v[j];"),
    ("output read before the state update",
     """                step_forward(variant, S, K, V, k + (t * H + h) * K, v + (t * H + h) * V,
                             g + (t * H + h) * gK, beta[t * H + h], w, a);
                read_out(S, K, V, q + (t * H + h) * K, scale, o + (t * H + h) * V);""",
     """                read_out(S, K, V, q + (t * H + h) * K, scale, o + (t * H + h) * V);
                step_forward(variant, S, K, V, k + (t * H + h) * K, v + (t * H + h) * V,
                             g + (t * H + h) * gK, beta[t * H + h], w, a);"""),
    ("scale dropped from the read-out",
     "acc += S[c * V + j] * (scale * q[c]);", "acc += S[c * V + j] * q[c];"),
    ("read-out through S instead of S^T (transposed operand)",
     "for (int64_t c = 0; c < K; ++c) acc += S[c * V + j] * (scale * q[c]);",
     "for (int64_t c = 0; c < K; ++c) acc += S[(c * V + j) % V * V + (c * V + j) / V % V] * (scale * q[c]);"),
    ("GDN dk loses the P dS^T k term",
     "dkt[c] = bt_ * dsv - alpha * bt_ * (y[c] + pdx);",
     "dkt[c] = bt_ * dsv - alpha * bt_ * (y[c]);"),
    ("GDN dg loses the chain factor alpha",
     "dgt[0] = alpha * da;", "dgt[0] = da;"),
    ("GDN dbeta ignores the decay",
     "for (int64_t j = 0; j < V; ++j) db += x[j] * (vt[j] - alpha * w[j]);",
     "for (int64_t j = 0; j < V; ++j) db += x[j] * (vt[j] - w[j]);"),
    ("KDA state gradient not decayed",
     "for (int64_t j = 0; j < V; ++j) dS[c * V + j] = a[c] * dD[c * V + j];",
     "for (int64_t j = 0; j < V; ++j) dS[c * V + j] = dD[c * V + j];"),
    ("chunk count rounds down",
     "int64_t nc = (len + bt - 1) / bt;", "int64_t nc = len / bt + (len > 0);"),
    ("chunk offsets inclusive instead of exclusive",
     "chunk_offsets[n] = (int32_t)row;",
     "chunk_offsets[n] = (int32_t)(row + (cu[n + 1] > cu[n]));"),
]


def _pins():
    yield lambda: pins.test_hand_worked_example("gdn_hand_T2_K2_V2.json")
    yield lambda: pins.test_hand_worked_example("kda_hand_T2_K2_V2.json")
    yield pins.test_chunk_meta_golden
    for v in (0, 1):
        yield lambda v=v: pins.test_I1_beta_zero_is_pure_decay(v)
        yield lambda v=v: pins.test_I2_unit_beta_recovers_value(v)
        yield lambda v=v: pins.test_I3_brute_force_transition_products(v, 5)
        yield lambda v=v: pins.test_I9_backward_finite_differences(v, (16, 16))


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(name, old, new, tmp_path, monkeypatch):
    src = open(oracle._SRC).read()
    assert src.count(old) == 1, "mutation site not found: " + name
    mpath = tmp_path / "mutant.c"
    mpath.write_text(src.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-o", str(so),
                    str(mpath), "-lm"], check=True)
    monkeypatch.setattr(oracle, "_lib", oracle.bind(ctypes.CDLL(str(so))))
    caught = 0
    for pin in _pins():
        try:
            pin()
        except AssertionError:
            caught += 1
    assert caught > 0, "no pin caught: " + name
