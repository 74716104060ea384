"""The parity checker itself (tests/parity.py), on the CPU: it must accept an output whose
error is the kernels' measured rounding level, and reject local damage that the single
global rel-Frobenius norm lets through at full size."""
import numpy as np
import pytest

from parity import ROW_C, check, local_errors, relF

TOL = 5e-3
T, H, V = 4096, 16, 128          # the 4,096-token, 16-head, d = 128 forward


def _ref_and_noisy(seed=0, level=2.9e-3):
    rng = np.random.default_rng(seed)
    ref = rng.standard_normal((T, H, V)).astype(np.float32)
    # a correct bf16 kernel: relative error about 2.9e-3 spread over every element
    noisy = ref * (1.0 + level * rng.standard_normal(ref.shape).astype(np.float32))
    return ref, noisy


CU = np.array([0, T], dtype=np.int64)


def test_accepts_rounding_level_noise():
    ref, got = _ref_and_noisy()
    eg, eu, er = check("o", got, ref, TOL, cu=CU)
    assert eg < TOL and eu < TOL and er < ROW_C * TOL


def test_zeroed_row_of_one_head_passes_global_norm_but_fails_local_bars():
    ref, got = _ref_and_noisy(seed=1)
    got[1234, 5, :] = 0.0
    assert relF(got, ref) <= TOL                     # the old, global-only check accepts it
    eu, lab, er, rlab = local_errors(got, ref, CU)
    assert lab == (0, 5) and eu > TOL                # the per-unit bar rejects it
    assert rlab == ((0, 5), 1234) and er > ROW_C * TOL   # and so does the per-row bar
    with pytest.raises(AssertionError, match=r"unit \(0, 5\)"):
        check("o", got, ref, TOL, cu=CU)


def test_one_bad_row_inside_a_short_sequence_of_a_varlen_batch():
    rng = np.random.default_rng(2)
    cu = np.array([0, 1, 64, 65, 2000, 2001, 4096], dtype=np.int64)
    ref = rng.standard_normal((T, 2, V))
    got = ref * (1.0 + 2.9e-3 * rng.standard_normal(ref.shape))
    check("o", got, ref, TOL, cu=cu)
    got[64, 1, :] *= 1.05                            # the one-token sequence of head 1, 5% off
    eu, lab, er, rlab = local_errors(got, ref, cu)
    assert lab == (2, 1) and eu > TOL
    with pytest.raises(AssertionError):
        check("o", got, ref, TOL, cu=cu)


def test_one_scaled_state_row_fails_the_state_check():
    rng = np.random.default_rng(3)
    ref = rng.standard_normal((4, 16, 128, 128))
    got = ref * (1.0 + 2e-3 * rng.standard_normal(ref.shape))
    check("ht", got, ref, TOL)
    got[3, 15, 7] *= 1.2                              # one key row of the last state, 20% off
    assert relF(got, ref) <= TOL
    with pytest.raises(AssertionError, match=r"unit \(3, 15\)"):
        check("ht", got, ref, TOL)


def test_non_finite_values_fail():
    ref, got = _ref_and_noisy(seed=4)
    got[0, 0, 0] = np.nan
    with pytest.raises(AssertionError):
        check("o", got, ref, TOL, cu=CU)


def test_reduction_gradients_take_the_wider_unit_bar():
    """dg-like tensors: an absolute error at 2e-3 of the tensor's scale on every value passes
    even where one unit's values are small; a zeroed value of a normal unit still fails."""
    rng = np.random.default_rng(5)
    cu = np.array([0, 1, 64, 200], dtype=np.int64)
    ref = 0.05 * rng.standard_normal((200, 4))
    ref[0, 2] = 0.01                                  # a one-token unit with a small value
    got = ref + 1e-4 * rng.standard_normal(ref.shape)
    got[0, 2] += 1.5e-4
    check("dg", got, ref, TOL, cu=cu)
    with pytest.raises(AssertionError):
        check("o", got, ref, TOL, cu=cu)              # the plain unit bar would reject it
    got[100, 1] = 0.0
    with pytest.raises(AssertionError):
        check("dg", got, ref, TOL, cu=cu)
