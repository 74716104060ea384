"""Parity checks shared by the GPU tests (numpy only, so the CPU suite can test them).

A single rel-Frobenius norm over a whole output hides local damage: at 4,096 tokens x 16
heads one wrong token row of one head moves it by only 1/sqrt(65,536) = 3.9e-3.  So every
comparison here applies the bar at three levels:

  global   ||got - ref||_F / ||ref||_F <= tol over the live rows of the whole tensor;
  unit     the same bar per (sequence, head) unit u: the rows bos..eos-1 of one head (for
           token-major tensors) or one [K, V] state (for [N, H, K, V] tensors):
               ||got_u - ref_u||_F <= tol * max(||ref_u||_F, rms * sqrt(rows of u));
  row      per token row (or state row) r of a unit u:
               ||got_r - ref_r|| <= ROW_C * tol * max(||ref_r||, rms_u, rms),
           where rms_u = ||ref_u||_F / sqrt(rows of u) is the unit's root-mean-square row
           norm and rms the whole tensor's.  The floors keep rows and units whose values
           nearly cancel, or have decayed far below the tensor's scale (a state after
           hundreds of tokens of pure decay is ~1e-100, which fp32 flushes to zero), from
           failing on rounding noise that is tiny against the tensor's own scale.

ROW_C = 4.  Why that constant: the kernels' error is a sum of many independent bf16 (or
fp32) operand roundings, so its size per row follows the size of the row's terms.  Rows of
V = 128 elements with errors of a common scale have norms within about +-12% of their mean
(sqrt(2 / 128)); over 65,536 rows the largest lands about 1.6x above the mean.  Rows with
larger terms than their result (cancellation) have larger relative errors, which the
max(||ref_r||, rms_u) floor absorbs.  A factor of 4 on the bar leaves that margin and
still rejects any row whose error is more than 2% of the unit's typical row (4 x 5e-3 at
bf16): a zeroed, swapped or shifted row of one head fails, while the global bar alone
accepts a zeroed row at that size.
"""
from __future__ import annotations

import numpy as np

ROW_C = 4.0
# Per-token scalar gradients that are inner products over the whole [K, V] state (dg and dbeta:
# the last row of a chunk carries e^{gamma_c} <dS', S>, 16,384 products whose sum often nearly
# cancels).  Their error is that of the bf16 state gradient times the state norms, not a
# fraction of the (possibly small) result: measured up to 3e-3 absolute on last rows whose
# values range from 0.02 to 0.9 (the largest value of the tensor is such a term).  So their
# unit bar is ROW_C x tol against the tensor-scale floor, and their row bar
# ROW_C x tol x max(|ref_r|, rms_u, rms, peak) with peak the tensor's largest |value|: an
# absolute bar at 2% of the state-term scale, which a zeroed or swapped value of typical size
# (a tenth of the peak or more) still fails.
REDUCTIONS = ("dg", "dbeta")
RECORD = []        # (name, global, worst unit, worst row ratio, bar) of every check, in order


def relF(got, want) -> float:
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    den = np.linalg.norm(want)
    return float(np.linalg.norm(got - want) / (den if den > 0 else 1.0))


def _units_tokens(x, cu):
    """(label, rows) for every live (sequence, head) unit of a token-major tensor [T, H, ...];
    rows has shape [len, D] (D = 1 for [T, H] tensors)."""
    x = np.asarray(x)
    H = x.shape[1]
    for n in range(len(cu) - 1):
        bos, eos = int(cu[n]), int(cu[n + 1])
        if eos <= bos:
            continue
        for h in range(H):
            yield (n, h), x[bos:eos, h].reshape(eos - bos, -1)


def _units_states(x):
    """(label, rows) for every [K, V] state of an [N, H, K, V] tensor."""
    x = np.asarray(x)
    for n in range(x.shape[0]):
        for h in range(x.shape[1]):
            yield (n, h), x[n, h].reshape(x.shape[2], -1)


def local_errors(got, ref, cu=None, reduction=False):
    """Worst unit ratio ||e_u|| / max(||ref_u||, rms sqrt(rows_u)) and worst row ratio
    ||e_r|| / max(||ref_r||, rms_u, rms).

    cu: cu_seqlens for token-major tensors, None for [N, H, K, V] state tensors.
    Returns (worst_unit, unit_label, worst_row, (unit_label, row))."""
    gi = _units_states(got) if cu is None else _units_tokens(got, cu)
    ri = _units_states(ref) if cu is None else _units_tokens(ref, cu)
    units = list(zip(gi, ri))
    rows_all = sum(r.shape[0] for (_, _), (_, r) in units)
    ss_all = sum(float(np.sum(np.square(r, dtype=np.float64))) for (_, _), (_, r) in units)
    rms_all = np.sqrt(ss_all / max(rows_all, 1))
    # reductions: the largest row norm of the tensor joins the row floor
    peak = max((float(np.max(np.linalg.norm(r.astype(np.float64), axis=1))) for (_, _), (_, r) in units
                if r.shape[0] > 0), default=0.0) if reduction else 0.0
    worst_u, wu_lab, worst_r, wr_lab = 0.0, None, 0.0, None
    for (lab, g), (_, r) in units:
        g = g.astype(np.float64)
        r = r.astype(np.float64)
        err = g - r
        den = max(np.linalg.norm(r), rms_all * np.sqrt(r.shape[0]))
        eu = float(np.linalg.norm(err) / den) if den > 0 else float(np.linalg.norm(err))
        if not np.isfinite(eu) or eu > worst_u:
            worst_u, wu_lab = eu, lab
        rn = np.linalg.norm(r, axis=1)
        rms = max(np.linalg.norm(r) / np.sqrt(r.shape[0]), rms_all, peak)
        scale = np.maximum(rn, rms)
        en = np.linalg.norm(err, axis=1)
        ratio = np.where(scale > 0, en / np.where(scale > 0, scale, 1.0), en)
        i = int(np.argmax(np.where(np.isfinite(ratio), ratio, np.inf)))
        if not np.isfinite(ratio[i]) or ratio[i] > worst_r:
            worst_r, wr_lab = float(ratio[i]), (lab, i)
    return worst_u, wu_lab, worst_r, wr_lab


def check(name, got, ref, tol, cu=None, row_c=ROW_C, reduction=None):
    """Assert the global, per-unit and per-row bars; returns the three measured values.
    reduction: the tensor is one of REDUCTIONS (default: judged from the name's last word)."""
    if reduction is None:
        reduction = name.split()[-1] in REDUCTIONS
    eg = relF(got, ref)
    eu, lu, er, lr = local_errors(got, ref, cu, reduction)
    RECORD.append((name, eg, eu, er, tol))
    unit_tol = row_c * tol if reduction else tol
    assert eg <= tol, f"{name}: rel-Frobenius {eg:.3e} > {tol}"
    assert eu <= unit_tol, f"{name}: unit {lu} error {eu:.3e} of the unit scale > {unit_tol}"
    assert er <= row_c * tol, (f"{name}: unit {lr[0]} row {lr[1]}: error {er:.3e} of the row "
                               f"scale > {row_c} x {tol}")
    return eg, eu, er
