"""Helpers of the GPU parity tests: tolerance check, host copies, oracle calls."""
from __future__ import annotations

import numpy as np

# |y - y_ref| <= 1e-2 * (|y_ref| + rms(y_ref)), elementwise, rms over the whole tensor:
# bf16 output rounding contributes at most 2^-9 |y_ref| and fp32 accumulation over
# K <= 16384 terms about 1e-6 * rms, so a correct kernel sits ~20x inside the bound
# while a dropped term, a wrong row or a wrong weight lands far outside it.
REL_TOL = 1e-2


def tol_report(y, y_ref):
    y = np.asarray(y, dtype=np.float64)
    y_ref = np.asarray(y_ref, dtype=np.float64)
    rms = float(np.sqrt(np.mean(y_ref ** 2))) if y_ref.size else 0.0
    err = np.abs(y - y_ref)
    bound = REL_TOL * (np.abs(y_ref) + rms)
    bad = err > bound
    worst = float(np.max(err / np.maximum(bound, 1e-300))) if y.size else 0.0
    return int(bad.sum()), worst


def assert_close(y, y_ref, what=""):
    nbad, worst = tol_report(y, y_ref)
    assert nbad == 0, f"{what}: {nbad} of {np.size(y_ref)} elements outside tolerance (worst {worst:.3g}x bound)"
    return worst


def to_f64(oracle, t):
    from split_switched_decode_gb300 import inputs
    return oracle.bf16_to_f64(inputs.bits(t))


def topk_gap(logits_row, k):
    """Smallest gap between adjacent sorted logits among the top k+1 (near-tie size)."""
    s = np.sort(np.asarray(logits_row, dtype=np.float64))[::-1][: k + 1]
    return float(np.min(np.abs(np.diff(s)))) if s.size > 1 else float("inf")
