"""Parity tolerance of the CUDA path against the double-precision oracle.

The bound is a max-norm relative error: max_i |got_i - ref_i| / max(max_i |ref_i|, 1e-3), at most 1e-4
for fp32 inputs and 2e-2 for bf16 inputs (fp32 state and accumulation). The elementwise variant
max_i(|got_i - ref_i| / max(|ref_i|, 1e-3)) is computed alongside on every comparison and recorded
(``REPORT``; written as JSON at the end of the session when SSM_PARITY_REPORT names a file);
tests/test_tolerance_reading.py shows that no fp32 evaluation of the recurrence can meet that variant at
1e-4, so it cannot be the bound, and it is recorded, not gated: on outputs near the 1e-3 floor it measures
rounding, not correctness (sums over channels such as dB and dC, and bf16 outputs of the SSD layer whose
operands are rounded to bf16, reach 1e-2 and above there while their max-norm errors stay within bound).
"""
import os

import numpy as np

TOL = {"f32": 1e-4, "bf16": 2e-2}

REPORT = []  # (test id, max-norm error, elementwise error, number of elements)


def _pair(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    return got, ref


def rel_err(got, ref):
    """Max-norm relative error (the gate); the elementwise error of the same pair is recorded in REPORT."""
    got, ref = _pair(got, ref)
    if ref.size == 0:
        return 0.0
    diff = np.abs(got - ref)
    mx = float(np.max(diff) / max(float(np.max(np.abs(ref))), 1e-3))
    ew = float(np.max(diff / np.maximum(np.abs(ref), 1e-3)))
    REPORT.append((os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0], mx, ew, int(ref.size)))
    return mx


def rel_err_elementwise(got, ref):
    got, ref = _pair(got, ref)
    if ref.size == 0:
        return 0.0
    return float(np.max(np.abs(got - ref) / np.maximum(np.abs(ref), 1e-3)))


def last_elementwise():
    """Elementwise error of the most recent rel_err() comparison."""
    return REPORT[-1][2] if REPORT else 0.0
