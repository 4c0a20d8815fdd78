"""Parity tolerance of the CUDA path against the double-precision oracle.

The bound is a max-norm relative error: max_i |got_i - ref_i| / max(max_i |ref_i|, 1e-3), at most 1e-4
for fp32 inputs and 2e-2 for bf16 inputs (fp32 state and accumulation). The elementwise variant
max_i(|got_i - ref_i| / max(|ref_i|, 1e-3)) is reported alongside; tests/test_tolerance_reading.py shows
that no fp32 evaluation of the recurrence can meet that variant at 1e-4, so it cannot be the bound.
"""
import numpy as np

TOL = {"f32": 1e-4, "bf16": 2e-2}


def rel_err(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    if ref.size == 0:
        return 0.0
    return float(np.max(np.abs(got - ref)) / max(float(np.max(np.abs(ref))), 1e-3))


def rel_err_elementwise(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    if ref.size == 0:
        return 0.0
    return float(np.max(np.abs(got - ref) / np.maximum(np.abs(ref), 1e-3)))
