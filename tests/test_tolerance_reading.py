"""Why the parity bound is a max-norm relative error.

The bound reads max|y_gpu - y_ref| / max(|y_ref|, 1e-3). Read elementwise (each |error| divided by its own
max(|y_ref_i|, 1e-3)), it would ask for about 1e-7 absolute accuracy on every output near zero. A
correctly rounded float32 evaluation of one decode step already misses that: outputs are sums of 16
products of order one, so their float32 rounding is a few 1e-8 to 1e-7 absolute. The max-norm reading
(one maximum over the whole tensor, divided by max(max|y_ref|, 1e-3)) is met by float32 with three
orders of magnitude to spare. This test keeps that evidence: float32 numpy against the fp64 oracle.
"""
import numpy as np

import ssm_inputs
from tolerance import TOL, rel_err, rel_err_elementwise


def test_fp32_rounding_fails_elementwise_but_meets_max_norm(orc):
    rng = np.random.default_rng(0)
    batch, D, N = 32, 256, 16
    state = rng.standard_normal((batch, D, N)).astype(np.float32)
    x = rng.standard_normal((batch, D)).astype(np.float32)
    dt = np.log1p(np.exp(rng.normal(-2.0, 1.0, (batch, D)))).astype(np.float32)
    B = rng.standard_normal((batch, N)).astype(np.float32)
    C = rng.standard_normal((batch, N)).astype(np.float32)
    A_log = ssm_inputs.a_log_s4d(D, N)
    ref_state, ref_y = orc.scan_step(state.astype(np.float64), x, dt, A_log, B, C, disc="euler")
    # float32 evaluation of the same step, every operation rounded to float32
    A = (-np.exp(A_log.astype(np.float64))).astype(np.float32)
    abar = np.exp((dt[..., None] * A[None]).astype(np.float32)).astype(np.float32)
    bx = ((dt * x)[..., None] * B[:, None, :]).astype(np.float32)
    h = (abar * state + bx).astype(np.float32)
    y = np.zeros((batch, D), np.float32)
    for n in range(N):
        y = (y + C[:, None, n] * h[..., n]).astype(np.float32)
    assert rel_err(y, ref_y) < TOL["f32"] / 100
    assert rel_err(h, ref_state) < TOL["f32"] / 100
    assert rel_err_elementwise(y, ref_y) > TOL["f32"]
