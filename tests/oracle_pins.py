"""Pins of the CPU oracle to facts fixed outside it: values the pages print for their worked examples,
closed forms, invariants, and independent evaluations (the 1-semiseparable matrix, the convolution
kernel of a time-invariant system, the associative combine).

Every pin takes an ``oracle.Oracle`` handle, so the same pins run against the real build and against
builds with planted mistakes (tests/test_oracle_mutants.py), each of which must fail at least one pin.
"""
import math

import numpy as np

import oracle as oracle_mod
from golden_io import half_unit, load


def _softplus(z):
    return math.log1p(math.exp(z))


def _chan1(seq, dtype=np.float64):
    """[L] -> [1, L, 1] (one batch element, one channel)."""
    return np.asarray(seq, dtype).reshape(1, -1, 1)


def _bc(rows):
    """list of N-vectors per step -> [1, L, N]."""
    return np.asarray(rows, np.float64).reshape(1, len(rows), -1)


def _close(got, want, tol, what):
    got, want = np.asarray(got, np.float64), np.asarray(want, np.float64)
    err = np.max(np.abs(got - want)) if got.size else 0.0
    assert err <= tol, f"{what}: got {got}, want {want} (|diff| {err:.3g} > {tol:.3g})"


def _rel(got, want, tol, what):
    got, want = np.asarray(got, np.float64), np.asarray(want, np.float64)
    err = np.max(np.abs(got - want) / np.abs(want))
    assert err <= tol, f"{what}: got {got}, want {want} (rel {err:.3g} > {tol:.3g})"


def _step_abar(orc, dt, A_log, disc):
    """Abar of one step: start from state 1, input 0."""
    N = len(A_log)
    st, _ = orc.scan_step(np.ones((1, 1, N)), np.zeros((1, 1)), np.full((1, 1), dt),
                          np.asarray(A_log, np.float64).reshape(1, N), np.zeros((1, N)),
                          np.zeros((1, N)), disc=disc, f64=True)
    return st.reshape(N)


def _step_bbar(orc, dt, A_log, B, disc):
    """Bbar of one step: start from state 0, input 1."""
    N = len(A_log)
    st, _ = orc.scan_step(np.zeros((1, 1, N)), np.ones((1, 1)), np.full((1, 1), dt),
                          np.asarray(A_log, np.float64).reshape(1, N), np.asarray(B, np.float64).reshape(1, N),
                          np.zeros((1, N)), disc=disc, f64=True)
    return st.reshape(N)


# --- "Mathematical Prerequisites for Mamba": leaky bucket, closed form h(t) = 1 - e^{-t} -------------

def pin_leaky_bucket_closed_form(orc):
    g = load("leaky_bucket.txt")
    L = 64
    ones = np.ones(L)
    y, st = orc.scan_fwd(_chan1(ones), _chan1(ones), np.zeros((1, 1)), _bc([[1.0]] * L), _bc([[1.0]] * L),
                         disc="zoh", f64=True)
    exact = 1.0 - np.exp(-np.arange(1, L + 1, dtype=np.float64))
    _close(y[0, :, 0], exact, 1e-13, "leaky bucket vs 1 - e^-t")
    _close(st[0, 0, 0], exact[-1], 1e-13, "leaky bucket final state")
    _close(y[0, :4, 0], g["h"], 5e-4, "leaky bucket vs printed samples")
    _close(_step_abar(orc, 1.0, [0.0], "zoh"), g["abar"], 5e-4, "Abar at Delta = 1")
    _close(_step_bbar(orc, 1.0, [0.0], [1.0], "zoh"), g["bbar"], 5e-4, "Bbar at Delta = 1")


def pin_ema_identity(orc):
    """ZOH with A = -1, B = 1: Abar + Bbar = 1, so h_t = Abar h_{t-1} + (1 - Abar) x_t (an exponential
    moving average), "Mathematical Prerequisites for Mamba" s5."""
    rng = np.random.default_rng(11)
    L = 40
    x = rng.standard_normal(L)
    dt = rng.uniform(0.01, 3.0, L)
    y, _ = orc.scan_fwd(_chan1(x), _chan1(dt), np.zeros((1, 1)), _bc([[1.0]] * L), _bc([[1.0]] * L),
                        disc="zoh", f64=True)
    h = y[0, :, 0]
    prev = 0.0
    for t in range(L):
        a = math.exp(-dt[t])
        want = a * prev + (1.0 - a) * x[t]
        assert abs(h[t] - want) <= 1e-13 * max(1.0, abs(want)), f"EMA form broken at t={t}"
        lo, hi = min(prev, x[t]), max(prev, x[t])
        assert lo - 1e-15 <= h[t] <= hi + 1e-15, "EMA step is not a convex combination"
        prev = h[t]


# --- "State Space Models & Mamba" chapter: scalar Euler traces --------------------------------------

def _scalar_euler(orc, xs, bias):
    dts = [_softplus(xv + bias) for xv in xs]
    L = len(xs)
    y, _ = orc.scan_fwd(_chan1(xs), _chan1(dts), np.zeros((1, 1)), _bc([[1.0]] * L), _bc([[1.0]] * L),
                        disc="euler", f64=True)
    return y[0, :, 0], dts


def pin_euler_scalar_trace(orc):
    g = load("euler_scalar_trace.txt")
    h, dts = _scalar_euler(orc, g["x"], g["bias"][0])
    _rel(h, g["h"], 2e-15, "16-digit Euler trace")
    _close(dts, g["delta"], 5e-7, "trace Delta")
    abars = [_step_abar(orc, d, [0.0], "euler")[0] for d in dts]
    _close(abars[1:], g["abar_2_4"], 5e-7, "trace Abar_2..4")
    _close(abars[0], math.exp(-dts[0]), 1e-15, "trace Abar_1 = exp(-Delta_1)")


def _printed(got, g, graw, key, drift, what):
    """Within the print's own rounding plus a relative drift from rounded intermediates."""
    want = np.asarray(g[key])
    tol = np.asarray(half_unit(graw[key])) + drift * np.abs(want)
    err = np.abs(np.asarray(got) - want)
    assert np.all(err <= tol), f"{what}: got {got}, want {want} (|diff| {err} > {tol})"


def pin_active_recall_traces(orc):
    g = load("active_recall_traces.txt")
    graw = load("active_recall_traces.txt", raw=True)
    h3, _ = _scalar_euler(orc, g["q3_x"], g["q3_bias"][0])
    _printed(h3, g, graw, "q3_h", 1e-5, "Q3 trace")
    h4, d4 = _scalar_euler(orc, g["q4_x"], g["q4_bias"][0])
    _printed(h4, g, graw, "q4_h", 1e-5, "Q4 trace")
    _printed(d4, g, graw, "q4_delta", 0.0, "Q4 Delta")


# --- "Understanding Mamba": time-invariant and selective ZOH examples ---------------------------------

def _lti_setup(g):
    A = np.asarray(g["A"])
    A_log = np.log(-A).reshape(1, -1)
    return A_log


def pin_lti_zoh_example(orc):
    g = load("lti_zoh_n2.txt")
    A_log = _lti_setup(g)
    x = g["x"]
    L = len(x)
    B = _bc([g["B"]] * L)
    C = _bc([g["C"]] * L)
    dt = [g["delta"][0]] * L
    y, _ = orc.scan_fwd(_chan1(x), _chan1(dt), A_log, B, C, disc="zoh", f64=True)
    _close(y[0, :, 0], g["y"], 5e-4, "LTI y")
    for t in range(L):
        _, st = orc.scan_fwd(_chan1(x[:t + 1]), _chan1(dt[:t + 1]), A_log, B[:, :t + 1], C[:, :t + 1],
                             disc="zoh", f64=True)
        _close(st[0, 0], g[f"h{t + 1}"], 5e-4, f"LTI h{t + 1}")
    _close(_step_abar(orc, 1.0, A_log[0], "zoh"), g["abar"], 5e-4, "LTI Abar")
    _close(_step_bbar(orc, 1.0, A_log[0], g["B"], "zoh"), g["bbar"], 5e-4, "LTI Bbar")


def pin_convolution_view(orc):
    """Time-invariant case: y = x * K with K_i = C Abar^i Bbar ("Understanding Mamba" s3.1)."""
    g = load("lti_zoh_n2.txt")
    A_log = _lti_setup(g)
    L = 4
    B = _bc([g["B"]] * L)
    C = _bc([g["C"]] * L)
    dt = [1.0] * L
    impulse = [1.0, 0.0, 0.0, 0.0]
    K, _ = orc.scan_fwd(_chan1(impulse), _chan1(dt), A_log, B, C, disc="zoh", f64=True)
    K = K[0, :, 0]
    _close(K, g["K"], 5e-4, "impulse response vs printed taps")
    y, _ = orc.scan_fwd(_chan1(g["x"]), _chan1(dt), A_log, B, C, disc="zoh", f64=True)
    _close(y[0, :, 0], np.convolve(g["x"], K)[:L], 1e-14, "scan vs numpy.convolve with its own taps")
    # longer random time-invariant system against the independent kernel evaluation
    rng = np.random.default_rng(5)
    L, N = 50, 4
    A_log = rng.uniform(-1.0, 1.0, N)
    Bv, Cv = rng.standard_normal(N), rng.standard_normal(N)
    xs = rng.standard_normal(L)
    for disc in ("zoh", "euler"):
        y, _ = orc.scan_fwd(_chan1(xs), _chan1([0.3] * L), A_log.reshape(1, N), _bc([Bv] * L),
                            _bc([Cv] * L), disc=disc, f64=True)
        ref, _ = oracle_mod.lti_conv(xs, 0.3, A_log, Bv, Cv, disc=disc)
        _close(y[0, :, 0], ref, 1e-12 * max(1.0, np.abs(ref).max()), f"scan vs convolution kernel ({disc})")


def pin_selective_zoh_example(orc):
    g = load("selective_zoh_n2.txt")
    A_log = np.log(-np.asarray(g["A"])).reshape(1, -1)
    x = g["x"]
    L = len(x)
    dts = [_softplus(2.0 * v) for v in x]
    _close(dts, g["delta"], 5e-4, "selective Delta")
    BC = _bc([[0.4 * v, 0.4 * v] for v in x])
    y, _ = orc.scan_fwd(_chan1(x), _chan1(dts), A_log, BC, BC, disc="zoh", f64=True)
    _close(y[0, :, 0], g["y"], 5e-4, "selective y")
    for t in range(L):
        _, st = orc.scan_fwd(_chan1(x[:t + 1]), _chan1(dts[:t + 1]), A_log, BC[:, :t + 1], BC[:, :t + 1],
                             disc="zoh", f64=True)
        _close(st[0, 0], g[f"h{t + 1}"], 5e-4, f"selective h{t + 1}")
        _close(_step_abar(orc, dts[t], A_log[0], "zoh"), g[f"abar{t + 1}"], 5e-4, f"selective Abar{t + 1}")


def _combine(P, Q):
    """(a_i, b_i) . (a_j, b_j) = (a_i a_j, a_j b_i + b_j), i before j ("Understanding Mamba" Eq. (8))."""
    return (P[0] * Q[0], Q[0] * P[1] + Q[1])


def pin_combine_tree(orc):
    g = load("combine_tree.txt")
    pairs = list(zip(g["pairs_a"], g["pairs_b"]))
    P12 = _combine(pairs[0], pairs[1])
    P34 = _combine(pairs[2], pairs[3])
    P14 = _combine(P12, P34)
    _close(P12, g["P12"], 2e-3, "P12")
    _close(P34, g["P34"], 2e-3, "P34")
    _close(P14, g["P14"], 2e-3, "P14")
    # the oracle's exact pairs for state channel 0 of the selective example
    sel = load("selective_zoh_n2.txt")
    A_log = np.log(-np.asarray(sel["A"])).reshape(1, -1)
    x = sel["x"]
    dts = [_softplus(2.0 * v) for v in x]
    exact = []
    for t in range(4):
        a = _step_abar(orc, dts[t], A_log[0], "zoh")[0]
        bx = _step_bbar(orc, dts[t], A_log[0], [0.4 * x[t], 0.4 * x[t]], "zoh")[0] * x[t]
        exact.append((a, bx))
    _close([p[0] for p in exact], g["pairs_a"], 5e-4, "oracle Abar pairs")
    _close([p[1] for p in exact], g["pairs_b"], 5e-4, "oracle Bbar x pairs")
    tree = _combine(_combine(exact[0], exact[1]), _combine(exact[2], exact[3]))
    fold = exact[0]
    for p in exact[1:]:
        fold = _combine(fold, p)
    BC = _bc([[0.4 * v, 0.4 * v] for v in x])
    _, st = orc.scan_fwd(_chan1(x), _chan1(dts), A_log, BC, BC, disc="zoh", f64=True)
    _close(tree[1], st[0, 0, 0], 1e-14, "tree combine vs oracle state")
    _close(fold[1], st[0, 0, 0], 1e-14, "left fold vs oracle state")
    _close(st[0, 0, 0], g["h4"], 5e-4, "h4")


def pin_small_delta_limit(orc):
    g = load("small_delta.txt")
    A_log = np.log(-np.asarray(g["A"]))
    dt = g["delta"][0]
    _close(_step_abar(orc, dt, A_log, "zoh"), g["abar"], 5e-6, "small-Delta Abar")
    bz = _step_bbar(orc, dt, A_log, g["B"], "zoh")
    _close(bz, g["bbar"], 5e-6, "small-Delta ZOH Bbar")
    be = _step_bbar(orc, dt, A_log, g["B"], "euler")
    _close(be, g["delta_b"], 1e-15, "Euler Bbar = Delta B")
    # ZOH Bbar = Delta B + O(Delta^2): |Bbar_zoh - Delta B| <= |A| Delta^2 |B| / 2
    bound = np.abs(np.asarray(g["A"])) * dt * dt * np.abs(np.asarray(g["B"])) / 2
    assert np.all(np.abs(bz - be) <= bound * 1.0001), "ZOH and Euler do not agree to second order"
    assert np.all(np.abs(bz - be) >= bound * 0.98), "ZOH second-order term has the wrong size"


def pin_unit_input_two_step(orc):
    g = load("unit_input_two_step.txt")
    dts = g["delta"]
    Bs = _bc([[1.0 / d] for d in dts])   # Euler Bbar = Delta B = 1
    y, _ = orc.scan_fwd(_chan1(g["u"]), _chan1(dts), np.zeros((1, 1)), Bs, _bc([[1.0]] * 2),
                        disc="euler", f64=True)
    exact = [5.0, 5.0 * math.exp(-0.05) + 5.0]
    _close(y[0, :, 0], exact, 1e-13, "two-step exact")
    _close(y[0, :, 0], g["h"], g["page_rounding"][0], "two-step vs page")


# --- invariants -----------------------------------------------------------------------------------

def pin_delta_limits(orc):
    """Delta -> 0 leaves the state as it is; ZOH with Delta -> infinity resets it to -B x / A (to x when
    A = -1, B = 1: "resets to the current input"); Euler then gives Delta B x (no such limit)."""
    rng = np.random.default_rng(3)
    batch, L, D, N = 2, 5, 3, 4
    A_log = rng.uniform(-0.5, 1.5, (D, N))
    A = -np.exp(A_log)
    h0 = rng.standard_normal((batch, D, N))
    x = rng.standard_normal((batch, L, D))
    B = rng.standard_normal((batch, L, N))
    C = rng.standard_normal((batch, L, N))
    for disc in ("euler", "zoh"):
        y, st = orc.scan_fwd(x, np.full((batch, L, D), 1e-30), A_log, B, C, disc=disc, h0=h0, f64=True)
        _close(st, h0, 1e-14, f"Delta -> 0 keeps the state ({disc})")
        want = np.einsum("bln,bdn->bld", C, h0)
        _close(y, want, 1e-13, f"Delta -> 0 readout ({disc})")
    big = 1e4
    y, st = orc.scan_fwd(x, np.full((batch, L, D), big), A_log, B, C, disc="zoh", h0=h0, f64=True)
    want = -B[:, -1, None, :] * x[:, -1, :, None] / A[None]
    _close(st, want, 1e-12, "ZOH Delta -> inf resets to -B x / A")
    ones = np.ones((batch, L, N))
    _, st = orc.scan_fwd(x, np.full((batch, L, D), big), np.zeros((D, N)), ones, ones, disc="zoh",
                         h0=h0, f64=True)
    _close(st, np.broadcast_to(x[:, -1, :, None], st.shape), 1e-12, "reset to the current input")
    _, st = orc.scan_fwd(x, np.full((batch, L, D), 50.0), A_log, B, C, disc="euler", h0=h0, f64=True)
    want = 50.0 * B[:, -1, None, :] * x[:, -1, :, None]
    _close(st, want, 1e-12 * np.abs(want).max(), "Euler with a large step gives Delta B x")


def pin_brute_force_1ss(orc):
    """Sequential oracle == the 1-semiseparable matrix product on tiny random inputs, both modes."""
    rng = np.random.default_rng(7)
    for trial in range(4):
        batch, L, D, N = 2, int(rng.integers(1, 40)), int(rng.integers(1, 4)), int(rng.integers(1, 5))
        x = rng.standard_normal((batch, L, D))
        dt = np.log1p(np.exp(rng.normal(-1.0, 1.0, (batch, L, D))))
        A_log = rng.uniform(-1.0, 1.5, (D, N))
        B = rng.standard_normal((batch, L, N))
        C = rng.standard_normal((batch, L, N))
        h0 = rng.standard_normal((batch, D, N)) if trial % 2 else None
        for disc in ("euler", "zoh"):
            y, st = orc.scan_fwd(x, dt, A_log, B, C, disc=disc, h0=h0, f64=True)
            yb, sb = oracle_mod.scan_1ss(x, dt, A_log, B, C, disc=disc, h0=h0)
            scale = max(1.0, np.abs(yb).max())
            _close(y, yb, 1e-12 * scale, f"oracle vs 1-SS y ({disc}, trial {trial})")
            _close(st, sb, 1e-12 * max(1.0, np.abs(sb).max()), f"oracle vs 1-SS state ({disc})")


def pin_split_and_step(orc):
    """fwd over [0, L) == fwd over [0, k) then fwd from that state over [k, L) == fwd then step calls
    (associativity of the step, "Understanding Mamba" s7.1); a subset of channels agrees with the full
    evaluation."""
    rng = np.random.default_rng(9)
    batch, L, D, N, k = 2, 30, 3, 4, 17
    x = rng.standard_normal((batch, L, D))
    dt = np.log1p(np.exp(rng.normal(-1.0, 1.0, (batch, L, D))))
    A_log = rng.uniform(-1.0, 1.5, (D, N))
    B = rng.standard_normal((batch, L, N))
    C = rng.standard_normal((batch, L, N))
    for disc in ("euler", "zoh"):
        y, st = orc.scan_fwd(x, dt, A_log, B, C, disc=disc, f64=True)
        y1, s1 = orc.scan_fwd(x[:, :k], dt[:, :k], A_log, B[:, :k], C[:, :k], disc=disc, f64=True)
        y2, s2 = orc.scan_fwd(x[:, k:], dt[:, k:], A_log, B[:, k:], C[:, k:], disc=disc, h0=s1, f64=True)
        _close(np.concatenate([y1, y2], 1), y, 1e-13, f"split fwd y ({disc})")
        _close(s2, st, 1e-13, f"split fwd state ({disc})")
        s = s1.copy()
        for t in range(k, L):
            s, yt = orc.scan_step(s, x[:, t], dt[:, t], A_log, B[:, t], C[:, t], disc=disc, f64=True)
            _close(yt, y[:, t], 1e-13, f"step y at t={t} ({disc})")
        _close(s, st, 1e-13, f"step state ({disc})")
        chans = [5, 0, 3]
        ys, ss = orc.scan_fwd(x, dt, A_log, B, C, disc=disc, channels=chans, f64=True)
        for i, c in enumerate(chans):
            b, d = divmod(c, D)
            _close(ys[i], y[b, :, d], 0.0, "channel subset y")
            _close(ss[i], st[b, d], 0.0, "channel subset state")


# --- layer pieces around the scan ------------------------------------------------------------------------

def pin_softplus_inside_scan(orc):
    """The chapter's 16-digit trace with Delta_t = softplus(x_t - 5) formed by the scan itself from the raw
    projection x_t and the bias -5 ("Understanding Mamba" Eq. (6): softplus(b_Delta + w_Delta x_t)), for the
    prefill and for four decode steps in a row."""
    g = load("euler_scalar_trace.txt")
    xs = np.asarray(g["x"], np.float64)
    L = len(xs)
    y, _ = orc.scan_fwd(_chan1(xs), _chan1(xs), np.zeros((1, 1)), _bc([[1.0]] * L), _bc([[1.0]] * L),
                        disc="euler", f64=True, delta_bias=np.asarray(g["bias"], np.float64), delta_softplus=True)
    _rel(y[0, :, 0], g["h"], 2e-15, "trace with in-scan softplus")
    st = np.zeros((1, 1, 1))
    hs = []
    for t in range(L):
        st, yt = orc.scan_step(st, xs[t].reshape(1, 1), xs[t].reshape(1, 1), np.zeros((1, 1)), np.ones((1, 1)),
                               np.ones((1, 1)), disc="euler", f64=True, delta_bias=np.asarray(g["bias"], np.float64),
                               delta_softplus=True)
        hs.append(yt[0, 0])
    _rel(hs, g["h"], 2e-15, "trace with in-step softplus")


def pin_feedthrough_and_gate(orc):
    """Closed forms of y_out = (C h + D x) * SiLU(z), SiLU(v) = v sigma(v) ("Understanding Mamba" Eq. (1)/(3),
    s2.1: D is a direct pipe from x to the output, added after everything else; Eq. (9), s8.1: the gate)."""
    rng = np.random.default_rng(3)
    L = 5
    x = rng.standard_normal(L)
    z = rng.standard_normal(L)
    ones, zeros = _bc([[1.0]] * L), _bc([[0.0]] * L)
    dt = _chan1(np.full(L, 0.3))
    # C = 0: the bucket never reaches the output, only the pipe does
    y, _ = orc.scan_fwd(_chan1(x), dt, np.zeros((1, 1)), ones, zeros, disc="zoh", f64=True, D_skip=np.array([0.5]))
    _close(y[0, :, 0], 0.5 * x, 1e-15, "feedthrough alone")
    y, _ = orc.scan_fwd(_chan1(x), dt, np.zeros((1, 1)), ones, zeros, disc="zoh", f64=True, D_skip=np.array([0.5]),
                        z=_chan1(z))
    _close(y[0, :, 0], 0.5 * x * z / (1.0 + np.exp(-z)), 1e-15, "gated feedthrough")
    # one step from rest: x = 1, raw delta 0 -> Delta = softplus(0) = ln 2, A = -1, B = C = 1, Euler: h = ln 2
    y, _ = orc.scan_fwd(_chan1([1.0]), _chan1([0.0]), np.zeros((1, 1)), _bc([[1.0]]), _bc([[1.0]]), disc="euler",
                        f64=True, delta_softplus=True, D_skip=np.array([0.5]), z=_chan1([1.0]))
    _close(y[0, 0, 0], (0.5 + math.log(2.0)) / (1.0 + math.exp(-1.0)), 1e-15, "one gated step")
    # SiLU(0) = 0 closes the gate; a large positive z passes y through, a large negative one blocks it
    base, _ = orc.scan_fwd(_chan1(x), dt, np.zeros((1, 1)), ones, ones, disc="zoh", f64=True)
    for zv, want in ((0.0, 0.0), (60.0, 60.0), (-60.0, 0.0)):
        y, _ = orc.scan_fwd(_chan1(x), dt, np.zeros((1, 1)), ones, ones, disc="zoh", f64=True,
                            z=_chan1(np.full(L, zv)))
        _close(y[0, :, 0], base[0, :, 0] * want, 1e-12 * max(1.0, abs(want)), f"gate at z = {zv}")


# --- backward pass (gradients of the prefill scan) -------------------------------------------------------
# The pages fix only that the backward pass recomputes h ("State Space Models & Mamba" chapter, the fused-
# kernel paragraph); the gradients themselves are fixed by the forward definition, so they are pinned to
# central finite differences of the forward oracle, to the adjoint of the convolution view, and to closed
# forms of one step.

def _bwd_problem(rng, batch, L, D, N, A_lo, A_hi, dt_lo, dt_hi):
    x = rng.standard_normal((batch, L, D))
    dt = rng.uniform(dt_lo, dt_hi, (batch, L, D))
    A_log = np.log(rng.uniform(A_lo, A_hi, (D, N)))
    B = rng.standard_normal((batch, L, N))
    C = rng.standard_normal((batch, L, N))
    dy = rng.standard_normal((batch, L, D))
    h0 = rng.standard_normal((batch, D, N))
    dfinal = rng.standard_normal((batch, D, N))
    return x, dt, A_log, B, C, dy, h0, dfinal


def _fd_check(orc, disc, x, dt, A_log, B, C, dy, h0, dfinal, tol, what):
    g = orc.scan_bwd(x, dt, A_log, B, C, dy, disc=disc, h0=h0, dfinal=dfinal, f64=True)
    inputs = {"x": x, "dt": dt, "A_log": A_log, "B": B, "C": C, "h0": h0}

    def J(vals):
        y, f = orc.scan_fwd(vals["x"], vals["dt"], vals["A_log"], vals["B"], vals["C"], disc=disc, h0=vals["h0"],
                            f64=True)
        return float(np.sum(y * dy) + np.sum(f * dfinal))
    for name, key in (("x", "dx"), ("dt", "ddelta"), ("A_log", "dA_log"), ("B", "dB"), ("C", "dC"), ("h0", "dh0")):
        arr = inputs[name]
        fd = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            eps = 1e-6 * max(1.0, abs(arr[idx]))
            vals = dict(inputs)
            p = arr.copy(); p[idx] += eps
            m = arr.copy(); m[idx] -= eps
            vals[name] = p; jp = J(vals)
            vals[name] = m; jm = J(vals)
            fd[idx] = (jp - jm) / (2.0 * eps)
        scale = max(np.abs(fd).max(), 1e-300)
        _close(g[key], fd, tol * scale, f"{what}: {key} vs central differences ({disc})")


def pin_bwd_finite_differences(orc):
    """Every gradient equals the central difference of sum(dy y) + sum(dfinal final_state) computed with the
    forward oracle, both discretisations, with an initial state; a second case keeps |delta A| below 1e-3,
    where the ZOH gradient in A goes through its small-argument series."""
    rng = np.random.default_rng(21)
    for disc in ("euler", "zoh"):
        _fd_check(orc, disc, *_bwd_problem(rng, 2, 6, 2, 3, 0.3, 3.0, 0.05, 0.7), 1e-7, "random")
    _fd_check(orc, "zoh", *_bwd_problem(rng, 1, 5, 2, 3, 1e-3, 1e-2, 0.01, 0.1), 1e-6, "small delta A")


def pin_bwd_convolution_adjoint(orc):
    """Time-invariant case (fixed delta, B, C; zero initial state): y = x * K ("Understanding Mamba" s3.1), so
    dJ/dx_j = sum_{t >= j} dy_t K_{t-j}, the correlation of dy with the kernel's taps."""
    rng = np.random.default_rng(22)
    L, N = 12, 3
    A_log = rng.uniform(-1.0, 1.0, N)
    Bv, Cv = rng.standard_normal(N), rng.standard_normal(N)
    x, dy = rng.standard_normal(L), rng.standard_normal(L)
    for disc in ("euler", "zoh"):
        _, K = oracle_mod.lti_conv(x, 0.4, A_log, Bv, Cv, disc=disc)
        want = np.array([np.sum(dy[j:] * K[:L - j]) for j in range(L)])
        g = orc.scan_bwd(_chan1(x), _chan1(np.full(L, 0.4)), A_log.reshape(1, N), np.tile(Bv, (1, L, 1)),
                         np.tile(Cv, (1, L, 1)), _chan1(dy), disc=disc, f64=True)
        _close(g["dx"][0, :, 0], want, 1e-12 * np.abs(want).max(), f"dx as the correlation with K ({disc})")


def pin_bwd_one_step(orc):
    """One step, one entry, by hand: h = a h0 + bf B x, y = C h, J = dy y + df h, lambda = C dy + df:
    dx = lambda bf B, dh0 = lambda a, dC = dy h, dB = lambda bf x, and
    ddelta = lambda (A a h0 + B x) (Euler, bf = delta) or lambda (A a h0 + a B x) (ZOH, bf = (a - 1)/A)."""
    x, dt, A, h0, Bv, Cv, dy, df = 0.7, 0.3, -1.5, 0.4, 1.2, -0.8, 0.9, 0.25
    a = math.exp(dt * A)
    lam = Cv * dy + df
    for disc, bf, dd, dA in (
            ("euler", dt, lam * (A * a * h0 + Bv * x), lam * h0 * dt * a),
            ("zoh", (a - 1.0) / A, lam * (A * a * h0 + a * Bv * x),
             lam * h0 * dt * a + lam * x * Bv * (dt * A * a - (a - 1.0)) / (A * A))):
        h = a * h0 + bf * Bv * x
        g = orc.scan_bwd(_chan1([x]), _chan1([dt]), np.full((1, 1), math.log(-A)), _bc([[Bv]]), _bc([[Cv]]),
                         _chan1([dy]), disc=disc, h0=np.full((1, 1, 1), h0), dfinal=np.full((1, 1, 1), df), f64=True)
        for key, want in (("dx", lam * bf * Bv), ("dh0", lam * a), ("dC", dy * h), ("dB", lam * bf * x),
                          ("ddelta", dd), ("dA_log", dA * A)):
            _close(np.ravel(g[key])[0], want, 1e-14, f"one step {key} ({disc})")


def pin_bwd_split(orc):
    """Reverse-time associativity: the gradients over [0, L) equal those of [k, L) (started from the state at
    k) followed by those of [0, k) with dfinal = the second half's dJ/dh0; dA_log and the per-step gradients
    add up piecewise."""
    rng = np.random.default_rng(23)
    x, dt, A_log, B, C, dy, h0, dfinal = _bwd_problem(rng, 2, 20, 3, 4, 0.3, 3.0, 0.05, 0.7)
    k = 8
    for disc in ("euler", "zoh"):
        g = orc.scan_bwd(x, dt, A_log, B, C, dy, disc=disc, h0=h0, dfinal=dfinal, f64=True)
        _, s1 = orc.scan_fwd(x[:, :k], dt[:, :k], A_log, B[:, :k], C[:, :k], disc=disc, h0=h0, f64=True)
        g2 = orc.scan_bwd(x[:, k:], dt[:, k:], A_log, B[:, k:], C[:, k:], dy[:, k:], disc=disc, h0=s1,
                          dfinal=dfinal, f64=True)
        g1 = orc.scan_bwd(x[:, :k], dt[:, :k], A_log, B[:, :k], C[:, :k], dy[:, :k], disc=disc, h0=h0,
                          dfinal=g2["dh0"], f64=True)
        for key in ("dx", "ddelta", "dB", "dC"):
            _close(np.concatenate([g1[key], g2[key]], 1), g[key], 1e-12, f"split {key} ({disc})")
        _close(g1["dA_log"] + g2["dA_log"], g["dA_log"], 1e-12, f"split dA_log ({disc})")
        _close(g1["dh0"], g["dh0"], 1e-12, f"split dh0 ({disc})")


def pin_bwd_channel_subset(orc):
    """The per-channel outputs of a channel subset equal the full evaluation's (dx, ddelta, dh0), and the
    per-channel contributions add up to the full dA_log, dB and dC."""
    rng = np.random.default_rng(24)
    batch, L, D, N = 2, 9, 3, 4
    x, dt, A_log, B, C, dy, h0, dfinal = _bwd_problem(rng, batch, L, D, N, 0.3, 3.0, 0.05, 0.7)
    g = orc.scan_bwd(x, dt, A_log, B, C, dy, disc="zoh", h0=h0, dfinal=dfinal, f64=True)
    chans = [4, 1, 5, 0, 2, 3]
    gs = orc.scan_bwd(x, dt, A_log, B, C, dy, disc="zoh", h0=h0.reshape(batch * D, N)[chans],
                      dfinal=dfinal.reshape(batch * D, N)[chans], channels=chans, f64=True)
    dA = np.zeros((D, N))
    dB = np.zeros((batch, L, N))
    dC = np.zeros((batch, L, N))
    for i, c in enumerate(chans):
        b, d = divmod(c, D)
        _close(gs["dx"][i], g["dx"][b, :, d], 1e-14, "subset dx")
        _close(gs["ddelta"][i], g["ddelta"][b, :, d], 1e-14, "subset ddelta")
        _close(gs["dh0"][i], g["dh0"][b, d], 1e-14, "subset dh0")
        dA[d] += gs["dA_log"][i]
        dB[b] += gs["dB"][i]
        dC[b] += gs["dC"][i]
    _close(dA, g["dA_log"], 1e-13, "subset dA_log sum")
    _close(dB, g["dB"], 1e-13, "subset dB sum")
    _close(dC, g["dC"], 1e-13, "subset dC sum")


# --- Mamba-2 SSD layer (scalar A per head) -----------------------------------------------------------------

def _ssd_problem(rng, batch, L, H, P, N):
    x = rng.standard_normal((batch, L, H, P))
    dt = np.log1p(np.exp(rng.normal(-1.0, 1.0, (batch, L, H))))
    A_log = rng.uniform(-1.0, 1.5, H)
    B = rng.standard_normal((batch, L, N))
    C = rng.standard_normal((batch, L, N))
    h0 = rng.standard_normal((batch, H, P, N))
    return x, dt, A_log, B, C, h0


def pin_ssd_is_the_scan_with_shared_decay(orc):
    """A = a I per head is the diagonal scan with A_log[d, n] = A_log[h] for all n and delta shared by the
    head's P channels (d = h P + p): ssd_fwd equals scan_fwd on those broadcast arguments."""
    rng = np.random.default_rng(41)
    batch, L, H, P, N = 2, 19, 3, 4, 5
    x, dt, A_log, B, C, h0 = _ssd_problem(rng, batch, L, H, P, N)
    for disc in ("euler", "zoh"):
        y, st = orc.ssd_fwd(x, dt, A_log, B, C, disc=disc, h0=h0, f64=True)
        ym, sm = orc.scan_fwd(x.reshape(batch, L, H * P), np.repeat(dt, P, axis=2), np.repeat(A_log, P)[:, None]
                              * np.ones((1, N)), B, C, disc=disc, h0=h0.reshape(batch, H * P, N), f64=True)
        _close(y.reshape(batch, L, H * P), ym, 1e-13 * max(1.0, np.abs(ym).max()), f"ssd vs diagonal scan y ({disc})")
        _close(st.reshape(batch, H * P, N), sm, 1e-13 * max(1.0, np.abs(sm).max()), f"ssd vs diagonal scan state ({disc})")


def pin_ssd_chunked_duality(orc):
    """The recurrence and the chunked masked-matrix evaluation are the same function for every chunk size
    ("Mathematical Prerequisites for Mamba" s7: the recurrent and the matrix-multiply algorithms compute the
    same output; SSD uses matrix products inside chunks and the recurrence between them)."""
    rng = np.random.default_rng(42)
    batch, L, H, P, N = 2, 23, 2, 3, 4
    x, dt, A_log, B, C, h0 = _ssd_problem(rng, batch, L, H, P, N)
    for disc in ("euler", "zoh"):
        y, st = orc.ssd_fwd(x, dt, A_log, B, C, disc=disc, h0=h0, f64=True)
        for Q in (1, 4, 8, 23, 64):
            yc, sc = oracle_mod.ssd_chunked(x, dt, A_log, B, C, Q, disc=disc, h0=h0)
            _close(yc, y, 1e-12 * max(1.0, np.abs(y).max()), f"chunked (Q = {Q}) vs recurrence y ({disc})")
            _close(sc, st, 1e-12 * max(1.0, np.abs(st).max()), f"chunked (Q = {Q}) vs recurrence state ({disc})")


def pin_ssd_running_example(orc):
    """The pages' 1-SS numerical check: Abar = e^-1 (printed 0.368), Bbar = 1 - e^-1 (0.632), x = 1 gives
    h = 0.632, 0.865, 0.950, 0.982 (closed form 1 - e^-t), here in every entry of a P x N head state."""
    g = load("leaky_bucket.txt")
    L, P, N = 12, 2, 3
    y, st = orc.ssd_fwd(np.ones((1, L, 1, P)), np.ones((1, L, 1)), np.zeros(1), np.ones((1, L, N)),
                        np.full((1, L, N), 1.0 / N), disc="zoh", f64=True)
    exact = 1.0 - np.exp(-np.arange(1, L + 1, dtype=np.float64))
    for p in range(P):
        _close(y[0, :, 0, p], exact, 1e-13, "SSD running example vs 1 - e^-t")
    _close(st[0, 0], np.full((P, N), exact[-1]), 1e-13, "SSD running example final state")
    _close(y[0, :4, 0, 0], g["h"], 5e-4, "SSD running example vs printed samples")


ALL_PINS = [
    pin_leaky_bucket_closed_form, pin_ema_identity, pin_euler_scalar_trace, pin_active_recall_traces,
    pin_lti_zoh_example, pin_convolution_view, pin_selective_zoh_example, pin_combine_tree,
    pin_small_delta_limit, pin_unit_input_two_step, pin_delta_limits, pin_brute_force_1ss,
    pin_split_and_step, pin_softplus_inside_scan, pin_feedthrough_and_gate, pin_bwd_finite_differences,
    pin_bwd_convolution_adjoint, pin_bwd_one_step, pin_bwd_split, pin_bwd_channel_subset,
    pin_ssd_is_the_scan_with_shared_decay,
    pin_ssd_chunked_duality, pin_ssd_running_example,
]
