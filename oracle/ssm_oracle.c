/*
 * ssm_oracle.c -- plain, slow, sequential double-precision oracle for the selective scan.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the library path links, loads or calls this file.
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg use it.
 *
 * What it computes (one channel (b,d) at a time, time strictly sequential):
 *
 *   A[n]   = -exp(A_log[d,n])                     "Selective State Space Models" (aiwiki entry):
 *                                                   A is stored as -exp(A_log), reference loop
 *   abar   = exp(delta[b,t,d] * A[n])              "Understanding Mamba" s2.2, Eq. (2) (first half);
 *                                                   the same exact Abar is kept in the first-order form
 *                                                   ("State Space Models & Mamba" chapter, scalar
 *                                                   selective recurrence and its code)
 *   bbar*x = Euler: delta * B[b,t,n] * x[b,t,d]    aiwiki entry (dt * B, named there as the form Mamba uses);
 *                                                   chapter's Euler-simplified Bbar = delta * B
 *            ZOH:   expm1(delta*A[n]) / A[n] * B[b,t,n] * x[b,t,d]
 *                                                   "Understanding Mamba" s2.2 Eq. (2) second half,
 *                                                   written as (Abar - 1)/A * B as in its discretize()
 *                                                   example; "Mathematical Prerequisites for Mamba" s5
 *            ZOH at A[n] == 0: delta * B * x       (continuous extension of (e^z - 1)/z -> 1; the
 *                                                   chapter states the ZOH form only for A != 0)
 *   h[n]   = abar * h[n] + bbar*x                  "Understanding Mamba" s2.3, Eq. (3)
 *   y[b,t,d] = sum_n C[b,t,n] * h[n]               Eq. (3) readout with the feedthrough D set to 0
 *                                                   (s2.1); aiwiki reference loop (state @ C_t)
 *   h starts at 0 (or at h0 when given)             "Understanding Mamba" s3.1 (h_{-1} = 0)
 *   final_state[b,d,:] = h after the last step      aiwiki reference loop keeps a [B, D, N] state
 *
 * The _ex entry points add the layer pieces around the scan that the pages define next to it:
 *   delta  = softplus(delta_raw + bias[d])          "Understanding Mamba" s5.1, Eq. (6) (softplus of the
 *            (when asked; softplus(v) = ln(1+e^v))    projection plus its bias b_Delta)
 *   y_out  = (sum_n C h + Dskip[d] * x) * SiLU(z)   Eq. (1)/(3) feedthrough D x, "one independent, final
 *            SiLU(v) = v * sigma(v)                  + D * x_t" (s2.1); the gate y (.) SiLU(z) of Eq. (9)
 *                                                    (s8.1); each piece optional (bias 0, Dskip 0, no z)
 *
 * Layouts (all row-major, dense): x, delta: [batch, L, D]; B, C: [batch, L, N]; A_log: [D, N];
 * h0 / final_state: [batch, D, N] (or [n_chan, N] with a channel list, see below).
 * Inputs arrive as float (fp32 values, or bf16 values widened exactly to fp32 by the caller) or,
 * with is_f64 = 1, as double (used to feed the pages' worked examples exactly); every arithmetic
 * step below runs in double.
 *
 * A channel list `chan` (flat ids b*D + d, n_chan of them) selects which channels to evaluate;
 * chan == NULL means all batch*D channels in order. Outputs are per listed channel:
 * y_out[k*L + t], state_out[k*N + n].
 *
 * Parallelism: OpenMP over independent channels only; each channel is one sequential loop.
 */
#include <math.h>
#include <stdlib.h>
#include <stddef.h>
#include <stdint.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_EULER = 0, ORACLE_ZOH = 1 };
#define ORACLE_MAX_N 256

/* Read element i of an input array that holds float (is_f64 == 0) or double (is_f64 == 1). */
static double ld(const void *p, int64_t i, int is_f64)
{
    return is_f64 ? ((const double *)p)[i] : (double)((const float *)p)[i];
}

/* Discretised input term Bbar*x for one state entry (see the header comment for the sources). */
static double oracle_bbar_x(double dlt, double a_n, double b_n, double x, int disc)
{
    if (disc == ORACLE_ZOH) {
        if (a_n == 0.0) return dlt * b_n * x;      /* limit of expm1(z)/z -> 1 as A -> 0 */
        return expm1(dlt * a_n) / a_n * b_n * x;
    }
    return dlt * b_n * x;
}

/* delta as the recurrence uses it: the given value, or softplus(raw + bias[d]) computed as
   max(v, 0) + log1p(exp(-|v|)) (the same function, without overflow for large v). */
static double oracle_delta(double raw, const double *bias, int64_t d, int softplus)
{
    double v = raw + (bias ? bias[d] : 0.0);
    if (!softplus) return v;
    return (v > 0.0 ? v : 0.0) + log1p(exp(-fabs(v)));
}

/* The output of one channel at one step: read-out plus feedthrough, times the SiLU gate when z is given. */
static double oracle_output(double yssm, double x, const double *dskip, int64_t d, const void *z, int64_t zi,
                            int is_f64)
{
    double out = yssm + (dskip ? dskip[d] * x : 0.0);
    if (z) {
        double zv = ld(z, zi, is_f64);
        out *= zv / (1.0 + exp(-zv));
    }
    return out;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Prefill scan over whole sequences. Returns 0 on success, -1 on a bad argument.
 * h0 may be NULL (zero initial state); when given it is indexed like state_out (per listed channel).
 */
int oracle_scan_fwd_ex(const void *x, const void *delta, const void *A_log,
                       const void *B, const void *C, const double *h0,
                       const double *delta_bias, int delta_softplus, const double *dskip, const void *z,
                       int64_t batch, int64_t L, int64_t D, int64_t N, int disc, int is_f64,
                       const int64_t *chan, int64_t n_chan,
                       double *y_out, double *state_out)
{
    if (batch < 0 || L < 0 || D < 0 || N < 1 || N > ORACLE_MAX_N) return -1;
    if (disc != ORACLE_EULER && disc != ORACLE_ZOH) return -1;
    int64_t total = chan ? n_chan : batch * D;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t k = 0; k < total; ++k) {
        int64_t flat = chan ? chan[k] : k;
        if (flat < 0 || flat >= batch * D) { bad = 1; continue; }
        int64_t b = flat / D, d = flat % D;
        double h[ORACLE_MAX_N];
        double A[ORACLE_MAX_N];
        for (int64_t n = 0; n < N; ++n) {
            A[n] = -exp(ld(A_log, d * N + n, is_f64));
            h[n] = h0 ? h0[k * N + n] : 0.0;
        }
        for (int64_t t = 0; t < L; ++t) {
            double xt = ld(x, (b * L + t) * D + d, is_f64);
            double dt = oracle_delta(ld(delta, (b * L + t) * D + d, is_f64), delta_bias, d, delta_softplus);
            int64_t bc = (b * L + t) * N;
            double yt = 0.0;
            for (int64_t n = 0; n < N; ++n) {
                double abar = exp(dt * A[n]);
                h[n] = abar * h[n] + oracle_bbar_x(dt, A[n], ld(B, bc + n, is_f64), xt, disc);
                yt += ld(C, bc + n, is_f64) * h[n];
            }
            y_out[k * L + t] = oracle_output(yt, xt, dskip, d, z, (b * L + t) * D + d, is_f64);
        }
        for (int64_t n = 0; n < N; ++n) state_out[k * N + n] = h[n];
    }
    return bad ? -1 : 0;
}

int oracle_scan_fwd(const void *x, const void *delta, const void *A_log,
                    const void *B, const void *C, const double *h0,
                    int64_t batch, int64_t L, int64_t D, int64_t N, int disc, int is_f64,
                    const int64_t *chan, int64_t n_chan,
                    double *y_out, double *state_out)
{
    return oracle_scan_fwd_ex(x, delta, A_log, B, C, h0, 0, 0, 0, 0, batch, L, D, N, disc, is_f64, chan, n_chan,
                              y_out, state_out);
}

/*
 * One recurrent decode step ("Understanding Mamba" s3.2 / s10.1: the same Eq. (3) body applied to a
 * carried state). state: [n_chan, N] doubles, updated in place; x_t, delta_t: [batch, D];
 * B_t, C_t: [batch, N]; y_t: [n_chan].
 */
int oracle_scan_step_ex(double *state, const void *x_t, const void *delta_t, const void *A_log,
                        const void *B_t, const void *C_t,
                        const double *delta_bias, int delta_softplus, const double *dskip, const void *z_t,
                        int64_t batch, int64_t D, int64_t N, int disc, int is_f64,
                        const int64_t *chan, int64_t n_chan, double *y_t)
{
    if (batch < 0 || D < 0 || N < 1 || N > ORACLE_MAX_N) return -1;
    if (disc != ORACLE_EULER && disc != ORACLE_ZOH) return -1;
    int64_t total = chan ? n_chan : batch * D;
    int bad = 0;
#pragma omp parallel for schedule(static) reduction(| : bad)
    for (int64_t k = 0; k < total; ++k) {
        int64_t flat = chan ? chan[k] : k;
        if (flat < 0 || flat >= batch * D) { bad = 1; continue; }
        int64_t b = flat / D, d = flat % D;
        double xt = ld(x_t, b * D + d, is_f64);
        double dt = oracle_delta(ld(delta_t, b * D + d, is_f64), delta_bias, d, delta_softplus);
        double yt = 0.0;
        for (int64_t n = 0; n < N; ++n) {
            double A = -exp(ld(A_log, d * N + n, is_f64));
            double abar = exp(dt * A);
            double hn = abar * state[k * N + n] + oracle_bbar_x(dt, A, ld(B_t, b * N + n, is_f64), xt, disc);
            state[k * N + n] = hn;
            yt += ld(C_t, b * N + n, is_f64) * hn;
        }
        y_t[k] = oracle_output(yt, xt, dskip, d, z_t, b * D + d, is_f64);
    }
    return bad ? -1 : 0;
}

int oracle_scan_step(double *state, const void *x_t, const void *delta_t, const void *A_log,
                     const void *B_t, const void *C_t,
                     int64_t batch, int64_t D, int64_t N, int disc, int is_f64,
                     const int64_t *chan, int64_t n_chan, double *y_t)
{
    return oracle_scan_step_ex(state, x_t, delta_t, A_log, B_t, C_t, 0, 0, 0, 0, batch, D, N, disc, is_f64, chan,
                               n_chan, y_t);
}

/*
 * ---- Backward pass (gradients of the prefill scan) ---------------------------------------------------
 *
 * The pages say only that the backward pass recomputes the states h instead of storing them ("State
 * Space Models & Mamba" chapter, the paragraph on the fused kernel). What it must produce is fixed by
 * the forward definition above: the gradients of
 *     J = sum_{b,t,d} dy[b,t,d] * y[b,t,d] + sum_{b,d,n} dfinal[b,d,n] * final_state[b,d,n]
 * with respect to x, delta, A_log, B, C and h0, for the plain scan (no softplus, feedthrough or gate).
 * This oracle keeps every h_t of the channel (it is the plain reading, not the memory-saving one) and runs
 * the adjoint recurrence of h_t = abar_t h_{t-1} + bbar_t x_t backwards in time:
 *     lambda_t = C_t dy_t + abar_{t+1} lambda_{t+1},    lambda_{L-1} = C_{L-1} dy_{L-1} + dfinal
 * (lambda_t = dJ/dh_t), and for every step and entry
 *     dx_t     += lambda_t bbar_t                 (bbar_t = delta_t B_t (Euler) or expm1(delta_t A)/A B_t)
 *     d abar_t  = lambda_t h_{t-1}                d bbar_t = lambda_t x_t
 *     dC_t     += dy_t h_t
 *     ddelta_t += d abar_t A abar_t + d bbar_t (Euler: B_t; ZOH: abar_t B_t)
 *     dA       += d abar_t delta_t abar_t + (ZOH only) d bbar_t B_t delta_t^2 f(delta_t A)
 *     dB_t     += d bbar_t (Euler: delta_t; ZOH: expm1(delta_t A)/A)
 * where f(w) = (w e^w - expm1(w)) / w^2 is d/dA [expm1(delta A)/A] / delta^2 (limit 1/2 at A = 0, the
 * same continuous extension the forward uses for bbar there), and finally dh0 = abar_0 lambda_0 and
 * dA_log = dA * A (A = -exp(A_log)).
 */

/* f(w) = (w e^w - expm1(w)) / w^2, with its Taylor series 1/2 + w/3 + w^2/8 + w^3/30 near 0 where the
   difference cancels. */
static double oracle_zoh_dA_factor(double w)
{
    if (fabs(w) < 1e-3) return 0.5 + w * (1.0 / 3.0 + w * (1.0 / 8.0 + w / 30.0));
    return (w * exp(w) - expm1(w)) / (w * w);
}

/* bbar / B for one entry: delta (Euler), expm1(delta A)/A (ZOH; delta where A == 0). */
static double oracle_bfac(double dlt, double a_n, int disc)
{
    if (disc == ORACLE_ZOH && a_n != 0.0) return expm1(dlt * a_n) / a_n;
    return dlt;
}

/*
 * Gradients for the listed channels (chan as in oracle_scan_fwd_ex). Per listed channel k:
 *   dx_out[k*L + t], ddelta_out[k*L + t]      gradients of that channel's x and delta
 *   dA_log_out[k*N + n]                        that channel's contribution to dA_log[d, n] (the caller
 *                                              sums the contributions of the batch elements)
 *   dB_out[(k*L + t)*N + n], dC_out[...]       that channel's contribution to dB[b,t,n], dC[b,t,n]
 *                                              (the caller sums over d); either may be NULL
 *   dh0_out[k*N + n]                           dJ/dh0 (NULL: not wanted)
 * dy: [batch, L, D] like x; dfinal, h0: [n_chan, N] doubles or NULL (zero).
 */
int oracle_scan_bwd(const void *x, const void *delta, const void *A_log, const void *B, const void *C,
                    const double *h0, const void *dy, const double *dfinal,
                    int64_t batch, int64_t L, int64_t D, int64_t N, int disc, int is_f64,
                    const int64_t *chan, int64_t n_chan,
                    double *dx_out, double *ddelta_out, double *dA_log_out, double *dB_out, double *dC_out,
                    double *dh0_out)
{
    if (batch < 0 || L < 0 || D < 0 || N < 1 || N > ORACLE_MAX_N) return -1;
    if (disc != ORACLE_EULER && disc != ORACLE_ZOH) return -1;
    int64_t total = chan ? n_chan : batch * D;
    int bad = 0;
#pragma omp parallel reduction(| : bad)
    {
        double *H = (double *)malloc((size_t)(L > 0 ? L : 1) * (size_t)N * sizeof(double));  /* h_t, t < L */
        if (!H) bad = 1;
#pragma omp for schedule(dynamic, 1)
        for (int64_t k = 0; k < total; ++k) {
            int64_t flat = chan ? chan[k] : k;
            if (!H || flat < 0 || flat >= batch * D) { bad = 1; continue; }
            int64_t b = flat / D, d = flat % D;
            double A[ORACLE_MAX_N], h[ORACLE_MAX_N], lam[ORACLE_MAX_N], mu[ORACLE_MAX_N], dA[ORACLE_MAX_N];
            for (int64_t n = 0; n < N; ++n) {
                A[n] = -exp(ld(A_log, d * N + n, is_f64));
                h[n] = h0 ? h0[k * N + n] : 0.0;
                mu[n] = dfinal ? dfinal[k * N + n] : 0.0;   /* dJ/dh_{L-1} from the final state */
                dA[n] = 0.0;
            }
            /* forward, keeping every state */
            for (int64_t t = 0; t < L; ++t) {
                double xt = ld(x, (b * L + t) * D + d, is_f64);
                double dt = ld(delta, (b * L + t) * D + d, is_f64);
                for (int64_t n = 0; n < N; ++n) {
                    h[n] = exp(dt * A[n]) * h[n] + oracle_bfac(dt, A[n], disc) * ld(B, (b * L + t) * N + n, is_f64) * xt;
                    H[t * N + n] = h[n];
                }
            }
            /* backward */
            for (int64_t t = L - 1; t >= 0; --t) {
                double xt = ld(x, (b * L + t) * D + d, is_f64);
                double dt = ld(delta, (b * L + t) * D + d, is_f64);
                double dyt = ld(dy, (b * L + t) * D + d, is_f64);
                double gx = 0.0, gdt = 0.0;
                for (int64_t n = 0; n < N; ++n) {
                    int64_t bc = (b * L + t) * N + n;
                    double Bn = ld(B, bc, is_f64), Cn = ld(C, bc, is_f64);
                    double abar = exp(dt * A[n]);
                    double bfac = oracle_bfac(dt, A[n], disc);
                    double hprev = t > 0 ? H[(t - 1) * N + n] : (h0 ? h0[k * N + n] : 0.0);
                    lam[n] = Cn * dyt + mu[n];
                    double g_abar = lam[n] * hprev;
                    double g_bbar = lam[n] * xt;          /* gradient of bbar = bfac * B */
                    gx += lam[n] * bfac * Bn;
                    gdt += g_abar * A[n] * abar;
                    dA[n] += g_abar * dt * abar;
                    if (disc == ORACLE_ZOH) {
                        gdt += g_bbar * abar * Bn;
                        dA[n] += g_bbar * Bn * dt * dt * oracle_zoh_dA_factor(dt * A[n]);
                    } else {
                        gdt += g_bbar * Bn;
                    }
                    if (dB_out) dB_out[(k * L + t) * N + n] = g_bbar * bfac;
                    if (dC_out) dC_out[(k * L + t) * N + n] = dyt * H[t * N + n];
                    mu[n] = abar * lam[n];
                }
                dx_out[k * L + t] = gx;
                ddelta_out[k * L + t] = gdt;
            }
            for (int64_t n = 0; n < N; ++n) {
                dA_log_out[k * N + n] = dA[n] * A[n];
                if (dh0_out) dh0_out[k * N + n] = mu[n];
            }
        }
        free(H);
    }
    return bad ? -1 : 0;
}

/*
 * ---- Mamba-2 structured state space duality (SSD) layer: the scan with A = a * I -----------------------
 *
 * "Mamba and Mamba-2" as the chapter describes it ("State Space Models & Mamba" chapter, the Mamba-2
 * paragraph; "Mathematical Prerequisites for Mamba" s7 and the paragraph after it): the state matrix is a
 * scalar times the identity, one scalar per head, so every channel of a head shares one decay per step and
 * the head's state is a matrix [P, N] (P channels of the head, N state entries each):
 *   A_h      = -exp(A_log[h])
 *   abar     = exp(delta[b,t,h] * A_h)                      one decay per (step, head)
 *   coef     = delta (Euler) or expm1(delta A_h) / A_h (ZOH; delta where A_h == 0)
 *   S[p][n]  = abar * S[p][n] + coef * B[b,t,n] * x[b,t,h,p]
 *   y[b,t,h,p] = sum_n C[b,t,n] * S[p][n]
 * with S = h0 (or 0) before the first step and final_state = S after the last. This is the plain
 * recurrence; the chunked (masked matrix product) evaluation of the same function lives in the tests.
 * Layouts: x, y [batch, L, H, P]; delta [batch, L, H]; A_log [H]; B, C [batch, L, N] (one group shared by
 * the heads); h0, final_state [batch, H, P, N] (doubles).
 */
int oracle_ssd_fwd(const void *x, const void *delta, const void *A_log, const void *B, const void *C,
                   const double *h0, int64_t batch, int64_t L, int64_t H, int64_t P, int64_t N, int disc,
                   int is_f64, double *y_out, double *state_out)
{
    if (batch < 0 || L < 0 || H < 0 || P < 1 || N < 1 || P > ORACLE_MAX_N || N > ORACLE_MAX_N) return -1;
    if (disc != ORACLE_EULER && disc != ORACLE_ZOH) return -1;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t k = 0; k < batch * H; ++k) {
        int64_t b = k / H, hh = k % H;
        double *S = (double *)malloc((size_t)(P * N) * sizeof(double));
        if (!S) { bad = 1; continue; }
        double A = -exp(ld(A_log, hh, is_f64));
        for (int64_t i = 0; i < P * N; ++i) S[i] = h0 ? h0[k * P * N + i] : 0.0;
        for (int64_t t = 0; t < L; ++t) {
            double dt = ld(delta, (b * L + t) * H + hh, is_f64);
            double abar = exp(dt * A);
            double coef = oracle_bfac(dt, A, disc);
            for (int64_t p = 0; p < P; ++p) {
                double xv = ld(x, ((b * L + t) * H + hh) * P + p, is_f64);
                double yv = 0.0;
                for (int64_t n = 0; n < N; ++n) {
                    S[p * N + n] = abar * S[p * N + n] + coef * ld(B, (b * L + t) * N + n, is_f64) * xv;
                    yv += ld(C, (b * L + t) * N + n, is_f64) * S[p * N + n];
                }
                y_out[((b * L + t) * H + hh) * P + p] = yv;
            }
        }
        for (int64_t i = 0; i < P * N; ++i) state_out[k * P * N + i] = S[i];
        free(S);
    }
    return bad ? -1 : 0;
}
