/*
 * oracle.c -- plain, slow, sequential float64 CPU reference for the selective
 * state-space scan.  TEST INFRASTRUCTURE ONLY: the product path (the CUDA
 * library under selective_scan_mamba_gb300/) never links, loads or calls this
 * file; only the tests, the smoke check and the CPU-baseline leg of the bench
 * do.  It shares no header, helper, table or constant with the CUDA path.
 *
 * Every routine is the definition written out, in the order the pages state
 * it, with no blocking, fusion or reordering:
 *
 *   - "From S4 to Mamba-3" (ssmbench case study), section 03/System,
 *     mamba_minimal.py entry: Mamba-1 is an input-dependent (Delta, B, C)
 *     selective scan run as an explicit time loop, with an incremental step()
 *     for decoding.
 *   - same page, mamba2_minimal.py entry: a scalar A per head turns the
 *     recurrence into SSD, computed as chunked decayed-attention matmuls with a
 *     carried (N, P) state, next to a sequential scan used as its reference.
 *   - same page, s4_minimal.py entry and "Likely questions" Q01: exact ZOH for a
 *     diagonal A gives B-bar = Delta*B*(e^z - 1)/z with z = Delta*a, with the
 *     Taylor series 1 + z/2 + z^2/6 used for |z| < 1e-4.
 *   - same page, mamba3_minimal.py entry and section 04/Approach: the
 *     exponential-Euler rule (A-bar = exp(Delta*A), B-bar = Delta*B) is the
 *     form Mamba-3 reduces to at lambda = 1, theta = 0; it is the default here.
 *
 * Readings where the pages leave a step open (each listed in the design notes):
 *   - Delta = softplus(delta + bias) when softplus is requested, computed here
 *     in the overflow-safe form max(v,0) + log1p(exp(-|v|)).
 *   - the output uses the state after step t: y_t = C_t . h_t + D x_t;
 *   - the skip term is added before the gate: y = (C.h + D x) * SiLU(z);
 *   - a missing initial state means zeros.
 *
 * Layouts (row-major, last index fastest) are the library's:
 *   Mamba-1 : x, delta, z, y [batch, dim, seqlen]; B, C [batch, ngroups, dstate,
 *             seqlen]; A [dim, dstate]; D, bias [dim]; h0, h_final [batch, dim,
 *             dstate]; channel d reads group d / (dim / ngroups).
 *   SSD     : x, z, y [batch, seqlen, nheads, headdim]; dt [batch, seqlen,
 *             nheads]; B, C [batch, seqlen, ngroups, dstate]; A, D, bias
 *             [nheads]; h0, h_final [batch, nheads, headdim, dstate]; head h
 *             reads group h / (nheads / ngroups).
 *   Step    : state [batch, nheads, headdim, dstate]; x, z, y [batch, nheads,
 *             headdim]; dt [batch, nheads]; B, C [batch, ngroups, dstate];
 *             A [nheads] (a_per_state = 0) or [nheads, dstate] (= 1).
 */
#include <math.h>
#include <stddef.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_DISC_EXP_EULER 0
#define ORACLE_DISC_ZOH 1

/* softplus(v) = log(1 + e^v), written in a form that neither overflows for
 * large v nor loses the small result for very negative v. */
double oracle_softplus(double v) {
    double m = v > 0.0 ? v : 0.0;
    return m + log1p(exp(-fabs(v)));
}

/* phi1(z) = (e^z - 1) / z, the ZOH input factor; for |z| < 1e-4 the pages use
 * the Taylor polynomial 1 + z/2 + z^2/6 to avoid 0/0 ("From S4 to Mamba-3",
 * Likely questions Q01). */
double oracle_phi1(double z) {
    if (fabs(z) < 1e-4) return 1.0 + z / 2.0 + z * z / 6.0;
    return (exp(z) - 1.0) / z;
}

static double silu(double v) { return v / (1.0 + exp(-v)); }

static double step_delta(double raw, const double* bias, int idx, int use_softplus) {
    double v = raw + (bias ? bias[idx] : 0.0);
    return use_softplus ? oracle_softplus(v) : v;
}

/* Discretised input weight for one (Delta, a) pair: Delta under
 * exponential-Euler, Delta * phi1(Delta * a) under ZOH. */
static double input_weight(double delta, double a, int disc) {
    if (disc == ORACLE_DISC_ZOH) return delta * oracle_phi1(delta * a);
    return delta;
}

/* Mamba-1 selective scan ("From S4 to Mamba-3", 03/System, mamba_minimal.py):
 * for every (b, d) run the recurrence over time, for every state n:
 *   h[n] <- exp(Delta_t A[d,n]) h[n] + w(Delta_t, A[d,n]) B[n,t] x_t
 *   y_t  = sum_n C[n,t] h[n] + D[d] x_t, then y_t *= SiLU(z_t).          */
int oracle_mamba1_scan(int batch, int dim, int dstate, int seqlen, int ngroups,
                       const double* x, const double* delta, const double* delta_bias,
                       int delta_softplus, const double* A, const double* B, const double* C,
                       const double* Dskip, const double* z, const double* h0, int disc,
                       double* y, double* h_final) {
    if (batch < 0 || dim <= 0 || dstate <= 0 || seqlen < 0 || ngroups <= 0 || dim % ngroups)
        return 1;
    int per_group = dim / ngroups;
#pragma omp parallel for collapse(2) schedule(static)
    for (int b = 0; b < batch; ++b) {
        for (int d = 0; d < dim; ++d) {
            int g = d / per_group;
            double* h = (double*)malloc(sizeof(double) * (size_t)dstate);
            size_t row = ((size_t)b * dim + d) * (size_t)seqlen;
            for (int n = 0; n < dstate; ++n)
                h[n] = h0 ? h0[((size_t)b * dim + d) * dstate + n] : 0.0;
            for (int t = 0; t < seqlen; ++t) {
                double dt = step_delta(delta[row + t], delta_bias, d, delta_softplus);
                double xt = x[row + t];
                double acc = 0.0;
                for (int n = 0; n < dstate; ++n) {
                    double a = A[(size_t)d * dstate + n];
                    size_t bc = (((size_t)b * ngroups + g) * dstate + n) * (size_t)seqlen + t;
                    h[n] = exp(dt * a) * h[n] + input_weight(dt, a, disc) * B[bc] * xt;
                    acc += C[bc] * h[n];
                }
                if (Dskip) acc += Dskip[d] * xt;
                if (z) acc *= silu(z[row + t]);
                y[row + t] = acc;
            }
            if (h_final)
                for (int n = 0; n < dstate; ++n)
                    h_final[((size_t)b * dim + d) * dstate + n] = h[n];
            free(h);
        }
    }
    return 0;
}

/* Reverse-mode derivative of oracle_mamba1_scan (exponential-Euler only): given
 * dy [batch, dim, L] and dh_final [batch, dim, N] (nullable = zero), the gradients
 * of  sum_t dy_t y_t + sum_n dh_final[n] h_final[n]  with respect to every input.
 * The pages train every model with this scan inside ("From S4 to Mamba-3",
 * 03/System: one shared trainer; 05/Evaluation: per-model training-step latency),
 * so the derivative of the recurrence is part of the path; it is the chain rule
 * applied to the forward definition above, walked backwards in time:
 *   G_t[n]   = g[n] + do_t C_t[n]          (dL/dh_t; g carries the later steps)
 *   dC_t[n] += do_t h_t[n],  dB_t[n] += G_t[n] Delta_t x_t
 *   dx_t    += sum_n G_t[n] Delta_t B_t[n] (+ do_t D)
 *   dDelta_t = sum_n G_t[n] (B_t[n] x_t + h_{t-1}[n] E_t[n] A[n]),  E_t = exp(Delta_t A)
 *   dA[n]   += G_t[n] h_{t-1}[n] E_t[n] Delta_t,   g[n] = G_t[n] E_t[n]
 * with do_t = dy_t SiLU(z_t), dz_t = dy_t o_t SiLU'(z_t) where o_t is the pre-gate
 * output, d(delta)_t = dDelta_t sigmoid(delta_t + bias) under softplus, and
 * dh0 = g after step 0.  dA, dD and dbias are summed over the batch; dB and dC over
 * the channels of a group.  Gradient pointers for absent inputs may be NULL. */
int oracle_mamba1_scan_bwd(int batch, int dim, int dstate, int seqlen, int ngroups,
                           const double* x, const double* delta, const double* delta_bias,
                           int delta_softplus, const double* A, const double* B,
                           const double* C, const double* Dskip, const double* z,
                           const double* h0, const double* dy, const double* dh_final,
                           double* dx, double* ddelta, double* dA, double* dB, double* dC,
                           double* dD, double* dz, double* dbias, double* dh0) {
    if (batch < 0 || dim <= 0 || dstate <= 0 || seqlen < 0 || ngroups <= 0 || dim % ngroups)
        return 1;
    int per_group = dim / ngroups;
    size_t L = (size_t)seqlen, N = (size_t)dstate;
    memset(dA, 0, sizeof(double) * (size_t)dim * N);
    memset(dB, 0, sizeof(double) * (size_t)batch * ngroups * N * L);
    memset(dC, 0, sizeof(double) * (size_t)batch * ngroups * N * L);
    if (dD) memset(dD, 0, sizeof(double) * (size_t)dim);
    if (dbias) memset(dbias, 0, sizeof(double) * (size_t)dim);
    double* hs = (double*)malloc(sizeof(double) * (L + 1) * N);  /* h_{t-1} for t = 0..L */
    double* o = (double*)malloc(sizeof(double) * (L ? L : 1));
    double* g = (double*)malloc(sizeof(double) * N);
    for (int b = 0; b < batch; ++b) {
        for (int d = 0; d < dim; ++d) {
            int gr = d / per_group;
            size_t row = ((size_t)b * dim + d) * L;
            /* forward again, keeping every state and the pre-gate output */
            for (size_t n = 0; n < N; ++n) hs[n] = h0 ? h0[((size_t)b * dim + d) * N + n] : 0.0;
            for (size_t t = 0; t < L; ++t) {
                double dt = step_delta(delta[row + t], delta_bias, d, delta_softplus);
                double acc = 0.0;
                for (size_t n = 0; n < N; ++n) {
                    size_t bc = (((size_t)b * ngroups + gr) * N + n) * L + t;
                    double a = A[(size_t)d * N + n];
                    hs[(t + 1) * N + n] = exp(dt * a) * hs[t * N + n] + dt * B[bc] * x[row + t];
                    acc += C[bc] * hs[(t + 1) * N + n];
                }
                if (Dskip) acc += Dskip[d] * x[row + t];
                o[t] = acc;
            }
            /* backwards in time */
            for (size_t n = 0; n < N; ++n) g[n] = dh_final ? dh_final[((size_t)b * dim + d) * N + n] : 0.0;
            for (size_t tt = L; tt-- > 0;) {
                double v = delta[row + tt] + (delta_bias ? delta_bias[d] : 0.0);
                double dt = delta_softplus ? oracle_softplus(v) : v;
                double xt = x[row + tt];
                double dout = dy[row + tt];
                if (z) {
                    double zt = z[row + tt];
                    double sg = 1.0 / (1.0 + exp(-zt));
                    dz[row + tt] = dy[row + tt] * o[tt] * sg * (1.0 + zt * (1.0 - sg));
                    dout = dy[row + tt] * silu(zt);
                }
                double dxt = Dskip ? dout * Dskip[d] : 0.0;
                if (dD) dD[d] += dout * xt;
                double ddt = 0.0;
                for (size_t n = 0; n < N; ++n) {
                    size_t bc = (((size_t)b * ngroups + gr) * N + n) * L + tt;
                    double a = A[(size_t)d * N + n];
                    double E = exp(dt * a);
                    double Gt = g[n] + dout * C[bc];
                    double hprev = hs[tt * N + n];
                    dC[bc] += dout * hs[(tt + 1) * N + n];
                    dB[bc] += Gt * dt * xt;
                    dxt += Gt * dt * B[bc];
                    ddt += Gt * (B[bc] * xt + hprev * E * a);
                    dA[(size_t)d * N + n] += Gt * hprev * E * dt;
                    g[n] = Gt * E;
                }
                dx[row + tt] = dxt;
                double dv = delta_softplus ? ddt / (1.0 + exp(-v)) : ddt;
                ddelta[row + tt] = dv;
                if (dbias) dbias[d] += dv;
            }
            if (dh0)
                for (size_t n = 0; n < N; ++n) dh0[((size_t)b * dim + d) * N + n] = g[n];
        }
    }
    free(hs);
    free(o);
    free(g);
    return 0;
}

/* Mamba-3 scan ("From S4 to Mamba-3", 03/System, mamba3_minimal.py; 04/Approach,
 * "Complex transitions for state tracking"): a complex diagonal transition
 * A = A_re + i A_im per (channel, state) (A_re = -exp(a) < 0, A_im = theta) with a
 * data-dependent exponential-trapezoidal rule.  The pages fix only that the rule blends
 * the two ends of each step with a weight lambda_t and reduces to exponential-Euler at
 * lambda = 1, theta = 0; the reading taken here is the trapezoid over [t-1, t] with the
 * left end decayed by the step's transition:
 *   Abar_t[n] = exp(Delta_t A[n])                       (complex)
 *   h_t[n]    = Abar_t h_{t-1} + (1 - lambda_t) Delta_t Abar_t B_{t-1}[n] x_{t-1}
 *               + lambda_t Delta_t B_t[n] x_t           (the t-1 term is 0 at t = 0)
 *   y_t       = (Re sum_n C_t[n] h_t[n] + D x_t) * SiLU(z_t).
 * States are complex, stored as (re, im) pairs: h0, h_final [batch, dim, N, 2].
 * lambda: [batch, dim, L].  Other layouts as oracle_mamba1_scan. */
int oracle_mamba3_scan(int batch, int dim, int dstate, int seqlen, int ngroups,
                       const double* x, const double* delta, const double* delta_bias,
                       int delta_softplus, const double* A_re, const double* A_im,
                       const double* lam, const double* B, const double* C, const double* Dskip,
                       const double* z, const double* h0, double* y, double* h_final) {
    if (batch < 0 || dim <= 0 || dstate <= 0 || seqlen < 0 || ngroups <= 0 || dim % ngroups)
        return 1;
    int per_group = dim / ngroups;
    size_t N = (size_t)dstate, L = (size_t)seqlen;
#pragma omp parallel for collapse(2) schedule(static)
    for (int b = 0; b < batch; ++b) {
        for (int d = 0; d < dim; ++d) {
            int g = d / per_group;
            size_t row = ((size_t)b * dim + d) * L;
            double* hr = (double*)malloc(sizeof(double) * N * 2);
            double* hi = hr + N;
            for (size_t n = 0; n < N; ++n) {
                size_t k = (((size_t)b * dim + d) * N + n) * 2;
                hr[n] = h0 ? h0[k] : 0.0;
                hi[n] = h0 ? h0[k + 1] : 0.0;
            }
            for (size_t t = 0; t < L; ++t) {
                double dt = step_delta(delta[row + t], delta_bias, d, delta_softplus);
                double lt = lam[row + t];
                double xt = x[row + t];
                double xp = t > 0 ? x[row + t - 1] : 0.0;
                double acc = 0.0;
                for (size_t n = 0; n < N; ++n) {
                    size_t bc = (((size_t)b * ngroups + g) * N + n) * L + t;
                    double mag = exp(dt * A_re[(size_t)d * N + n]);
                    double ang = dt * A_im[(size_t)d * N + n];
                    double ar = mag * cos(ang), ai = mag * sin(ang);
                    double up = t > 0 ? B[bc - 1] * xp : 0.0;   /* B_{t-1} x_{t-1} */
                    double cur = B[bc] * xt;                   /* B_t x_t */
                    /* Abar (h + (1 - lambda) Delta u_{t-1}) + lambda Delta u_t */
                    double pr = hr[n] + (1.0 - lt) * dt * up;
                    double pi = hi[n];
                    hr[n] = ar * pr - ai * pi + lt * dt * cur;
                    hi[n] = ar * pi + ai * pr;
                    acc += C[bc] * hr[n];
                }
                if (Dskip) acc += Dskip[d] * xt;
                if (z) acc *= silu(z[row + t]);
                y[row + t] = acc;
            }
            if (h_final)
                for (size_t n = 0; n < N; ++n) {
                    size_t k = (((size_t)b * dim + d) * N + n) * 2;
                    h_final[k] = hr[n];
                    h_final[k + 1] = hi[n];
                }
            free(hr);
        }
    }
    return 0;
}

/* S4D ("From S4 to Mamba-3", 03/System, s4_minimal.py; Likely questions Q01): a linear
 * time-invariant SSM with a complex diagonal A per (channel, state), discretised by exact
 * ZOH with Delta = exp(log_dt) per channel:
 *   Abar[n] = exp(Delta A[n]),  Bbar[n] = Delta B[n] phi1(Delta A[n]),  phi1(z) = (e^z - 1)/z
 * (the Taylor polynomial 1 + z/2 + z^2/6 for |z| < 1e-4, as the pages state), and
 *   recurrent form:    h_t = Abar h_{t-1} + Bbar u_t,  y_t = Re sum_n C[n] h_t[n] + D u_t
 *   convolution form:  y = K * u + D u,  K_l = Re sum_n C[n] Bbar[n] Abar[n]^l
 * (equal from a zero state; the pages test one against the other).  A, B, C complex
 * (re, im) pairs: A [dim, N, 2], B, C [dim, N, 2]; u, y [batch, dim, L]; h0, h_final
 * [batch, dim, N, 2]. */
static void s4d_discretise(double dt, double ar, double ai, double br, double bi,
                           double* abr, double* abi, double* bbr, double* bbi) {
    double zr = dt * ar, zi = dt * ai;
    double ex = exp(zr);
    *abr = ex * cos(zi);
    *abi = ex * sin(zi);
    double pr, pi;  /* phi1(z) */
    if (sqrt(zr * zr + zi * zi) < 1e-4) {
        /* 1 + z/2 + z^2/6 */
        pr = 1.0 + zr / 2.0 + (zr * zr - zi * zi) / 6.0;
        pi = zi / 2.0 + (2.0 * zr * zi) / 6.0;
    } else {
        /* (e^z - 1) / z with e^z - 1 = expm1(zr) cos(zi) - 2 sin^2(zi/2) + i e^zr sin(zi) */
        double s2 = sin(zi / 2.0);
        double nr = expm1(zr) * cos(zi) - 2.0 * s2 * s2;
        double ni = ex * sin(zi);
        double den = zr * zr + zi * zi;
        pr = (nr * zr + ni * zi) / den;
        pi = (ni * zr - nr * zi) / den;
    }
    /* Bbar = Delta B phi1 */
    *bbr = dt * (br * pr - bi * pi);
    *bbi = dt * (br * pi + bi * pr);
}

int oracle_s4d_kernel(int dim, int dstate, int seqlen, const double* log_dt, const double* A,
                      const double* B, const double* C, double* K) {
    if (dim <= 0 || dstate <= 0 || seqlen < 0) return 1;
    size_t N = (size_t)dstate, L = (size_t)seqlen;
    for (int d = 0; d < dim; ++d) {
        double dt = exp(log_dt[d]);
        for (size_t l = 0; l < L; ++l) K[(size_t)d * L + l] = 0.0;
        for (size_t n = 0; n < N; ++n) {
            size_t k = ((size_t)d * N + n) * 2;
            double abr, abi, bbr, bbi;
            s4d_discretise(dt, A[k], A[k + 1], B[k], B[k + 1], &abr, &abi, &bbr, &bbi);
            /* w = C Bbar, then w Abar^l for l = 0, 1, ... */
            double wr = C[k] * bbr - C[k + 1] * bbi, wi = C[k] * bbi + C[k + 1] * bbr;
            for (size_t l = 0; l < L; ++l) {
                K[(size_t)d * L + l] += wr;
                double nr = wr * abr - wi * abi;
                wi = wr * abi + wi * abr;
                wr = nr;
            }
        }
    }
    return 0;
}

int oracle_s4d_recurrent(int batch, int dim, int dstate, int seqlen, const double* u,
                         const double* log_dt, const double* A, const double* B, const double* C,
                         const double* Dskip, const double* h0, double* y, double* h_final) {
    if (batch < 0 || dim <= 0 || dstate <= 0 || seqlen < 0) return 1;
    size_t N = (size_t)dstate, L = (size_t)seqlen;
#pragma omp parallel for collapse(2) schedule(static)
    for (int b = 0; b < batch; ++b) {
        for (int d = 0; d < dim; ++d) {
            double dt = exp(log_dt[d]);
            size_t row = ((size_t)b * dim + d) * L;
            for (size_t t = 0; t < L; ++t) y[row + t] = Dskip ? Dskip[d] * u[row + t] : 0.0;
            for (size_t n = 0; n < N; ++n) {
                size_t k = ((size_t)d * N + n) * 2;
                size_t hk = (((size_t)b * dim + d) * N + n) * 2;
                double abr, abi, bbr, bbi;
                s4d_discretise(dt, A[k], A[k + 1], B[k], B[k + 1], &abr, &abi, &bbr, &bbi);
                double hr = h0 ? h0[hk] : 0.0, hi = h0 ? h0[hk + 1] : 0.0;
                for (size_t t = 0; t < L; ++t) {
                    double nr = abr * hr - abi * hi + bbr * u[row + t];
                    hi = abr * hi + abi * hr + bbi * u[row + t];
                    hr = nr;
                    y[row + t] += C[k] * hr - C[k + 1] * hi;
                }
                if (h_final) {
                    h_final[hk] = hr;
                    h_final[hk + 1] = hi;
                }
            }
        }
    }
    return 0;
}

/* Mamba-2 sequential scan, the reference the pages test the chunked form
 * against ("From S4 to Mamba-3", 03/System, mamba2_minimal.py): scalar A per
 * head, state h[p, n] per (batch, head):
 *   h[p,n] <- exp(Delta_t A_h) h[p,n] + w(Delta_t, A_h) x_t[p] B_t[n]
 *   y_t[p] = sum_n C_t[n] h[p,n] + D_h x_t[p], then gated.                 */
int oracle_ssd_sequential(int batch, int seqlen, int nheads, int headdim, int dstate,
                          int ngroups, const double* x, const double* dt,
                          const double* dt_bias, int dt_softplus, const double* A,
                          const double* B, const double* C, const double* Dskip,
                          const double* z, const double* h0, int disc, double* y,
                          double* h_final) {
    if (batch < 0 || seqlen < 0 || nheads <= 0 || headdim <= 0 || dstate <= 0 || ngroups <= 0 ||
        nheads % ngroups)
        return 1;
    int per_group = nheads / ngroups;
    size_t PN = (size_t)headdim * dstate;
#pragma omp parallel for collapse(2) schedule(static)
    for (int b = 0; b < batch; ++b) {
        for (int hd = 0; hd < nheads; ++hd) {
            int g = hd / per_group;
            double* h = (double*)malloc(sizeof(double) * PN);
            for (size_t i = 0; i < PN; ++i)
                h[i] = h0 ? h0[((size_t)b * nheads + hd) * PN + i] : 0.0;
            for (int t = 0; t < seqlen; ++t) {
                double d_t = step_delta(dt[((size_t)b * seqlen + t) * nheads + hd], dt_bias, hd,
                                        dt_softplus);
                double decay = exp(d_t * A[hd]);
                double w = input_weight(d_t, A[hd], disc);
                const double* xt = x + (((size_t)b * seqlen + t) * nheads + hd) * headdim;
                const double* Bt = B + (((size_t)b * seqlen + t) * ngroups + g) * dstate;
                const double* Ct = C + (((size_t)b * seqlen + t) * ngroups + g) * dstate;
                double* yt = y + (((size_t)b * seqlen + t) * nheads + hd) * headdim;
                const double* zt = z ? z + (((size_t)b * seqlen + t) * nheads + hd) * headdim : NULL;
                for (int p = 0; p < headdim; ++p) {
                    double acc = 0.0;
                    for (int n = 0; n < dstate; ++n) {
                        double* hp = h + (size_t)p * dstate + n;
                        *hp = decay * *hp + w * xt[p] * Bt[n];
                        acc += Ct[n] * *hp;
                    }
                    if (Dskip) acc += Dskip[hd] * xt[p];
                    if (zt) acc *= silu(zt[p]);
                    yt[p] = acc;
                }
            }
            if (h_final) memcpy(h_final + ((size_t)b * nheads + hd) * PN, h, sizeof(double) * PN);
            free(h);
        }
    }
    return 0;
}

/* Mamba-2 chunked SSD ("From S4 to Mamba-3", 03/System, mamba2_minimal.py, and
 * 04/Approach "Chunked SSD with a sequential reference"): the sequence is cut
 * into chunks of Q steps (the last one may be shorter).  Inside a chunk, with
 * s_t the running sum of Delta*A_h from the chunk start up to and including t:
 *   decayed attention  y_t += sum_{s<=t} (C_t . B_s) exp(s_t - s_s) w_s x_s
 *   carried state      y_t += exp(s_t) C_t . h_in
 *   chunk state        S    = sum_s exp(s_end - s_s) w_s x_s B_s^T   (P x N)
 *   state passing      h_out = exp(s_end) h_in + S
 * followed by the skip term and the gate.  This is written independently of
 * oracle_ssd_sequential and must agree with it. */
int oracle_ssd_chunked(int batch, int seqlen, int nheads, int headdim, int dstate, int ngroups,
                       int chunk, const double* x, const double* dt, const double* dt_bias,
                       int dt_softplus, const double* A, const double* B, const double* C,
                       const double* Dskip, const double* z, const double* h0, int disc,
                       double* y, double* h_final) {
    if (batch < 0 || seqlen < 0 || nheads <= 0 || headdim <= 0 || dstate <= 0 || ngroups <= 0 ||
        nheads % ngroups || chunk <= 0)
        return 1;
    int per_group = nheads / ngroups;
    size_t PN = (size_t)headdim * dstate;
#pragma omp parallel for collapse(2) schedule(static)
    for (int b = 0; b < batch; ++b) {
        for (int hd = 0; hd < nheads; ++hd) {
            int g = hd / per_group;
            double* h = (double*)malloc(sizeof(double) * PN);      /* carried state */
            double* S = (double*)malloc(sizeof(double) * PN);      /* chunk state   */
            double* cum = (double*)malloc(sizeof(double) * (size_t)chunk);
            double* w = (double*)malloc(sizeof(double) * (size_t)chunk);
            for (size_t i = 0; i < PN; ++i)
                h[i] = h0 ? h0[((size_t)b * nheads + hd) * PN + i] : 0.0;
            for (int c0 = 0; c0 < seqlen; c0 += chunk) {
                int q = seqlen - c0 < chunk ? seqlen - c0 : chunk;
                /* running sums of Delta*A inside the chunk, and input weights */
                double run = 0.0;
                for (int i = 0; i < q; ++i) {
                    int t = c0 + i;
                    double d_t = step_delta(dt[((size_t)b * seqlen + t) * nheads + hd], dt_bias,
                                            hd, dt_softplus);
                    run += d_t * A[hd];
                    cum[i] = run;
                    w[i] = input_weight(d_t, A[hd], disc);
                }
                /* outputs of the chunk */
                for (int i = 0; i < q; ++i) {
                    int t = c0 + i;
                    const double* Ct = C + (((size_t)b * seqlen + t) * ngroups + g) * dstate;
                    for (int p = 0; p < headdim; ++p) {
                        double acc = 0.0;
                        for (int j = 0; j <= i; ++j) {        /* decayed attention */
                            int s = c0 + j;
                            const double* Bs = B + (((size_t)b * seqlen + s) * ngroups + g) * dstate;
                            double cb = 0.0;
                            for (int n = 0; n < dstate; ++n) cb += Ct[n] * Bs[n];
                            double xs = x[(((size_t)b * seqlen + s) * nheads + hd) * headdim + p];
                            acc += cb * exp(cum[i] - cum[j]) * w[j] * xs;
                        }
                        double ch = 0.0;                      /* carried state */
                        for (int n = 0; n < dstate; ++n) ch += Ct[n] * h[(size_t)p * dstate + n];
                        acc += exp(cum[i]) * ch;
                        size_t yi = (((size_t)b * seqlen + t) * nheads + hd) * headdim + p;
                        if (Dskip) acc += Dskip[hd] * x[yi];
                        if (z) acc *= silu(z[yi]);
                        y[yi] = acc;
                    }
                }
                /* chunk state and state passing */
                for (size_t i = 0; i < PN; ++i) S[i] = 0.0;
                for (int j = 0; j < q; ++j) {
                    int s = c0 + j;
                    double f = exp(cum[q - 1] - cum[j]) * w[j];
                    const double* Bs = B + (((size_t)b * seqlen + s) * ngroups + g) * dstate;
                    const double* xs = x + (((size_t)b * seqlen + s) * nheads + hd) * headdim;
                    for (int p = 0; p < headdim; ++p)
                        for (int n = 0; n < dstate; ++n)
                            S[(size_t)p * dstate + n] += f * xs[p] * Bs[n];
                }
                double chunk_decay = exp(cum[q - 1]);
                for (size_t i = 0; i < PN; ++i) h[i] = chunk_decay * h[i] + S[i];
            }
            if (h_final) memcpy(h_final + ((size_t)b * nheads + hd) * PN, h, sizeof(double) * PN);
            free(h);
            free(S);
            free(cum);
            free(w);
        }
    }
    return 0;
}

/* One decoding step ("From S4 to Mamba-3", 03/System: the incremental step()
 * of mamba_minimal.py and the O(1)-state recurrent decode).  The state is
 * updated in place:
 *   h[p,n] <- exp(Delta A) h[p,n] + w(Delta, A) x[p] B[n]
 *   y[p]    = sum_n C[n] h[p,n] + D x[p], then gated,
 * with A = A[h] (a_per_state = 0, Mamba-2 form) or A[h, n] (a_per_state = 1,
 * Mamba-1 form). */
int oracle_state_update(int batch, int nheads, int headdim, int dstate, int ngroups,
                        int a_per_state, double* state, const double* x, const double* dt,
                        const double* dt_bias, int dt_softplus, const double* A, const double* B,
                        const double* C, const double* Dskip, const double* z, int disc,
                        double* y) {
    if (batch < 0 || nheads <= 0 || headdim <= 0 || dstate <= 0 || ngroups <= 0 ||
        nheads % ngroups)
        return 1;
    int per_group = nheads / ngroups;
#pragma omp parallel for collapse(2) schedule(static)
    for (int b = 0; b < batch; ++b) {
        for (int hd = 0; hd < nheads; ++hd) {
            int g = hd / per_group;
            double d_t = step_delta(dt[(size_t)b * nheads + hd], dt_bias, hd, dt_softplus);
            const double* Bb = B + ((size_t)b * ngroups + g) * dstate;
            const double* Cb = C + ((size_t)b * ngroups + g) * dstate;
            for (int p = 0; p < headdim; ++p) {
                size_t xi = ((size_t)b * nheads + hd) * headdim + p;
                double* hrow = state + xi * dstate;
                double acc = 0.0;
                for (int n = 0; n < dstate; ++n) {
                    double a = a_per_state ? A[(size_t)hd * dstate + n] : A[hd];
                    hrow[n] = exp(d_t * a) * hrow[n] + input_weight(d_t, a, disc) * x[xi] * Bb[n];
                    acc += Cb[n] * hrow[n];
                }
                if (Dskip) acc += Dskip[hd] * x[xi];
                if (z) acc *= silu(z[xi]);
                y[xi] = acc;
            }
        }
    }
    return 0;
}

/* Number of OpenMP threads a parallel region here will use (1 without OpenMP). */
int oracle_num_threads(void) {
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Sets the number of OpenMP threads the parallel regions here use (timing harness only:
 * the results do not depend on it, every row is computed by one thread in order).
 * n < 1 restores the default.  Without OpenMP this does nothing. */
void oracle_set_num_threads(int n) {
#ifdef _OPENMP
    extern void omp_set_num_threads(int);
    extern int omp_get_num_procs(void);
    omp_set_num_threads(n >= 1 ? n : omp_get_num_procs());
#else
    (void)n;
#endif
}
