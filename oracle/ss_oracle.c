/*
 * Selective state space scan (S6): plain fp64 CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously-correct
 * definition that the CUDA library is checked against.  Only the test suite,
 * the smoke check and the benchmark's CPU-baseline leg may load it; the
 * product path never calls it and has no CPU fallback.
 *
 * It shares no code with the CUDA library: its own loops, its own bf16
 * widening, its own softplus and SiLU, all in double precision.
 *
 * What it computes, per batch row b and channel d, sequentially in t
 * (the equations of "State Space Models and Mamba", multigrid.ai/learn/mamba-ssm,
 * section "Selective state", equations delta_t, A_t, h_t; readout y_t = C h_t
 * from section "It is a linear recurrence"):
 *
 *     x      = delta_raw[b,d,t] + delta_bias[d]          (bias optional)
 *     dt     = softplus(x)            if softplus_flag, else x
 *     Abar_n = exp(dt * A[d,n])
 *     h_n    = Abar_n * h_n + dt * B[b,n,t] * u[b,d,t]   for n < N
 *              (zero-order hold: (exp(dt A) - 1)/A in place of dt)
 *     y      = sum_n C[b,n,t] * h_n + D[d] * u[b,d,t]     (D optional)
 *     y      = y * silu(z[b,d,t])                          (z optional)
 *
 * The D skip term follows the four-matrix statement of the model (A, B, C
 * and D) in "State space models and Mamba: reading long sequences without
 * attention" (ai-trend.me), section "Core idea".  The SiLU gate is branch B
 * of the Mamba block, "What a Mamba block actually contains" (multigrid.ai)
 * and the block description in "Mamba: Linear-Time Sequence Modeling with
 * Selective State Spaces" (azimuth.plus); the gate multiplies the whole
 * branch-A output, so it is applied after the D term.
 *
 * The decode step (sso_state_update) is the same body for one token, with h
 * read from and written back to a persistent state: the "recurrence mode"
 * of the same pages.
 *
 * Layouts (row-major, C order):
 *   u, delta, z, y : (batch, dim, seqlen)     L contiguous
 *   B, C           : (batch, dstate, seqlen)  shared by every channel
 *   A              : (dim, dstate)            fp32
 *   D, delta_bias  : (dim)                    fp32
 *   state          : (batch, dim, dstate)
 * Input dtype (u, delta, B, C, z) is fp32 or bf16 (raw 16-bit patterns);
 * every value is widened exactly to double before use.
 *
 * Channel subsets: every entry point takes an optional list of flattened
 * channel indices c = b*dim + d, so that a few channels of a very large
 * problem can be computed one by one.  Outputs are packed by list position.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#include <stdlib.h>

#define SSO_F32 0
#define SSO_BF16 1

static double sso_widen(const void* p, int64_t i, int dtype) {
    if (dtype == SSO_F32) return (double)((const float*)p)[i];
    uint32_t bits = ((uint32_t)((const uint16_t*)p)[i]) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* softplus(x) = log(1 + exp(x)), in the overflow-free form max(x,0) + log1p(exp(-|x|)). */
static double sso_softplus(double x) {
    return (x > 0.0 ? x : 0.0) + log1p(exp(-fabs(x)));
}

/* silu(z) = z * sigmoid(z) = z / (1 + exp(-z)). */
static double sso_silu(double z) {
    return z / (1.0 + exp(-z));
}

/* Input weight of the zero-order-hold discretisation: (exp(dt A) - 1) / A, which
 * tends to dt as A -> 0.  With it the update is the exact solution of
 * dh/dt = A h + B x over a step of length dt with x held constant (the
 * "principled discretization" behind Theorem 1 of "Mamba: Linear-Time Sequence
 * Modeling with Selective State Spaces", azimuth.plus). */
static double sso_zoh_weight(double dt, double A) {
    return A != 0.0 ? expm1(dt * A) / A : dt;
}

/* One time step of one channel.  h has dstate entries and is updated in place.
 * Returns y.  Index arithmetic is done by the callers.  zoh selects the input
 * weight: dt (Euler, the equations as printed) or sso_zoh_weight. */
static double sso_step(double* h, int64_t dstate,
                       double u, double draw, double bias, int softplus_flag,
                       const float* A_row, double Dd,
                       const void* B, const void* C, int64_t bc_base, int64_t bc_stride,
                       int has_z, double z, int dtype, int zoh) {
    double x = draw + bias;
    double dt = softplus_flag ? sso_softplus(x) : x;
    double y = 0.0;
    for (int64_t n = 0; n < dstate; ++n) {
        double Bn = sso_widen(B, bc_base + n * bc_stride, dtype);
        double Cn = sso_widen(C, bc_base + n * bc_stride, dtype);
        double Abar = exp(dt * (double)A_row[n]);
        double wdt = zoh ? sso_zoh_weight(dt, (double)A_row[n]) : dt;
        h[n] = Abar * h[n] + wdt * Bn * u;
        y += Cn * h[n];
    }
    y += Dd * u;
    if (has_z) y *= sso_silu(z);
    return y;
}

/*
 * Full-sequence scan over the listed channels.
 *   chans == NULL  ->  all batch*dim channels in order (nchans ignored).
 *   h0   (nullable): (nchans, dstate) initial state; zeros when NULL.
 *   y             : (nchans, seqlen) output.
 *   h_last (nullable): (nchans, dstate) final state.
 * Returns 0, or -1 on a bad argument.
 */
int sso_scan(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen, int dtype,
             const void* u, const void* delta, const float* A, const void* B, const void* C,
             const float* D, const void* z, const float* delta_bias, int softplus_flag,
             const int64_t* chans, int64_t nchans, const double* h0,
             double* y, double* h_last, int nthreads, int zoh) {
    if (batch < 0 || dim < 0 || dstate < 0 || seqlen < 0) return -1;
    if (dtype != SSO_F32 && dtype != SSO_BF16) return -1;
    int64_t total = batch * dim;
    if (chans == NULL) nchans = total;
    if (nthreads < 1) nthreads = 1;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads) reduction(|:bad)
    for (int64_t i = 0; i < nchans; ++i) {
        int64_t c = chans ? chans[i] : i;
        if (c < 0 || c >= total) { bad = 1; continue; }
        int64_t b = c / dim, d = c % dim;
        double* h = (double*)malloc(sizeof(double) * (size_t)(dstate > 0 ? dstate : 1));
        for (int64_t n = 0; n < dstate; ++n) h[n] = h0 ? h0[i * dstate + n] : 0.0;
        double bias = delta_bias ? (double)delta_bias[d] : 0.0;
        double Dd = D ? (double)D[d] : 0.0;
        for (int64_t t = 0; t < seqlen; ++t) {
            int64_t ix = c * seqlen + t;                   /* (b, d, t) */
            double uu = sso_widen(u, ix, dtype);
            double dr = sso_widen(delta, ix, dtype);
            double zz = z ? sso_widen(z, ix, dtype) : 0.0;
            y[i * seqlen + t] = sso_step(h, dstate, uu, dr, bias, softplus_flag, A + d * dstate, Dd,
                                         B, C, b * dstate * seqlen + t, seqlen,
                                         z != NULL, zz, dtype, zoh);
        }
        if (h_last)
            for (int64_t n = 0; n < dstate; ++n) h_last[i * dstate + n] = h[n];
        free(h);
    }
    return bad ? -1 : 0;
}

/*
 * One decode step (recurrence mode) over the listed channels.
 *   u, delta, z : (batch, dim)       B, C : (batch, dstate)
 *   state       : (nchans, dstate) in/out, fp64
 *   y           : (nchans)
 */
int sso_state_update(int64_t batch, int64_t dim, int64_t dstate, int dtype,
                     double* state, const void* u, const void* delta, const float* A,
                     const void* B, const void* C, const float* D, const void* z,
                     const float* delta_bias, int softplus_flag,
                     const int64_t* chans, int64_t nchans, double* y, int nthreads, int zoh) {
    if (batch < 0 || dim < 0 || dstate < 0) return -1;
    if (dtype != SSO_F32 && dtype != SSO_BF16) return -1;
    int64_t total = batch * dim;
    if (chans == NULL) nchans = total;
    if (nthreads < 1) nthreads = 1;
    int bad = 0;
#pragma omp parallel for schedule(static) num_threads(nthreads) reduction(|:bad)
    for (int64_t i = 0; i < nchans; ++i) {
        int64_t c = chans ? chans[i] : i;
        if (c < 0 || c >= total) { bad = 1; continue; }
        int64_t b = c / dim, d = c % dim;
        double uu = sso_widen(u, c, dtype);
        double dr = sso_widen(delta, c, dtype);
        double zz = z ? sso_widen(z, c, dtype) : 0.0;
        y[i] = sso_step(state + i * dstate, dstate, uu, dr, delta_bias ? (double)delta_bias[d] : 0.0,
                        softplus_flag, A + d * dstate, D ? (double)D[d] : 0.0,
                        B, C, b * dstate, 1, z != NULL, zz, dtype, zoh);
    }
    return bad ? -1 : 0;
}

/* Exposed for pins on the step-size map: dt for one raw value. */
double sso_delta(double draw, double bias, int softplus_flag) {
    double x = draw + bias;
    return softplus_flag ? sso_softplus(x) : x;
}

/*
 * Causal depthwise convolution of width 4 with an optional SiLU, the short
 * convolution in front of the SSM ("What a Mamba block actually contains",
 * multigrid.ai: a four-wide depthwise conv1d before the selective SSM;
 * "Mamba: Linear-Time Sequence Modeling with Selective State Spaces",
 * azimuth.plus: branch 1 is projection -> 1D convolution of kernel size 4 ->
 * SiLU -> SSM).  Per batch row b, channel d and step t:
 *
 *     s      = bias[d] + sum_{k=0..3} w[d,k] * x[b,d,t-3+k]     (x = 0 before t = 0)
 *     out    = silu(s) if silu_flag, else s
 *
 * so w[d,3] weighs the current step and w[d,0] the step three back.
 *   x   : (batch, dim, seqlen), fp32 or bf16 bit patterns
 *   w   : (dim, 4) fp32;   bias : (dim) fp32 or NULL
 *   out : (batch, dim, seqlen) double
 */
int sso_conv1d(int64_t batch, int64_t dim, int64_t seqlen, int dtype, const void* x, const float* w,
               const float* bias, int silu_flag, double* out, int nthreads) {
    if (batch < 0 || dim < 0 || seqlen < 0) return -1;
    if (dtype != SSO_F32 && dtype != SSO_BF16) return -1;
    if (nthreads < 1) nthreads = 1;
    int64_t rows = batch * dim;
#pragma omp parallel for schedule(static) num_threads(nthreads)
    for (int64_t c = 0; c < rows; ++c) {
        int64_t d = c % dim;
        for (int64_t t = 0; t < seqlen; ++t) {
            double s = bias ? (double)bias[d] : 0.0;
            for (int64_t k = 0; k < 4; ++k) {
                int64_t src = t - 3 + k;
                if (src >= 0) s += (double)w[d * 4 + k] * sso_widen(x, c * seqlen + src, dtype);
            }
            out[c * seqlen + t] = silu_flag ? sso_silu(s) : s;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------ backward */

static double sso_sigmoid(double x) {
    return 1.0 / (1.0 + exp(-x));
}

/* d/dA of the zero-order-hold weight (exp(dt A) - 1)/A, i.e. (dt exp(dt A) - w)/A.
 * That form cancels for small dt*A; there it is dt^2 times the series
 * 1/2 + y/3 + y^2/8 + y^3/30 (y = dt*A), the derivative of (e^y - 1)/y. */
static double sso_zoh_weight_dA(double dt, double A) {
    double y = dt * A;
    if (fabs(y) < 1e-3) return dt * dt * (0.5 + y * (1.0 / 3.0 + y * (1.0 / 8.0 + y / 30.0)));
    return (dt * exp(y) - expm1(y) / A) / A;
}

/*
 * Backward pass of sso_scan: the gradient of
 *
 *     Loss = sum_{b,d,t} dy[b,d,t] * y[b,d,t]  +  sum_{b,d,n} dlast[b,d,n] * h_last[b,d,n]
 *
 * with respect to every input, i.e. the vector-Jacobian product of the forward
 * map above with the cotangents (dy, dlast).  The pages fix only the principle
 * ("Mamba: Linear-Time Sequence Modeling with Selective State Spaces",
 * azimuth.plus, the "Recomputation" technique; "Mamba State Space Models:
 * Fixed State, Linear Time", deepnoodle.ai, "Fixed state instead of a growing
 * cache"): the states are not stored by the forward pass but recomputed.  Here
 * each channel's states are recomputed by a forward sweep, then the chain
 * rule is applied step by step in reverse time.  With
 *     e = exp(dt A[n]),  w = dt (Euler) or (e - 1)/A[n] (zero-order hold),
 *     h_t = e h_{t-1} + w B_t u_t,  s_t = sum_n C_t h_t + D u_t,  y_t = s_t silu(z_t),
 * and mu[n] the gradient reaching h_t from later steps (dlast at t = L-1):
 *     ds     = dy silu(z),           dz = dy s silu'(z)
 *     lam[n] = mu[n] + C_t[n] ds     (total gradient of h_t[n])
 *     dC_t  += ds h_t,  dD += ds u,  du = D ds + sum_n lam w B_t
 *     dB_t  += lam w u
 *     ddt    = sum_n lam (h_{t-1} e A + B_t u dw/ddt)     dw/ddt = 1 or e
 *     dA    += lam (h_{t-1} e dt + B_t u dw/dA)             dw/dA  = 0 or sso_zoh_weight_dA
 *     ddelta = ddt softplus'(x) = ddt sigmoid(x)   (ddt when the flag is off),  dbias += ddelta
 *     mu[n]  = e lam                 (carried to step t-1; dh0 = mu after t = 0)
 *
 * Arguments follow sso_scan.  Cotangents: dy (nchans, seqlen) and dlast
 * (nchans, dstate, nullable = 0), both double.  Per-channel outputs, packed by
 * list position: du, ddelta (nchans, seqlen); dz (nchans, seqlen, nullable,
 * only with z); dA_part (nchans, dstate), dD_part, dbias_part (nchans) are this
 * channel's terms of dA[d,:], dD[d], ddelta_bias[d] (the caller sums over
 * batch rows); dh0 (nchans, dstate, nullable).  dB, dC (batch, dstate, seqlen),
 * nullable: zeroed, then the listed channels' terms are added.
 */
int sso_scan_bwd(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen, int dtype,
                 const void* u, const void* delta, const float* A, const void* B, const void* C,
                 const float* D, const void* z, const float* delta_bias, int softplus_flag,
                 const int64_t* chans, int64_t nchans, const double* h0,
                 const double* dy, const double* dlast,
                 double* du, double* ddelta, double* dz, double* dA_part, double* dD_part,
                 double* dbias_part, double* dh0, double* dB, double* dC, int nthreads, int zoh) {
    if (batch < 0 || dim < 0 || dstate < 0 || seqlen < 0) return -1;
    if (dtype != SSO_F32 && dtype != SSO_BF16) return -1;
    int64_t total = batch * dim;
    if (chans == NULL) nchans = total;
    if (nthreads < 1) nthreads = 1;
    const int64_t N = dstate, L = seqlen;
    if (dB) memset(dB, 0, sizeof(double) * (size_t)(batch * N * L));
    if (dC) memset(dC, 0, sizeof(double) * (size_t)(batch * N * L));
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads) reduction(|:bad)
    for (int64_t i = 0; i < nchans; ++i) {
        int64_t c = chans ? chans[i] : i;
        if (c < 0 || c >= total) { bad = 1; continue; }
        int64_t b = c / dim, d = c % dim;
        const float* Ad = A + d * N;
        double bias = delta_bias ? (double)delta_bias[d] : 0.0;
        double Dd = D ? (double)D[d] : 0.0;
        /* hist[t * N + n] = h_{t-1}[n] for t = 0..L (hist row 0 = h0, row L = h_last) */
        double* hist = (double*)calloc((size_t)((L + 1) * N + 1), sizeof(double));
        double* dts = (double*)malloc(sizeof(double) * (size_t)(L + 1));
        double* mu = (double*)calloc((size_t)(N + 1), sizeof(double));
        double* dBc = (double*)calloc((size_t)(N * L + 1), sizeof(double));
        double* dCc = (double*)calloc((size_t)(N * L + 1), sizeof(double));
        double* dAc = (double*)calloc((size_t)(N + 1), sizeof(double));
        for (int64_t n = 0; n < N; ++n) hist[n] = h0 ? h0[i * N + n] : 0.0;

        /* forward sweep: recompute dt_t and every state */
        for (int64_t t = 0; t < L; ++t) {
            int64_t ix = c * L + t;
            double x = sso_widen(delta, ix, dtype) + bias;
            double dt = softplus_flag ? sso_softplus(x) : x;
            double uu = sso_widen(u, ix, dtype);
            dts[t] = dt;
            for (int64_t n = 0; n < N; ++n) {
                double Bn = sso_widen(B, b * N * L + n * L + t, dtype);
                double e = exp(dt * (double)Ad[n]);
                double w = zoh ? sso_zoh_weight(dt, (double)Ad[n]) : dt;
                hist[(t + 1) * N + n] = e * hist[t * N + n] + w * Bn * uu;
            }
        }

        /* reverse sweep */
        for (int64_t n = 0; n < N; ++n) mu[n] = dlast ? dlast[i * N + n] : 0.0;
        double dDc = 0.0, dbc = 0.0;
        for (int64_t t = L - 1; t >= 0; --t) {
            int64_t ix = c * L + t;
            double x = sso_widen(delta, ix, dtype) + bias;
            double dt = dts[t];
            double uu = sso_widen(u, ix, dtype);
            const double* hp = hist + t * N;          /* h_{t-1} */
            const double* hc = hist + (t + 1) * N;    /* h_t */
            double s = Dd * uu;
            for (int64_t n = 0; n < N; ++n) s += sso_widen(C, b * N * L + n * L + t, dtype) * hc[n];
            double ds = dy[i * L + t];
            if (z) {
                double zz = sso_widen(z, ix, dtype);
                double sg = sso_sigmoid(zz);
                ds = dy[i * L + t] * zz * sg;
                if (dz) dz[i * L + t] = dy[i * L + t] * s * sg * (1.0 + zz * (1.0 - sg));
            }
            dDc += ds * uu;
            double duv = Dd * ds, ddt = 0.0;
            for (int64_t n = 0; n < N; ++n) {
                double An = (double)Ad[n];
                double Bn = sso_widen(B, b * N * L + n * L + t, dtype);
                double Cn = sso_widen(C, b * N * L + n * L + t, dtype);
                double e = exp(dt * An);
                double w = zoh ? sso_zoh_weight(dt, An) : dt;
                double lam = mu[n] + Cn * ds;
                dCc[n * L + t] = ds * hc[n];
                dBc[n * L + t] = lam * w * uu;
                duv += lam * w * Bn;
                ddt += lam * (hp[n] * e * An + Bn * uu * (zoh ? e : 1.0));
                dAc[n] += lam * (hp[n] * e * dt + (zoh ? Bn * uu * sso_zoh_weight_dA(dt, An) : 0.0));
                mu[n] = e * lam;
            }
            double dx = softplus_flag ? ddt * sso_sigmoid(x) : ddt;
            du[i * L + t] = duv;
            ddelta[i * L + t] = dx;
            dbc += dx;
        }
        for (int64_t n = 0; n < N; ++n) {
            dA_part[i * N + n] = dAc[n];
            if (dh0) dh0[i * N + n] = mu[n];
        }
        dD_part[i] = dDc;
        dbias_part[i] = dbc;
        if (dB || dC) {
#pragma omp critical(sso_bwd_bc)
            for (int64_t k = 0; k < N * L; ++k) {
                if (dB) dB[b * N * L + k] += dBc[k];
                if (dC) dC[b * N * L + k] += dCc[k];
            }
        }
        free(hist); free(dts); free(mu); free(dBc); free(dCc); free(dAc);
    }
    return bad ? -1 : 0;
}
