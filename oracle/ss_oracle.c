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
