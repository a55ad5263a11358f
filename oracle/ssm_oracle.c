/*
 * ssm_oracle.c -- plain fp64 CPU statement of the selective scan.
 *
 * TEST INFRASTRUCTURE ONLY (tests/, the smoke check and the bench's CPU
 * baseline).  Nothing here is blocked, fused or reordered: every function is
 * the defining loop, channel by channel, token by token, state by state.
 * See ssm_oracle.h for the sources and the reading of the discretisation.
 *
 * Parity status of each function (what pins it, outside of itself):
 *   oracle_scan_fwd  -- pinned: LTI convolution kernel (brute force and FFT),
 *                       the materialised time-varying kernel, L=1 closed
 *                       form, geometric-series closed form, Delta->0 and
 *                       Delta->inf limits, library softplus/sigmoid.
 *   oracle_scan_step -- pinned: equals the first token of the LTI closed
 *                       form; steps chained L times equal the forward.
 *   oracle_scan_bwd  -- pinned: central finite differences of the forward,
 *                       and the adjoint identity <dy, J v> = <J^T dy, v>.
 */
#include "ssm_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* softplus(x) = log(1 + e^x).  For x > 0 the same value is written as
 * x + log(1 + e^-x) so that e^x never overflows; both are exact identities. */
double oracle_softplus(double x) {
    if (x > 0.0) return x + log1p(exp(-x));
    return log1p(exp(x));
}

/* logistic sigmoid, sigma(x) = 1 / (1 + e^-x) */
static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

double oracle_silu(double z) { return z * sigmoid(z); }

/* The per-token selective update of one channel, shared by the forward and
 * the step so that both state the same thing:
 *   delta = softplus(delta_raw + bias)
 *   h[n]  = exp(delta * A[n]) * h[n] + delta * B[n] * u
 *   ys    = sum_n C[n] h[n] + Dskip * u                  (pre-gate output)
 * Strides let B and C be read along the L axis. */
static double token_update(int64_t N, double u, double dr, double bias,
                           const double* A, const double* Bv, const double* Cv,
                           int64_t bc_stride, double Dskip, double* h) {
    double delta = oracle_softplus(dr + bias);
    double ys = 0.0;
    for (int64_t n = 0; n < N; ++n) {
        double a = exp(delta * A[n]);
        h[n] = a * h[n] + delta * Bv[n * bc_stride] * u;
        ys += Cv[n * bc_stride] * h[n];
    }
    return ys + Dskip * u;
}

void oracle_conv_silu(int64_t Bt, int64_t D, int64_t L, int64_t K, const double* x,
                      const double* conv_w, const double* conv_b, double* u) {
    for (int64_t b = 0; b < Bt; ++b)
        for (int64_t d = 0; d < D; ++d) {
            const int64_t row = (b * D + d) * L;
            for (int64_t t = 0; t < L; ++t) {
                double s = conv_b ? conv_b[d] : 0.0;
                for (int64_t k = 0; k < K; ++k) {
                    const int64_t tt = t - (K - 1) + k;
                    if (tt >= 0) s += conv_w[d * K + k] * x[row + tt];
                }
                u[row + t] = oracle_silu(s);
            }
        }
}

/* Reverse mode of oracle_conv_silu ("Mamba Architecture Explained", section
 * "The Architecture in Practice": the branch's Conv1D and SiLU before the
 * selective SSM), given du = dLoss/du.  With pre[t] = conv_b + sum_k
 * conv_w[k] x[t-(K-1)+k] (x before token 0 is 0) and u = silu(pre):
 *   dpre[t]      = du[t] silu'(pre[t]),  silu'(p) = s (1 + p (1 - s)), s = 1 / (1 + e^-p)
 *   dx[t]        = sum_k conv_w[k] dpre[t+(K-1)-k]      (terms past the end absent)
 *   dconv_w[d,k] = sum_{b,t} dpre[t] x[t-(K-1)+k]
 *   dconv_b[d]   = sum_{b,t} dpre[t]
 * dconv_b nullable. */
void oracle_conv_silu_bwd(int64_t Bt, int64_t D, int64_t L, int64_t K, const double* x,
                          const double* conv_w, const double* conv_b, const double* du,
                          double* dx, double* dconv_w, double* dconv_b) {
    double* dpre = (double*)malloc((size_t)(L > 0 ? L : 1) * sizeof(double));
    for (int64_t d = 0; d < D; ++d) {
        for (int64_t k = 0; k < K; ++k) dconv_w[d * K + k] = 0.0;
        if (dconv_b) dconv_b[d] = 0.0;
    }
    for (int64_t b = 0; b < Bt; ++b)
        for (int64_t d = 0; d < D; ++d) {
            const int64_t row = (b * D + d) * L;
            for (int64_t t = 0; t < L; ++t) {
                double p = conv_b ? conv_b[d] : 0.0;
                for (int64_t k = 0; k < K; ++k) {
                    const int64_t tt = t - (K - 1) + k;
                    if (tt >= 0) p += conv_w[d * K + k] * x[row + tt];
                }
                const double sg = 1.0 / (1.0 + exp(-p));
                dpre[t] = du[row + t] * sg * (1.0 + p * (1.0 - sg));
            }
            for (int64_t t = 0; t < L; ++t) {
                double acc = 0.0;
                for (int64_t k = 0; k < K; ++k) {
                    const int64_t tt = t + (K - 1) - k;
                    if (tt < L) acc += conv_w[d * K + k] * dpre[tt];
                }
                dx[row + t] = acc;
                for (int64_t k = 0; k < K; ++k) {
                    const int64_t tt = t - (K - 1) + k;
                    if (tt >= 0) dconv_w[d * K + k] += dpre[t] * x[row + tt];
                }
                if (dconv_b) dconv_b[d] += dpre[t];
            }
        }
    free(dpre);
}

void oracle_scan_fwd(int64_t Bt, int64_t D, int64_t N, int64_t L,
                     const double* u, const double* delta_raw, const double* A,
                     const double* Bm, const double* Cm,
                     const double* Dv, const double* z,
                     const double* delta_bias, const double* h0,
                     double* y, double* hL) {
    double* h = (double*)malloc((size_t)(N > 0 ? N : 1) * sizeof(double));
    for (int64_t b = 0; b < Bt; ++b) {
        for (int64_t d = 0; d < D; ++d) {
            const int64_t row = (b * D + d) * L;
            for (int64_t n = 0; n < N; ++n) h[n] = h0 ? h0[(b * D + d) * N + n] : 0.0;
            const double bias = delta_bias ? delta_bias[d] : 0.0;
            const double Dskip = Dv ? Dv[d] : 0.0;
            for (int64_t t = 0; t < L; ++t) {
                const double* Bt_ = Bm + b * N * L + t;   /* B[b, :, t], stride L */
                const double* Ct_ = Cm + b * N * L + t;
                double ys = token_update(N, u[row + t], delta_raw[row + t], bias,
                                         A + d * N, Bt_, Ct_, L, Dskip, h);
                y[row + t] = z ? ys * oracle_silu(z[row + t]) : ys;
            }
            if (hL)
                for (int64_t n = 0; n < N; ++n) hL[(b * D + d) * N + n] = h[n];
        }
    }
    free(h);
}

void oracle_scan_step(int64_t Bt, int64_t D, int64_t N,
                      const double* u, const double* delta_raw, const double* A,
                      const double* Bm, const double* Cm,
                      const double* Dv, const double* z,
                      const double* delta_bias,
                      double* state, double* y) {
    for (int64_t b = 0; b < Bt; ++b) {
        for (int64_t d = 0; d < D; ++d) {
            const int64_t i = b * D + d;
            double ys = token_update(N, u[i], delta_raw[i], delta_bias ? delta_bias[d] : 0.0,
                                     A + d * N, Bm + b * N, Cm + b * N, 1,
                                     Dv ? Dv[d] : 0.0, state + i * N);
            y[i] = z ? ys * oracle_silu(z[i]) : ys;
        }
    }
}

/* Reverse mode, derived by hand from the forward loop above (the pages give
 * no backward).  With g_t = dy_t * silu(z_t) and lambda_t the total
 * derivative with respect to h_t:
 *   lambda_L = g_L C_L + dhL,  lambda_t = g_t C_t + a_{t+1} lambda_{t+1}
 *   dC_t += g_t h_t                 dB_t += lambda_t delta_t u_t
 *   du_t  = g_t D + sum_n lambda_t delta_t B_t
 *   ddelta_t = sum_n lambda_t (A a_t h_{t-1} + B_t u_t)
 *   dA   += lambda_t delta_t a_t h_{t-1}
 *   dz_t  = dy_t ys_t silu'(z_t),   silu'(z) = s(z) (1 + z (1 - s(z)))
 *   ddelta_raw_t = ddelta_t * sigmoid(delta_raw_t + bias)
 *   dh0   = a_1 lambda_1                                                    */
void oracle_scan_bwd(int64_t Bt, int64_t D, int64_t N, int64_t L,
                     const double* u, const double* delta_raw, const double* A,
                     const double* Bm, const double* Cm,
                     const double* Dv, const double* z,
                     const double* delta_bias, const double* h0,
                     const double* dy, const double* dhL,
                     double* du, double* ddelta_raw, double* dA, double* dB, double* dC,
                     double* dD, double* dz, double* ddelta_bias, double* dh0) {
    const int64_t Nn = N > 0 ? N : 1;
    /* forward record for one channel: h_t (t = 0..L, row 0 is h0), a_t, delta_t, ys_t */
    double* hs = (double*)malloc((size_t)((L + 1) * Nn) * sizeof(double));
    double* as = (double*)malloc((size_t)((L > 0 ? L : 1) * Nn) * sizeof(double));
    double* dl = (double*)malloc((size_t)(L > 0 ? L : 1) * sizeof(double));
    double* ys = (double*)malloc((size_t)(L > 0 ? L : 1) * sizeof(double));
    double* lam = (double*)malloc((size_t)Nn * sizeof(double));

    memset(dA, 0, (size_t)(D * N) * sizeof(double));
    memset(dB, 0, (size_t)(Bt * N * L) * sizeof(double));
    memset(dC, 0, (size_t)(Bt * N * L) * sizeof(double));
    if (dD) memset(dD, 0, (size_t)D * sizeof(double));
    if (ddelta_bias) memset(ddelta_bias, 0, (size_t)D * sizeof(double));

    for (int64_t b = 0; b < Bt; ++b) {
        for (int64_t d = 0; d < D; ++d) {
            const int64_t row = (b * D + d) * L;
            const double bias = delta_bias ? delta_bias[d] : 0.0;
            const double Dskip = Dv ? Dv[d] : 0.0;
            const double* Ad = A + d * N;
            /* forward, keeping everything the reverse pass needs */
            for (int64_t n = 0; n < N; ++n) hs[n] = h0 ? h0[(b * D + d) * N + n] : 0.0;
            for (int64_t t = 0; t < L; ++t) {
                double delta = oracle_softplus(delta_raw[row + t] + bias);
                dl[t] = delta;
                double acc = 0.0;
                for (int64_t n = 0; n < N; ++n) {
                    double a = exp(delta * Ad[n]);
                    double Bv = Bm[(b * N + n) * L + t];
                    as[t * N + n] = a;
                    hs[(t + 1) * N + n] = a * hs[t * N + n] + delta * Bv * u[row + t];
                    acc += Cm[(b * N + n) * L + t] * hs[(t + 1) * N + n];
                }
                ys[t] = acc + Dskip * u[row + t];
            }
            /* reverse */
            for (int64_t n = 0; n < N; ++n) lam[n] = dhL ? dhL[(b * D + d) * N + n] : 0.0;
            for (int64_t t = L - 1; t >= 0; --t) {
                const double zt = z ? z[row + t] : 0.0;
                const double gate = z ? oracle_silu(zt) : 1.0;
                const double g = dy[row + t] * gate;
                if (dz) {
                    if (z) {
                        double s = sigmoid(zt);
                        dz[row + t] = dy[row + t] * ys[t] * s * (1.0 + zt * (1.0 - s));
                    } else {
                        dz[row + t] = 0.0;
                    }
                }
                if (dD) dD[d] += g * u[row + t];
                const double delta = dl[t];
                double du_t = g * Dskip;
                double ddelta = 0.0;
                for (int64_t n = 0; n < N; ++n) {
                    const double Cv = Cm[(b * N + n) * L + t];
                    const double Bv = Bm[(b * N + n) * L + t];
                    /* lambda currently holds a_{t+1} lambda_{t+1} (or dhL) */
                    lam[n] += g * Cv;
                    const double a = as[t * N + n];
                    const double hprev = hs[t * N + n];
                    dC[(b * N + n) * L + t] += g * hs[(t + 1) * N + n];
                    dB[(b * N + n) * L + t] += lam[n] * delta * u[row + t];
                    du_t += lam[n] * delta * Bv;
                    ddelta += lam[n] * (Ad[n] * a * hprev + Bv * u[row + t]);
                    dA[d * N + n] += lam[n] * delta * a * hprev;
                    lam[n] *= a; /* becomes a_t lambda_t, the carry into t-1 */
                }
                du[row + t] = du_t;
                const double ddr = ddelta * sigmoid(delta_raw[row + t] + bias);
                ddelta_raw[row + t] = ddr;
                if (ddelta_bias) ddelta_bias[d] += ddr;
            }
            if (dh0)
                for (int64_t n = 0; n < N; ++n) dh0[(b * D + d) * N + n] = lam[n];
        }
    }
    free(hs); free(as); free(dl); free(ys); free(lam);
}
