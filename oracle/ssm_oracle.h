/*
 * ssm_oracle.h -- plain, slow, fp64 CPU statement of the selective scan.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, the smoke check and the bench's
 * CPU-baseline leg may load this library.  It shares no code, header, table
 * or helper with the CUDA library under selective_state_space_123_b300/.
 *
 * Sources (page title, section):
 *  - "State Space Models (SSMs) & Mamba" (aidatadrop), section "State-Space
 *    Models (SSMs): A Resurgent Paradigm for Sequence Modeling": the
 *    continuous system h'(t) = A h(t) + B u(t), y(t) = C h(t) + D u(t).
 *  - same page, section "The Magic of Selective Scan: Content-Aware Memory",
 *    and "Mamba: How Selective State Spaces Achieve 5x Faster Inference Than
 *    Transformers", section "The selective mechanism: input-dependent SSM
 *    parameters": B, C and the step Delta are per-token inputs, A is fixed.
 *  - the pages do not print the discretisation.  The reading used here is
 *    zero-order hold on the diagonal A with an Euler input term:
 *    dA = exp(Delta*A), h_t = dA*h_{t-1} + Delta*B_t*u_t,
 *    y_t = (sum_n C_t[n] h_t[n] + D u_t) * silu(z_t),
 *    Delta = softplus(Delta_raw + Delta_bias).
 *
 * Layouts (row-major, contiguous, all double):
 *   u, delta_raw, z, y, du, ddelta_raw, dz, dy : (Bt, D, L)   L fastest
 *   Bm, Cm, dB, dC                             : (Bt, N, L)   shared by channels
 *   A, dA                                      : (D, N)
 *   Dv, delta_bias, dD, ddelta_bias            : (D)
 *   h0, hL, dh0, dhL, state                    : (Bt, D, N)
 * Nullable pointers are marked; a null input means "absent" (zero bias,
 * zero initial state, no D term, no gate).
 */
#ifndef SSM_ORACLE_H
#define SSM_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* softplus(x) = log(1 + e^x), written in the overflow-free form. */
double oracle_softplus(double x);

/* silu(z) = z / (1 + e^-z). */
double oracle_silu(double z);

/* The block's local-processing step before the scan ("Mamba Architecture
 * Explained", section "The Architecture in Practice": a 1-D convolution with
 * a SiLU activation, per channel; "The convolution trick is gone -- what
 * now?": one branch goes through a Conv1D and then the selective SSM).
 * Reading: causal depthwise convolution of width K with left zero padding,
 * so that the output keeps length L:
 *   u[b,d,t] = silu(conv_b[d] + sum_{k<K} conv_w[d,k] * x[b,d,t-(K-1)+k]),
 * x at t < 0 being 0.  x, u: (Bt, D, L); conv_w: (D, K); conv_b: (D), nullable. */
void oracle_conv_silu(int64_t Bt, int64_t D, int64_t L, int64_t K, const double* x,
                      const double* conv_w, const double* conv_b /* nullable */, double* u);
/* Reverse mode of oracle_conv_silu given du (see ssm_oracle.c); dconv_b nullable. */
void oracle_conv_silu_bwd(int64_t Bt, int64_t D, int64_t L, int64_t K, const double* x,
                          const double* conv_w, const double* conv_b, const double* du,
                          double* dx, double* dconv_w, double* dconv_b);

/* Forward selective scan over the whole sequence, sequential in t. */
void oracle_scan_fwd(int64_t Bt, int64_t D, int64_t N, int64_t L,
                     const double* u, const double* delta_raw, const double* A,
                     const double* Bm, const double* Cm,
                     const double* Dv /* nullable */, const double* z /* nullable */,
                     const double* delta_bias /* nullable */, const double* h0 /* nullable */,
                     double* y, double* hL /* nullable */);

/* One recurrent step (single token): state (Bt,D,N) is updated in place.
 * Token tensors drop L: u, delta_raw, z, y are (Bt,D); Bm, Cm are (Bt,N). */
void oracle_scan_step(int64_t Bt, int64_t D, int64_t N,
                      const double* u, const double* delta_raw, const double* A,
                      const double* Bm, const double* Cm,
                      const double* Dv /* nullable */, const double* z /* nullable */,
                      const double* delta_bias /* nullable */,
                      double* state, double* y);

/* Reverse-mode derivative of oracle_scan_fwd for upstream dy (and dhL).
 * Every gradient output is overwritten.  du, ddelta_raw, dA, dB, dC are
 * required; dD, dz, ddelta_bias, dh0 may be null (not computed). */
void oracle_scan_bwd(int64_t Bt, int64_t D, int64_t N, int64_t L,
                     const double* u, const double* delta_raw, const double* A,
                     const double* Bm, const double* Cm,
                     const double* Dv, const double* z,
                     const double* delta_bias, const double* h0,
                     const double* dy, const double* dhL /* nullable */,
                     double* du, double* ddelta_raw, double* dA, double* dB, double* dC,
                     double* dD, double* dz, double* ddelta_bias, double* dh0);

#ifdef __cplusplus
}
#endif
#endif
