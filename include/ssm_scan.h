/*
 * ssm_scan.h -- C ABI of libssmscan.so: the selective scan of the Mamba
 * selective state space model on one B300 GPU (sm_103a).
 *
 * What is computed (per batch b, channel d, state n, token t):
 *
 *   delta_t = softplus(delta_raw[b,d,t] + delta_bias[d])
 *   h_t[n]  = exp(delta_t * A[d,n]) * h_{t-1}[n] + delta_t * B[b,n,t] * u[b,d,t]
 *   y[b,d,t] = (sum_n C[b,n,t] h_t[n] + D[d] u[b,d,t]) * silu(z[b,d,t])
 *   hL[b,d,n] = h_L[n],   h_0 = h0[b,d,n] (or 0)
 *
 * Sources (page title, section):
 *  - "State Space Models (SSMs) & Mamba" (aidatadrop): section "State-Space
 *    Models (SSMs): A Resurgent Paradigm for Sequence Modeling" gives the
 *    continuous system h' = A h + B u, y = C h + D u; section "The Magic of
 *    Selective Scan: Content-Aware Memory" makes B, C and the step Delta
 *    functions of the input token while A stays fixed; section "The Payoff:
 *    Linear Scaling and Lightning-Fast Inference" gives the constant-memory
 *    recurrent step.
 *  - "Mamba: How Selective State Spaces Achieve 5x Faster Inference Than
 *    Transformers", section "The selective mechanism: input-dependent SSM
 *    parameters": B, C and Delta are computed per token; training runs the
 *    recurrence as a parallel prefix scan; inference is a pure recurrence.
 *  - "The convolution trick is gone -- what now?" (Mamba lesson 2): the scan
 *    keeps the recurrence on chip and writes back only the final state.
 *  - "Mamba Architecture Explained", section "The Architecture in Practice":
 *    the SSM output is gated by SiLU of a second branch (z here).
 *  The pages do not print the discretisation; this library reads it as
 *  dA = exp(Delta A) with input term Delta B u, the gate applied after the
 *  D skip term.
 *
 * Layouts: row-major, contiguous, token axis fastest.
 *   u, delta_raw, z, y, dy, du, ddelta_raw, dz : (batch, dim, seqlen)
 *   B, C, dB, dC                               : (batch, dstate, seqlen), shared by all channels
 *   A, dA                                      : (dim, dstate)   fp32
 *   D, delta_bias, dD, ddelta_bias             : (dim)           fp32
 *   h0, hL, dhL, dh0, decode state             : (batch, dim, dstate) fp32
 *
 * Conventions for every entry point:
 *  - All pointers are DEVICE pointers except the shape struct, and must be
 *    16-byte aligned.  The caller owns and allocates every buffer, including
 *    the workspace; the library never allocates, frees or synchronises
 *    (except ssm_get_status, which synchronises the stream it is given).
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and runs asynchronously.  Argument errors are detected on the
 *    host before anything is enqueued and returned synchronously.  Errors
 *    detected on the device (a bounded wait that expired) are written to the
 *    status word in the workspace and read with ssm_get_status; so are
 *    packed-sequence starts out of order (ssm_scan_fwd_varlen).
 *  - Gradient outputs are overwritten, never accumulated into.
 *  - Return value: SSM_OK (0) or one of the negative SSM_ERR_* codes.
 */
#ifndef SSM_SCAN_H
#define SSM_SCAN_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SSM_API __attribute__((visibility("default")))
#else
#define SSM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef void* ssm_stream_t; /* a cudaStream_t */

typedef enum { SSM_F32 = 0, SSM_BF16 = 1 } ssm_dtype;

typedef struct {
    int64_t batch;     /* Bt >= 0 */
    int64_t dim;       /* D  >= 0 channels */
    int64_t dstate;    /* N, 1 <= N <= 64 */
    int64_t seqlen;    /* L >= 0 */
    int32_t in_dtype;  /* ssm_dtype of u, delta_raw, z, B, C (and dy in backward) */
    int32_t out_dtype; /* ssm_dtype of y (and du, ddelta_raw, dz in backward) */
} ssm_shape;

enum {
    SSM_OK = 0,
    SSM_ERR_NULL = -1,        /* a required pointer is NULL */
    SSM_ERR_SHAPE = -2,       /* negative size, dstate outside 1..64, or size overflow */
    SSM_ERR_DTYPE = -3,       /* in_dtype / out_dtype not an ssm_dtype */
    SSM_ERR_ALIGN = -4,       /* a pointer is not 16-byte aligned */
    SSM_ERR_WORKSPACE = -5,   /* workspace NULL or smaller than ssm_scan_workspace_bytes */
    SSM_ERR_CUDA = -6,        /* a CUDA runtime call failed (launch, attribute query) */
    SSM_ERR_TIMEOUT = -7,     /* device side: a bounded wait expired; outputs undefined */
    SSM_ERR_UNSUPPORTED = -8, /* valid request the library does not implement */
    SSM_ERR_SEQLENS = -9      /* device side: packed-sequence starts not 0 <= ... <= seqlen */
};

/* Bytes of device workspace the call needs for this shape on the current
 * device: for_backward = 0 for ssm_scan_fwd (and its _conv and _varlen forms),
 * 1 for ssm_scan_bwd (and _varlen), 2 for ssm_scan_fwd_bidir, 3 for
 * ssm_scan_bwd_bidir, 4 for ssm_scan_bwd_conv.  Always at
 * least 256 (the status word lives at offset 0).  Returns 0 for an invalid
 * shape. */
SSM_API size_t ssm_scan_workspace_bytes(const ssm_shape* shape, int for_backward);

/* Forward selective scan over the whole sequence.
 *   u, delta_raw, B, C : in_dtype, required.     A : fp32 (dim, dstate), required.
 *   D, z, delta_bias, h0 : nullable (absent term / no gate / zero bias / zero state).
 *   y  : out_dtype (batch, dim, seqlen), required.
 *   hL : fp32 (batch, dim, dstate), nullable (final state not written).
 *   workspace : >= ssm_scan_workspace_bytes(shape, 0) bytes of device memory.
 * Long sequences with few channels are split into segments whose carried
 * state is combined between two passes ("write back only the final state
 * per tile", Mamba lesson 2); the result is the same recurrence. */
SSM_API int ssm_scan_fwd(const ssm_shape* shape, const void* u, const void* delta_raw,
                 const float* A, const void* B, const void* C, const float* D,
                 const void* z, const float* delta_bias, const float* h0,
                 void* y, float* hL, void* workspace, size_t ws_bytes,
                 ssm_stream_t stream);

/* ssm_scan_fwd fed by the block's local-processing step ("Mamba Architecture
 * Explained", section "The Architecture in Practice": a 1-D convolution with
 * a SiLU activation before the selective SSM; "The convolution trick is gone
 * -- what now?": one branch goes through a Conv1D and then the selective
 * SSM).  Instead of u the call takes the branch input x and computes, per
 * channel, a causal depthwise convolution of width conv_k with left zero
 * padding, then SiLU:
 *   u[b,d,t] = silu(conv_b[d] + sum_{k<conv_k} conv_w[d,k] * x[b,d,t-(conv_k-1)+k])
 * (x at t < 0 is 0), inside the scan kernel; u never reaches HBM.
 *   x : in_dtype (batch, dim, seqlen), required (layout of u).
 *   conv_w : fp32 (dim, conv_k), required; conv_b : fp32 (dim), nullable (no bias).
 *   conv_k : 1..4 (else SSM_ERR_SHAPE).
 * Everything else as ssm_scan_fwd (same workspace size).  Built for 9 to 16
 * states and rows of seqlen * element size a multiple of 16 bytes; other
 * shapes return SSM_ERR_UNSUPPORTED before anything is enqueued. */
SSM_API int ssm_scan_fwd_conv(const ssm_shape* shape, const void* x, const float* conv_w,
                 const float* conv_b, int conv_k, const void* delta_raw, const float* A,
                 const void* B, const void* C, const float* D, const void* z,
                 const float* delta_bias, const float* h0, void* y, float* hL,
                 void* workspace, size_t ws_bytes, ssm_stream_t stream);

/* ssm_scan_fwd (or ssm_scan_fwd_conv) over packed sequences ("Mamba
 * Architecture Explained", section "Problem 3: Ecosystem maturity": packing
 * several sequences into one row needs its own kernel support).  Every batch
 * row holds the same nseq >= 1 sequences back to back: sequence s covers
 * tokens [cu_seqlens[s], cu_seqlens[s+1]), with
 * 0 = cu_seqlens[0] <= cu_seqlens[1] <= ... <= cu_seqlens[nseq] = seqlen
 * (empty sequences allowed).  Each sequence is scanned on its own: its state
 * starts at h0[s] (zero when h0 is NULL) and, with conv_w given, its
 * convolution window starts from zeros; nothing crosses a start.
 *   cu_seqlens : int32 (nseq + 1), device memory (4-byte alignment is
 *     enough for this one pointer), required.  Start values
 *     that break the order above are reported as SSM_ERR_SEQLENS in the
 *     workspace status word (ssm_get_status); the outputs are then undefined,
 *     and no access goes outside the buffers.
 *   u : in_dtype (batch, dim, seqlen): u itself (conv_w NULL) or the conv
 *     branch input x (conv_w given; conv_b, conv_k as in ssm_scan_fwd_conv).
 *   h0 : fp32 (nseq, batch, dim, dstate), nullable.
 *   hL : fp32 (nseq, batch, dim, dstate), nullable: every sequence's final
 *     state (an empty sequence's is its initial state).
 * Everything else as ssm_scan_fwd (same workspace size).  Built for 9 to 16
 * states and rows of seqlen * element size a multiple of 16 bytes (pad the
 * packed row with a last sequence); other shapes return SSM_ERR_UNSUPPORTED
 * before anything is enqueued. */
SSM_API int ssm_scan_fwd_varlen(const ssm_shape* shape, const void* u, const int32_t* cu_seqlens,
                 int nseq, const float* conv_w, const float* conv_b, int conv_k,
                 const void* delta_raw, const float* A, const void* B, const void* C,
                 const float* D, const void* z, const float* delta_bias, const float* h0,
                 void* y, float* hL, void* workspace, size_t ws_bytes, ssm_stream_t stream);

/* Bidirectional scan ("Mamba Architecture Explained", section "Frequently
 * Asked Questions": the standard scan is causal, bidirectional SSM variants
 * run a second scan the other way).  Two selective scans over the same u
 * and gate z, each with its own parameters: the left-to-right scan of
 * ssm_scan_fwd with (delta_raw, A, B, C, D, delta_bias, h0), and a
 * right-to-left scan with (delta_raw_r, A_r, B_r, C_r, D_r, delta_bias_r,
 * h0_r) whose state runs from token seqlen-1 down to token 0:
 *   h_r[t] = exp(delta_r[t] A_r) h_r[t+1] + delta_r[t] B_r[t] u[t],  h_r[seqlen] = h0_r
 *   y[t] = (C[t].h[t] + D u[t]) silu(z[t]) + (C_r[t].h_r[t] + D_r u[t]) silu(z[t]).
 * (The same pointers for both directions give the weight-tied variant.)
 *   Shapes and dtypes as ssm_scan_fwd, per direction; z nullable (no gate).
 *   hL : the left-to-right state after token seqlen-1; hL_r : the
 *     right-to-left state after token 0; both fp32 (batch, dim, dstate), nullable.
 *   workspace : >= ssm_scan_workspace_bytes(shape, 2) bytes (it holds the
 *     right-to-left pass's fp32 output, batch * dim * seqlen floats).
 * Runs as two kernels (right to left, then left to right adding the first's
 * output); long sequences are not split into segments.  Built for 9 to 16
 * states and rows of seqlen * element size a multiple of 16 bytes; other
 * shapes return SSM_ERR_UNSUPPORTED before anything is enqueued. */
SSM_API int ssm_scan_fwd_bidir(const ssm_shape* shape, const void* u, const void* z,
                 const void* delta_raw, const float* A, const void* B, const void* C,
                 const float* D, const float* delta_bias, const float* h0,
                 const void* delta_raw_r, const float* A_r, const void* B_r, const void* C_r,
                 const float* D_r, const float* delta_bias_r, const float* h0_r,
                 void* y, float* hL, float* hL_r, void* workspace, size_t ws_bytes,
                 ssm_stream_t stream);

/* Reverse mode of ssm_scan_fwd_bidir (the pages give no backward; it is the
 * exact derivative of the two scans above).  The right-to-left scan is the
 * left-to-right scan of the token-reversed sequence, so its reverse mode is
 * ssm_scan_bwd run on token-reversed copies of its inputs (made in the
 * workspace), with its per-token gradients reversed back; u and z feed both
 * directions, so du and dz are the sums of the two directions' gradients.
 *   Inputs: those of ssm_scan_fwd_bidir (both directions' parameters, u, z
 *     nullable) plus dy : in_dtype (batch, dim, seqlen), required, and the
 *     upstream gradients of the two final states, dhL (of hL) and dhL_r (of
 *     hL_r) : fp32 (batch, dim, dstate), nullable (= 0).
 *   Outputs (overwritten):
 *     du : out_dtype, required;  dz : out_dtype, nullable (zeros without z);
 *     per direction (suffix _r: right to left) ddelta_raw : out_dtype,
 *     required; dA (dim, dstate), dB, dC (batch, dstate, seqlen) : fp32,
 *     required; dD, ddelta_bias (dim), dh0 (batch, dim, dstate) : fp32,
 *     nullable.  dh0_r is the gradient of h0_r, the right-to-left state
 *     before token seqlen-1.
 * workspace : >= ssm_scan_workspace_bytes(shape, 3) bytes (it holds the
 * reversed copies, both directions' fp32 per-token gradients and one
 * ssm_scan_bwd workspace); device errors of either direction are reported
 * through its status word.  Any state size and sequence length that
 * ssm_scan_bwd accepts. */
SSM_API int ssm_scan_bwd_bidir(const ssm_shape* shape, const void* u, const void* z,
                 const void* delta_raw, const float* A, const void* B, const void* C,
                 const float* D, const float* delta_bias, const float* h0,
                 const void* delta_raw_r, const float* A_r, const void* B_r, const void* C_r,
                 const float* D_r, const float* delta_bias_r, const float* h0_r,
                 const void* dy, const float* dhL, const float* dhL_r, void* du, void* dz,
                 void* ddelta_raw, float* dA, float* dB, float* dC, float* dD,
                 float* ddelta_bias, float* dh0, void* ddelta_raw_r, float* dA_r,
                 float* dB_r, float* dC_r, float* dD_r, float* ddelta_bias_r, float* dh0_r,
                 void* workspace, size_t ws_bytes, ssm_stream_t stream);

/* Reverse mode of ssm_scan_fwd (the pages give no backward; it is the exact
 * derivative of the recurrence above).  Inputs are the forward inputs plus
 *   dy  : in_dtype (batch, dim, seqlen), required;   dhL : fp32, nullable (= 0).
 * Outputs (overwritten):
 *   du, ddelta_raw : out_dtype, required.   dz : out_dtype, nullable.
 *   dA (dim,dstate), dB, dC (batch,dstate,seqlen) : fp32, required
 *     (dB and dC are sums over all channels).
 *   dD, ddelta_bias (dim), dh0 (batch,dim,dstate) : fp32, nullable.
 *   ddelta_raw is the derivative with respect to delta_raw (before softplus).
 * workspace : >= ssm_scan_workspace_bytes(shape, 1) bytes.  The backward
 * reruns the forward recurrence itself (with the derivative of the state
 * with respect to A beside it); nothing from ssm_scan_fwd is needed.  Long
 * sequences with too few channels to fill the GPU ("Mamba: Linear-Time
 * Sequence Modeling with Selective State Spaces", section "Key points":
 * sequences up to a million tokens) are cut into segments run side by side,
 * each given its initial state, the adjoint entering from its right and the
 * dA tangent crossing its boundaries by summary passes and carries over the
 * segments (workspace sized for them); the results are the same reverse
 * mode. */
SSM_API int ssm_scan_bwd(const ssm_shape* shape, const void* u, const void* delta_raw,
                 const float* A, const void* B, const void* C, const float* D,
                 const void* z, const float* delta_bias, const float* h0,
                 const void* dy, const float* dhL,
                 void* du, void* ddelta_raw, float* dA, float* dB, float* dC,
                 float* dD, void* dz, float* ddelta_bias, float* dh0,
                 void* workspace, size_t ws_bytes, ssm_stream_t stream);

/* ssm_scan_bwd over packed sequences: the reverse mode of ssm_scan_fwd_varlen
 * without the conv prologue ("Mamba Architecture Explained", section
 * "Problem 3: Ecosystem maturity": training on packed sequences needs its
 * own kernel support).  Every packed sequence gets its own reverse mode:
 * its per-token gradients land in its token range, dh0[s] is the gradient of
 * its initial state h0[s], dhL[s] the upstream gradient of its final state,
 * and nothing flows across a start; dA, dD, ddelta_bias are summed over all
 * sequences, dB and dC over all channels.
 *   cu_seqlens, nseq : as for ssm_scan_fwd_varlen (device int32, nseq + 1
 *     starts; starts out of order are reported as SSM_ERR_SEQLENS in the
 *     workspace status word, outputs then undefined, no access out of bounds).
 *   h0, dhL, dh0 : fp32 (nseq, batch, dim, dstate), nullable; an empty
 *     sequence gets dh0[s] = dhL[s] (zero when dhL is NULL).
 *   Everything else as ssm_scan_bwd (same workspace size).  Built for 9 to 16
 *   states and rows of seqlen * element size a multiple of 16 bytes; other
 *   shapes return SSM_ERR_UNSUPPORTED before anything is enqueued. */
SSM_API int ssm_scan_bwd_varlen(const ssm_shape* shape, const void* u, const int32_t* cu_seqlens,
                 int nseq, const void* delta_raw, const float* A, const void* B, const void* C,
                 const float* D, const void* z, const float* delta_bias, const float* h0,
                 const void* dy, const float* dhL, void* du, void* ddelta_raw, float* dA,
                 float* dB, float* dC, float* dD, void* dz, float* ddelta_bias, float* dh0,
                 void* workspace, size_t ws_bytes, ssm_stream_t stream);

/* Reverse mode of ssm_scan_fwd_conv: the scan's reverse mode with u formed
 * from the branch input x inside both sweeps ("Mamba Architecture
 * Explained", section "The Architecture in Practice": the branch's Conv1D
 * and SiLU before the selective SSM), then the prologue's own reverse mode.
 * With pre[t] = conv_b[d] + sum_{k<conv_k} conv_w[d,k] x[t-(conv_k-1)+k]
 * (x before token 0 is 0) and u = silu(pre), from the scan's du:
 *   dx[t] = sum_k conv_w[d,k] dpre[t+(conv_k-1)-k],  dpre = du silu'(pre)
 *   dconv_w[d,k] = sum_{b,t} dpre[t] x[t-(conv_k-1)+k],  dconv_b[d] = sum_{b,t} dpre[t]
 *   x, conv_w, conv_b, conv_k : as for ssm_scan_fwd_conv (conv_b nullable).
 *   dx : out_dtype (batch, dim, seqlen), required (replaces du).
 *   dconv_w : fp32 (dim, conv_k), required;  dconv_b : fp32 (dim), nullable.
 *   Everything else as ssm_scan_bwd.  workspace >= ssm_scan_workspace_bytes(
 *   shape, 4) bytes (it also holds the scan's du in fp32, so that dx is
 *   rounded once).  Built for
 *   9 to 16 states and rows of seqlen * element size a multiple of 16 bytes;
 *   other shapes return SSM_ERR_UNSUPPORTED before anything is enqueued. */
SSM_API int ssm_scan_bwd_conv(const ssm_shape* shape, const void* x, const float* conv_w,
                 const float* conv_b, int conv_k, const void* delta_raw, const float* A,
                 const void* B, const void* C, const float* D, const void* z,
                 const float* delta_bias, const float* h0, const void* dy, const float* dhL,
                 void* dx, void* ddelta_raw, float* dA, float* dB, float* dC, float* dD,
                 void* dz, float* ddelta_bias, float* dh0, float* dconv_w, float* dconv_b,
                 void* workspace, size_t ws_bytes, ssm_stream_t stream);

/* One recurrent (decode) step for a single token per sequence, with the
 * state updated in place ("Mamba: How Selective State Spaces ...", section
 * "The selective mechanism": constant memory per generated token).
 *   u, delta_raw, z, y : (batch, dim);  B, C : (batch, dstate);  in_dtype / out_dtype.
 *   A : fp32 (dim, dstate), required.  D, z, delta_bias : nullable.
 *   state : fp32 (batch, dim, dstate), read and overwritten with the new state.
 *   status : nullable device int32 (4-byte aligned).  If a bounded wait in
 *     the kernel expires, SSM_ERR_TIMEOUT is written there (only if it still
 *     holds SSM_OK) and y and the state are left partly updated, i.e.
 *     undefined.  Read and clear it with ssm_get_status(status, stream) (a
 *     256-byte workspace whose first word is the status serves as well).
 *     With status NULL an expired wait is not reported.
 * Needs no workspace. */
SSM_API int ssm_scan_step(int64_t batch, int64_t dim, int64_t dstate, int32_t in_dtype,
                  int32_t out_dtype, const void* u, const void* delta_raw,
                  const float* A, const void* B, const void* C, const float* D,
                  const void* z, const float* delta_bias, float* state, void* y,
                  int32_t* status, ssm_stream_t stream);

/* Synchronise `stream`, then return the device status word held in
 * `workspace` (SSM_OK, SSM_ERR_TIMEOUT or SSM_ERR_SEQLENS) and reset it to SSM_OK.  Returns
 * SSM_ERR_CUDA if the synchronisation itself fails, SSM_ERR_NULL for a NULL
 * workspace. */
SSM_API int ssm_get_status(void* workspace, ssm_stream_t stream);

/* Human-readable text of a status code (static storage, never NULL). */
SSM_API const char* ssm_strerror(int code);

/* Size in bytes of the fixed scratch array ssm_scan_fwd_noalloc runs in
 * (32 MiB). */
#define SSM_NOALLOC_SCRATCH_BYTES 33554432

/* ssm_scan_fwd for callers that cannot allocate device memory.  The method's
 * description has no counterpart to this entry point; it exists for callers
 * that are handed only their input and output buffers and may not allocate on the device
 * themselves (a plug-in inside a host engine whose allocator owns all device
 * memory, or a latency-bound loop that must not call cudaMalloc after
 * start-up, since it can synchronise the device and take unbounded time).
 * Arguments are those of ssm_scan_fwd without the workspace; nothing is
 * allocated or freed.
 *  - The scratch is a fixed array of SSM_NOALLOC_SCRATCH_BYTES (32 MiB)
 *    inside the library.  A shape whose ssm_scan_workspace_bytes(shape, 0)
 *    exceeds it is rejected with SSM_ERR_WORKSPACE before anything is
 *    enqueued (at 16 states that is about 262,000 tokens summed over the
 *    batch).
 *  - Every call looks up the array's device address on the current device
 *    (cudaGetSymbolAddress; a host-side lookup once the library's device code
 *    is loaded, so a new CUDA context after cudaDeviceReset gets its own
 *    address).  With CUDA's default lazy module loading the FIRST call on
 *    each device (or context) loads the library's device code and so reserves
 *    the 32 MiB there, which can allocate and synchronise: make one warm-up
 *    call at start-up, before any stream capture.  The array then stays
 *    reserved on that device until the process exits.
 *  - Every call shares the one array: calls whose work overlaps on the GPU
 *    (different streams, or several host threads) race and corrupt each
 *    other's results; issue them in order on one stream.  Each call rewrites
 *    all the scratch it reads, so earlier contents do not matter.
 *  - The device status word lives in that scratch and is not reachable by the
 *    caller; an expired device-side wait leaves y and hL undefined. */
SSM_API int ssm_scan_fwd_noalloc(const ssm_shape* shape, const void* u, const void* delta_raw,
                 const float* A, const void* B, const void* C, const float* D,
                 const void* z, const float* delta_bias, const float* h0,
                 void* y, float* hL, ssm_stream_t stream);

/* DIAGNOSTIC, not part of the scan: a failure-detection self test for the
 * test suite and for a caller who wants to check that expired device waits
 * reach the status word on their system.  Launches one block that waits on a device
 * flag nothing ever sets, giving up after `spin_limit` polls; the expired
 * wait is reported through the workspace status word (SSM_ERR_TIMEOUT, read
 * with ssm_get_status).  No copy is in flight while it waits. */
SSM_API int ssm_debug_expired_wait(void* workspace, size_t ws_bytes, int64_t spin_limit,
                           ssm_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* SSM_SCAN_H */
