// ssm_kernels.cuh -- launch parameters shared between the host dispatcher
// (ssm_api.cu) and the kernels.  Internal to libssmscan.so.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace ssm {

constexpr int kT = 64;              // tokens per chunk (one TMA tile along L)
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;  // bounded waits: 2 s

// Forward-kernel layout per NT (threads per channel).  Per compute warp an
// exchange buffer holds, per channel, the NT partial read-outs of one
// super-block.  With two lanes per channel a row is 40 floats (10 16-byte
// chunks, 8 used) and chunk f of channel cw sits at slot f ^ (cw & 3): the
// eight lanes of a quarter warp then reach eight distinct bank groups both
// when they store their partials (chunks 4g .. 4g+3) and when they read
// the partials of their own tokens (chunks 4gg + 2g + h); other NT pad the
// rows by 16 bytes.
template <int NT>
struct FwdLayout {
    static constexpr int CW = 32 / NT;             // channels per compute warp
    static constexpr int TPL = 8;                  // tokens each lane finishes per super-block
    static constexpr int SB = TPL * NT;            // tokens per super-block
    static constexpr int YROW = NT * SB + (NT == 2 ? 8 : 4);   // floats per channel row
    static constexpr int XY_FLOATS = CW * YROW;
    // float offset in channel cw's row of the partial read-out at position f
    // (f = lane-in-channel * SB + token, a multiple of 4 for a chunk start)
    static __host__ __device__ constexpr int xoff(int cw, int f) {
        return NT == 2 ? (((f >> 2) ^ (cw & 3)) << 2) + (f & 3) : f;
    }
    static constexpr int kMaxWarps = 7;    // compute warps per CTA at most (+ the producer: 256 threads)
    static constexpr int kMinBlocks = 1;   // launch bound: up to 255 registers, no spills
};
constexpr int kFwdMaxStages = 6;
constexpr int kMaxSmemPerCta = 226 * 1024;   // dynamic shared memory per CTA (227 KB on sm_103a, less the static part)

// Forward scan parameters.  Layouts are the public ones (see ssm_scan.h);
// `bc` is the prepared copy of B and C: (batch, seqlen, 2*NP) fp32 with
// [0, NP) = ln2 * B[b, n, t] and [NP, 2NP) = C[b, n, t], zero for n >= N.
// Marker in a segment's sum of delta2 (segmented plan): the carry drops the
// state coming into the segment (the tail search found its decay below
// 2^-40, or a packed sequence starts inside the segment).
constexpr float kTailSat = 1e30f;

struct FwdParams {
    int64_t Bt, D, L;
    int N;
    const void* u;
    const void* dr;
    const void* z;          // nullable
    const float* A;
    const float* Dv;        // nullable
    const float* bias;      // nullable
    const float* h0;        // nullable
    const float* bc;
    void* y;
    float* hL;              // nullable
    // segmented plan (nseg > 1): the sequence is cut into nseg segments of
    // seg_chunks chunks; pass 1 writes per-segment summaries, the carry
    // kernel turns them into per-segment initial states, pass 2 writes y.
    int64_t seg_chunks;
    int nseg;
    int seg0;               // segment of blockIdx.z = 0 (the right-to-left summary pass: 1)
    float* hin;             // (nseg, Bt, D, NP) initial state of each segment (pass 2)
    float* hloc;            // (nseg, Bt, D, NP) end state from a zero start (pass 1)
    float* sumd;            // (nseg, Bt, D) sum of delta/ln2 over the segment (pass 1)
    // pass 1 with a tail search (nullable): first chunk each (segment, batch
    // row, channel tile) must run, (nseg, Bt, tiles); sumd is then written by
    // the search, or by pass 1 where it runs the whole segment
    const int* tstart;
    int stages;             // depth of the shared-memory ring (<= kFwdMaxStages)
    // conv prologue (the kernel instantiated with CONV): u is computed from
    // the branch input x (passed as `u`) by a causal depthwise convolution of
    // width conv_k <= 4 and SiLU; conv_w (D, conv_k), conv_b (D) nullable
    const float* conv_w;
    const float* conv_b;
    int conv_k;
    // packed sequences (the kernel instantiated with VARLEN): every batch row
    // holds nseq sequences, sequence s at tokens [cu_seqlens[s],
    // cu_seqlens[s+1]); the state restarts at each start (from h0[s], h0 then
    // (nseq, Bt, D, N)) and hL receives every sequence's final state (nseq,
    // Bt, D, N)
    const int* cu_seqlens;
    int nseq;
    // bidirectional forward (the kernel instantiated with DIR = 2): the other
    // direction's gated output (Bt, D, L) fp32, added to y
    const float* yadd;
    int* status;
    uint64_t timeout_ns;
};

// Backward-kernel layout per (NT, NP): per compute warp a transpose buffer
// of 8 tokens x CW channels x NP states for the cross-channel sums of dB and
// dC.  In a token row, lane L's G states are KC = G/4 16-byte chunks; chunk k
// sits at slot 32k + (L ^ s(k)), so that the lanes of one quarter warp write
// eight distinct bank groups, and rows are padded so that the reads of one
// quarter warp (the same 4 states of up to 32/NP tokens' channels) hit
// disjoint banks too.
template <int NT, int NP>
struct BwdLayout {
    static constexpr int CW = 32 / NT;             // channels per compute warp
    static constexpr int G = NP / NT;              // states per lane
    static constexpr int SB = 8 * NT;              // tokens per super-block
    static constexpr int KC = G / 4;               // 16-byte chunks per lane and token
    static constexpr int TPAD = NP == 8 ? 8 : NP == 16 ? (NT == 2 ? 8 : 16) : 4;
    static constexpr int TROW = CW * NP + TPAD;    // floats per token row of the transpose buffer
    static constexpr int TBUF = 8 * TROW;          // floats per warp
    // float offset of lane L's chunk k inside a token row
    static __host__ __device__ constexpr int chunk(int L, int k) {
        return 4 * (KC == 1 ? L : 32 * k + (L ^ (KC == 2 ? 4 * k : 2 * k)));
    }
    static constexpr int kMaxWarps = 7;            // compute warps per CTA at most
};

// Backward parameters (both sweeps).
struct BwdParams {
    int64_t Bt, D, L;
    int N;
    const void* u;
    const void* dr;
    const void* z;          // nullable
    const void* dy;
    const float* A;
    const float* Dv;        // nullable
    const float* bias;      // nullable
    const float* h0;        // nullable
    const float* dhL;       // nullable
    const float* bc;        // prepared B/C (see FwdParams)
    float* phi;             // (Bt*D, L) fp32 workspace, written by the forward sweep
    float* hfin;            // (Bt*D, NP) fp32 workspace: final state
    float* hck;             // (Bt*D, nchunks, NP) fp32 workspace: state at the end of each chunk
    float* hprev;           // fp32 inputs: (Bt*D, L, NP) fp32 workspace, the state each
                            // token's update starts from
    void* du;
    void* ddr;
    void* dz;               // nullable
    float* dA;              // accumulated with atomics (zeroed by the host)
    float* dB;              // accumulated with atomics (zeroed by the host)
    float* dC;              // accumulated with atomics (zeroed by the host)
    float* dD;              // nullable, accumulated (zeroed by the host)
    float* dbias;           // nullable, accumulated (zeroed by the host)
    float* dh0;             // nullable
    int stages;             // depth of the shared-memory ring (<= kFwdMaxStages)
    // segmented plan (nseg > 1, grid z = segment; 0 or 1: whole rows): the
    // sequence is cut into nseg segments of seg_chunks chunks
    int64_t seg_chunks;
    int nseg;
    const float* hin;       // (nseg, Bt, D, NP) state before each segment (the forward's carry)
    const float* lam_in;    // (nseg, Bt, D, NP) a_{t1} lambda_{t1} entering each segment from the right
    float* lam_loc;         // (nseg, Bt, D, NP) the same from a zero start (adjoint summary)
    float* sumd;            // (nseg, Bt, D) sum of delta/ln2 over a segment (adjoint summary)
    const int* kstop;       // (nseg, Bt, tiles) nullable: chunk after the last one the adjoint
                            // summary needs (head search; sumd then holds its saturation marks)
    float* gp;              // (nseg, Bt, D, NP) sum_t g_t C_t P_t, P_t = decay since the segment start
    float* mend;            // (nseg, Bt, D, NP) dA tangent / ln2 at the segment end from a zero start
    // conv prologue (the kernel instantiated with CONV): u is computed from
    // the branch input x (passed as `u`) by a causal depthwise convolution of
    // width conv_k <= 4 and SiLU; conv_w (D, conv_k), conv_b (D) nullable
    const float* conv_w;
    const float* conv_b;
    int conv_k;
    // packed sequences (the kernel instantiated with VARLEN): every batch row
    // holds nseq sequences, sequence s at tokens [cu_seqlens[s],
    // cu_seqlens[s+1]); the state restarts at each start (from h0[s], h0 then
    // (nseq, Bt, D, N)) and hL receives every sequence's final state (nseq,
    // Bt, D, N)
    const int* cu_seqlens;
    int nseq;
    // bidirectional forward (the kernel instantiated with DIR = 2): the other
    // direction's gated output (Bt, D, L) fp32, added to y
    const float* yadd;
    int* status;
    uint64_t timeout_ns;
};

struct StepParams {
    int64_t Bt, D;
    int N;
    const void* u;
    const void* dr;
    const void* z;
    const float* A;
    const float* Dv;
    const float* bias;
    const void* B;
    const void* C;
    float* state;
    void* y;
    int* status;            // nullable: SSM_ERR_TIMEOUT on an expired wait
};

}  // namespace ssm
