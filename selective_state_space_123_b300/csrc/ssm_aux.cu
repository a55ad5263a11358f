// ssm_aux.cu -- the kernels around the forward scan:
//   * prep_bc:   B, C (batch, N, L) -> fp32 (batch, L, 2*NP) with ln2 folded
//                into B (the scan then uses delta/ln2 throughout);
//   * tail:      where each segment's summary pass may start (segmented plan);
//   * head:      where the segmented backward's adjoint summary may stop;
//   * carry:     per-segment initial states of the segmented forward,
//                h_in[s+1] = 2^(A * sum_delta2[s]) * h_in[s] + h_loc[s];
//   * varlen_prep: checks packed-sequence starts, final states of empty ones;
//   * tangent carry: the segmented backward's dA terms across segments;
//   * expired_wait: the failure-detection self test (a wait nothing ends).
#include "ssm_common.cuh"
#include "ssm_kernels.cuh"
#include "ssm_internal.h"

namespace ssm {

// ------------------------------------------------------------- prep_bc ---
template <typename TIN>
__global__ void prep_bc_kernel(int64_t Bt, int N, int NP, int64_t L, const TIN* __restrict__ B,
                               const TIN* __restrict__ C, float* __restrict__ out, int* status) {
    // first kernel of every call on a workspace: clear its status word
    if (status && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0 && threadIdx.y == 0) *status = 0;
    __shared__ float tb[64][33];
    __shared__ float tc[64][33];
    const int tx = threadIdx.x, ty = threadIdx.y;   // 32 x 8
    const int64_t b = blockIdx.y;
    const int64_t t0 = (int64_t)blockIdx.x * 32;
    for (int n = ty; n < N; n += 8) {
        const int64_t t = t0 + tx;
        float vb = 0.0f, vc = 0.0f;
        if (t < L) {
            vb = Elem<TIN>::to_f(B[(b * N + n) * L + t]);
            vc = Elem<TIN>::to_f(C[(b * N + n) * L + t]);
        }
        tb[n][tx] = vb;
        tc[n][tx] = vc;
    }
    __syncthreads();
    for (int r = ty; r < 32; r += 8) {
        const int64_t t = t0 + r;
        if (t >= L) break;
        float* o = out + (b * L + t) * (2 * NP);
        for (int j = tx; j < 2 * NP; j += 32) {
            float v = 0.0f;
            if (j < NP) {
                if (j < N) v = kLn2 * tb[j][r];
            } else if (j - NP < N) {
                v = tc[j - NP][r];
            }
            o[j] = v;
        }
    }
}

// The same for bf16 inputs whose rows are 16-byte aligned (L % 8 = 0) and at
// most 16 states: a CTA of 256 threads takes 64 tokens of one batch row,
// reads 8 tokens of one (B or C, state) row per 16-byte load, transposes
// through shared memory (rows padded to 65 floats, so that both the loads'
// stores and the output's reads hit 32 distinct banks per warp) and writes
// whole 16-byte chunks of the output rows.
constexpr int kPrepT = 64;
constexpr int kPrepPitch = kPrepT + 1;
__global__ void __launch_bounds__(256) prep_bc16_kernel(int64_t Bt, int N, int64_t L,
                                                        const __nv_bfloat16* __restrict__ B,
                                                        const __nv_bfloat16* __restrict__ C,
                                                        float* __restrict__ out, int* status) {
    constexpr int NP = 16;
    if (status && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *status = 0;
    __shared__ float tile[2 * NP * kPrepPitch];   // [B or C][state][token]
    const int tid = threadIdx.x;
    const int64_t b = blockIdx.y;
    const int64_t t0 = (int64_t)blockIdx.x * kPrepT;
    {
        // task = (B or C, state, group of 8 tokens): 2 x 16 x 8 = 256 tasks
        const int c8 = tid & 7;
        const int n = (tid >> 3) & (NP - 1);
        const int which = tid >> 7;
        const int64_t t = t0 + c8 * 8;
        float v[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
        if (n < N && t < L) {   // L % 8 = 0: the 8 tokens are all in the row
            const __nv_bfloat16* src = (which ? C : B) + (b * N + n) * L + t;
            const uint4 w = *reinterpret_cast<const uint4*>(src);
            v[0] = bf_lo(w.x); v[1] = bf_hi(w.x); v[2] = bf_lo(w.y); v[3] = bf_hi(w.y);
            v[4] = bf_lo(w.z); v[5] = bf_hi(w.z); v[6] = bf_lo(w.w); v[7] = bf_hi(w.w);
        }
        const float sc = which ? 1.0f : kLn2;
        float* row = tile + (which * NP + n) * kPrepPitch + c8 * 8;
#pragma unroll
        for (int q = 0; q < 8; ++q) row[q] = v[q] * sc;
    }
    __syncthreads();
    // output: 64 token rows x 8 chunks of 4 floats (B' states 0..15, then C)
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int idx = tid + 256 * k;
        const int r = idx >> 3, j4 = idx & 7;
        const int64_t t = t0 + r;
        if (t < L) {
            const float* col = tile + (j4 * 4) * kPrepPitch + r;
            *reinterpret_cast<float4*>(out + (b * L + t) * (2 * NP) + j4 * 4) =
                make_float4(col[0], col[kPrepPitch], col[2 * kPrepPitch], col[3 * kPrepPitch]);
        }
    }
}

cudaError_t launch_prep_bc(int tin, int64_t Bt, int N, int NP, int64_t L, const void* B,
                           const void* C, float* out, int* status, cudaStream_t st) {
    if (tin == SSM_BF16 && NP == 16 && N <= 16 && L % 8 == 0) {
        dim3 grid16((unsigned)((L + kPrepT - 1) / kPrepT), (unsigned)Bt);
        prep_bc16_kernel<<<grid16, 256, 0, st>>>(Bt, N, L, static_cast<const __nv_bfloat16*>(B),
                                                 static_cast<const __nv_bfloat16*>(C), out, status);
        return cudaGetLastError();
    }
    dim3 grid((unsigned)((L + 31) / 32), (unsigned)Bt), block(32, 8);
    if (tin == SSM_BF16)
        prep_bc_kernel<__nv_bfloat16><<<grid, block, 0, st>>>(
            Bt, N, NP, L, static_cast<const __nv_bfloat16*>(B), static_cast<const __nv_bfloat16*>(C), out, status);
    else
        prep_bc_kernel<float><<<grid, block, 0, st>>>(Bt, N, NP, L, static_cast<const float*>(B),
                                                      static_cast<const float*>(C), out, status);
    return cudaGetLastError();
}

// --------------------------------------------------------------- carry ---
// reverse: the right-to-left scan of the bidirectional form, whose state
// runs from the last segment to the first (h0 enters the last segment).
__global__ void carry_kernel(int64_t Bt, int64_t D, int N, int NP, int nseg, const float* __restrict__ A,
                             const float* __restrict__ h0, const float* __restrict__ hloc,
                             const float* __restrict__ sumd, float* __restrict__ hin, bool reverse) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;   // (b, d, n)
    if (i >= Bt * D * NP) return;
    const int n = (int)(i % NP);
    const int64_t row = i / NP;
    const int64_t d = row % D;
    const int64_t seg_stride = Bt * D;
    const float a = n < N ? A[d * N + n] : 0.0f;
    float h = (h0 && n < N) ? h0[row * N + n] : 0.0f;
    for (int j = 0; j < nseg; ++j) {
        const int s = reverse ? nseg - 1 - j : j;
        hin[(s * seg_stride + row) * NP + n] = h;
        if (j + 1 < nseg) {
            const float sd = sumd[s * seg_stride + row];
            h = (sd >= kTailSat ? 0.0f : ex2(a * sd) * h) + hloc[(s * seg_stride + row) * NP + n];
        }
    }
}

// Packed sequences: block 0 checks the starts; every block takes a share of
// the sequences and gives each empty one its initial state as final state
// (the scan kernels write the others).  per_seq = Bt * D * N floats.
__global__ void varlen_prep_kernel(const int* __restrict__ cu, int nseq, int64_t L, int64_t per_seq,
                                   const float* __restrict__ h0, float* __restrict__ hL,
                                   int* status) {
    if (blockIdx.x == 0) {
        for (int s = threadIdx.x; s <= nseq; s += blockDim.x) {
            const int64_t v = cu[s];
            const bool bad = v < 0 || v > L || (s == 0 && v != 0) || (s == nseq && v != L) ||
                             (s > 0 && v < (int64_t)cu[s - 1]);
            if (bad) set_status(status, SSM_ERR_SEQLENS);
        }
    }
    if (!hL) return;
    for (int s = blockIdx.x; s < nseq; s += gridDim.x) {
        if (cu[s] != cu[s + 1]) continue;
        float* o = hL + (int64_t)s * per_seq;
        const float* i0 = h0 ? h0 + (int64_t)s * per_seq : nullptr;
        for (int64_t i = threadIdx.x; i < per_seq; i += blockDim.x) o[i] = i0 ? i0[i] : 0.0f;
    }
}

cudaError_t launch_varlen_prep(const int* cu, int nseq, int64_t L, int64_t per_seq, const float* h0,
                               float* hL, int* status, cudaStream_t st) {
    const int blocks = nseq < 1184 ? (nseq > 0 ? nseq : 1) : 1184;
    varlen_prep_kernel<<<blocks, 256, 0, st>>>(cu, nseq, L, per_seq, h0, hL, status);
    return cudaGetLastError();
}

// Tail search for the segmented plan.  Pass 1 needs each segment's end
// state from a zero start, h_end = sum_t P(t -> end) delta_t u_t B_t, where
// the decay of state n from token t to the segment's end is
// P = 2^(A_n * S_t), S_t = sum of delta2 over the tokens after t.  Once the
// slowest state's decay, 2^(max_n A_n * S_t), is below 2^-kTailLog2, the
// earlier tokens change h_end by less than 2^-40 of the state at that point,
// far below fp32 resolution, so pass 1 may start after them (the hot-path
// table's truncation option, with the full segment as the fallback).  The
// search walks delta backwards from each segment's end (one warp per
// channel, 16-byte loads) until that point or the segment's start, and
// writes per (segment, batch row, channel tile) the earliest chunk any
// channel of the tile needs, and per saturated channel kTailSat into sumd,
// so that the carry drops the incoming state (2^(A * kTailSat) = 0 for
// A < 0).  Where a tile needs its whole segment, pass 1 writes the exact
// sums.  Segments 0 .. nseg-2 (whole chunks); L * sizeof(TIN) % 16 == 0.
constexpr float kTailLog2 = 40.0f;

template <typename TIN>
__global__ void __launch_bounds__(1024) tail_kernel(const FwdParams p, int CH, int* __restrict__ tstart,
                                                    float* __restrict__ sumd) {
    constexpr bool ACCURATE = sizeof(TIN) == 4;
    constexpr int VEC = 16 / (int)sizeof(TIN);        // tokens per 16-byte load
    constexpr int LOADS = 4;                            // loads per lane per step
    constexpr int STEP = LOADS * 32 * VEC;              // tokens per warp step
    const int tile = blockIdx.x;
    const int64_t b = blockIdx.y;
    const int seg = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nwarps = blockDim.x >> 5;
    const int64_t c_begin = (int64_t)seg * p.seg_chunks;
    const int64_t c_end = c_begin + p.seg_chunks;       // segments 0 .. nseg-2 are full
    const int64_t s0 = c_begin * kT, s1 = c_end * kT;
    if (p.cu_seqlens) {
        // packed sequences: a segment holding a sequence start needs only the
        // tokens from its last start on (the carry then drops the incoming
        // state); the condition is the same for the whole block
        int lo = 0, hi = p.nseq;   // first start at or after the segment's end
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if ((int64_t)p.cu_seqlens[mid] < s1) lo = mid + 1;
            else hi = mid;
        }
        if (lo > 0 && (int64_t)p.cu_seqlens[lo - 1] >= s0) {
            if (threadIdx.x == 0)
                tstart[((int64_t)seg * p.Bt + b) * gridDim.x + tile] =
                    (int)((int64_t)p.cu_seqlens[lo - 1] / kT);
            return;
        }
    }
    __shared__ int cmin;
    if (threadIdx.x == 0) cmin = (int)(c_end - c_begin);
    __syncthreads();
    const TIN* dr = static_cast<const TIN*>(p.dr);
    int my_min = (int)(c_end - c_begin);               // chunk offsets within the segment
    for (int c = warp; c < CH; c += nwarps) {
        const int64_t d = (int64_t)tile * CH + c;
        if (d >= p.D) break;
        if (*reinterpret_cast<volatile int*>(&cmin) == 0) break;   // the tile needs its whole segment
        const int64_t row = b * p.D + d;
        float amax = -INFINITY;
        for (int n = 0; n < p.N; ++n) amax = fmaxf(amax, p.A[d * p.N + n]);
        const float bias2 = p.bias ? p.bias[d] * kLog2e : 0.0f;
        const TIN* rp = dr + row * p.L;
        double tot = 0.0;
        int64_t t0 = s0;
        bool sat = false;
        for (int64_t hi = s1; hi > s0; hi -= STEP) {
            const int64_t lo = hi - STEP > s0 ? hi - STEP : s0;
            float part = 0.0f;
#pragma unroll
            for (int j = 0; j < LOADS; ++j) {
                const int64_t t = lo + (int64_t)(j * 32 + lane) * VEC;
                if (t < hi) {
                    float v[VEC];
                    if constexpr (sizeof(TIN) == 2) {
                        const uint4 w = *reinterpret_cast<const uint4*>(rp + t);
                        v[0] = bf_lo(w.x); v[1] = bf_hi(w.x); v[2] = bf_lo(w.y); v[3] = bf_hi(w.y);
                        v[4] = bf_lo(w.z); v[5] = bf_hi(w.z); v[6] = bf_lo(w.w); v[7] = bf_hi(w.w);
                    } else {
                        const float4 w = *reinterpret_cast<const float4*>(rp + t);
                        v[0] = w.x; v[1] = w.y; v[2] = w.z; v[3] = w.w;
                    }
#pragma unroll
                    for (int q = 0; q < VEC; ++q) part += softplus2<ACCURATE>(fmaf(v[q], kLog2e, bias2));
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
            tot += (double)part;
            if (amax < 0.0f && (double)amax * tot <= -(double)kTailLog2) {
                t0 = lo;
                sat = true;
                break;
            }
        }
        const int need = (int)((t0 - s0) / kT);
        if (need < my_min) my_min = need;
        if (lane == 0) {
            if (sat) sumd[(int64_t)seg * p.Bt * p.D + row] = kTailSat;
            if (need == 0) atomicMin(&cmin, 0);
        }
    }
    if (lane == 0) atomicMin(&cmin, my_min);
    __syncthreads();
    if (threadIdx.x == 0)
        tstart[((int64_t)seg * p.Bt + b) * gridDim.x + tile] = (int)c_begin + cmin;
}

// The mirror for the backward's adjoint summary: the adjoint a segment
// passes to its left neighbour, a_{t0} lambda_{t0}, weighs token t's g_t C_t
// by the decay from t0 through t, 2^(A_n * S'_t) with S'_t = sum of delta2
// over tokens t0 .. t; once the slowest state's decay is below 2^-kTailLog2
// the later tokens do not matter.  The search walks delta forward from each
// segment's start (one warp per channel) and writes per (segment, batch
// row, channel tile) the chunk after the last one any channel of the tile
// needs, and per saturated channel kTailSat into sumd (the carry then drops
// the adjoint entering the segment from the right).  Segments 1 .. nseg-1
// (the last one may end with a partial chunk); L * sizeof(TIN) % 16 == 0.
template <typename TIN>
__global__ void __launch_bounds__(1024) head_kernel(const BwdParams p, int CH, int* __restrict__ kstop,
                                                    float* __restrict__ sumd) {
    constexpr bool ACCURATE = sizeof(TIN) == 4;
    constexpr int VEC = 16 / (int)sizeof(TIN);        // tokens per 16-byte load
    constexpr int LOADS = 4;                            // loads per lane per step
    constexpr int STEP = LOADS * 32 * VEC;              // tokens per warp step
    const int tile = blockIdx.x;
    const int64_t b = blockIdx.y;
    const int seg = blockIdx.z + 1;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nwarps = blockDim.x >> 5;
    const int64_t nchunks = (p.L + kT - 1) / kT;
    const int64_t c_begin = (int64_t)seg * p.seg_chunks;
    const int64_t c_end = min(nchunks, c_begin + p.seg_chunks);
    const int64_t s0 = c_begin * kT, s1 = min(p.L, c_end * kT);
    if (p.cu_seqlens) {
        // packed sequences: a segment in which a sequence ends (a start in
        // (s0, s1]) needs only the tokens up to its first end, and passes on
        // nothing from its right; the condition is the same for the whole block
        int lo = 0, hi = p.nseq;   // first start after s0
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if ((int64_t)p.cu_seqlens[mid] <= s0) lo = mid + 1;
            else hi = mid;
        }
        const int64_t c = lo < p.nseq ? (int64_t)p.cu_seqlens[lo] : p.L;
        if (c <= s1 && c < p.L) {
            for (int i = threadIdx.x; i < CH; i += blockDim.x) {
                const int64_t d = (int64_t)tile * CH + i;
                if (d < p.D) sumd[(int64_t)seg * p.Bt * p.D + b * p.D + d] = kTailSat;
            }
            if (threadIdx.x == 0)
                kstop[((int64_t)seg * p.Bt + b) * gridDim.x + tile] = (int)((c - 1) / kT + 1);
            return;
        }
    }
    __shared__ int cmax;
    if (threadIdx.x == 0) cmax = 0;
    __syncthreads();
    const TIN* dr = static_cast<const TIN*>(p.dr);
    const int whole = (int)(c_end - c_begin);           // chunk counts from the segment's start
    int my_max = 0;
    for (int c = warp; c < CH; c += nwarps) {
        const int64_t d = (int64_t)tile * CH + c;
        if (d >= p.D) break;
        if (*reinterpret_cast<volatile int*>(&cmax) == whole) break;   // the tile needs its whole segment
        const int64_t row = b * p.D + d;
        float amax = -INFINITY;
        for (int n = 0; n < p.N; ++n) amax = fmaxf(amax, p.A[d * p.N + n]);
        const float bias2 = p.bias ? p.bias[d] * kLog2e : 0.0f;
        const TIN* rp = dr + row * p.L;
        double tot = 0.0;
        int64_t t1 = s1;
        bool sat = false;
        for (int64_t lo = s0; lo < s1; lo += STEP) {
            const int64_t hi = lo + STEP < s1 ? lo + STEP : s1;
            float part = 0.0f;
#pragma unroll
            for (int j = 0; j < LOADS; ++j) {
                const int64_t t = lo + (int64_t)(j * 32 + lane) * VEC;
                if (t < hi) {
                    float v[VEC];
                    if constexpr (sizeof(TIN) == 2) {
                        const uint4 w = *reinterpret_cast<const uint4*>(rp + t);
                        v[0] = bf_lo(w.x); v[1] = bf_hi(w.x); v[2] = bf_lo(w.y); v[3] = bf_hi(w.y);
                        v[4] = bf_lo(w.z); v[5] = bf_hi(w.z); v[6] = bf_lo(w.w); v[7] = bf_hi(w.w);
                    } else {
                        const float4 w = *reinterpret_cast<const float4*>(rp + t);
                        v[0] = w.x; v[1] = w.y; v[2] = w.z; v[3] = w.w;
                    }
#pragma unroll
                    for (int q = 0; q < VEC; ++q)
                        if (t + q < hi) part += softplus2<ACCURATE>(fmaf(v[q], kLog2e, bias2));
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
            tot += (double)part;
            if (amax < 0.0f && (double)amax * tot <= -(double)kTailLog2) {
                t1 = hi;
                sat = true;
                break;
            }
        }
        const int need = (int)((t1 - s0 + kT - 1) / kT);
        if (need > my_max) my_max = need;
        if (lane == 0) {
            if (sat) sumd[(int64_t)seg * p.Bt * p.D + row] = kTailSat;
            if (need == whole) atomicMax(&cmax, whole);
        }
    }
    if (lane == 0) atomicMax(&cmax, my_max);
    __syncthreads();
    if (threadIdx.x == 0)
        kstop[((int64_t)seg * p.Bt + b) * gridDim.x + tile] = (int)c_begin + cmax;
}

cudaError_t launch_head(int tin, const BwdParams& p, int CH, unsigned tiles, int* kstop, float* sumd,
                        cudaStream_t st) {
    const dim3 grid(tiles, (unsigned)p.Bt, (unsigned)(p.nseg - 1));
    if (tin == SSM_BF16)
        head_kernel<__nv_bfloat16><<<grid, 1024, 0, st>>>(p, CH, kstop, sumd);
    else
        head_kernel<float><<<grid, 1024, 0, st>>>(p, CH, kstop, sumd);
    return cudaGetLastError();
}

cudaError_t launch_tail(int tin, const FwdParams& p, int CH, unsigned tiles, int* tstart, float* sumd,
                        cudaStream_t st) {
    const dim3 grid(tiles, (unsigned)p.Bt, (unsigned)(p.nseg - 1));
    if (tin == SSM_BF16)
        tail_kernel<__nv_bfloat16><<<grid, 1024, 0, st>>>(p, CH, tstart, sumd);
    else
        tail_kernel<float><<<grid, 1024, 0, st>>>(p, CH, tstart, sumd);
    return cudaGetLastError();
}

cudaError_t launch_carry(int64_t Bt, int64_t D, int N, int NP, int nseg, const float* A,
                         const float* h0, const float* hloc, const float* sumd, float* hin,
                         cudaStream_t st, bool reverse) {
    const int64_t total = Bt * D * NP;
    carry_kernel<<<(unsigned)((total + 255) / 256), 256, 0, st>>>(Bt, D, N, NP, nseg, A, h0, hloc,
                                                                  sumd, hin, reverse);
    return cudaGetLastError();
}


// ------------------------------------------------------ tangent carry ---
// Segmented backward: the forward sweep runs segment s with the tangent
// m = dh/dA (in units of 1/ln2) from zero, so the tangent of the whole
// sequence there is m_loc + P * m_in[s], with P the decay since the
// segment's start and m_in[s] = m_end[s-1] + 2^(A sumd[s-1]) m_in[s-1],
// m_in[0] = 0 (sumd = the forward summary's sum of delta/ln2, kTailSat where
// the decay is below fp32 resolution).  The missing dA terms are
// sum_s m_in[s] * gp[s] (gp = sum_t g_t C_t P_t, plus dhL P_L in the last
// segment), summed over the batch rows: one thread per (channel, state),
// added after the sweep's own atomics on the same stream.
__global__ void tangent_carry_kernel(int64_t Bt, int64_t D, int N, int NP, int nseg,
                                     const float* __restrict__ A, const float* __restrict__ sumd,
                                     const float* __restrict__ mend, const float* __restrict__ gp,
                                     float* __restrict__ dA) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;   // (d, n)
    if (i >= D * N) return;
    const int64_t d = i / N;
    const int n = (int)(i % N);
    const float a = A[i];
    const int64_t seg_stride = Bt * D;
    float acc = 0.0f;
    for (int64_t b = 0; b < Bt; ++b) {
        const int64_t row = b * D + d;
        float m = 0.0f;
        for (int s = 1; s < nseg; ++s) {
            const int64_t prev = (int64_t)(s - 1) * seg_stride + row;
            const float sd = sumd[prev];
            m = fmaf(sd >= kTailSat ? 0.0f : ex2(a * sd), m, mend[prev * NP + n]);
            acc = fmaf(m, gp[((int64_t)s * seg_stride + row) * NP + n], acc);
        }
    }
    dA[i] += kLn2 * acc;
}

cudaError_t launch_tangent_carry(int64_t Bt, int64_t D, int N, int NP, int nseg, const float* A,
                                 const float* sumd, const float* mend, const float* gp, float* dA,
                                 cudaStream_t st) {
    const int64_t total = D * N;
    if (total == 0 || nseg < 2) return cudaSuccess;
    tangent_carry_kernel<<<(unsigned)((total + 255) / 256), 256, 0, st>>>(Bt, D, N, NP, nseg, A, sumd,
                                                                          mend, gp, dA);
    return cudaGetLastError();
}


// -------------------------------------------------------- expired wait ---
// A single CTA arms an mbarrier that nothing will ever complete and waits on
// it with a poll limit; no copy is in flight.  The expired wait is reported
// through the status word, exactly like a stalled pipeline in the scan.
__global__ void expired_wait_kernel(int* status, int64_t spin_limit, uint64_t timeout_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        if (!mbar_wait(&bar, 0, timeout_ns, spin_limit)) set_status(status, SSM_ERR_TIMEOUT);
    }
}

cudaError_t launch_expired_wait(int* status, int64_t spin_limit, cudaStream_t st) {
    expired_wait_kernel<<<1, 32, 0, st>>>(status, spin_limit, kDefaultTimeoutNs);
    return cudaGetLastError();
}

}  // namespace ssm
