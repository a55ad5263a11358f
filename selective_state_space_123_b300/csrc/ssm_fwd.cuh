// ssm_fwd.cuh -- forward selective-scan kernel (templated; instantiated in
// the ssm_fwd_*.cu translation units) plus the small helper kernels of the
// forward path.
//
// What one CTA does (sources: "The convolution trick is gone -- what now?",
// Mamba lesson 2: keep the recurrence on chip, write back only the final
// state; "State Space Models (SSMs) & Mamba", section "Hardware-Aware
// Parallelism": the recurrence is a scan over the sequence):
//   * it owns CH = 32 W / NT channels of one batch row (W <= 7 compute warps,
//     chosen by the host planner) for a whole segment of the sequence
//     (normally the whole sequence);
//   * a producer warp streams 64-token chunks of u, delta_raw, z (TMA, 128-B
//     swizzle) and of the prepared B/C tile into a multi-stage shared-memory
//     ring guarded by mbarriers;
//   * each compute thread keeps G = NP/NT states of one channel in
//     registers; the NT threads of a channel split the per-token work
//     (softplus, gate, D skip) and exchange it with warp shuffles;
//   * per token and state: dA = 2^(delta2 * A) on the MUFU (delta2 = delta /
//     ln 2, so no extra scaling), h = dA h + delta u B, y += C h, in packed
//     f32x2 arithmetic.  With fp32 inputs the state is carried compensated
//     (comp_update: two floats, the decay as 2^x - 1 on the FMA pipe) so that
//     long sequences and long memories keep fp32-level agreement.
// SUMMARY = true is pass 1 of the segmented plan for very long sequences: no
// read-out, the kernel records each segment's end state from a zero start and
// the segment's sum of delta2 (the decay of the carried state over the
// segment is 2^(A * sum)); it starts at the chunk a tail search found (the
// earlier tokens' decay to the segment end is below 2^-40).
// Variants, each its own instantiation ("Mamba Architecture Explained"):
//   CONV = true   the raw tile holds the conv branch input x; u = silu(causal
//                 depthwise conv of x) is formed per lane from the tile
//                 (section "The Architecture in Practice");
//   VARLEN = true packed sequences: the state restarts at every start in
//                 cu_seqlens (section "Problem 3: Ecosystem maturity");
//   DIR = 1 / 2   the bidirectional scan's right-to-left pass (chunks,
//                 super-blocks and tokens in reverse order) and its
//                 left-to-right pass, which adds the first pass's output
//                 (section "Frequently Asked Questions").
#pragma once

#include "ssm_common.cuh"
#include "ssm_kernels.cuh"

namespace ssm {

template <int NP>
constexpr int bc_tile_bytes() { return kT * 2 * NP * 4; }

// 8 consecutive tokens [tb, tb+8) of local channel c from a raw tile of
// `ch` channel rows (TMA 128-byte swizzle; fp32 tiles are two boxes of 32
// tokens, each ch x 128 bytes).
template <typename TIN>
__device__ __forceinline__ void load_raw8r(const uint8_t* tile, int ch, int c, int tb,
                                           float (&v)[8]) {
    if constexpr (sizeof(TIN) == 2) {
        const uint4 w = *reinterpret_cast<const uint4*>(tile + swz128(c, tb * 2));
        v[0] = bf_lo(w.x); v[1] = bf_hi(w.x); v[2] = bf_lo(w.y); v[3] = bf_hi(w.y);
        v[4] = bf_lo(w.z); v[5] = bf_hi(w.z); v[6] = bf_lo(w.w); v[7] = bf_hi(w.w);
    } else {
        const uint8_t* box = tile + (tb / 32) * (ch * 128);
        const int cb = (tb % 32) * 4;
        const float4 a = *reinterpret_cast<const float4*>(box + swz128(c, cb));
        const float4 b = *reinterpret_cast<const float4*>(box + swz128(c, cb + 16));
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
}
template <typename TIN, int CH>
__device__ __forceinline__ void load_raw8(const uint8_t* tile, int c, int tb, float (&v)[8]) {
    load_raw8r<TIN>(tile, CH, c, tb, v);
}

// Store 8 consecutive outputs of one row; `nv` of them are inside the row.
template <typename TOUT>
__device__ __forceinline__ void store_out8(void* y, int64_t off, const float (&v)[8], int nv,
                                           bool vec_ok) {
    if (nv <= 0) return;
    if constexpr (sizeof(TOUT) == 2) {
        __nv_bfloat16* yp = reinterpret_cast<__nv_bfloat16*>(y) + off;
        if (vec_ok && nv >= 8) {
            uint4 w;
            w.x = pack_bf16x2(v[0], v[1]); w.y = pack_bf16x2(v[2], v[3]);
            w.z = pack_bf16x2(v[4], v[5]); w.w = pack_bf16x2(v[6], v[7]);
            *reinterpret_cast<uint4*>(yp) = w;
        } else {
#pragma unroll
            for (int q = 0; q < 8; ++q)
                if (q < nv) yp[q] = __float2bfloat16_rn(v[q]);
        }
    } else {
        float* yp = reinterpret_cast<float*>(y) + off;
        if (vec_ok && nv >= 8) {
            reinterpret_cast<float4*>(yp)[0] = make_float4(v[0], v[1], v[2], v[3]);
            reinterpret_cast<float4*>(yp)[1] = make_float4(v[4], v[5], v[6], v[7]);
        } else {
#pragma unroll
            for (int q = 0; q < 8; ++q)
                if (q < nv) yp[q] = v[q];
        }
    }
}

// Plain (non-TMA) fill of one raw tile of `ch` rows, used when rows are not
// 16-byte aligned (seqlen * element size not a multiple of 16).  Same
// swizzled layout as the TMA tiles.
template <typename TIN>
__device__ __forceinline__ void fill_raw_tile_r(uint8_t* tile, int ch, const void* src,
                                                int64_t row0, int64_t rows_valid, int64_t L,
                                                int64_t t0, int lane) {
    const TIN* s = reinterpret_cast<const TIN*>(src);
    for (int idx = lane; idx < ch * kT; idx += 32) {
        const int c = idx / kT, t = idx % kT;
        TIN v = TIN(0.0f);
        if (c < rows_valid && t0 + t < L) v = s[(row0 + c) * L + t0 + t];
        uint8_t* dst;
        if constexpr (sizeof(TIN) == 2) {
            dst = tile + swz128(c, t * 2);
        } else {
            dst = tile + (t / 32) * (ch * 128) + swz128(c, (t % 32) * 4);
        }
        *reinterpret_cast<TIN*>(dst) = v;
    }
}
template <typename TIN, int CH>
__device__ __forceinline__ void fill_raw_tile(uint8_t* tile, const void* src, int64_t row0,
                                              int64_t rows_valid, int64_t L, int64_t t0,
                                              int lane) {
    fill_raw_tile_r<TIN>(tile, CH, src, row0, rows_valid, L, t0, lane);
}

// First s in [0, nseq) with cu[s] >= t (nseq if none); a bounded binary
// search, also on unsorted input.
__device__ __forceinline__ int seq_lower_bound(const int* cu, int nseq, int64_t t) {
    int lo = 0, hi = nseq;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if ((int64_t)cu[mid] < t) lo = mid + 1;
        else hi = mid;
    }
    return lo;
}

// No restart inside a super-block.
struct NoRestart {
    template <typename H>
    __device__ __forceinline__ void operator()(int, H&) const {}
};

// One state's update in the compensated form used for fp32 inputs.  The state
// is hi + lo (two floats).  With e = 2^x - 1 (x = delta2 * A, exp2m1_accurate)
// the update is h + (e h + xin): when the decay is close to 1 this keeps the
// forgetting rate e to its own relative accuracy (2^x rounded to fp32 would
// keep only that of 1), and the rounding error of adding the small increment
// to hi is recovered exactly (TwoSum) into lo, so that it does not pile up
// over the ~1/(delta |A|) tokens the state remembers.  For e < -1/2 (the
// state forgets within a few tokens, nothing accumulates) the plain form
// (1 + e) h + xin is used, 1 + e being exact there.
__device__ __forceinline__ void comp_update_e(float e, float xin, float& hi, float& lo) {
    const float a = 1.0f + e;
    const float plain = fmaf(a, hi, xin);
    const float inc = fmaf(e, hi, xin);
    const float s = hi + inc;
    const float bb = s - hi;
    const float err = (hi - (s - bb)) + (inc - bb);
    const bool fast = e < -0.5f;
    lo = fmaf(e, lo, lo) + (fast ? 0.0f : err);
    hi = fast ? plain : s;
}
// the same from x = delta2 * A
__device__ __forceinline__ void comp_update(float x, float xin, float& hi, float& lo) {
    comp_update_e(exp2m1_accurate(x), xin, hi, lo);
}

// The recurrence over one super-block of SB tokens for one lane's G states.
//   d2, du: delta/ln2 and delta2*u of the SB tokens (registers)
//   bcb:    prepared B/C row of the super-block's first token at this lane's states
//   hl:     low parts of the compensated state (ACCURATE only; unused otherwise)
// With RESTART, tokens whose bit is set in `rmask` begin a packed sequence:
// `restart(tt, h)` replaces the state (h and hl) before that token's update.
// With REV the tokens are taken from the last to the first.
template <int NP, int G, int SB, bool SUMMARY, bool ACCURATE, bool REV = false,
          bool RESTART = false, typename F = NoRestart>
__device__ __forceinline__ void fwd_chain(const float (&d2)[SB], const float (&du)[SB],
                                          const float* bcb, const f2 (&Ap)[G / 2],
                                          f2 (&h)[G / 2], f2 (&hl)[G / 2], float (&yp)[SB],
                                          uint32_t rmask = 0, F restart = F()) {
    constexpr int Q = G / 4;
#pragma unroll
    for (int t0 = 0; t0 < SB; ++t0) {
        const int tt = REV ? SB - 1 - t0 : t0;
        if constexpr (RESTART) {
            if ((rmask >> tt) & 1u) restart(tt, h);
        }
        const f2 d2p = pk(d2[tt], d2[tt]), dup = pk(du[tt], du[tt]);
        const float* bcrow = bcb + tt * (2 * NP);
        f2 acc = pk(0.0f, 0.0f);
#pragma unroll
        for (int q4 = 0; q4 < Q; ++q4) {
            const ulonglong2 Bq = *reinterpret_cast<const ulonglong2*>(bcrow + 4 * q4);
            if constexpr (ACCURATE) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int j = 2 * q4 + e;
                    float x0, x1, i0, i1, h0, h1, l0, l1;
                    upk(mul2(d2p, Ap[j]), x0, x1);
                    upk(mul2(dup, e ? Bq.y : Bq.x), i0, i1);
                    upk(h[j], h0, h1);
                    upk(hl[j], l0, l1);
                    comp_update(x0, i0, h0, l0);
                    comp_update(x1, i1, h1, l1);
                    h[j] = pk(h0, h1);
                    hl[j] = pk(l0, l1);
                }
            } else {
                const f2 a0 = ex2x2(mul2(d2p, Ap[2 * q4]));
                const f2 a1 = ex2x2(mul2(d2p, Ap[2 * q4 + 1]));
                h[2 * q4] = fma2(a0, h[2 * q4], mul2(dup, Bq.x));
                h[2 * q4 + 1] = fma2(a1, h[2 * q4 + 1], mul2(dup, Bq.y));
            }
            if (!SUMMARY) {
                const ulonglong2 Cq = *reinterpret_cast<const ulonglong2*>(bcrow + NP + 4 * q4);
                acc = fma2(Cq.x, h[2 * q4], acc);
                acc = fma2(Cq.y, h[2 * q4 + 1], acc);
                if constexpr (ACCURATE) {
                    acc = fma2(Cq.x, hl[2 * q4], acc);
                    acc = fma2(Cq.y, hl[2 * q4 + 1], acc);
                }
            }
        }
        if (!SUMMARY) {
            float lo, hi;
            upk(acc, lo, hi);
            yp[tt] = lo + hi;
        }
    }
}

// Forward kernel.  blockDim.x = 32 * (W + 1): W compute warps and one
// producer warp (the last).  A CTA owns CH = W * 32 / NT channels of one
// batch row for one segment of the sequence.  Per super-block of SB = TPL *
// NT tokens each lane computes softplus and delta * u of its own TPL tokens
// and gathers the channel's other tokens from its NT - 1 partner lanes by
// shuffles, runs the recurrence over the SB tokens for its G = NP / NT
// states, writes its per-token partial read-outs to the warp's exchange
// buffer, and then finishes its own TPL tokens (sum over the NT lanes, D
// skip, SiLU gate, store).  All exchange stays inside the warp.
template <int NP, int NT, typename TIN, typename TOUT, bool SUMMARY, bool TMA_RAW, bool CONV = false,
          bool VARLEN = false, int DIR = 0>
__global__ void __launch_bounds__(32 * (FwdLayout<NT>::kMaxWarps + 1), FwdLayout<NT>::kMinBlocks)
fwd_kernel(const FwdParams p, const __grid_constant__ CUtensorMap tm_u,
           const __grid_constant__ CUtensorMap tm_dr, const __grid_constant__ CUtensorMap tm_z,
           const __grid_constant__ CUtensorMap tm_bc, const __grid_constant__ CUtensorMap tm_ya) {
    using Lay = FwdLayout<NT>;
    constexpr int G = NP / NT;
    constexpr int CW = Lay::CW;
    constexpr int SB = Lay::SB;
    constexpr int TPL = Lay::TPL;     // tokens each lane finishes per super-block
    constexpr int EB = (int)sizeof(TIN);
    constexpr int NRAW = SUMMARY ? 2 : 3;
    constexpr int BCB = bc_tile_bytes<NP>();
    // the left-to-right pass of the bidirectional scan streams the other
    // direction's fp32 output through the ring as a fourth tile
    constexpr bool YTILE = DIR == 2;
    constexpr bool ACCURATE = EB == 4;
    static_assert(G == 4 || G == 8 || G == 16, "states per thread");
    static_assert(NT == 1 || NT == 2 || NT == 4, "threads per channel");

    const int W = (int)(blockDim.x / 32) - 1;
    const int CH = W * CW;
    const int RAW = CH * kT * EB;
    const int RAWF = YTILE ? CH * kT * 4 : 0;
    const int STAGE = NRAW * RAW + RAWF + BCB;
    const int BCOFF = NRAW * RAW + RAWF;   // the B/C tile's offset in a stage
    const int STAGES = p.stages;

    extern __shared__ uint8_t smem_dyn[];
    uint8_t* smem = align_smem_1024(smem_dyn);
    float* xy_all = reinterpret_cast<float*>(smem + STAGES * STAGE);
    __shared__ __align__(8) uint64_t full_bar[kFwdMaxStages];
    __shared__ __align__(8) uint64_t empty_bar[kFwdMaxStages];

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int64_t b = blockIdx.y;
    const int64_t d0 = (int64_t)blockIdx.x * CH;
    const int seg = (int)blockIdx.z + p.seg0;
    const int64_t L = p.L;
    const int64_t nchunks = (L + kT - 1) / kT;
    const int64_t k_seg = (int64_t)seg * p.seg_chunks;
    const int64_t k_end = min(nchunks, k_seg + p.seg_chunks);
    // a summary starts where the tail search found that the segment's end
    // state no longer depends on earlier tokens (their decay is below 2^-40)
    int64_t k_begin =
        (SUMMARY && p.tstart)
            ? max(k_seg, min(k_end - 1, (int64_t)p.tstart[((int64_t)seg * p.Bt + blockIdx.y) * gridDim.x + blockIdx.x]))
            : k_seg;
    if constexpr (VARLEN && SUMMARY) {
        // packed: the segment's end state depends only on the tokens from the
        // last sequence start inside the segment on
        const int j = seq_lower_bound(p.cu_seqlens, p.nseq, k_end * kT);
        if (j > 0) {
            const int64_t ls = p.cu_seqlens[j - 1];
            if (ls >= k_seg * kT && ls < k_end * kT) k_begin = max(k_begin, ls / kT);
        }
    }
    const bool has_z = !SUMMARY && p.z != nullptr;

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], W);
        }
        fence_mbar_init();
    }
    __syncthreads();

    // ------------------------------------------------------ producer warp
    if (warp == W) {
        if (lane == 0) {
            prefetch_tmap(&tm_bc);
            if (TMA_RAW) {
                prefetch_tmap(&tm_u);
                prefetch_tmap(&tm_dr);
                if (has_z) prefetch_tmap(&tm_z);
                if (YTILE) prefetch_tmap(&tm_ya);
            }
        }
        constexpr int BOXES = kT * EB / 128;   // 128-byte TMA boxes per tile row
        constexpr int BOX_T = 128 / EB;        // tokens per box
        const int64_t row0 = b * p.D + d0;
        const int64_t rows_valid = (int64_t)min((int64_t)CH, p.D - d0);
        for (int64_t i = 0; i < k_end - k_begin; ++i) {
            const int64_t k = DIR == 1 ? k_end - 1 - i : k_begin + i;   // right to left: last chunk first
            const int s = (int)(i % STAGES);
            if (i >= STAGES) {
                bool ok = true;
                if (lane == 0)
                    ok = mbar_wait(&empty_bar[s], (uint32_t)(((i / STAGES) - 1) & 1), p.timeout_ns);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) {
                    if (lane == 0) set_status(p.status, SSM_ERR_TIMEOUT);
                    return;
                }
            }
            uint8_t* st = smem + s * STAGE;
            const int32_t t0 = (int32_t)(k * kT);
            if (TMA_RAW) {
                if (lane == 0) {
                    mbar_arrive_expect_tx(&full_bar[s], (uint32_t)((has_z ? 3 : 2) * RAW + RAWF + BCB));
#pragma unroll
                    for (int bx = 0; bx < BOXES; ++bx) {
                        const int32_t x = t0 + bx * BOX_T;
                        tma_load_2d(st + bx * CH * 128, &tm_u, &full_bar[s], x, (int32_t)row0);
                        tma_load_2d(st + RAW + bx * CH * 128, &tm_dr, &full_bar[s], x, (int32_t)row0);
                        if (has_z)
                            tma_load_2d(st + 2 * RAW + bx * CH * 128, &tm_z, &full_bar[s], x,
                                        (int32_t)row0);
                    }
                    if (YTILE) {
                        // fp32 rows: two boxes of 32 tokens per chunk
#pragma unroll
                        for (int bx = 0; bx < 2; ++bx)
                            tma_load_2d(st + NRAW * RAW + bx * CH * 128, &tm_ya, &full_bar[s],
                                        t0 + bx * 32, (int32_t)row0);
                    }
                    tma_load_2d(st + BCOFF, &tm_bc, &full_bar[s], 0, (int32_t)(b * L + t0));
                }
            } else {
                fill_raw_tile_r<TIN>(st, CH, p.u, row0, rows_valid, L, t0, lane);
                fill_raw_tile_r<TIN>(st + RAW, CH, p.dr, row0, rows_valid, L, t0, lane);
                if (has_z) fill_raw_tile_r<TIN>(st + 2 * RAW, CH, p.z, row0, rows_valid, L, t0, lane);
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive_expect_tx(&full_bar[s], BCB);
                    tma_load_2d(st + BCOFF, &tm_bc, &full_bar[s], 0, (int32_t)(b * L + t0));
                }
            }
        }
        return;
    }

    // ---------------------------------------------------- compute warps
    const int cw = lane / NT;          // channel within the warp
    const int g = lane % NT;           // state group
    const int c = warp * CW + cw;      // channel within the CTA
    const int64_t d = d0 + c;
    const bool ch_ok = d < p.D;
    const int64_t row = b * p.D + d;
    const int N = p.N;
    float* xy = xy_all + warp * Lay::XY_FLOATS;   // this warp's exchange buffer
    const int src_base = lane & ~(NT - 1);         // lane g = 0 of this channel

    f2 Ap[G / 2], h[G / 2];
    f2 hl[G / 2];   // low parts of the compensated state (fp32 inputs), else zero
#pragma unroll
    for (int j = 0; j < G / 2; ++j) {
        const int n0 = g * G + 2 * j, n1 = n0 + 1;
        const float a0 = (ch_ok && n0 < N) ? p.A[d * N + n0] : 0.0f;
        const float a1 = (ch_ok && n1 < N) ? p.A[d * N + n1] : 0.0f;
        Ap[j] = pk(a0, a1);
        hl[j] = pk(0.0f, 0.0f);
        float h0v = 0.0f, h1v = 0.0f;
        if (!SUMMARY && ch_ok) {
            if (p.hin) {
                const float* hs = p.hin + ((int64_t)seg * p.Bt * p.D + row) * NP;
                h0v = hs[n0];
                h1v = hs[n1];
            } else if (p.h0) {
                if (n0 < N) h0v = p.h0[row * N + n0];
                if (n1 < N) h1v = p.h0[row * N + n1];
            }
        }
        h[j] = pk(h0v, h1v);
    }
    const float bias2 = (p.bias && ch_ok) ? p.bias[d] * kLog2e : 0.0f;
    const float Dd = (p.Dv && ch_ok) ? p.Dv[d] : 0.0f;
    const bool vec_out = ((L * (int64_t)sizeof(TOUT)) % 16) == 0;
    double sum_d2 = 0.0;
    // conv prologue: weights right-aligned to width 4 (leading zeros for a
    // narrower kernel) and the last 3 branch inputs before the current chunk
    float cw4[4] = {0.0f, 0.0f, 0.0f, 0.0f}, cbias = 0.0f, xhalo[3] = {0.0f, 0.0f, 0.0f};
    if constexpr (CONV) {
        if (ch_ok) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {   // static indices: the weights stay in registers
                const int kk = q - (4 - p.conv_k);
                if (kk >= 0) cw4[q] = p.conv_w[d * p.conv_k + kk];
            }
            cbias = p.conv_b ? p.conv_b[d] : 0.0f;
            const int64_t t0 = k_begin * kT;   // a segment starting inside the sequence
            const TIN* xr = static_cast<const TIN*>(p.u) + row * L;
#pragma unroll
            for (int q = 0; q < 3; ++q)
                if (t0 - 3 + q >= 0) xhalo[q] = Elem<TIN>::to_f(xr[t0 - 3 + q]);
        }
    }
    // packed sequences: every thread walks the sequence starts in token
    // order (the same walk in all threads, so branches on it are uniform).
    // sp = index of the first start after the last token scanned, next_start
    // = that start, cur_start = start of the sequence being scanned.
    int sp = 0;
    int64_t next_start = INT64_MAX, cur_start = 0;
    bool seg_restart = false;   // a sequence starts inside this segment
    if constexpr (VARLEN) {
        const int* cu = p.cu_seqlens;
        sp = seq_lower_bound(cu, p.nseq, k_begin * kT);
        next_start = sp < p.nseq ? (int64_t)cu[sp] : INT64_MAX;
        cur_start = sp > 0 ? (int64_t)cu[sp - 1] : 0;
        const int j = seq_lower_bound(cu, p.nseq, k_seg * kT);
        seg_restart = j < p.nseq && (int64_t)cu[j] < min(k_end * kT, L);
    }
    // a sequence starting at token t: write the final state of the one that
    // ended at t - 1 (pass 2), then start from h0 of the new one (or zero)
    auto restart = [&](int64_t t, f2 (&hh)[G / 2]) {
        if constexpr (VARLEN) {
            const int* cu = p.cu_seqlens;
            const int last = p.nseq - 1;
            if (!SUMMARY && ch_ok && p.hL && t > 0) {
                const int sf = min(max(sp - 1, 0), last);
                float* hfin = p.hL + ((int64_t)sf * p.Bt * p.D + row) * N;
#pragma unroll
                for (int j = 0; j < G / 2; ++j) {
                    float lo, hi;
                    upk(ACCURATE ? add2(hh[j], hl[j]) : hh[j], lo, hi);
                    const int n0 = g * G + 2 * j;
                    if (n0 < N) hfin[n0] = lo;
                    if (n0 + 1 < N) hfin[n0 + 1] = hi;
                }
            }
            while (sp < p.nseq && (int64_t)cu[sp] <= t) ++sp;
            const int sn = min(max(sp - 1, 0), last);
            const float* hs = (p.h0 && ch_ok) ? p.h0 + ((int64_t)sn * p.Bt * p.D + row) * N : nullptr;
#pragma unroll
            for (int j = 0; j < G / 2; ++j) {
                const int n0 = g * G + 2 * j;
                hh[j] = pk((hs && n0 < N) ? hs[n0] : 0.0f, (hs && n0 + 1 < N) ? hs[n0 + 1] : 0.0f);
                hl[j] = pk(0.0f, 0.0f);
            }
            next_start = sp < p.nseq ? (int64_t)cu[sp] : INT64_MAX;
        }
    };
    bool dead = false;   // a bounded wait expired: stop working (warp-uniform)

    for (int64_t i = 0; i < k_end - k_begin && !dead; ++i) {
        const int64_t k = DIR == 1 ? k_end - 1 - i : k_begin + i;
        const int s = (int)(i % STAGES);
        const bool ok = __all_sync(
            0xffffffffu, mbar_wait(&full_bar[s], (uint32_t)((i / STAGES) & 1), p.timeout_ns));
        if (!ok) {
            if (lane == 0) set_status(p.status, SSM_ERR_TIMEOUT);
            dead = true;
            break;
        }
        const uint8_t* st = smem + s * STAGE;
        const float* bct = reinterpret_cast<const float*>(st + BCOFF);
        const int nvalid = (int)min((int64_t)kT, L - k * kT);

#pragma unroll 1
        for (int sbi = 0; sbi < kT / SB; ++sbi) {
            const int sb = DIR == 1 ? kT / SB - 1 - sbi : sbi;
            if (sb * SB >= nvalid) {
                if (DIR == 1) continue;   // right to left: padded super-blocks come first
                break;
            }
            const int64_t t_sb = k * kT + sb * SB;
            uint32_t rmask = 0;   // tokens of this super-block that start a sequence
            if constexpr (VARLEN) {
                if (next_start < t_sb + SB) {
                    for (int j = sp; j < p.nseq; ++j) {
                        const int64_t cs = p.cu_seqlens[j];
                        if (cs >= t_sb + SB || cs >= L) break;
                        if (cs >= t_sb) rmask |= 1u << (int)(cs - t_sb);
                        else sp = j + 1;   // out of order (invalid starts): skip for good
                    }
                    next_start = sp < p.nseq ? (int64_t)p.cu_seqlens[sp] : INT64_MAX;
                }
            }

            // 1. each lane computes delta2 = softplus / ln2 and delta2 * u of its
            //    own TPL tokens, then gathers all SB tokens of the channel from
            //    the NT lanes with shuffles (one softplus per token)
            const int tb = sb * SB + g * TPL;
            float uo[TPL];
            float d2[SB], du[SB];
            {
                float dv[TPL], d2o[TPL], duo[TPL];
#pragma unroll
                for (int k8 = 0; k8 < TPL / 8; ++k8) {
                    float t8[8], r8[8];
                    load_raw8r<TIN>(st, CH, c, tb + 8 * k8, t8);
                    load_raw8r<TIN>(st + RAW, CH, c, tb + 8 * k8, r8);
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        uo[8 * k8 + q] = t8[q];
                        dv[8 * k8 + q] = r8[q];
                    }
                }
                if constexpr (CONV) {
                    // the tile holds the branch input x: u = silu(conv of x);
                    // the 3 inputs before this lane's first token come from
                    // the tile, or from the previous chunk at token 0
                    float prev[8];
                    load_raw8r<TIN>(st, CH, c, tb >= 8 ? tb - 8 : 0, prev);
                    float xw[TPL + 3];
#pragma unroll
                    for (int q = 0; q < 3; ++q) xw[q] = tb > 0 ? prev[5 + q] : xhalo[q];
#pragma unroll
                    for (int q = 0; q < TPL; ++q) xw[3 + q] = uo[q];
                    // taps before the token's sequence start (kmin of them) read zero
                    auto conv_tok = [&](int q, int kmin) {
                        float a = fmaf(cw4[0], kmin > 0 ? 0.0f : xw[q], cbias);
                        a = fmaf(cw4[1], kmin > 1 ? 0.0f : xw[q + 1], a);
                        a = fmaf(cw4[2], kmin > 2 ? 0.0f : xw[q + 2], a);
                        a = fmaf(cw4[3], xw[q + 3], a);
                        uo[q] = a * rcp(1.0f + ex2(-kLog2e * a));
                    };
                    bool masked = false;
                    if constexpr (VARLEN) {
                        if (rmask != 0 || cur_start > t_sb - 3) {
#pragma unroll
                            for (int q = 0; q < TPL; ++q) {
                                const int r = g * TPL + q;   // token within the super-block
                                const uint32_t m = rmask & ((2u << r) - 1u);
                                const int64_t st0 = m ? t_sb + (31 - __clz(m)) : cur_start;
                                conv_tok(q, (int)(st0 - (t_sb + r)) + 3);
                            }
                            masked = true;
                        }
                    }
                    if (!masked) {
#pragma unroll
                        for (int q = 0; q < TPL; ++q) conv_tok(q, 0);
                    }
                }
                const bool full = nvalid == kT;   // warp-uniform: no padded token
                float s8 = 0.0f;
#pragma unroll
                for (int q = 0; q < TPL; ++q) {
                    float dd = softplus2<ACCURATE>(fmaf(dv[q], kLog2e, bias2));
                    if (!full && tb + q >= nvalid) dd = 0.0f;
                    d2o[q] = dd;
                    duo[q] = dd * uo[q];
                    if (SUMMARY) s8 += dd;
                }
                if (SUMMARY) sum_d2 += (double)s8;   // this lane's own tokens
#pragma unroll
                for (int jj = 0; jj < NT; ++jj) {
#pragma unroll
                    for (int q = 0; q < TPL; ++q) {
                        d2[TPL * jj + q] = NT == 1 ? d2o[q] : __shfl_sync(0xffffffffu, d2o[q], src_base + jj);
                        du[TPL * jj + q] = NT == 1 ? duo[q] : __shfl_sync(0xffffffffu, duo[q], src_base + jj);
                    }
                }
            }
            // 2. the recurrence over the SB tokens for this lane's G states
            float yp[SB];
            bool restarted = false;
            if constexpr (VARLEN) {
                if (rmask != 0) {
                    fwd_chain<NP, G, SB, SUMMARY, ACCURATE, false, true>(
                        d2, du, bct + sb * SB * (2 * NP) + g * G, Ap, h, hl, yp, rmask,
                        [&](int tt, f2 (&hh)[G / 2]) { restart(t_sb + tt, hh); });
                    cur_start = t_sb + (31 - __clz(rmask));
                    restarted = true;
                }
            }
            if (!restarted)
                fwd_chain<NP, G, SB, SUMMARY, ACCURATE, DIR == 1>(
                    d2, du, bct + sb * SB * (2 * NP) + g * G, Ap, h, hl, yp);

            if (!SUMMARY) {
                // 3. partial read-outs through the buffer (one lane per channel:
                //    the lane's own sums); finish the own tokens
                float* yb = xy + cw * Lay::YROW;
                if (NT > 1) {
#pragma unroll
                    for (int q = 0; q < SB; q += 4)
                        *reinterpret_cast<float4*>(yb + Lay::xoff(cw, g * SB + q)) =
                            make_float4(yp[q], yp[q + 1], yp[q + 2], yp[q + 3]);
                    __syncwarp();
                }
#pragma unroll
                for (int k8 = 0; k8 < TPL / 8; ++k8) {
                    float yt[8];
                    if (NT == 1) {
#pragma unroll
                        for (int q = 0; q < 8; ++q) yt[q] = yp[8 * k8 + q];
                    }
#pragma unroll
                    for (int gg = 0; gg < (NT > 1 ? NT : 0); ++gg) {
                        const float4 a = *reinterpret_cast<const float4*>(yb + Lay::xoff(cw, gg * SB + g * TPL + 8 * k8));
                        const float4 bq = *reinterpret_cast<const float4*>(yb + Lay::xoff(cw, gg * SB + g * TPL + 8 * k8 + 4));
                        if (gg == 0) {
                            yt[0] = a.x; yt[1] = a.y; yt[2] = a.z; yt[3] = a.w;
                            yt[4] = bq.x; yt[5] = bq.y; yt[6] = bq.z; yt[7] = bq.w;
                        } else {
                            yt[0] += a.x; yt[1] += a.y; yt[2] += a.z; yt[3] += a.w;
                            yt[4] += bq.x; yt[5] += bq.y; yt[6] += bq.z; yt[7] += bq.w;
                        }
                    }
                    float zv[8];
                    if (has_z) load_raw8r<TIN>(st + 2 * RAW, CH, c, tb + 8 * k8, zv);
                    float out[8];
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        float v = fmaf(Dd, uo[8 * k8 + q], yt[q]);
                        if (has_z) v *= zv[q] * rcp(1.0f + ex2(-kLog2e * zv[q]));
                        out[q] = v;
                    }
                    if constexpr (YTILE) {
                        // the right-to-left scan's gated output of these tokens,
                        // from the ring (zeros past the row's end)
                        float ya[8];
                        load_raw8r<float>(st + NRAW * RAW, CH, c, tb + 8 * k8, ya);
#pragma unroll
                        for (int q = 0; q < 8; ++q) out[q] += ya[q];
                    }
                    if (ch_ok)
                        store_out8<TOUT>(p.y, row * L + k * kT + tb + 8 * k8, out,
                                         nvalid - (tb + 8 * k8), vec_out);
                }
                __syncwarp();   // before the next super-block overwrites the buffer
            }
        }
        if constexpr (CONV) {
            // the chunk's last 3 inputs start the next chunk's convolution
            float last[8];
            load_raw8r<TIN>(st, CH, c, kT - 8, last);
#pragma unroll
            for (int q = 0; q < 3; ++q) xhalo[q] = last[5 + q];
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[s]);
    }
    if (dead) return;

    if (SUMMARY) {
        // one thread per channel records the segment's sum of delta2 (each
        // lane summed its own tokens)
        double tot = sum_d2;
#pragma unroll
        for (int o = 1; o < NT; o <<= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
        if (ch_ok) {
            float* hsum = p.hloc + ((int64_t)seg * p.Bt * p.D + row) * NP + g * G;
#pragma unroll
            for (int j = 0; j < G / 2; ++j) {
                float lo, hi;
                upk(ACCURATE ? add2(h[j], hl[j]) : h[j], lo, hi);
                hsum[2 * j] = lo;
                hsum[2 * j + 1] = hi;
            }
            // a summary over the whole segment has the exact sum; a shortened one
            // keeps the search's saturation marker
            // (a sequence starting inside the segment cuts the carried state off)
            if (g == 0 && (seg_restart || k_begin == k_seg))
                p.sumd[(int64_t)seg * p.Bt * p.D + row] = seg_restart ? kTailSat : (float)tot;
        }
    } else if ((DIR == 1 ? k_seg == 0 : k_end == nchunks) && p.hL && ch_ok) {
        // the last sequence's final state (packed: the one holding token L-1;
        // right to left: the state after token 0, in the first segment)
        const int64_t sf = VARLEN ? (int64_t)min(max(sp - 1, 0), p.nseq - 1) : 0;
        float* hfin = p.hL + (sf * p.Bt * p.D + row) * N;
#pragma unroll
        for (int j = 0; j < G / 2; ++j) {
            float lo, hi;
            upk(ACCURATE ? add2(h[j], hl[j]) : h[j], lo, hi);
            const int n0 = g * G + 2 * j;
            if (n0 < N) hfin[n0] = lo;
            if (n0 + 1 < N) hfin[n0 + 1] = hi;
        }
    }
}

}  // namespace ssm
