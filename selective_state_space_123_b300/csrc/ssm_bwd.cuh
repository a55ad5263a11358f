// ssm_bwd.cuh -- reverse mode of the selective scan (templated; instantiated
// in the ssm_bwd_*.cu translation units).
//
// The pages give no backward pass; this is the exact derivative of the
// recurrence of "State Space Models (SSMs) & Mamba" (sections "State-Space
// Models (SSMs): A Resurgent Paradigm" and "The Magic of Selective Scan"),
// in natural units:
//   g_t      = dy_t silu(z_t)                     (dy_t if there is no gate)
//   lambda_t = g_t C_t + a_{t+1} lambda_{t+1},     lambda_L = g_L C_L + dhL
//   du_t     = g_t D + delta_t sum_n lambda_t B_t
//   ddelta_t = sum_n lambda_t (A a_t h_{t-1} + B_t u_t)
//   dB_t     = sum_d lambda_t delta_t u_t,   dC_t = sum_d g_t h_t
//   dA       = sum_{b,t} lambda_t delta_t a_t h_{t-1},   dh0 = a_1 lambda_1
//   dz_t     = dy_t (sum_n C_t h_t + D u_t) silu'(z_t)
//
// Two streaming sweeps per channel tile, neither of which keeps per-token
// states:
//  * bwd_fwd_kernel runs the recurrence forward from h0 and, beside h, the
//    tangent m = dh/dA (m_t = a_t m_{t-1} + delta_t a_t h_{t-1}), so that
//    dA = sum_t g_t C_t m_t + dhL m_L needs no reverse pass.  It also emits
//    dz, dC (reduced over the tile's channels, then added to global memory),
//    the final state, and one fp32 number per token,
//        phi_t = g_t sum_n A_n C_t[n] a_t[n] h_{t-1}[n].
//  * bwd_rev_kernel walks the sequence backwards carrying lambda.  The one
//    term of ddelta that needs h, Q_t = sum_n A_n lambda_t a_t h_{t-1}, is
//    rebuilt from per-token scalars: substituting the two recurrences gives
//    Q_t = Q_{t+1} + phi_t - rho_t with
//        rho_t = delta_t u_t sum_n A_n a_{t+1}[n] lambda_{t+1}[n] B_t[n]
//    and Q after the last token = psi = sum_n A_n dhL[n] h_L[n], hence
//        ddelta_t = psi + sum_{s>=t} (phi_s - rho_s) + u_t sum_n lambda_t B_t.
//    Both increments shrink with the decay a, so states that forget quickly
//    add no large, cancelling terms to the fp32 suffix sum.  The sum runs
//    over scalars per (channel, token); at every chunk boundary it is reset
//    to its exact value, computed from lambda and the state at the end of the
//    previous chunk (stored by the forward sweep, N floats per 64 tokens), so
//    rounding never accumulates over more than one chunk.
// Units: as in the forward kernel, delta2 = delta / ln2 and the prepared B
// is ln2 * B, so delta * B * u = delta2 * u * B'.  Gradients are written in
// natural units.
#pragma once

#include "ssm_fwd.cuh"

namespace ssm {

__device__ __forceinline__ void red_add_v4(float* addr, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};"
                 ::"l"(addr), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}

// Sum the W warps' partials of one chunk (red[w][n][t]) and add them to
// out[(b*N + n)*L + t0 + t] for n < N, t < nvalid, scaled by `scale`.
template <int NP>
__device__ __forceinline__ void flush_red(const float* red, int W, float* out, int64_t b, int N,
                                          int64_t L, int64_t t0, int nvalid, float scale,
                                          int tid, int nthreads) {
    const bool vec = (L % 4) == 0;
    for (int idx = tid; idx < NP * (kT / 4); idx += nthreads) {
        const int n = idx / (kT / 4);
        const int t = (idx % (kT / 4)) * 4;
        if (n >= N || t >= nvalid) continue;
        float s[4] = {0.f, 0.f, 0.f, 0.f};
        for (int w = 0; w < W; ++w) {
            const float4 v = *reinterpret_cast<const float4*>(red + (w * NP + n) * kT + t);
            s[0] += v.x; s[1] += v.y; s[2] += v.z; s[3] += v.w;
        }
        float* o = out + (b * N + n) * L + t0 + t;
        if (vec && t + 4 <= nvalid) {
            red_add_v4(o, s[0] * scale, s[1] * scale, s[2] * scale, s[3] * scale);
        } else {
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (t + q < nvalid) atomicAdd(o + q, s[q] * scale);
        }
    }
}

// Cross-channel sum of one group of 8 tokens through the warp's transpose
// buffer (token rows of CW channels x NP states, laid out as BwdLayout says):
// lane tasks are (token, group of 4 states); each sums the CW channels'
// float4s and writes the 4 sums to the warp's chunk buffer redw[n][t].
template <int NP, int CW>
__device__ __forceinline__ void transpose_reduce(const float* tb, float* redw, int t_first, int lane) {
    using Lay = BwdLayout<32 / CW, NP>;
    constexpr int NT = 32 / CW;
    constexpr int TASKS = 8 * NP / 4;
    for (int task = lane; task < TASKS; task += 32) {
        const int t = task / (NP / 4);
        const int q = task % (NP / 4);
        const int g = q / Lay::KC, kc = q % Lay::KC;    // the lane within a channel and its chunk
        const float* src = tb + t * Lay::TROW;
        f2 s01 = pk(0.0f, 0.0f), s23 = pk(0.0f, 0.0f);
#pragma unroll
        for (int c = 0; c < CW; ++c) {
            const ulonglong2 v = *reinterpret_cast<const ulonglong2*>(src + Lay::chunk(c * NT + g, kc));
            s01 = add2(s01, v.x);
            s23 = add2(s23, v.y);
        }
        float a0, a1, a2, a3;
        upk(s01, a0, a1);
        upk(s23, a2, a3);
        float* o = redw + (q * 4) * kT + t_first + t;
        o[0] = a0;
        o[kT] = a1;
        o[2 * kT] = a2;
        o[3 * kT] = a3;
    }
}

// Issue the loads of one stage (producer warp).  Raw tiles at slots 0..3
// (u, delta_raw, z, dy) of RAW bytes each, then (PHI: the reverse sweep) the
// fp32 per-token tile of RAWF bytes, then the B/C tile.
template <typename TIN, int NP, bool PHI, bool TMA_RAW>
__device__ __forceinline__ void bwd_load_stage(
    uint8_t* st, uint64_t* bar, const BwdParams& p, const CUtensorMap* tm_u,
    const CUtensorMap* tm_dr, const CUtensorMap* tm_z, const CUtensorMap* tm_dy,
    const CUtensorMap* tm_phi, const CUtensorMap* tm_bc, int64_t b, int64_t row0,
    int64_t rows_valid, int64_t k, bool has_z, int lane, int CH) {
    constexpr int EB = (int)sizeof(TIN);
    constexpr int BOXES = kT * EB / 128, BOX_T = 128 / EB;
    const int RAW = CH * kT * EB;
    const int RAWF = CH * kT * 4;
    constexpr int BCB = bc_tile_bytes<NP>();
    const int64_t L = p.L;
    const int32_t t0 = (int32_t)(k * kT);
    uint8_t* phi_dst = st + 4 * RAW;
    uint8_t* bc_dst = st + 4 * RAW + (PHI ? RAWF : 0);
    if (TMA_RAW) {
        if (lane == 0) {
            const uint32_t bytes = (has_z ? 4 : 3) * RAW + (PHI ? RAWF : 0) + BCB;
            mbar_arrive_expect_tx(bar, bytes);
#pragma unroll
            for (int bx = 0; bx < BOXES; ++bx) {
                const int32_t x = t0 + bx * BOX_T;
                tma_load_2d(st + bx * CH * 128, tm_u, bar, x, (int32_t)row0);
                tma_load_2d(st + RAW + bx * CH * 128, tm_dr, bar, x, (int32_t)row0);
                if (has_z) tma_load_2d(st + 2 * RAW + bx * CH * 128, tm_z, bar, x, (int32_t)row0);
                tma_load_2d(st + 3 * RAW + bx * CH * 128, tm_dy, bar, x, (int32_t)row0);
            }
            if (PHI) {
#pragma unroll
                for (int bx = 0; bx < 2; ++bx)
                    tma_load_2d(phi_dst + bx * CH * 128, tm_phi, bar, t0 + bx * 32, (int32_t)row0);
            }
            tma_load_2d(bc_dst, tm_bc, bar, 0, (int32_t)(b * L + t0));
        }
    } else {
        fill_raw_tile_r<TIN>(st, CH, p.u, row0, rows_valid, L, t0, lane);
        fill_raw_tile_r<TIN>(st + RAW, CH, p.dr, row0, rows_valid, L, t0, lane);
        if (has_z) fill_raw_tile_r<TIN>(st + 2 * RAW, CH, p.z, row0, rows_valid, L, t0, lane);
        fill_raw_tile_r<TIN>(st + 3 * RAW, CH, p.dy, row0, rows_valid, L, t0, lane);
        if (PHI) fill_raw_tile_r<float>(phi_dst, CH, p.phi, row0, rows_valid, L, t0, lane);
        __syncwarp();
        if (lane == 0) {
            mbar_arrive_expect_tx(bar, BCB);
            tma_load_2d(bc_dst, tm_bc, bar, 0, (int32_t)(b * L + t0));
        }
    }
}

// Producer warp: stream the chunks k_begin .. k_end-1 (forward or reverse
// order) through the ring, and add each finished chunk's cross-channel sums
// (the W warps' slices of the double-buffered chunk buffer) to `out` with
// vector atomics: the flush of chunk i-1 follows the loads of chunk i, so the
// compute warps never wait for it and never meet at a CTA barrier (out null:
// no sums, nothing to flush).  Gives up (status set) if a bounded wait
// expires.
template <typename TIN, int NP, bool REV, bool TMA_RAW, bool PHI = REV>
__device__ __forceinline__ void bwd_producer(uint8_t* smem, int STAGES, int STAGE,
                                             uint64_t* full_bar, uint64_t* empty_bar,
                                             uint64_t* rfull, uint64_t* rempty, const float* red,
                                             int W, float* out, float scale,
                                             const BwdParams& p, const CUtensorMap* tm_u,
                                             const CUtensorMap* tm_dr, const CUtensorMap* tm_z,
                                             const CUtensorMap* tm_dy, const CUtensorMap* tm_phi,
                                             const CUtensorMap* tm_bc, int64_t b, int64_t d0,
                                             bool has_z, int lane, int CH, int64_t k_begin,
                                             int64_t k_end) {
    if (lane == 0) {
        prefetch_tmap(tm_bc);
        if (TMA_RAW) {
            prefetch_tmap(tm_u);
            prefetch_tmap(tm_dr);
            if (has_z) prefetch_tmap(tm_z);
            prefetch_tmap(tm_dy);
            if (PHI) prefetch_tmap(tm_phi);
        }
    }
    const int64_t L = p.L;
    const int64_t nloc = k_end - k_begin;
    const int64_t row0 = b * p.D + d0;
    const int64_t rows_valid = (int64_t)min((int64_t)CH, p.D - d0);
    const int N = p.N;
    // flush of the chunk processed i-th: wait until all W warps wrote their
    // slices, add them up, then hand the buffer back to the compute warps
    auto flush = [&](int64_t i) -> bool {
        const int buf = (int)(i & 1);
        bool ok = true;
        if (lane == 0) ok = mbar_wait(&rfull[buf], (uint32_t)((i >> 1) & 1), p.timeout_ns);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) return false;
        const int64_t k = REV ? k_end - 1 - i : k_begin + i;
        const int nvalid = (int)min((int64_t)kT, L - k * kT);
        flush_red<NP>(red + (size_t)buf * W * NP * kT, W, out, b, N, L, k * kT, nvalid, scale, lane, 32);
        __syncwarp();
        if (lane == 0) mbar_arrive(&rempty[buf]);
        return true;
    };
    for (int64_t i = 0; i < nloc; ++i) {
        const int64_t k = REV ? k_end - 1 - i : k_begin + i;
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
        bwd_load_stage<TIN, NP, PHI, TMA_RAW>(smem + s * STAGE, &full_bar[s], p, tm_u, tm_dr, tm_z,
                                              tm_dy, tm_phi, tm_bc, b, row0, rows_valid, k, has_z,
                                              lane, CH);
        if (out && i >= 1 && !flush(i - 1)) {
            if (lane == 0) set_status(p.status, SSM_ERR_TIMEOUT);
            return;
        }
    }
    if (out && nloc >= 1 && !flush(nloc - 1)) {
        if (lane == 0) set_status(p.status, SSM_ERR_TIMEOUT);
    }
}

// Per-token quantities the chain loop needs for this lane's 8 tokens:
// delta2 = delta / ln2, delta2 * u and g = dy * silu(z) (dy without a gate).
// Tokens past the end, and channels past D (whose tile rows belong to the
// next batch row), get zeros and so contribute nothing.
template <typename TIN, bool ACCURATE>
__device__ __forceinline__ void token_prep(const uint8_t* st, int CH, int c, int tb, int nvalid,
                                           bool has_z, bool ch_ok, float bias2, float (&d2)[8],
                                           float (&du)[8], float (&gq)[8]) {
    const int RAW = CH * kT * (int)sizeof(TIN);
    float uv[8], dv[8], gy[8];
    load_raw8r<TIN>(st, CH, c, tb, uv);
    load_raw8r<TIN>(st + RAW, CH, c, tb, dv);
    load_raw8r<TIN>(st + 3 * RAW, CH, c, tb, gy);
    float zv[8];
    if (has_z) load_raw8r<TIN>(st + 2 * RAW, CH, c, tb, zv);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        d2[q] = softplus2<ACCURATE>(fmaf(dv[q], kLog2e, bias2));
        du[q] = d2[q] * uv[q];
        gq[q] = has_z ? gy[q] * zv[q] * rcp(1.0f + ex2(-kLog2e * zv[q])) : gy[q];
        if (tb + q >= nvalid || !ch_ok) {
            d2[q] = 0.0f;
            du[q] = 0.0f;
            gq[q] = 0.0f;
        }
    }
}

// token_prep with u given (the conv prologue forms it from the branch input).
template <typename TIN, bool ACCURATE>
__device__ __forceinline__ void token_prep_u(const uint8_t* st, int CH, int c, int tb, int nvalid,
                                             bool has_z, bool ch_ok, float bias2, const float (&uv)[8],
                                             float (&d2)[8], float (&du)[8], float (&gq)[8]) {
    const int RAW = CH * kT * (int)sizeof(TIN);
    float dv[8], gy[8];
    load_raw8r<TIN>(st + RAW, CH, c, tb, dv);
    load_raw8r<TIN>(st + 3 * RAW, CH, c, tb, gy);
    float zv[8];
    if (has_z) load_raw8r<TIN>(st + 2 * RAW, CH, c, tb, zv);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        d2[q] = softplus2<ACCURATE>(fmaf(dv[q], kLog2e, bias2));
        du[q] = d2[q] * uv[q];
        gq[q] = has_z ? gy[q] * zv[q] * rcp(1.0f + ex2(-kLog2e * zv[q])) : gy[q];
        if (tb + q >= nvalid || !ch_ok) {
            d2[q] = 0.0f;
            du[q] = 0.0f;
            gq[q] = 0.0f;
        }
    }
}

// The conv prologue of the backward: the tile's slot 0 holds the branch
// input x, and this lane's 8 tokens [tb, tb + 8) of the chunk starting at
// token t_chunk get u = silu(conv_b + sum_k w_k x[t - 3 + k]) (weights
// right-aligned to width 4).  The 3 inputs before tb come from the tile, or
// at tb = 0 from global memory (xrow; zeros before token 0): the reverse
// sweep meets the chunks last to first, so no halo is carried over.
template <typename TIN>
__device__ __forceinline__ void conv_u8(const uint8_t* st, int CH, int c, int tb, int64_t t_chunk,
                                        const TIN* xrow, const float (&cw4)[4], float cb,
                                        float (&u)[8]) {
    float xv[8];
    load_raw8r<TIN>(st, CH, c, tb, xv);
    float xw[11];
    if (tb >= 8) {
        float pv[8];
        load_raw8r<TIN>(st, CH, c, tb - 8, pv);
        xw[0] = pv[5];
        xw[1] = pv[6];
        xw[2] = pv[7];
    } else {
#pragma unroll
        for (int q = 0; q < 3; ++q) {
            const int64_t t = t_chunk + tb - 3 + q;
            xw[q] = (xrow && t >= 0) ? Elem<TIN>::to_f(xrow[t]) : 0.0f;
        }
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) xw[3 + q] = xv[q];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        float a = fmaf(cw4[0], xw[q], cb);
        a = fmaf(cw4[1], xw[q + 1], a);
        a = fmaf(cw4[2], xw[q + 2], a);
        a = fmaf(cw4[3], xw[q + 3], a);
        u[q] = a * rcp(1.0f + ex2(-kLog2e * a));
    }
}

// Load the conv weights of channel d right-aligned to width 4 (leading zeros
// for a narrower kernel), its bias, and the row of x for the halo loads.
template <typename TIN>
__device__ __forceinline__ void conv_setup(const BwdParams& p, bool ch_ok, int64_t d, int64_t row,
                                           float (&cw4)[4], float& cb, const TIN*& xrow) {
#pragma unroll
    for (int q = 0; q < 4; ++q) cw4[q] = 0.0f;
    cb = 0.0f;
    xrow = nullptr;
    if (!ch_ok) return;
#pragma unroll
    for (int q = 0; q < 4; ++q) {   // static indices: the weights stay in registers
        const int kk = q - (4 - p.conv_k);
        if (kk >= 0) cw4[q] = p.conv_w[d * p.conv_k + kk];
    }
    cb = p.conv_b ? p.conv_b[d] : 0.0f;
    xrow = static_cast<const TIN*>(p.u) + row * p.L;
}

// Sum over the NT lanes of a channel (every lane gets the sum).
template <int NT, int V>
__device__ __forceinline__ void allreduce_nt(float (&v)[V]) {
#pragma unroll
    for (int o = 1; o < NT; o <<= 1)
#pragma unroll
        for (int q = 0; q < V; ++q) v[q] += __shfl_xor_sync(0xffffffffu, v[q], o);
}

// Store this lane's G partials of one token into the token's row of the
// transpose buffer.
template <int NT, int NP>
__device__ __forceinline__ void put_tr(float* row, int lane, const f2 (&v)[NP / NT / 2]) {
    using Lay = BwdLayout<NT, NP>;
#pragma unroll
    for (int j = 0; j < Lay::KC; ++j) {
        float a, bb, cc, dd;
        upk(v[2 * j], a, bb);
        upk(v[2 * j + 1], cc, dd);
        *reinterpret_cast<float4*>(row + Lay::chunk(lane, j)) = make_float4(a, bb, cc, dd);
    }
}

// Packed sequences (VARLEN): the sequence holding token t is the last s with
// cu_seqlens[s] <= t (empty sequences are skipped that way).
__device__ __forceinline__ int seq_of_token(const int* cu, int nseq, int64_t t) {
    return max(seq_lower_bound(cu, nseq, t + 1) - 1, 0);
}

// A compile-time flag passed to a generic lambda: the token loops of the
// packed sweeps are instantiated twice, with the per-token start test for
// the 8-token groups that hold a start and without it for all others.
template <bool V>
struct Flag {
    static constexpr bool value = V;
};

// The sequence starts in (0, L) met by a sweep, super-block by super-block,
// walked incrementally instead of searched for in every super-block: one
// compare per super-block, a load of cu only where a start is passed.
// bits(lo) returns bit i (0 <= i < SB) set when token lo + i is a start; lo
// must not decrease between calls (StartsUp) or increase (StartsDown).  The
// index stays in [-1, nseq] and moves at most nseq times in all, also on
// unsorted input, and every bit set lies inside the window.
struct StartsUp {
    const int* cu;
    int nseq, j;
    int64_t L, c;
    __device__ __forceinline__ void init(const int* cu_, int nseq_, int64_t L_, int64_t t) {
        cu = cu_; nseq = nseq_; L = L_;
        j = seq_lower_bound(cu, nseq, t);
        c = j < nseq ? (int64_t)cu[j] : INT64_MAX;
    }
    __device__ __forceinline__ void step() { ++j; c = j < nseq ? (int64_t)cu[j] : INT64_MAX; }
    template <int SB>
    __device__ __forceinline__ uint32_t bits(int64_t lo) {
        while (c < lo) step();
        uint32_t m = 0;
        while (c < lo + SB) {
            if (c > 0 && c < L) m |= 1u << (int)(c - lo);
            step();
        }
        return m;
    }
};
struct StartsDown {
    const int* cu;
    int nseq, j;
    int64_t L, c;
    // t: above every window of the sweep
    __device__ __forceinline__ void init(const int* cu_, int nseq_, int64_t L_, int64_t t) {
        cu = cu_; nseq = nseq_; L = L_;
        j = seq_lower_bound(cu, nseq, t) - 1;
        c = j >= 0 ? (int64_t)cu[j] : INT64_MIN;
    }
    __device__ __forceinline__ void step() { --j; c = j >= 0 ? (int64_t)cu[j] : INT64_MIN; }
    template <int SB>
    __device__ __forceinline__ uint32_t bits(int64_t lo) {
        while (c >= lo + SB) step();
        uint32_t m = 0;
        while (c >= lo) {
            if (c > 0 && c < L) m |= 1u << (int)(c - lo);
            step();
        }
        return m;
    }
};

// ===================================================== forward sweep ===
// blockDim.x = 32 * (W + 1): W compute warps and one producer warp (the last).
// VARLEN: packed sequences restart inside the row (cu_seqlens); at a start
// the ending sequence's dhL term enters dA, its psi = sum_n A dhL h_end is
// added to phi of its last token (so the reverse sweep's suffix sum restarts
// from zero there), and h, m start again from the new sequence's h0 and 0.
// SEG: the sequence is cut into p.nseg segments (grid z), each run from its
// initial state p.hin[seg] with the tangent m from zero; besides adding its
// local dA terms, a segment records the tangent at its end (p.mend) and
// GP = sum_t g_t C_t P_t (p.gp), P_t = the decay from the segment's start
// through token t (plus dhL P_L in the last segment), from which a carry
// adds the dA terms of the tangent flowing in from earlier segments.  With
// packed sequences a start inside the segment adds dhL[ending] P to GP and
// sets P to 0 (the tangent from outside ends there); psi of a sequence that
// ends with the segment's last token is added by this segment, not by the
// next one, which would race with this segment's store of that token.
template <int NP, int NT, typename TIN, typename TOUT, bool TMA_RAW, bool VARLEN = false,
          bool SEG = false, bool CONV = false>
__global__ void __launch_bounds__(32 * (BwdLayout<NT, NP>::kMaxWarps + 1), 1)
bwd_fwd_kernel(const BwdParams p, const __grid_constant__ CUtensorMap tm_u,
               const __grid_constant__ CUtensorMap tm_dr, const __grid_constant__ CUtensorMap tm_z,
               const __grid_constant__ CUtensorMap tm_dy, const __grid_constant__ CUtensorMap tm_bc) {
    using Lay = BwdLayout<NT, NP>;
    constexpr int G = Lay::G;
    constexpr int CW = Lay::CW;
    constexpr int SB = Lay::SB;
    constexpr int EB = (int)sizeof(TIN);
    constexpr int BCB = bc_tile_bytes<NP>();
    constexpr bool ACCURATE = EB == 4;
    static_assert(G % 4 == 0 && G <= 16, "states per thread");

    const int W = (int)(blockDim.x / 32) - 1;
    const int CH = W * CW;
    const int RAW = CH * kT * EB;
    const int STAGE = 4 * RAW + BCB;
    const int STAGES = p.stages;

    extern __shared__ uint8_t smem_dyn[];
    uint8_t* smem = align_smem_1024(smem_dyn);
    float* red = reinterpret_cast<float*>(smem + STAGES * STAGE);
    float* trb = red + 2 * W * NP * kT;                // after the two chunk buffers
    __shared__ __align__(8) uint64_t full_bar[kFwdMaxStages];
    __shared__ __align__(8) uint64_t empty_bar[kFwdMaxStages];
    __shared__ __align__(8) uint64_t rfull[2];     // chunk buffer written by all W warps
    __shared__ __align__(8) uint64_t rempty[2];    // chunk buffer added up by the producer

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int64_t b = blockIdx.y;
    const int64_t d0 = (int64_t)blockIdx.x * CH;
    const int64_t L = p.L;
    const int64_t nchunks = (L + kT - 1) / kT;
    const bool has_z = p.z != nullptr;
    // this CTA's chunks: its segment's (all of them without segments)
    const int seg = (int)blockIdx.z;
    const int nseg = p.nseg > 1 ? p.nseg : 1;
    const int64_t seg_chunks = p.nseg > 1 ? p.seg_chunks : nchunks;
    const int64_t k_begin = (int64_t)seg * seg_chunks;
    const int64_t k_end = min(nchunks, k_begin + seg_chunks);
    const bool last_seg = seg == nseg - 1;

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], W);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&rfull[s], W);
            mbar_init(&rempty[s], 1);
        }
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == W) {
        bwd_producer<TIN, NP, false, TMA_RAW>(smem, STAGES, STAGE, full_bar, empty_bar, rfull, rempty,
                                              red, W, p.dC, 1.0f, p, &tm_u, &tm_dr, &tm_z, &tm_dy,
                                              nullptr, &tm_bc, b, d0, has_z, lane, CH, k_begin, k_end);
        return;
    }

    const int cw = lane / NT;
    const int g = lane % NT;
    const int c = warp * CW + cw;
    const int64_t d = d0 + c;
    const bool ch_ok = d < p.D;
    const int64_t row = b * p.D + d;
    const int N = p.N;
    float* tb = trb + warp * Lay::TBUF;

    // packed sequences: per-sequence state arrays are (nseq, Bt, D, N)
    const int64_t seq_stride = p.Bt * p.D * (int64_t)N;
    const int s_first = VARLEN ? seq_of_token(p.cu_seqlens, p.nseq, 0) : 0;
    f2 Ap[G / 2], h[G / 2], m[G / 2], dAc[G / 2];
    f2 hl[ACCURATE ? G / 2 : 1];                     // fp32 inputs: low parts of the compensated state
    f2 Pd[SEG ? G / 2 : 1], GP[SEG ? G / 2 : 1];   // SEG: decay since the segment start, sum g C P
#pragma unroll
    for (int j = 0; j < G / 2; ++j) {
        const int n0 = g * G + 2 * j, n1 = n0 + 1;
        Ap[j] = pk((ch_ok && n0 < N) ? p.A[d * N + n0] : 0.0f,
                   (ch_ok && n1 < N) ? p.A[d * N + n1] : 0.0f);
        float h0v = 0.0f, h1v = 0.0f;
        if (SEG && seg > 0) {
            // the segment's initial state (padded states are zero there)
            if (ch_ok) {
                const float* hs = p.hin + ((int64_t)seg * p.Bt * p.D + row) * NP;
                h0v = hs[n0];
                h1v = hs[n1];
            }
        } else if (ch_ok && p.h0) {
            const float* hs = p.h0 + (int64_t)s_first * seq_stride;
            if (n0 < N) h0v = hs[row * N + n0];
            if (n1 < N) h1v = hs[row * N + n1];
        }
        h[j] = pk(h0v, h1v);
        if constexpr (ACCURATE) hl[j] = pk(0.0f, 0.0f);
        m[j] = pk(0.0f, 0.0f);
        dAc[j] = pk(0.0f, 0.0f);
        if constexpr (SEG) {
            Pd[j] = pk(1.0f, 1.0f);
            GP[j] = pk(0.0f, 0.0f);
        }
    }
    const float bias2 = (p.bias && ch_ok) ? p.bias[d] * kLog2e : 0.0f;
    const float Dd = (p.Dv && ch_ok) ? p.Dv[d] : 0.0f;
    const bool vec_out = ((L * (int64_t)sizeof(TOUT)) % 16) == 0;
    const bool vec_phi = (L % 4) == 0;
    // CONV: the tile's slot 0 holds the branch input x (u formed per token)
    float cw4[4], cbias;
    const TIN* xrow;
    if constexpr (CONV) conv_setup<TIN>(p, ch_ok, d, row, cw4, cbias, xrow);
    const int src_base = lane & ~(NT - 1);

    // A warp whose bounded wait expires records the error and stops working.
    bool dead = false;
    // The state at the end of every chunk: the reverse sweep re-anchors its
    // suffix sum with it.  With fp32 inputs the state before every token is
    // stored as well (the reverse sweep forms the h-dependent term of ddelta
    // from it directly).
    // the full state of pair j (hi + lo for fp32 inputs)
    auto full = [&](int j) -> f2 {
        if constexpr (ACCURATE) return add2(h[j], hl[j]);
        else return h[j];
    };
    auto store_anchor = [&](int64_t a) {
        float4* hc = reinterpret_cast<float4*>(p.hck + (row * nchunks + a) * NP + g * G);
#pragma unroll
        for (int j = 0; j < G / 4; ++j) {
            float x0, x1, x2, x3;
            upk(full(2 * j), x0, x1);
            upk(full(2 * j + 1), x2, x3);
            hc[j] = make_float4(x0, x1, x2, x3);
        }
    };
    StartsUp starts;
    if constexpr (VARLEN) starts.init(p.cu_seqlens, p.nseq, L, k_begin * kT);
    for (int64_t kl = 0; kl < k_end - k_begin; ++kl) {
        const int64_t k = k_begin + kl;        // the chunk; kl its place in this CTA's ring
        const int s = (int)(kl % STAGES);
        if (!dead) {
            const bool ok = __all_sync(
                0xffffffffu, mbar_wait(&full_bar[s], (uint32_t)((kl / STAGES) & 1), p.timeout_ns));
            if (!ok) {
                if (lane == 0) set_status(p.status, SSM_ERR_TIMEOUT);
                dead = true;
            }
        }
        const uint8_t* st = smem + s * STAGE;
        const float* bct = reinterpret_cast<const float*>(st + 4 * RAW);
        const int nvalid = (int)min((int64_t)kT, L - k * kT);
        // this chunk's cross-channel sums go to chunk buffer (kl & 1), free once
        // the producer has added up the chunk processed two before
        const int rb = (int)(kl & 1);
        if (!dead && kl >= 2) {
            const bool okr = __all_sync(0xffffffffu, mbar_wait(&rempty[rb], (uint32_t)(((kl >> 1) - 1) & 1), p.timeout_ns));
            if (!okr) {
                if (lane == 0) set_status(p.status, SSM_ERR_TIMEOUT);
                dead = true;
            }
        }
        float* redw = red + ((size_t)rb * W + warp) * NP * kT;

#pragma unroll 1
        for (int sb = 0; sb < kT / SB; ++sb) {
            if (dead || sb * SB >= nvalid) break;
            const int tbk = sb * SB + g * 8;   // this lane's 8 tokens
            float d2[8], du[8], gq[8], uo[8];
            if constexpr (CONV) {
                conv_u8<TIN>(st, CH, c, tbk, k * kT, xrow, cw4, cbias, uo);
                token_prep_u<TIN, ACCURATE>(st, CH, c, tbk, nvalid, has_z, ch_ok, bias2, uo, d2, du, gq);
            } else {
                token_prep<TIN, ACCURATE>(st, CH, c, tbk, nvalid, has_z, ch_ok, bias2, d2, du, gq);
            }
            // packed: tokens of this super-block that start a sequence, and
            // psi of an ending sequence to add to phi of its last own token
            const int64_t t_sb = k * kT + sb * SB;
            const uint32_t rmask = VARLEN ? starts.template bits<SB>(t_sb) : 0u;
            float psi_add[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) psi_add[q] = 0.0f;
            // restart before token t: close the sequence ending at t - 1, start
            // the one holding t; returns psi of the closed sequence
            auto restart = [&](int64_t t) -> float {
                const int se = seq_of_token(p.cu_seqlens, p.nseq, t - 1);
                const int sn = seq_of_token(p.cu_seqlens, p.nseq, t);
                const float* dh = (p.dhL && ch_ok) ? p.dhL + (int64_t)se * seq_stride + row * N : nullptr;
                const float* hs = (p.h0 && ch_ok) ? p.h0 + (int64_t)sn * seq_stride + row * N : nullptr;
                float psi = 0.0f;
#pragma unroll
                for (int jj = 0; jj < G / 2; ++jj) {
                    const int n0 = g * G + 2 * jj;
                    const f2 dhp = pk((dh && n0 < N) ? dh[n0] : 0.0f, (dh && n0 + 1 < N) ? dh[n0 + 1] : 0.0f);
                    dAc[jj] = fma2(dhp, m[jj], dAc[jj]);          // dhL[se] . dh/dA
                    if constexpr (SEG) {
                        GP[jj] = fma2(dhp, Pd[jj], GP[jj]);       // ... of the tangent from outside
                        Pd[jj] = pk(0.0f, 0.0f);
                    }
                    float x0, x1;
                    upk(mul2(mul2(Ap[jj], dhp), full(jj)), x0, x1);  // A dhL[se] h_end
                    psi += x0 + x1;
                    h[jj] = pk((hs && n0 < N) ? hs[n0] : 0.0f, (hs && n0 + 1 < N) ? hs[n0 + 1] : 0.0f);
                    if constexpr (ACCURATE) hl[jj] = pk(0.0f, 0.0f);
                    m[jj] = pk(0.0f, 0.0f);
                }
#pragma unroll
                for (int o = 1; o < NT; o <<= 1) psi += __shfl_xor_sync(0xffffffffu, psi, o);
                return psi;
            };

            float ys_own[8], ph_own[8];        // sums over n of this lane's tokens
#pragma unroll 1
            for (int j = 0; j < NT; ++j) {     // token group of lane j of the channel
                const int src = src_base + j;
                float D2[8], DU[8], GQ[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    D2[q] = NT == 1 ? d2[q] : __shfl_sync(0xffffffffu, d2[q], src);
                    DU[q] = NT == 1 ? du[q] : __shfl_sync(0xffffffffu, du[q], src);
                    GQ[q] = NT == 1 ? gq[q] : __shfl_sync(0xffffffffu, gq[q], src);
                }
                const int t_grp = sb * SB + j * 8;
                float yp[8], pp[8];
                auto tokens = [&](auto starts_here) {
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        if (decltype(starts_here)::value && ((rmask >> (j * 8 + q)) & 1u)) {
                            const float psi = restart(t_sb + j * 8 + q);
                            // psi belongs to the token before: an own token of
                            // this super-block, or one of the previous super-block
                            // that its owner (the channel's last lane, the thread
                            // that stored it) adds to in place
                            if (q > 0) {
                                if (g == j) psi_add[q - 1] += psi;
                            } else if (j > 0) {
                                if (g == j - 1) psi_add[7] += psi;
                            } else if (g == NT - 1 && ch_ok && !(SEG && t_sb == k_begin * kT)) {
                                atomicAdd(p.phi + row * L + t_sb - 1, psi);
                            }
                        }
                        if (ACCURATE && ch_ok && t_grp + q < nvalid) {
                            // h_{t-1} as this token's update uses it (after a restart)
                            float4* hp = reinterpret_cast<float4*>(
                                p.hprev + (row * L + k * kT + t_grp + q) * NP + g * G);
#pragma unroll
                            for (int jj = 0; jj < G / 4; ++jj) {
                                float x0, x1, x2, x3;
                                upk(full(2 * jj), x0, x1);
                                upk(full(2 * jj + 1), x2, x3);
                                hp[jj] = make_float4(x0, x1, x2, x3);
                            }
                        }
                        const float* bcrow = bct + (t_grp + q) * (2 * NP) + g * G;
                        const f2 d2p = pk(D2[q], D2[q]), dup = pk(DU[q], DU[q]), gqp = pk(GQ[q], GQ[q]);
                        f2 accy = pk(0.0f, 0.0f), accp = pk(0.0f, 0.0f);
                        f2 gh[G / 2];
#pragma unroll
                        for (int q4 = 0; q4 < G / 4; ++q4) {
                            const ulonglong2 Bq = *reinterpret_cast<const ulonglong2*>(bcrow + 4 * q4);
                            const ulonglong2 Cq = *reinterpret_cast<const ulonglong2*>(bcrow + NP + 4 * q4);
#pragma unroll
                            for (int e = 0; e < 2; ++e) {
                                const int jj = 2 * q4 + e;
                                const f2 Bj = e ? Bq.y : Bq.x;
                                const f2 Cj = e ? Cq.y : Cq.x;
                                f2 a, qv, hn;   // the decay, a_t h_{t-1} and h_t
                                if constexpr (ACCURATE) {
                                    // compensated state (see comp_update): qv and
                                    // h_t from the full state hi + lo
                                    float x0, x1, i0, i1, h0, h1, l0, l1;
                                    upk(mul2(d2p, Ap[jj]), x0, x1);
                                    upk(mul2(dup, Bj), i0, i1);
                                    upk(h[jj], h0, h1);
                                    upk(hl[jj], l0, l1);
                                    const float e0 = exp2m1_accurate(x0), e1 = exp2m1_accurate(x1);
                                    const float p0 = h0 + l0, p1 = h1 + l1;
                                    qv = pk(fmaf(e0, p0, p0), fmaf(e1, p1, p1));
                                    a = pk(1.0f + e0, 1.0f + e1);
                                    comp_update_e(e0, i0, h0, l0);
                                    comp_update_e(e1, i1, h1, l1);
                                    h[jj] = pk(h0, h1);
                                    hl[jj] = pk(l0, l1);
                                    hn = pk(h0 + l0, h1 + l1);
                                } else {
                                    a = ex2x2(mul2(d2p, Ap[jj]));
                                    qv = mul2(a, h[jj]);
                                    h[jj] = fma2(dup, Bj, qv);
                                    hn = h[jj];
                                }
                                m[jj] = fma2(a, m[jj], mul2(d2p, qv));   // dh/dA / ln2
                                accy = fma2(Cj, hn, accy);
                                accp = fma2(Ap[jj], mul2(Cj, qv), accp);
                                const f2 gC = mul2(gqp, Cj);
                                dAc[jj] = fma2(gC, m[jj], dAc[jj]);
                                if constexpr (SEG) {
                                    Pd[jj] = mul2(a, Pd[jj]);
                                    GP[jj] = fma2(gC, Pd[jj], GP[jj]);
                                }
                                gh[jj] = mul2(gqp, hn);                  // g_t h_t: dC partial
                            }
                        }
                        put_tr<NT, NP>(tb + q * Lay::TROW, lane, gh);
                        float lo, hi;
                        upk(accy, lo, hi);
                        yp[q] = lo + hi;
                        upk(accp, lo, hi);
                        pp[q] = lo + hi;
                    }
                };
                if (VARLEN && ((rmask >> (j * 8)) & 0xffu)) tokens(Flag<VARLEN>{});
                else tokens(Flag<false>{});
                __syncwarp();
                transpose_reduce<NP, CW>(tb, redw, t_grp, lane);
                allreduce_nt<NT, 8>(yp);
                allreduce_nt<NT, 8>(pp);
                if (j == g) {
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        ys_own[q] = yp[q];
                        ph_own[q] = pp[q];
                    }
                }
                __syncwarp();   // the transpose buffer is reused by the next group
            }

            if constexpr (VARLEN && SEG) {
                // a sequence ending with this segment's last token (the next
                // segment starts one): its psi goes to phi of that token here
                const int64_t tn = k_end * kT;
                if (!last_seg && k == k_end - 1 && t_sb + SB == tn && tn < L) {
                    const int lb = seq_lower_bound(p.cu_seqlens, p.nseq, tn);
                    if (lb < p.nseq && (int64_t)p.cu_seqlens[lb] == tn) {
                        const int se = seq_of_token(p.cu_seqlens, p.nseq, tn - 1);
                        const float* dh = (p.dhL && ch_ok) ? p.dhL + (int64_t)se * seq_stride + row * N : nullptr;
                        float psi = 0.0f;
#pragma unroll
                        for (int jj = 0; jj < G / 2; ++jj) {
                            const int n0 = g * G + 2 * jj;
                            const f2 dhp = pk((dh && n0 < N) ? dh[n0] : 0.0f, (dh && n0 + 1 < N) ? dh[n0 + 1] : 0.0f);
                            float x0, x1;
                            upk(mul2(mul2(Ap[jj], dhp), full(jj)), x0, x1);
                            psi += x0 + x1;
                        }
#pragma unroll
                        for (int o = 1; o < NT; o <<= 1) psi += __shfl_xor_sync(0xffffffffu, psi, o);
                        if (g == NT - 1) psi_add[7] += psi;
                    }
                }
            }
            // this lane's tokens: dz and phi
            float uv[8], gy[8], zv[8];
            if constexpr (CONV) {
#pragma unroll
                for (int q = 0; q < 8; ++q) uv[q] = uo[q];
            } else {
                load_raw8r<TIN>(st, CH, c, tbk, uv);
            }
            load_raw8r<TIN>(st + 3 * RAW, CH, c, tbk, gy);
            if (has_z) load_raw8r<TIN>(st + 2 * RAW, CH, c, tbk, zv);
            float dzv[8], phv[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                if (has_z) {
                    const float sz = rcp(1.0f + ex2(-kLog2e * zv[q]));
                    const float pre = fmaf(Dd, uv[q], ys_own[q]);
                    dzv[q] = gy[q] * pre * sz * fmaf(zv[q], 1.0f - sz, 1.0f);
                } else {
                    dzv[q] = 0.0f;
                }
                phv[q] = fmaf(gq[q], ph_own[q], psi_add[q]);
            }
            if (ch_ok) {
                const int64_t off = row * L + k * kT + tbk;
                if (p.dz) store_out8<TOUT>(p.dz, off, dzv, nvalid - tbk, vec_out);
                store_out8<float>(p.phi, off, phv, nvalid - tbk, vec_phi);
            }
        }
        if (!dead && ch_ok && k + 1 < nchunks) store_anchor(k);
        __syncwarp();
        if (lane == 0 && !dead) {
            mbar_arrive(&empty_bar[s]);
            mbar_arrive(&rfull[rb]);
        }
    }

    if (ch_ok && !dead) {
        // the last sequence's final-state gradient (packed: the one holding
        // token L-1); with segments only the last segment holds it
        const int s_last = VARLEN ? seq_of_token(p.cu_seqlens, p.nseq, L - 1) : 0;
        const float* dhl = (p.dhL && last_seg) ? p.dhL + (int64_t)s_last * seq_stride + row * N : nullptr;
        const int64_t segrow = ((int64_t)seg * p.Bt * p.D + row) * NP;
#pragma unroll
        for (int j = 0; j < G / 2; ++j) {
            const int n0 = g * G + 2 * j;
            float hl0, hl1, m0, m1, a0, a1;
            upk(full(j), hl0, hl1);
            upk(m[j], m0, m1);
            upk(dAc[j], a0, a1);
            if (last_seg) {
                p.hfin[row * NP + n0] = hl0;
                p.hfin[row * NP + n0 + 1] = hl1;
            }
            const float g0 = (dhl && n0 < N) ? dhl[n0] : 0.0f;
            const float g1 = (dhl && n0 + 1 < N) ? dhl[n0 + 1] : 0.0f;
            if (n0 < N) atomicAdd(p.dA + d * N + n0, kLn2 * fmaf(g0, m0, a0));
            if (n0 + 1 < N) atomicAdd(p.dA + d * N + n0 + 1, kLn2 * fmaf(g1, m1, a1));
            if constexpr (SEG) {
                // the carry's inputs: the tangent at this segment's end, and
                // sum g C P (+ dhL P_L) against the tangent flowing in
                float p0, p1, q0, q1;
                upk(Pd[j], p0, p1);
                upk(GP[j], q0, q1);
                p.mend[segrow + n0] = m0;
                p.mend[segrow + n0 + 1] = m1;
                p.gp[segrow + n0] = fmaf(g0, p0, q0);
                p.gp[segrow + n0 + 1] = fmaf(g1, p1, q1);
            }
        }
    }
}

// ===================================================== reverse sweep ===
// VARLEN: at the last token of a packed sequence the adjoint carried in from
// the next token is replaced by that sequence's dhL (after the next
// sequence's dh0 = a lambda has been written), and the suffix sum restarts
// from zero there (the ending sequence's psi is already in phi of that token).
// Segments (p.nseg > 1, grid z): a segment other than the last starts from
// the adjoint flowing in at its right end, p.lam_in[seg] = a_{t1} lambda_{t1}
// (t1 = the next segment's first token; the decay "after" the segment's
// last token is then 1), and its suffix sum from sum_n A lam_in h_{t1-1},
// with h_{t1-1} the forward sweep's state at the end of its last chunk.
template <int NP, int NT, typename TIN, typename TOUT, bool TMA_RAW, bool VARLEN = false,
          bool CONV = false>
__global__ void __launch_bounds__(32 * (BwdLayout<NT, NP>::kMaxWarps + 1), 1)
bwd_rev_kernel(const BwdParams p, const __grid_constant__ CUtensorMap tm_u,
               const __grid_constant__ CUtensorMap tm_dr, const __grid_constant__ CUtensorMap tm_z,
               const __grid_constant__ CUtensorMap tm_dy, const __grid_constant__ CUtensorMap tm_phi,
               const __grid_constant__ CUtensorMap tm_bc) {
    using Lay = BwdLayout<NT, NP>;
    constexpr int G = Lay::G;
    constexpr int CW = Lay::CW;
    constexpr int SB = Lay::SB;
    constexpr int EB = (int)sizeof(TIN);
    constexpr int BCB = bc_tile_bytes<NP>();
    constexpr bool ACCURATE = EB == 4;
    static_assert(G % 4 == 0 && G <= 16, "states per thread");

    const int W = (int)(blockDim.x / 32) - 1;
    const int CH = W * CW;
    const int RAW = CH * kT * EB;
    const int RAWF = CH * kT * 4;
    const int STAGE = 4 * RAW + RAWF + BCB;
    const int STAGES = p.stages;

    extern __shared__ uint8_t smem_dyn[];
    uint8_t* smem = align_smem_1024(smem_dyn);
    float* red = reinterpret_cast<float*>(smem + STAGES * STAGE);
    float* trb = red + 2 * W * NP * kT;                // after the two chunk buffers
    __shared__ __align__(8) uint64_t full_bar[kFwdMaxStages];
    __shared__ __align__(8) uint64_t empty_bar[kFwdMaxStages];
    __shared__ __align__(8) uint64_t rfull[2];     // chunk buffer written by all W warps
    __shared__ __align__(8) uint64_t rempty[2];    // chunk buffer added up by the producer

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int64_t b = blockIdx.y;
    const int64_t d0 = (int64_t)blockIdx.x * CH;
    const int64_t L = p.L;
    const int64_t nchunks = (L + kT - 1) / kT;
    const bool has_z = p.z != nullptr;
    // this CTA's chunks: its segment's (all of them without segments)
    const int seg = (int)blockIdx.z;
    const int nseg = p.nseg > 1 ? p.nseg : 1;
    const int64_t seg_chunks = p.nseg > 1 ? p.seg_chunks : nchunks;
    const int64_t k_begin = (int64_t)seg * seg_chunks;
    const int64_t k_end = min(nchunks, k_begin + seg_chunks);
    const bool last_seg = seg == nseg - 1;

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], W);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&rfull[s], W);
            mbar_init(&rempty[s], 1);
        }
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == W) {
        bwd_producer<TIN, NP, true, TMA_RAW>(smem, STAGES, STAGE, full_bar, empty_bar, rfull, rempty,
                                              red, W, p.dB, kLn2, p, &tm_u, &tm_dr, &tm_z, &tm_dy,
                                              &tm_phi, &tm_bc, b, d0, has_z, lane, CH, k_begin, k_end);
        return;
    }

    const int cw = lane / NT;
    const int g = lane % NT;
    const int c = warp * CW + cw;
    const int64_t d = d0 + c;
    const bool ch_ok = d < p.D;
    const int64_t row = b * p.D + d;
    const int N = p.N;
    float* tb = trb + warp * Lay::TBUF;

    // lambda starts at dhL, the decay "after the last token" is 1, and
    // psi = sum_n A dhL h_L starts the suffix sum (packed: dhL of the
    // sequence holding token L-1)
    const int64_t seq_stride = p.Bt * p.D * (int64_t)N;
    const int s_last = VARLEN ? seq_of_token(p.cu_seqlens, p.nseq, L - 1) : 0;
    const float* dhl_last = p.dhL ? p.dhL + (int64_t)s_last * seq_stride : nullptr;
    // the state after this CTA's last token: the final state, or the forward
    // sweep's state at the end of the segment's last chunk
    const float* hend = last_seg ? p.hfin + row * NP : p.hck + (row * nchunks + (k_end - 1)) * NP;
    const float* lin = last_seg ? nullptr : p.lam_in + ((int64_t)seg * p.Bt * p.D + row) * NP;
    f2 Ap[G / 2], lam[G / 2], anext[G / 2];
    float psi = 0.0f;
#pragma unroll
    for (int j = 0; j < G / 2; ++j) {
        const int n0 = g * G + 2 * j, n1 = n0 + 1;
        const float a0 = (ch_ok && n0 < N) ? p.A[d * N + n0] : 0.0f;
        const float a1 = (ch_ok && n1 < N) ? p.A[d * N + n1] : 0.0f;
        Ap[j] = pk(a0, a1);
        float l0 = 0.0f, l1 = 0.0f;
        if (ch_ok && lin) {
            l0 = lin[n0];
            l1 = lin[n1];
        } else if (ch_ok && dhl_last) {
            if (n0 < N) l0 = dhl_last[row * N + n0];
            if (n1 < N) l1 = dhl_last[row * N + n1];
        }
        lam[j] = pk(l0, l1);
        anext[j] = pk(1.0f, 1.0f);
        if (ch_ok) psi += a0 * l0 * hend[n0] + a1 * l1 * hend[n1];
    }
#pragma unroll
    for (int o = 1; o < NT; o <<= 1) psi += __shfl_xor_sync(0xffffffffu, psi, o);
    float carry = psi;                 // psi + sum of (phi - rho) over the later tokens
    const float bias2 = (p.bias && ch_ok) ? p.bias[d] * kLog2e : 0.0f;
    const float Dd = (p.Dv && ch_ok) ? p.Dv[d] : 0.0f;
    const bool vec_out = ((L * (int64_t)sizeof(TOUT)) % 16) == 0;
    const int src_base = lane & ~(NT - 1);
    float dD_acc = 0.0f, db_acc = 0.0f;
    float cw4[4], cbias;   // CONV: see the forward sweep
    const TIN* xrow;
    if constexpr (CONV) conv_setup<TIN>(p, ch_ok, d, row, cw4, cbias, xrow);
    bool dead = false;   // see the forward sweep
    // Re-anchor: the suffix sum equals sum_n A a_t lambda_t h_{t-1} at the
    // first token t of a chunk, with h_{t-1} the state the forward sweep
    // stored at the end of the chunk before.  Rounding in the running sum is
    // thereby confined to one chunk instead of random-walking over the
    // sequence.
    auto reanchor = [&](int64_t a) -> float {
        float part = 0.0f;
        if (ch_ok && !dead) {
            const float4* hc = reinterpret_cast<const float4*>(p.hck + (row * nchunks + a) * NP + g * G);
#pragma unroll
            for (int j = 0; j < G / 4; ++j) {
                const float4 hv = hc[j];
                float l0, l1, l2, l3;
                upk(mul2(mul2(Ap[2 * j], anext[2 * j]), lam[2 * j]), l0, l1);
                upk(mul2(mul2(Ap[2 * j + 1], anext[2 * j + 1]), lam[2 * j + 1]), l2, l3);
                part = fmaf(l0, hv.x, part);
                part = fmaf(l1, hv.y, part);
                part = fmaf(l2, hv.z, part);
                part = fmaf(l3, hv.w, part);
            }
        }
#pragma unroll
        for (int o = 1; o < NT; o <<= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
        return part;
    };

    StartsDown starts;
    if constexpr (VARLEN) starts.init(p.cu_seqlens, p.nseq, L, k_end * kT + 1);
    for (int64_t i = 0; i < k_end - k_begin; ++i) {
        const int64_t k = k_end - 1 - i;       // the chunk; i its place in this CTA's ring
        const int s = (int)(i % STAGES);
        if (!dead) {
            const bool ok = __all_sync(
                0xffffffffu, mbar_wait(&full_bar[s], (uint32_t)((i / STAGES) & 1), p.timeout_ns));
            if (!ok) {
                if (lane == 0) set_status(p.status, SSM_ERR_TIMEOUT);
                dead = true;
            }
        }
        const uint8_t* st = smem + s * STAGE;
        const uint8_t* phit = st + 4 * RAW;
        const float* bct = reinterpret_cast<const float*>(st + 4 * RAW + RAWF);
        const int nvalid = (int)min((int64_t)kT, L - k * kT);
        // this chunk's cross-channel sums go to chunk buffer (i & 1), free once
        // the producer has added up the chunk processed two before
        const int rb = (int)(i & 1);
        if (!dead && i >= 2) {
            const bool okr = __all_sync(0xffffffffu, mbar_wait(&rempty[rb], (uint32_t)(((i >> 1) - 1) & 1), p.timeout_ns));
            if (!okr) {
                if (lane == 0) set_status(p.status, SSM_ERR_TIMEOUT);
                dead = true;
            }
        }
        float* redw = red + ((size_t)rb * W + warp) * NP * kT;

#pragma unroll 1
        for (int sb = kT / SB - 1; sb >= 0; --sb) {
            if (dead) break;
            if (sb * SB >= nvalid) continue;
            const int tbk = sb * SB + g * 8;
            float d2[8], du[8], gq[8], uo[8];
            if constexpr (CONV) {
                conv_u8<TIN>(st, CH, c, tbk, k * kT, xrow, cw4, cbias, uo);
                token_prep_u<TIN, ACCURATE>(st, CH, c, tbk, nvalid, has_z, ch_ok, bias2, uo, d2, du, gq);
            } else {
                token_prep<TIN, ACCURATE>(st, CH, c, tbk, nvalid, has_z, ch_ok, bias2, d2, du, gq);
            }
            // packed: tokens of this super-block that end a sequence
            const int64_t t_sb = k * kT + sb * SB;
            const uint32_t emask = VARLEN ? starts.template bits<SB>(t_sb + 1) : 0u;

            float sb_own[8], sab_own[8];       // sum_n lambda B', sum_n A a_{t+1} lambda_{t+1} B'
            float qd_own[8];                   // fp32 inputs: Q of the own tokens, formed directly
#pragma unroll 1
            for (int j = NT - 1; j >= 0; --j) {
                const int src = src_base + j;
                float D2[8], DU[8], GQ[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    D2[q] = NT == 1 ? d2[q] : __shfl_sync(0xffffffffu, d2[q], src);
                    DU[q] = NT == 1 ? du[q] : __shfl_sync(0xffffffffu, du[q], src);
                    GQ[q] = NT == 1 ? gq[q] : __shfl_sync(0xffffffffu, gq[q], src);
                }
                const int t_grp = sb * SB + j * 8;
                float bp[8], abp[8], qd[8];
                auto tokens = [&](auto ends_here) {
#pragma unroll
                    for (int q = 7; q >= 0; --q) {
                        if (decltype(ends_here)::value && ((emask >> (j * 8 + q)) & 1u)) {
                            // token t ends sequence se, t + 1 starts sn: write
                            // dh0[sn] = a_{t+1} lambda_{t+1}, then carry dhL[se]
                            const int64_t t = t_sb + j * 8 + q;
                            const int sn = seq_of_token(p.cu_seqlens, p.nseq, t + 1);
                            const int se = seq_of_token(p.cu_seqlens, p.nseq, t);
                            const float* dh = (p.dhL && ch_ok) ? p.dhL + (int64_t)se * seq_stride + row * N : nullptr;
                            float* d0p = (p.dh0 && ch_ok) ? p.dh0 + (int64_t)sn * seq_stride + row * N : nullptr;
#pragma unroll
                            for (int jj = 0; jj < G / 2; ++jj) {
                                const int n0 = g * G + 2 * jj;
                                if (d0p) {
                                    float v0, v1;
                                    upk(mul2(anext[jj], lam[jj]), v0, v1);
                                    if (n0 < N) d0p[n0] = v0;
                                    if (n0 + 1 < N) d0p[n0 + 1] = v1;
                                }
                                lam[jj] = pk((dh && n0 < N) ? dh[n0] : 0.0f, (dh && n0 + 1 < N) ? dh[n0 + 1] : 0.0f);
                                anext[jj] = pk(1.0f, 1.0f);
                            }
                        }
                        const float* bcrow = bct + (t_grp + q) * (2 * NP) + g * G;
                        const f2 d2p = pk(D2[q], D2[q]), dup = pk(DU[q], DU[q]), gqp = pk(GQ[q], GQ[q]);
                        f2 accb = pk(0.0f, 0.0f), accab = pk(0.0f, 0.0f);
                        f2 ld[G / 2];
#pragma unroll
                        for (int q4 = 0; q4 < G / 4; ++q4) {
                            const ulonglong2 Bq = *reinterpret_cast<const ulonglong2*>(bcrow + 4 * q4);
                            const ulonglong2 Cq = *reinterpret_cast<const ulonglong2*>(bcrow + NP + 4 * q4);
#pragma unroll
                            for (int e = 0; e < 2; ++e) {
                                const int jj = 2 * q4 + e;
                                const f2 Bj = e ? Bq.y : Bq.x;
                                const f2 Cj = e ? Cq.y : Cq.x;
                                const f2 al = mul2(anext[jj], lam[jj]);   // a_{t+1} lambda_{t+1}
                                lam[jj] = fma2(gqp, Cj, al);
                                accb = fma2(lam[jj], Bj, accb);
                                accab = fma2(Ap[jj], mul2(al, Bj), accab);
                                ld[jj] = mul2(lam[jj], dup);              // dB partial / ln2
                                const f2 arg = mul2(d2p, Ap[jj]);
                                anext[jj] = ACCURATE ? exp2_accurate_x2(arg) : ex2x2(arg);
                            }
                        }
                        put_tr<NT, NP>(tb + q * Lay::TROW, lane, ld);
                        float lo, hi;
                        upk(accb, lo, hi);
                        bp[q] = lo + hi;
                        upk(accab, lo, hi);
                        abp[q] = lo + hi;
                        if constexpr (ACCURATE) {
                            // Q_t = sum_n A a_t lambda_t h_{t-1} from the stored state
                            float qacc = 0.0f;
                            if (ch_ok && t_grp + q < nvalid) {
                                const float4* hp = reinterpret_cast<const float4*>(
                                    p.hprev + (row * L + k * kT + t_grp + q) * NP + g * G);
#pragma unroll
                                for (int jj = 0; jj < G / 4; ++jj) {
                                    const float4 hv = hp[jj];
                                    float l0, l1, l2, l3;
                                    upk(mul2(mul2(Ap[2 * jj], anext[2 * jj]), lam[2 * jj]), l0, l1);
                                    upk(mul2(mul2(Ap[2 * jj + 1], anext[2 * jj + 1]), lam[2 * jj + 1]), l2, l3);
                                    qacc = fmaf(l0, hv.x, qacc);
                                    qacc = fmaf(l1, hv.y, qacc);
                                    qacc = fmaf(l2, hv.z, qacc);
                                    qacc = fmaf(l3, hv.w, qacc);
                                }
                            }
                            qd[q] = qacc;
                        }
                    }
                };
                if (VARLEN && ((emask >> (j * 8)) & 0xffu)) tokens(Flag<VARLEN>{});
                else tokens(Flag<false>{});
                __syncwarp();
                transpose_reduce<NP, CW>(tb, redw, t_grp, lane);
                allreduce_nt<NT, 8>(bp);
                allreduce_nt<NT, 8>(abp);
                if (ACCURATE) allreduce_nt<NT, 8>(qd);
                if (j == g) {
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        sb_own[q] = bp[q];
                        sab_own[q] = abp[q];
                        if (ACCURATE) qd_own[q] = qd[q];
                    }
                }
                __syncwarp();   // the transpose buffer is reused by the next group
            }

            // suffix sums of w = phi - rho over this lane's tokens, then over
            // the later lanes of the channel, then the later super-blocks
            const int RAWB = RAW;
            float phv[8], uv[8], dv[8];
            load_raw8r<float>(phit, CH, c, tbk, phv);
            if constexpr (CONV) {
#pragma unroll
                for (int q = 0; q < 8; ++q) uv[q] = uo[q];
            } else {
                load_raw8r<TIN>(st, CH, c, tbk, uv);
            }
            load_raw8r<TIN>(st + RAWB, CH, c, tbk, dv);
            float suf[8];
            float run = 0.0f;
            // packed: the suffix restarts at zero at a sequence's last token;
            // `top` = the highest own token at which it does (-1: none), above
            // which the tokens still take the carry from later tokens
            const uint32_t eown = VARLEN ? (emask >> (g * 8)) & 0xffu : 0u;
            const int top = VARLEN ? 31 - __clz((int)eown) : -1;
#pragma unroll
            for (int q = 7; q >= 0; --q) {
                if (VARLEN && ((eown >> q) & 1u)) run = 0.0f;
                run += phv[q] - du[q] * sab_own[q];
                suf[q] = run;
            }
            float qv[8];   // the suffix sum Q at each own token
            if (VARLEN) {
                // carry into each lane's tokens, lane NT-1 first: a lane passes
                // on its sum, plus what came in if it has no restart
                float R = carry, rin = carry;
#pragma unroll
                for (int gg = NT - 1; gg >= 0; --gg) {
                    if (g == gg) rin = R;
                    const float cand = run + (top < 0 ? R : 0.0f);
                    R = __shfl_sync(0xffffffffu, cand, src_base + gg);
                }
#pragma unroll
                for (int q = 0; q < 8; ++q) qv[q] = q > top ? rin + suf[q] : suf[q];
                carry = R;
            } else {
                float incl = run;
#pragma unroll
                for (int o = 1; o < NT; o <<= 1) {
                    const float v = __shfl_down_sync(0xffffffffu, incl, o, NT);
                    if (g + o < NT) incl += v;
                }
                const float excl = incl - run;
                const float total = __shfl_sync(0xffffffffu, incl, src_base);
#pragma unroll
                for (int q = 0; q < 8; ++q) qv[q] = carry + excl + suf[q];
                carry += total;
            }
            float duv[8], ddv[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float dd = (ACCURATE ? qd_own[q] : qv[q]) + uv[q] * sb_own[q] * kLog2e;
                const float sx = rcp(1.0f + ex2(-fmaf(dv[q], kLog2e, bias2)));  // d softplus / dx
                ddv[q] = dd * sx;
                duv[q] = fmaf(gq[q], Dd, d2[q] * sb_own[q]);
                if (tbk + q < nvalid) {
                    dD_acc = fmaf(gq[q], uv[q], dD_acc);
                    db_acc += ddv[q];
                }
            }
            if (ch_ok) {
                const int64_t off = row * L + k * kT + tbk;
                // CONV: du is an intermediate (the prologue's reverse mode
                // reads it), kept in fp32 so that dx is rounded once
                if constexpr (CONV) store_out8<float>(p.du, off, duv, nvalid - tbk, (L % 4) == 0);
                else store_out8<TOUT>(p.du, off, duv, nvalid - tbk, vec_out);
                store_out8<TOUT>(p.ddr, off, ddv, nvalid - tbk, vec_out);
            }
        }
        if (k > 0) carry = reanchor(k - 1);
        __syncwarp();
        if (lane == 0 && !dead) {
            mbar_arrive(&empty_bar[s]);
            mbar_arrive(&rfull[rb]);
        }
    }

#pragma unroll
    for (int o = 1; o < NT; o <<= 1) {
        dD_acc += __shfl_xor_sync(0xffffffffu, dD_acc, o);
        db_acc += __shfl_xor_sync(0xffffffffu, db_acc, o);
    }
    if (ch_ok && !dead) {
        if (g == 0) {
            if (p.dD) atomicAdd(p.dD + d, dD_acc);
            if (p.dbias) atomicAdd(p.dbias + d, db_acc);
        }
        if (p.dh0 && seg == 0) {
            // packed: dh0 of the sequence holding token 0
            float* d0p = p.dh0 + (VARLEN ? (int64_t)seq_of_token(p.cu_seqlens, p.nseq, 0) * seq_stride : 0);
#pragma unroll
            for (int j = 0; j < G / 2; ++j) {
                const int n0 = g * G + 2 * j;
                float v0, v1;
                upk(mul2(anext[j], lam[j]), v0, v1);
                if (n0 < N) d0p[row * N + n0] = v0;
                if (n0 + 1 < N) d0p[row * N + n0 + 1] = v1;
            }
        }
    }
}


// ============================================ adjoint summary (segments) ===
// For segment seg = blockIdx.z + 1 (segments 1 .. nseg-1): the reverse
// recurrence lambda_t = g_t C_t + a_{t+1} lambda_{t+1} from zero at the
// segment's right end down to its first token t0, giving
// p.lam_loc[seg] = a_{t0} lambda_{t0} (what the segment passes to its left
// neighbour from a zero start; the last segment starts from the final-state
// gradient dhL instead), and p.sumd[seg], the segment's sum of delta/ln2
// (its total decay is 2^(A sumd)).  A carry over the segments, from
// the last one down, then gives every segment the adjoint flowing in at its
// right end.  Same tiles and ring as the reverse sweep, without the per-token
// tile; nothing but the recurrence per state.  With a head search (p.kstop)
// the summary starts at the chunk where the decay from the segment's start
// has fallen below fp32 resolution for every channel of the tile; the sum
// of delta2 is then the search's (saturation marks) unless the whole segment
// ran.  VARLEN: at the last token of a packed sequence the adjoint restarts
// from that sequence's dhL (as in the reverse sweep); a segment in which a
// sequence ends passes on nothing from its right (the search marks it).
template <int NP, int NT, typename TIN, bool TMA_RAW, bool VARLEN = false>
__global__ void __launch_bounds__(32 * (BwdLayout<NT, NP>::kMaxWarps + 1), 1)
bwd_lam_kernel(const BwdParams p, const __grid_constant__ CUtensorMap tm_u,
               const __grid_constant__ CUtensorMap tm_dr, const __grid_constant__ CUtensorMap tm_z,
               const __grid_constant__ CUtensorMap tm_dy, const __grid_constant__ CUtensorMap tm_bc) {
    using Lay = BwdLayout<NT, NP>;
    constexpr int G = Lay::G;
    constexpr int CW = Lay::CW;
    constexpr int SB = Lay::SB;
    constexpr int EB = (int)sizeof(TIN);
    constexpr int BCB = bc_tile_bytes<NP>();
    constexpr bool ACCURATE = EB == 4;
    static_assert(G % 4 == 0 && G <= 16, "states per thread");

    const int W = (int)(blockDim.x / 32) - 1;
    const int CH = W * CW;
    const int RAW = CH * kT * EB;
    const int STAGE = 4 * RAW + BCB;
    const int STAGES = p.stages;

    extern __shared__ uint8_t smem_dyn[];
    uint8_t* smem = align_smem_1024(smem_dyn);
    __shared__ __align__(8) uint64_t full_bar[kFwdMaxStages];
    __shared__ __align__(8) uint64_t empty_bar[kFwdMaxStages];

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int64_t b = blockIdx.y;
    const int64_t d0 = (int64_t)blockIdx.x * CH;
    const int64_t L = p.L;
    const int64_t nchunks = (L + kT - 1) / kT;
    const bool has_z = p.z != nullptr;
    const int seg = (int)blockIdx.z + 1;
    const int64_t k_begin = (int64_t)seg * p.seg_chunks;
    const int64_t k_seg_end = min(nchunks, k_begin + p.seg_chunks);
    const int64_t k_end = p.kstop ? min(k_seg_end, (int64_t)p.kstop[((int64_t)seg * p.Bt + b) * gridDim.x + blockIdx.x])
                                  : k_seg_end;

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], W);
        }
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == W) {
        bwd_producer<TIN, NP, true, TMA_RAW, false>(smem, STAGES, STAGE, full_bar, empty_bar, nullptr,
                                                     nullptr, nullptr, W, nullptr, 0.0f, p, &tm_u,
                                                     &tm_dr, &tm_z, &tm_dy, nullptr, &tm_bc, b, d0,
                                                     has_z, lane, CH, k_begin, k_end);
        return;
    }

    const int cw = lane / NT;
    const int g = lane % NT;
    const int c = warp * CW + cw;
    const int64_t d = d0 + c;
    const bool ch_ok = d < p.D;
    const int64_t row = b * p.D + d;
    const int N = p.N;
    const int64_t seq_stride = p.Bt * p.D * (int64_t)N;
    // the last segment: dhL of the sequence holding token L-1
    const bool last_seg = seg == p.nseg - 1;
    const int s_last = (VARLEN && last_seg) ? seq_of_token(p.cu_seqlens, p.nseq, L - 1) : 0;
    const float* dhl = (last_seg && p.dhL && ch_ok) ? p.dhL + (int64_t)s_last * seq_stride + row * N : nullptr;
    f2 Ap[G / 2], lam[G / 2], anext[G / 2];
#pragma unroll
    for (int j = 0; j < G / 2; ++j) {
        const int n0 = g * G + 2 * j, n1 = n0 + 1;
        Ap[j] = pk((ch_ok && n0 < N) ? p.A[d * N + n0] : 0.0f,
                   (ch_ok && n1 < N) ? p.A[d * N + n1] : 0.0f);
        lam[j] = pk((dhl && n0 < N) ? dhl[n0] : 0.0f, (dhl && n1 < N) ? dhl[n1] : 0.0f);
        anext[j] = pk(1.0f, 1.0f);
    }
    const float bias2 = (p.bias && ch_ok) ? p.bias[d] * kLog2e : 0.0f;
    const int src_base = lane & ~(NT - 1);
    double sum_d2 = 0.0;   // this lane's own tokens
    bool dead = false;
    // packed: a sequence ends inside the segment (a start in (s0, s1])
    bool cut = false;
    if constexpr (VARLEN) {
        const int64_t s0 = k_begin * kT, s1 = min(L, k_seg_end * kT);
        const int lb = seq_lower_bound(p.cu_seqlens, p.nseq, s0 + 1);
        cut = lb < p.nseq && (int64_t)p.cu_seqlens[lb] <= s1 && (int64_t)p.cu_seqlens[lb] < L;
    }

    StartsDown starts;
    if constexpr (VARLEN) starts.init(p.cu_seqlens, p.nseq, L, k_end * kT + 1);
    for (int64_t i = 0; i < k_end - k_begin; ++i) {
        const int64_t k = k_end - 1 - i;
        const int s = (int)(i % STAGES);
        if (!dead) {
            const bool ok = __all_sync(
                0xffffffffu, mbar_wait(&full_bar[s], (uint32_t)((i / STAGES) & 1), p.timeout_ns));
            if (!ok) {
                if (lane == 0) set_status(p.status, SSM_ERR_TIMEOUT);
                dead = true;
            }
        }
        const uint8_t* st = smem + s * STAGE;
        const float* bct = reinterpret_cast<const float*>(st + 4 * RAW);
        const int nvalid = (int)min((int64_t)kT, L - k * kT);
#pragma unroll 1
        for (int sb = kT / SB - 1; sb >= 0; --sb) {
            if (dead) break;
            if (sb * SB >= nvalid) continue;
            const int tbk = sb * SB + g * 8;
            float d2[8], du[8], gq[8];
            token_prep<TIN, ACCURATE>(st, CH, c, tbk, nvalid, has_z, ch_ok, bias2, d2, du, gq);
            float s8 = 0.0f;
#pragma unroll
            for (int q = 0; q < 8; ++q) s8 += d2[q];
            sum_d2 += (double)s8;
            const int64_t t_sb = k * kT + sb * SB;
            const uint32_t emask = VARLEN ? starts.template bits<SB>(t_sb + 1) : 0u;
#pragma unroll 1
            for (int j = NT - 1; j >= 0; --j) {
                const int src = src_base + j;
                float D2[8], GQ[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    D2[q] = NT == 1 ? d2[q] : __shfl_sync(0xffffffffu, d2[q], src);
                    GQ[q] = NT == 1 ? gq[q] : __shfl_sync(0xffffffffu, gq[q], src);
                }
                const int t_grp = sb * SB + j * 8;
                auto tokens = [&](auto ends_here) {
#pragma unroll
                    for (int q = 7; q >= 0; --q) {
                        if (decltype(ends_here)::value && ((emask >> (j * 8 + q)) & 1u)) {
                            // token t ends sequence se: the adjoint restarts from dhL[se]
                            const int se = seq_of_token(p.cu_seqlens, p.nseq, t_sb + j * 8 + q);
                            const float* dh = (p.dhL && ch_ok) ? p.dhL + (int64_t)se * seq_stride + row * N : nullptr;
#pragma unroll
                            for (int jj = 0; jj < G / 2; ++jj) {
                                const int n0 = g * G + 2 * jj;
                                lam[jj] = pk((dh && n0 < N) ? dh[n0] : 0.0f, (dh && n0 + 1 < N) ? dh[n0 + 1] : 0.0f);
                                anext[jj] = pk(1.0f, 1.0f);
                            }
                        }
                        const float* crow = bct + (t_grp + q) * (2 * NP) + NP + g * G;
                        const f2 d2p = pk(D2[q], D2[q]), gqp = pk(GQ[q], GQ[q]);
#pragma unroll
                        for (int q4 = 0; q4 < G / 4; ++q4) {
                            const ulonglong2 Cq = *reinterpret_cast<const ulonglong2*>(crow + 4 * q4);
#pragma unroll
                            for (int e = 0; e < 2; ++e) {
                                const int jj = 2 * q4 + e;
                                const f2 Cj = e ? Cq.y : Cq.x;
                                lam[jj] = fma2(gqp, Cj, mul2(anext[jj], lam[jj]));
                                const f2 arg = mul2(d2p, Ap[jj]);
                                anext[jj] = ACCURATE ? exp2_accurate_x2(arg) : ex2x2(arg);
                            }
                        }
                    }
                };
                if (VARLEN && ((emask >> (j * 8)) & 0xffu)) tokens(Flag<VARLEN>{});
                else tokens(Flag<false>{});
            }
        }
        __syncwarp();
        if (lane == 0 && !dead) mbar_arrive(&empty_bar[s]);
    }

#pragma unroll
    for (int o = 1; o < NT; o <<= 1) sum_d2 += __shfl_xor_sync(0xffffffffu, sum_d2, o);
    if (ch_ok && !dead) {
        const int64_t segrow = (int64_t)seg * p.Bt * p.D + row;
#pragma unroll
        for (int j = 0; j < G / 2; ++j) {
            const int n0 = g * G + 2 * j;
            float v0, v1;
            upk(mul2(anext[j], lam[j]), v0, v1);
            p.lam_loc[segrow * NP + n0] = v0;
            p.lam_loc[segrow * NP + n0 + 1] = v1;
        }
        if (g == 0 && k_end == k_seg_end && !cut) p.sumd[segrow] = (float)sum_d2;
    }
}

}  // namespace ssm
