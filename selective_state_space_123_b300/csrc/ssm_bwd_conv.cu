// ssm_bwd_conv.cu -- the backward fed by the conv prologue: both sweeps form
// u from the branch input x per token (padded state size 16, 16-byte token
// rows, whole rows), and the prologue's own reverse mode, conv_bwd_kernel:
// dx, dconv_w, dconv_b from the sweeps' du.
#include "ssm_bwd_launch.cuh"

namespace ssm {

namespace {

// the sweeps write fp32 gradients (the prologue's pass rounds them once)
template <int NT>
cudaError_t conv_nt(int tin, const BwdParams& p, const BwdMaps& m, const BwdLaunch& lc,
                    cudaStream_t st) {
    return tin == SSM_BF16 ? launch_bwd_one<16, NT, __nv_bfloat16, float, true, false, true>(p, m, lc, st)
                           : launch_bwd_one<16, NT, float, float, true, false, true>(p, m, lc, st);
}

// The prologue's reverse mode over one tile of kConvTile tokens of one
// (batch, channel) row, 8 consecutive tokens per thread (16-byte loads and
// stores where the rows allow).  With pre[t] = conv_b + sum_k w[k] x[t-(K-1)+k] (x before token 0
// is 0) and u = silu(pre):
//   dpre[t] = du[t] silu'(pre[t]),  silu'(p) = s (1 + p (1 - s)), s = 1 / (1 + e^-p)
//   dx[t] = sum_k w[k] dpre[t+(K-1)-k] (terms past the end absent)
//   dconv_w[d,k] += sum_t dpre[t] x[t-(K-1)+k],  dconv_b[d] += sum_t dpre[t]
// x of the tile and the 3 tokens on each side, and dpre of the tile and the
// 3 tokens after it, go through shared memory; the weight and bias sums are
// reduced over the block and added once per tile.  The sweeps' gradients are
// fp32; with bf16 outputs the same pass also writes ddelta_raw and dz in the
// output type (cv_src -> cv_dst, nullable).  Rows of L % 8 != 0 (fp32 inputs
// with L % 8 = 4) and a group of 8 tokens that crosses a row's end take
// scalar accesses.
template <typename T> __device__ __forceinline__ T out_as(float v);
template <> __device__ __forceinline__ float out_as<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 out_as<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}

constexpr int kConvThreads = 256;
constexpr int kConvPer = 8;
constexpr int kConvTile = kConvThreads * kConvPer;

template <typename T> __device__ __forceinline__ void load8(const T* p, float (&v)[8]);
template <> __device__ __forceinline__ void load8<float>(const float* p, float (&v)[8]) {
    const float4 a = *reinterpret_cast<const float4*>(p);
    const float4 b = *reinterpret_cast<const float4*>(p + 4);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
template <> __device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16* p, float (&v)[8]) {
    const uint4 w = *reinterpret_cast<const uint4*>(p);
    v[0] = bf_lo(w.x); v[1] = bf_hi(w.x); v[2] = bf_lo(w.y); v[3] = bf_hi(w.y);
    v[4] = bf_lo(w.z); v[5] = bf_hi(w.z); v[6] = bf_lo(w.w); v[7] = bf_hi(w.w);
}
template <typename T> __device__ __forceinline__ void store8(T* p, const float (&v)[8]);
template <> __device__ __forceinline__ void store8<float>(float* p, const float (&v)[8]) {
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
    *reinterpret_cast<float4*>(p + 4) = make_float4(v[4], v[5], v[6], v[7]);
}
template <> __device__ __forceinline__ void store8<__nv_bfloat16>(__nv_bfloat16* p, const float (&v)[8]) {
    uint4 w;
    w.x = pack_bf16x2(v[0], v[1]);
    w.y = pack_bf16x2(v[2], v[3]);
    w.z = pack_bf16x2(v[4], v[5]);
    w.w = pack_bf16x2(v[6], v[7]);
    *reinterpret_cast<uint4*>(p) = w;
}

template <typename TIN, typename TOUT>
__global__ void __launch_bounds__(kConvThreads) conv_bwd_kernel(
    int64_t D, int64_t L, int K, const TIN* __restrict__ x, const float* __restrict__ conv_w,
    const float* __restrict__ conv_b, const float* __restrict__ du, TOUT* __restrict__ dx,
    float* __restrict__ dconv_w, float* __restrict__ dconv_b, const float* __restrict__ cv_src0,
    TOUT* __restrict__ cv_dst0, const float* __restrict__ cv_src1, TOUT* __restrict__ cv_dst1) {
    // x[t0-3 .. t0+TILE+3) and dpre[t0 .. t0+TILE+3), element i at P(i) =
    // i + i/32: a thread's 8 tokens are 8 floats apart from its neighbour's,
    // and the padding puts the 32 lanes' elements in 32 different banks
    __shared__ float xs[kConvTile + 6 + (kConvTile + 6) / 32 + 1];
    __shared__ float dps[kConvTile + 3 + (kConvTile + 3) / 32 + 1];
    __shared__ float red[kConvThreads / 32][5];
    auto P = [](int i) { return i + (i >> 5); };
    const int64_t row = blockIdx.x;                    // (batch, channel) row
    const int64_t d = row % D;
    const int64_t t0 = (int64_t)blockIdx.y * kConvTile;
    const int tid = threadIdx.x;
    const int64_t tt = t0 + (int64_t)tid * kConvPer;   // this thread's first token
    // 16-byte accesses when every row starts on a 16-byte boundary in every
    // type (L % 8 = 0) and the thread's 8 tokens are all in the row
    const bool full = (L % 8) == 0 && tt + kConvPer <= L;
    const TIN* xr = x + row * L;
    const float* dur = du + row * L;
    float w[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int k = 0; k < 4; ++k)
        if (k < K) w[k] = conv_w[d * K + k];
    const float cb = conv_b ? conv_b[d] : 0.0f;
    // x of the own tokens, and the halos (thread 0: the 3 before the tile;
    // the last thread: the 3 after it)
    float xv[8];
    if (full) {
        load8<TIN>(xr + tt, xv);
    } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) xv[q] = tt + q < L ? Elem<TIN>::to_f(xr[tt + q]) : 0.0f;
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) xs[P(3 + tid * kConvPer + q)] = xv[q];
    if (tid < 3) {
        const int64_t t = t0 - 3 + tid;
        xs[P(tid)] = t >= 0 ? Elem<TIN>::to_f(xr[t]) : 0.0f;
        const int64_t ta = t0 + kConvTile + tid;
        xs[P(3 + kConvTile + tid)] = ta < L ? Elem<TIN>::to_f(xr[ta]) : 0.0f;
    }
    __syncthreads();
    // dpre of the own tokens (and of the 3 tokens after the tile)
    auto dpre_at = [&](int i, float g) -> float {   // i = token index in the tile
        float pre = cb;
#pragma unroll
        for (int k = 0; k < 4; ++k)
            if (k < K) pre = fmaf(w[k], xs[P(i + 3 - (K - 1) + k)], pre);
        const float s = 1.0f / (1.0f + expf(-pre));
        return g * s * fmaf(pre, 1.0f - s, 1.0f);
    };
    float gv[8];
    if (full) {
        load8<float>(dur + tt, gv);
    } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) gv[q] = tt + q < L ? dur[tt + q] : 0.0f;
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) dps[P(tid * kConvPer + q)] = dpre_at(tid * kConvPer + q, gv[q]);
    if (tid < 3) {
        const int64_t ta = t0 + kConvTile + tid;
        dps[P(kConvTile + tid)] = ta < L ? dpre_at(kConvTile + tid, dur[ta]) : 0.0f;
    }
    __syncthreads();
    float pw[4] = {0.0f, 0.0f, 0.0f, 0.0f}, pb = 0.0f;
    if (tt < L) {
        float o[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int i = tid * kConvPer + q;
            float acc = 0.0f;
#pragma unroll
            for (int k = 0; k < 4; ++k)
                if (k < K) acc = fmaf(w[k], dps[P(i + (K - 1) - k)], acc);
            o[q] = acc;
            if (tt + q < L) {
                const float dp = dps[P(i)];
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    if (k < K) pw[k] = fmaf(dp, xs[P(i + 3 - (K - 1) + k)], pw[k]);
                pb += dp;
            }
        }
        TOUT* dxr = dx + row * L;
        if (full) {
            store8<TOUT>(dxr + tt, o);
        } else {
            for (int q = 0; q < 8; ++q)
                if (tt + q < L) dxr[tt + q] = out_as<TOUT>(o[q]);
        }
        const float* srcs[2] = {cv_src0, cv_src1};
        TOUT* dsts[2] = {cv_dst0, cv_dst1};
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            if (!srcs[j]) continue;
            float v[8];
            if (full) {
                load8<float>(srcs[j] + row * L + tt, v);
                store8<TOUT>(dsts[j] + row * L + tt, v);
            } else {
                for (int q = 0; q < 8; ++q)
                    if (tt + q < L) dsts[j][row * L + tt + q] = out_as<TOUT>(srcs[j][row * L + tt + q]);
            }
        }
    }
    // block sums: warp shuffles, then the warps' partials
    const int lane = tid & 31, warp = tid >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
        for (int k = 0; k < 4; ++k) pw[k] += __shfl_xor_sync(0xffffffffu, pw[k], o);
        pb += __shfl_xor_sync(0xffffffffu, pb, o);
    }
    if (lane == 0) {
#pragma unroll
        for (int k = 0; k < 4; ++k) red[warp][k] = pw[k];
        red[warp][4] = pb;
    }
    __syncthreads();
    if (tid < K + 1) {
        float s = 0.0f;
        for (int w8 = 0; w8 < kConvThreads / 32; ++w8) s += red[w8][tid == K ? 4 : tid];
        if (tid < K) atomicAdd(dconv_w + d * K + tid, s);
        else if (dconv_b) atomicAdd(dconv_b + d, s);
    }
}

template <typename TIN>
cudaError_t conv_bwd_tin(int tout, int64_t Bt, int64_t D, int64_t L, int K, const void* x,
                         const float* w, const float* b, const float* du, void* dx, float* dw,
                         float* db, const float* src0, void* dst0, const float* src1, void* dst1,
                         cudaStream_t st) {
    const dim3 grid((unsigned)(Bt * D), (unsigned)((L + kConvTile - 1) / kConvTile));
    if (tout == SSM_BF16)
        conv_bwd_kernel<TIN, __nv_bfloat16><<<grid, kConvThreads, 0, st>>>(
            D, L, K, static_cast<const TIN*>(x), w, b, du, static_cast<__nv_bfloat16*>(dx), dw, db,
            src0, static_cast<__nv_bfloat16*>(dst0), src1, static_cast<__nv_bfloat16*>(dst1));
    else
        conv_bwd_kernel<TIN, float><<<grid, kConvThreads, 0, st>>>(
            D, L, K, static_cast<const TIN*>(x), w, b, du, static_cast<float*>(dx), dw, db,
            src0, static_cast<float*>(dst0), src1, static_cast<float*>(dst1));
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_conv_np16(int NT, int tin, const BwdParams& p, const BwdMaps& m,
                                 const BwdLaunch& lc, cudaStream_t st) {
    switch (NT) {
        case 2: return conv_nt<2>(tin, p, m, lc, st);
        case 4: return conv_nt<4>(tin, p, m, lc, st);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_conv_bwd(int tin, int tout, int64_t Bt, int64_t D, int64_t L, int K,
                            const void* x, const float* conv_w, const float* conv_b,
                            const float* du, void* dx, float* dconv_w, float* dconv_b,
                            const float* ddr32, void* ddr, const float* dz32, void* dz,
                            cudaStream_t st) {
    if (Bt * D == 0 || L == 0) return cudaSuccess;
    return tin == SSM_BF16
               ? conv_bwd_tin<__nv_bfloat16>(tout, Bt, D, L, K, x, conv_w, conv_b, du, dx, dconv_w,
                                             dconv_b, ddr32, ddr, dz32, dz, st)
               : conv_bwd_tin<float>(tout, Bt, D, L, K, x, conv_w, conv_b, du, dx, dconv_w, dconv_b,
                                     ddr32, ddr, dz32, dz, st);
}

}  // namespace ssm
