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

// The prologue's reverse mode over one tile of TILE tokens of one (batch,
// channel) row, one token per thread and pass.  With pre[t] = conv_b +
// sum_k w[k] x[t-(K-1)+k] (x before token 0 is 0) and u = silu(pre):
//   dpre[t] = du[t] silu'(pre[t]),  silu'(p) = s (1 + p (1 - s)), s = 1 / (1 + e^-p)
//   dx[t] = sum_k w[k] dpre[t+(K-1)-k] (terms past the end absent)
//   dconv_w[d,k] += sum_t dpre[t] x[t-(K-1)+k],  dconv_b[d] += sum_t dpre[t]
// x of the tile and the 3 tokens before it, and dpre of the tile and the 3
// tokens after it, go through shared memory; the weight and bias sums are
// reduced over the block and added once per tile.  The sweeps' gradients are
// fp32; with bf16 outputs the same pass also writes ddelta_raw and dz in the
// output type (cv_src -> cv_dst, nullable).
template <typename T> __device__ __forceinline__ T out_as(float v);
template <> __device__ __forceinline__ float out_as<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 out_as<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}

constexpr int kConvTile = 1024;
constexpr int kConvThreads = 256;

template <typename TIN, typename TOUT>
__global__ void __launch_bounds__(kConvThreads) conv_bwd_kernel(
    int64_t D, int64_t L, int K, const TIN* __restrict__ x, const float* __restrict__ conv_w,
    const float* __restrict__ conv_b, const float* __restrict__ du, TOUT* __restrict__ dx,
    float* __restrict__ dconv_w, float* __restrict__ dconv_b, const float* __restrict__ cv_src0,
    TOUT* __restrict__ cv_dst0, const float* __restrict__ cv_src1, TOUT* __restrict__ cv_dst1) {
    __shared__ float xs[kConvTile + 6];     // x[t0-3 .. t0+TILE+3)
    __shared__ float dps[kConvTile + 3];    // dpre[t0 .. t0+TILE+3)
    __shared__ float red[kConvThreads / 32][5];
    const int64_t row = blockIdx.x;                    // (batch, channel) row
    const int64_t d = row % D;
    const int64_t t0 = (int64_t)blockIdx.y * kConvTile;
    const TIN* xr = x + row * L;
    float w[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int k = 0; k < 4; ++k)
        if (k < K) w[k] = conv_w[d * K + k];
    const float cb = conv_b ? conv_b[d] : 0.0f;
    for (int i = threadIdx.x; i < kConvTile + 6; i += kConvThreads) {
        const int64_t t = t0 - 3 + i;
        xs[i] = (t >= 0 && t < L) ? Elem<TIN>::to_f(xr[t]) : 0.0f;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < kConvTile + 3; i += kConvThreads) {
        const int64_t t = t0 + i;
        float v = 0.0f;
        if (t < L) {
            float pre = cb;
#pragma unroll
            for (int k = 0; k < 4; ++k)
                if (k < K) pre = fmaf(w[k], xs[i + 3 - (K - 1) + k], pre);
            const float s = 1.0f / (1.0f + expf(-pre));
            v = du[row * L + t] * s * fmaf(pre, 1.0f - s, 1.0f);
        }
        dps[i] = v;
    }
    __syncthreads();
    float pw[4] = {0.0f, 0.0f, 0.0f, 0.0f}, pb = 0.0f;
    for (int i = threadIdx.x; i < kConvTile; i += kConvThreads) {
        const int64_t t = t0 + i;
        if (t >= L) break;
        float acc = 0.0f;
#pragma unroll
        for (int k = 0; k < 4; ++k)
            if (k < K) acc = fmaf(w[k], dps[i + (K - 1) - k], acc);
        dx[row * L + t] = out_as<TOUT>(acc);
        if (cv_src0) cv_dst0[row * L + t] = out_as<TOUT>(cv_src0[row * L + t]);
        if (cv_src1) cv_dst1[row * L + t] = out_as<TOUT>(cv_src1[row * L + t]);
        const float dp = dps[i];
#pragma unroll
        for (int k = 0; k < 4; ++k)
            if (k < K) pw[k] = fmaf(dp, xs[i + 3 - (K - 1) + k], pw[k]);
        pb += dp;
    }
    // block sums: warp shuffles, then the warps' partials
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
        for (int k = 0; k < 4; ++k) pw[k] += __shfl_xor_sync(0xffffffffu, pw[k], o);
        pb += __shfl_xor_sync(0xffffffffu, pb, o);
    }
    if (lane == 0) {
        for (int k = 0; k < 4; ++k) red[warp][k] = pw[k];
        red[warp][4] = pb;
    }
    __syncthreads();
    if (threadIdx.x < K + 1) {
        float s = 0.0f;
        for (int w8 = 0; w8 < kConvThreads / 32; ++w8) s += red[w8][threadIdx.x == K ? 4 : threadIdx.x];
        if (threadIdx.x < K) atomicAdd(dconv_w + d * K + threadIdx.x, s);
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
