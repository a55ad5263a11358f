// ssm_bwd_conv.cu -- the backward fed by the conv prologue: both sweeps form
// u from the branch input x per token (padded state size 16, 16-byte token
// rows, whole rows), and the prologue's own reverse mode, conv_bwd_kernel:
// dx, dconv_w, dconv_b from the sweeps' du.
#include "ssm_bwd_launch.cuh"

namespace ssm {

namespace {

// the sweeps write ddelta_raw and dz in the output type and du in fp32 (the
// prologue's pass reads it and rounds dx once)
template <int NT, typename TIN>
cudaError_t conv_tin(int tout, const BwdParams& p, const BwdMaps& m, const BwdLaunch& lc,
                     cudaStream_t st) {
    return tout == SSM_BF16 ? launch_bwd_one<16, NT, TIN, __nv_bfloat16, true, false, true>(p, m, lc, st)
                            : launch_bwd_one<16, NT, TIN, float, true, false, true>(p, m, lc, st);
}
template <int NT>
cudaError_t conv_nt(int tin, int tout, const BwdParams& p, const BwdMaps& m, const BwdLaunch& lc,
                    cudaStream_t st) {
    return tin == SSM_BF16 ? conv_tin<NT, __nv_bfloat16>(tout, p, m, lc, st)
                           : conv_tin<NT, float>(tout, p, m, lc, st);
}

// The prologue's reverse mode over one tile of kConvTile tokens of one
// (batch, channel) row, 8 consecutive tokens per thread (16-byte loads and
// stores where the rows allow).  With pre[t] = conv_b + sum_k w[k] x[t-(K-1)+k] (x before token 0
// is 0) and u = silu(pre):
//   dpre[t] = du[t] silu'(pre[t]),  silu'(p) = s (1 + p (1 - s)), s = 1 / (1 + e^-p)
//   dx[t] = sum_k w[k] dpre[t+(K-1)-k] (terms past the end absent)
//   dconv_w[d,k] += sum_t dpre[t] x[t-(K-1)+k],  dconv_b[d] += sum_t dpre[t]
// Each thread keeps the x and dpre windows of its 8 tokens in registers;
// only the 3 x before them (from the previous thread) and the 3 dpre after
// them (from the next thread) go through shared memory, and the tile's
// first and last threads take those from global memory.  The weight and
// bias sums are reduced over the block and added once per tile.  du is the
// sweeps' fp32 output, so dx is rounded once.  Rows of L % 8 != 0 (fp32
// inputs with L % 8 = 4) and a group of 8 tokens that crosses a row's end
// take scalar accesses.
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
    float* __restrict__ dconv_w, float* __restrict__ dconv_b) {
    // the 3 last x and the 3 first dpre of every thread's tokens (stride 3:
    // the 32 lanes of a warp hit 32 different banks)
    __shared__ float x_tail[kConvThreads * 3];
    __shared__ float dp_head[kConvThreads * 3];
    __shared__ float red[kConvThreads / 32][5];
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
    // the taps aligned to a 4-token window ending at the token: tap m of
    // wa multiplies x[t-3+m] (zero for m < 4-K), tap m of wb multiplies
    // dpre[t+m] (zero for m >= K)
    float wa[4], wb[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        wa[m] = m >= 4 - K ? conv_w[d * K + m - (4 - K)] : 0.0f;
        wb[m] = m < K ? conv_w[d * K + K - 1 - m] : 0.0f;
    }
    const float cb = conv_b ? conv_b[d] : 0.0f;
    // xw[3 + q] = x of own token q, xw[0..2] = the 3 tokens before (zero
    // before token 0 and past the row's end)
    float xw[kConvPer + 3], g[kConvPer];
    // the tile's edges, loaded with the main loads so that a CTA waits for
    // global memory once: the first thread's 3 x before the tile, the last
    // thread's 3 x and du after it (zeros outside the row)
    float xh[3] = {0.0f, 0.0f, 0.0f}, xa[3] = {0.0f, 0.0f, 0.0f}, ga[3] = {0.0f, 0.0f, 0.0f};
    if (tid == 0) {
#pragma unroll
        for (int j = 0; j < 3; ++j) {
            const int64_t t = tt - 3 + j;
            if (t >= 0) xh[j] = Elem<TIN>::to_f(xr[t]);
        }
    }
    if (tid == kConvThreads - 1) {
#pragma unroll
        for (int j = 0; j < 3; ++j) {
            const int64_t t = tt + 8 + j;
            if (t < L) {
                xa[j] = Elem<TIN>::to_f(xr[t]);
                ga[j] = dur[t];
            }
        }
    }
    if (full) {
        float v[8];
        load8<TIN>(xr + tt, v);
#pragma unroll
        for (int q = 0; q < 8; ++q) xw[3 + q] = v[q];
        load8<float>(dur + tt, g);
    } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            xw[3 + q] = tt + q < L ? Elem<TIN>::to_f(xr[tt + q]) : 0.0f;
            g[q] = tt + q < L ? dur[tt + q] : 0.0f;
        }
    }
#pragma unroll
    for (int j = 0; j < 3; ++j) x_tail[tid * 3 + j] = xw[8 + j];
    __syncthreads();
#pragma unroll
    for (int j = 0; j < 3; ++j) xw[j] = tid > 0 ? x_tail[(tid - 1) * 3 + j] : xh[j];
    // dpre = du silu'(pre) from the 4-token window before each token
    auto dpre = [&](const float (&w4)[4], float gv) -> float {
        float pre = cb;
#pragma unroll
        for (int m = 0; m < 4; ++m) pre = fmaf(wa[m], w4[m], pre);
        const float sg = rcp(1.0f + ex2(-kLog2e * pre));
        return gv * sg * fmaf(pre, 1.0f - sg, 1.0f);
    };
    // dpw[q] = dpre of own token q, dpw[8..10] = of the 3 tokens after
    float dpw[kConvPer + 3];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const float w4[4] = {xw[q], xw[q + 1], xw[q + 2], xw[q + 3]};
        dpw[q] = dpre(w4, g[q]);
    }
#pragma unroll
    for (int j = 0; j < 3; ++j) dp_head[tid * 3 + j] = dpw[j];
    if (tid == kConvThreads - 1) {
        // the 3 tokens after the tile, from their own x and du
        float xe[6];
#pragma unroll
        for (int j = 0; j < 3; ++j) {
            xe[j] = xw[8 + j];
            xe[3 + j] = xa[j];
        }
#pragma unroll
        for (int j = 0; j < 3; ++j) {
            const float w4[4] = {xe[j], xe[j + 1], xe[j + 2], xe[j + 3]};
            dpw[8 + j] = dpre(w4, ga[j]);
        }
    }
    __syncthreads();
    if (tid < kConvThreads - 1) {
#pragma unroll
        for (int j = 0; j < 3; ++j) dpw[8 + j] = dp_head[(tid + 1) * 3 + j];
    }
    // dx, and the weight and bias sums (dpre is zero past the row's end)
    float o[8], pw[4] = {0.0f, 0.0f, 0.0f, 0.0f}, pb = 0.0f;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        float acc = 0.0f;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            acc = fmaf(wb[m], dpw[q + m], acc);
            pw[m] = fmaf(dpw[q], xw[q + m], pw[m]);
        }
        o[q] = acc;
        pb += dpw[q];
    }
    TOUT* dxr = dx + row * L;
    if (full) {
        store8<TOUT>(dxr + tt, o);
    } else {
#pragma unroll
        for (int q = 0; q < 8; ++q)
            if (tt + q < L) dxr[tt + q] = out_as<TOUT>(o[q]);
    }
    // block sums: warp shuffles, then the warps' partials; tap m of pw is
    // weight k = m - (4 - K)
    const int lane = tid & 31, warp = tid >> 5;
#pragma unroll
    for (int sh = 16; sh > 0; sh >>= 1) {
#pragma unroll
        for (int m = 0; m < 4; ++m) pw[m] += __shfl_xor_sync(0xffffffffu, pw[m], sh);
        pb += __shfl_xor_sync(0xffffffffu, pb, sh);
    }
    if (lane == 0) {
#pragma unroll
        for (int m = 0; m < 4; ++m) red[warp][m] = pw[m];
        red[warp][4] = pb;
    }
    __syncthreads();
    if (tid < K + 1) {
        const int slot = tid == K ? 4 : tid + 4 - K;
        float sum = 0.0f;
        for (int w8 = 0; w8 < kConvThreads / 32; ++w8) sum += red[w8][slot];
        if (tid < K) atomicAdd(dconv_w + d * K + tid, sum);
        else if (dconv_b) atomicAdd(dconv_b + d, sum);
    }
}

template <typename TIN>
cudaError_t conv_bwd_tin(int tout, int64_t Bt, int64_t D, int64_t L, int K, const void* x,
                         const float* w, const float* b, const float* du, void* dx, float* dw,
                         float* db, cudaStream_t st) {
    const dim3 grid((unsigned)(Bt * D), (unsigned)((L + kConvTile - 1) / kConvTile));
    if (tout == SSM_BF16)
        conv_bwd_kernel<TIN, __nv_bfloat16><<<grid, kConvThreads, 0, st>>>(
            D, L, K, static_cast<const TIN*>(x), w, b, du, static_cast<__nv_bfloat16*>(dx), dw, db);
    else
        conv_bwd_kernel<TIN, float><<<grid, kConvThreads, 0, st>>>(
            D, L, K, static_cast<const TIN*>(x), w, b, du, static_cast<float*>(dx), dw, db);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_conv_np16(int NT, int tin, int tout, const BwdParams& p, const BwdMaps& m,
                                 const BwdLaunch& lc, cudaStream_t st) {
    switch (NT) {
        case 2: return conv_nt<2>(tin, tout, p, m, lc, st);
        case 4: return conv_nt<4>(tin, tout, p, m, lc, st);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_conv_bwd(int tin, int tout, int64_t Bt, int64_t D, int64_t L, int K,
                            const void* x, const float* conv_w, const float* conv_b,
                            const float* du, void* dx, float* dconv_w, float* dconv_b,
                            cudaStream_t st) {
    if (Bt * D == 0 || L == 0) return cudaSuccess;
    return tin == SSM_BF16
               ? conv_bwd_tin<__nv_bfloat16>(tout, Bt, D, L, K, x, conv_w, conv_b, du, dx, dconv_w,
                                             dconv_b, st)
               : conv_bwd_tin<float>(tout, Bt, D, L, K, x, conv_w, conv_b, du, dx, dconv_w, dconv_b,
                                     st);
}

}  // namespace ssm
