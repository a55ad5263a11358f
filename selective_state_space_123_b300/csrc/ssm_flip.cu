// ssm_flip.cu -- token-order reversal and the combine step of the
// bidirectional scan's backward ("Mamba Architecture Explained", section
// "Frequently Asked Questions": the bidirectional variant runs a second scan
// right to left).  The right-to-left scan is the left-to-right scan of the
// token-reversed sequence, so its reverse mode is the ordinary backward run
// on reversed copies of its inputs, with its per-token gradients reversed
// back; du and dz are shared by the two directions and summed.
//   * flip_rows:  out[r, t] = in[r, L-1-t] for `rows` rows of L elements;
//   * bidir_combine: du = du_ltr + rev(du_rtl), dz likewise, ddelta_raw of
//     each direction, cast to the output type;
//   * fold_status: the first device error of an inner call into the outer
//     workspace's status word.
#include "ssm_common.cuh"
#include "ssm_internal.h"

namespace ssm {

// Reverse the order of 16-byte chunk lanes: element k of a chunk of V
// elements goes to V-1-k.
template <typename T>
struct Rev16;
template <>
struct Rev16<float> {
    static constexpr int V = 4;
    __device__ __forceinline__ static uint4 rev(uint4 w) { return make_uint4(w.w, w.z, w.y, w.x); }
};
template <>
struct Rev16<__nv_bfloat16> {
    static constexpr int V = 8;
    __device__ __forceinline__ static uint32_t sw(uint32_t x) { return (x >> 16) | (x << 16); }
    __device__ __forceinline__ static uint4 rev(uint4 w) {
        return make_uint4(sw(w.w), sw(w.z), sw(w.y), sw(w.x));
    }
};

// One thread per 16-byte chunk of the output when L is a multiple of the
// chunk (then a reversed chunk is again an aligned chunk), else one thread
// per element.
template <typename T, bool VEC>
__global__ void flip_rows_kernel(const T* __restrict__ in, T* __restrict__ out, int64_t rows,
                                 int64_t L) {
    constexpr int V = Rev16<T>::V;
    const int64_t per_row = VEC ? L / V : L;
    const int64_t total = rows * per_row;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = i / per_row, k = i - r * per_row;
        if (VEC) {
            const uint4 w = *reinterpret_cast<const uint4*>(in + r * L + (per_row - 1 - k) * V);
            *reinterpret_cast<uint4*>(out + r * L + k * V) = Rev16<T>::rev(w);
        } else {
            out[r * L + k] = in[r * L + (L - 1 - k)];
        }
    }
}

template <typename TOUT>
__device__ __forceinline__ void put(TOUT* p, float v);
template <>
__device__ __forceinline__ void put<float>(float* p, float v) { *p = v; }
template <>
__device__ __forceinline__ void put<__nv_bfloat16>(__nv_bfloat16* p, float v) {
    *p = __float2bfloat16_rn(v);
}

// Per element (r, t): du = du1[r,t] + du2[r,L-1-t], dz = dz1 + rev(dz2) (when
// dz is wanted), ddr = ddr1[r,t], ddr_r = ddr2[r,L-1-t].  The fp32 partials
// come from the two inner backward calls; the outputs take their type here.
template <typename TOUT>
__global__ void bidir_combine_kernel(int64_t rows, int64_t L, const float* __restrict__ du1,
                                     const float* __restrict__ du2, const float* __restrict__ dz1,
                                     const float* __restrict__ dz2, const float* __restrict__ ddr1,
                                     const float* __restrict__ ddr2, TOUT* __restrict__ du,
                                     TOUT* __restrict__ dz, TOUT* __restrict__ ddr,
                                     TOUT* __restrict__ ddr_r) {
    const int64_t total = rows * L;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = i / L, t = i - r * L;
        const int64_t j = r * L + (L - 1 - t);
        put<TOUT>(du + i, du1[i] + du2[j]);
        if (dz) put<TOUT>(dz + i, dz1[i] + dz2[j]);
        put<TOUT>(ddr + i, ddr1[i]);
        put<TOUT>(ddr_r + i, ddr2[j]);
    }
}

// The same 8 tokens at a time when L % 8 = 0 (then the mirrored group of 8
// tokens is again 32-byte aligned): 16-byte loads and stores, one index
// division per 8 tokens.
__device__ __forceinline__ void ld8f(const float* p, float (&v)[8]) {
    const float4 a = reinterpret_cast<const float4*>(p)[0];
    const float4 b = reinterpret_cast<const float4*>(p)[1];
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
template <typename TOUT>
__device__ __forceinline__ void st8(TOUT* p, const float (&v)[8]);
template <>
__device__ __forceinline__ void st8<float>(float* p, const float (&v)[8]) {
    reinterpret_cast<float4*>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4*>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
}
template <>
__device__ __forceinline__ void st8<__nv_bfloat16>(__nv_bfloat16* p, const float (&v)[8]) {
    *reinterpret_cast<uint4*>(p) = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                                              pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
}
template <typename TOUT>
__global__ void bidir_combine8_kernel(int64_t rows, int64_t L, const float* __restrict__ du1,
                                      const float* __restrict__ du2, const float* __restrict__ dz1,
                                      const float* __restrict__ dz2, const float* __restrict__ ddr1,
                                      const float* __restrict__ ddr2, TOUT* __restrict__ du,
                                      TOUT* __restrict__ dz, TOUT* __restrict__ ddr,
                                      TOUT* __restrict__ ddr_r) {
    const int64_t groups = L / 8;
    const int64_t total = rows * groups;
    for (int64_t gi = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; gi < total;
         gi += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = gi / groups;
        const int64_t t = (gi - r * groups) * 8;
        const int64_t i = r * L + t;            // tokens t .. t+7
        const int64_t j = r * L + (L - 8 - t);  // their mirrors, last to first
        float a[8], b[8], o[8];
        ld8f(du1 + i, a);
        ld8f(du2 + j, b);
#pragma unroll
        for (int q = 0; q < 8; ++q) o[q] = a[q] + b[7 - q];
        st8<TOUT>(du + i, o);
        if (dz) {
            ld8f(dz1 + i, a);
            ld8f(dz2 + j, b);
#pragma unroll
            for (int q = 0; q < 8; ++q) o[q] = a[q] + b[7 - q];
            st8<TOUT>(dz + i, o);
        }
        ld8f(ddr1 + i, a);
        st8<TOUT>(ddr + i, a);
        ld8f(ddr2 + j, b);
#pragma unroll
        for (int q = 0; q < 8; ++q) o[q] = b[7 - q];
        st8<TOUT>(ddr_r + i, o);
    }
}

__global__ void fold_status_kernel(int* outer, const int* inner) {
    const int v = *inner;
    if (v != SSM_OK) atomicCAS(outer, SSM_OK, v);
}

static unsigned grid_for(int64_t n, int threads) {
    int64_t b = (n + threads - 1) / threads;
    if (b > 148 * 16) b = 148 * 16;   // grid-stride beyond 16 CTAs per SM
    return (unsigned)(b > 0 ? b : 1);
}

cudaError_t launch_flip_rows(int dtype, const void* in, void* out, int64_t rows, int64_t L,
                             cudaStream_t st) {
    if (rows <= 0 || L <= 0) return cudaSuccess;
    const bool f32 = dtype == SSM_F32;
    const int V = f32 ? 4 : 8;
    const bool vec = (L % V) == 0;
    const int64_t n = rows * (vec ? L / V : L);
    const unsigned g = grid_for(n, 256);
    if (f32) {
        if (vec) flip_rows_kernel<float, true><<<g, 256, 0, st>>>(static_cast<const float*>(in), static_cast<float*>(out), rows, L);
        else flip_rows_kernel<float, false><<<g, 256, 0, st>>>(static_cast<const float*>(in), static_cast<float*>(out), rows, L);
    } else {
        using bf = __nv_bfloat16;
        if (vec) flip_rows_kernel<bf, true><<<g, 256, 0, st>>>(static_cast<const bf*>(in), static_cast<bf*>(out), rows, L);
        else flip_rows_kernel<bf, false><<<g, 256, 0, st>>>(static_cast<const bf*>(in), static_cast<bf*>(out), rows, L);
    }
    return cudaGetLastError();
}

cudaError_t launch_bidir_combine(int tout, int64_t rows, int64_t L, const float* du1,
                                 const float* du2, const float* dz1, const float* dz2,
                                 const float* ddr1, const float* ddr2, void* du, void* dz,
                                 void* ddr, void* ddr_r, cudaStream_t st) {
    if (rows <= 0 || L <= 0) return cudaSuccess;
    if (L % 8 == 0) {
        const unsigned g8 = grid_for(rows * (L / 8), 256);
        if (tout == SSM_F32)
            bidir_combine8_kernel<float><<<g8, 256, 0, st>>>(
                rows, L, du1, du2, dz1, dz2, ddr1, ddr2, static_cast<float*>(du),
                static_cast<float*>(dz), static_cast<float*>(ddr), static_cast<float*>(ddr_r));
        else
            bidir_combine8_kernel<__nv_bfloat16><<<g8, 256, 0, st>>>(
                rows, L, du1, du2, dz1, dz2, ddr1, ddr2, static_cast<__nv_bfloat16*>(du),
                static_cast<__nv_bfloat16*>(dz), static_cast<__nv_bfloat16*>(ddr),
                static_cast<__nv_bfloat16*>(ddr_r));
        return cudaGetLastError();
    }
    const unsigned g = grid_for(rows * L, 256);
    if (tout == SSM_F32)
        bidir_combine_kernel<float><<<g, 256, 0, st>>>(
            rows, L, du1, du2, dz1, dz2, ddr1, ddr2, static_cast<float*>(du), static_cast<float*>(dz),
            static_cast<float*>(ddr), static_cast<float*>(ddr_r));
    else
        bidir_combine_kernel<__nv_bfloat16><<<g, 256, 0, st>>>(
            rows, L, du1, du2, dz1, dz2, ddr1, ddr2, static_cast<__nv_bfloat16*>(du),
            static_cast<__nv_bfloat16*>(dz), static_cast<__nv_bfloat16*>(ddr),
            static_cast<__nv_bfloat16*>(ddr_r));
    return cudaGetLastError();
}

cudaError_t launch_fold_status(int* outer, const int* inner, cudaStream_t st) {
    fold_status_kernel<<<1, 1, 0, st>>>(outer, inner);
    return cudaGetLastError();
}

}  // namespace ssm
