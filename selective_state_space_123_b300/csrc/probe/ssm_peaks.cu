// ssm_peaks.cu -- register-only rate probes for the roofline of the scan
// kernels (libssmpeaks.so, separate from libssmscan.so).
//
// The forward scan does, per state update, one MUFU exponential (2^(delta A))
// and four FP32 operations (delta*A, delta*u*B, the state FMA, the read-out
// FMA).  Its roofline is therefore set by the MUFU ex2 rate and the FP32 pipe
// rate, which these kernels measure in units that do not depend on the clock:
// operations per SM clock cycle.  One CTA per SM; every thread runs eight
// independent dependency chains held in registers (no memory traffic inside
// the timed loop); each CTA reads %clock64 after a barrier at both ends and
// writes its cycle count, so rate = operations of the CTA / its cycles.
//
//   kind 0  ex2.approx.ftz.f32                    (MUFU)
//   kind 1  fma.rn.f32                            (FP32 pipe, one lane-op per thread)
//   kind 2  fma.rn.f32x2                          (FP32 pipe, two lane-ops per thread)
//   kind 3  the scan's update mix per pair of states: mul.f32x2 (delta*A),
//           two ex2, mul.f32x2 (delta*u*B), fma.f32x2 (state), fma.f32x2
//           (read-out); counted in state updates
//   kind 4  lg2.approx.ftz.f32                    (MUFU; softplus)
//   kind 5  rcp.approx.ftz.f32                    (MUFU; the SiLU gate)
#include <cstdint>
#include <cuda_runtime.h>

#include "../ssm_common.cuh"

#if defined(__GNUC__)
#define PEAKS_API extern "C" __attribute__((visibility("default")))
#else
#define PEAKS_API extern "C"
#endif

namespace {

using ssm::f2;

__device__ __forceinline__ void begin_clock(long long& t0) {
    __syncthreads();
    t0 = clock64();
}
__device__ __forceinline__ void end_clock(long long t0, long long* cycles) {
    __syncthreads();
    const long long t1 = clock64();
    if (threadIdx.x == 0) cycles[blockIdx.x] = t1 - t0;
}

__global__ void ex2_kernel(int iters, long long* cycles, float* sink) {
    float v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = 0.01f * (float)(threadIdx.x & 7) + 0.1f * (float)j;
    long long t0;
    begin_clock(t0);
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = ssm::ex2(-v[j]);   // stays in (0.5, 1]
    }
    end_clock(t0, cycles);
    float s = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) s += v[j];
    sink[(size_t)blockIdx.x * blockDim.x + threadIdx.x] = s;
}

__global__ void lg2_kernel(int iters, long long* cycles, float* sink) {
    float v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = 1.5f + 0.01f * (float)(threadIdx.x & 7) + 0.1f * (float)j;
    long long t0;
    begin_clock(t0);
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = 2.0f + ssm::lg2(v[j]);   // stays in [2.5, 3.6]
    }
    end_clock(t0, cycles);
    float s = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) s += v[j];
    sink[(size_t)blockIdx.x * blockDim.x + threadIdx.x] = s;
}

__global__ void rcp_kernel(int iters, long long* cycles, float* sink) {
    float v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = 1.5f + 0.01f * (float)(threadIdx.x & 7) + 0.1f * (float)j;
    long long t0;
    begin_clock(t0);
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = 1.0f + ssm::rcp(v[j]);   // stays in [1.3, 1.8]
    }
    end_clock(t0, cycles);
    float s = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) s += v[j];
    sink[(size_t)blockIdx.x * blockDim.x + threadIdx.x] = s;
}

__global__ void fma_kernel(int iters, long long* cycles, float* sink) {
    float v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = 1.0f + 0.001f * (float)(threadIdx.x + j);
    const float a = 0.999f, b = 1e-3f;
    long long t0;
    begin_clock(t0);
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = fmaf(v[j], a, b);
    }
    end_clock(t0, cycles);
    float s = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) s += v[j];
    sink[(size_t)blockIdx.x * blockDim.x + threadIdx.x] = s;
}

__global__ void fma2_kernel(int iters, long long* cycles, float* sink) {
    f2 v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
        v[j] = ssm::pk(1.0f + 0.001f * (float)(threadIdx.x + j), 1.0f - 0.001f * (float)j);
    const f2 a = ssm::pk(0.999f, 0.998f), b = ssm::pk(1e-3f, 2e-3f);
    long long t0;
    begin_clock(t0);
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = ssm::fma2(v[j], a, b);
    }
    end_clock(t0, cycles);
    float s = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        float lo, hi;
        ssm::upk(v[j], lo, hi);
        s += lo + hi;
    }
    sink[(size_t)blockIdx.x * blockDim.x + threadIdx.x] = s;
}

// 8 state pairs (16 states) of one channel per thread; per iteration one
// token: delta and delta*u change every token so nothing is hoisted.
__global__ void mix_kernel(int iters, long long* cycles, float* sink) {
    f2 h[8], A[8], Bv[8], Cv[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        h[j] = ssm::pk(0.0f, 0.0f);
        A[j] = ssm::pk(-1.4427f * (float)(2 * j + 1), -1.4427f * (float)(2 * j + 2));
        Bv[j] = ssm::pk(0.5f + 0.01f * (float)j, 0.4f);
        Cv[j] = ssm::pk(0.3f, 0.2f - 0.01f * (float)j);
    }
    float d2 = 0.01f + 1e-4f * (float)(threadIdx.x & 31), du = 0.02f;
    f2 acc = ssm::pk(0.0f, 0.0f);
    long long t0;
    begin_clock(t0);
    for (int i = 0; i < iters; ++i) {
        const f2 d2p = ssm::pk(d2, d2), dup = ssm::pk(du, du);
        f2 a = ssm::pk(0.0f, 0.0f);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const f2 dA = ssm::ex2x2(ssm::mul2(d2p, A[j]));
            h[j] = ssm::fma2(dA, h[j], ssm::mul2(dup, Bv[j]));
            a = ssm::fma2(Cv[j], h[j], a);
        }
        acc = ssm::add2(acc, a);
        d2 = fmaf(d2, 0.9999f, 1e-6f);
        du = fmaf(du, 0.9999f, 2e-6f);
    }
    end_clock(t0, cycles);
    float lo, hi;
    ssm::upk(acc, lo, hi);
    sink[(size_t)blockIdx.x * blockDim.x + threadIdx.x] = lo + hi;
}

}  // namespace

// Run probe `kind` (0..5, see above) with `blocks` CTAs of `threads` threads
// for `iters` loop iterations.  `cycles` (device, blocks int64) receives each
// CTA's clock cycles and `sink` (device, blocks * threads floats) the chains'
// final values.  Returns the operations (kind 3: state updates) one CTA
// performs, or -1 on a bad argument or launch failure.  Asynchronous on
// `stream`.
PEAKS_API long long ssm_peaks_launch(int kind, int blocks, int threads, int iters,
                                     long long* cycles, float* sink, void* stream) {
    if (kind < 0 || kind > 5 || blocks < 1 || threads < 32 || threads > 1024 || threads % 32 ||
        iters < 1 || !cycles || !sink)
        return -1;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const long long per_thread = (kind == 2 || kind == 3) ? 16LL * iters : 8LL * iters;
    switch (kind) {
        case 0: ex2_kernel<<<blocks, threads, 0, st>>>(iters, cycles, sink); break;
        case 1: fma_kernel<<<blocks, threads, 0, st>>>(iters, cycles, sink); break;
        case 2: fma2_kernel<<<blocks, threads, 0, st>>>(iters, cycles, sink); break;
        case 3: mix_kernel<<<blocks, threads, 0, st>>>(iters, cycles, sink); break;
        case 4: lg2_kernel<<<blocks, threads, 0, st>>>(iters, cycles, sink); break;
        default: rcp_kernel<<<blocks, threads, 0, st>>>(iters, cycles, sink); break;
    }
    if (cudaGetLastError() != cudaSuccess) return -1;
    return per_thread * threads;
}
