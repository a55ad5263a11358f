// ssm_aux.cu -- the small kernels around the forward scan:
//   * prep_bc:   B, C (batch, N, L) -> fp32 (batch, L, 2*NP) with ln2 folded
//                into B (the scan then uses delta/ln2 throughout);
//   * carry:     per-segment initial states of the segmented forward,
//                h_in[s+1] = 2^(A * sum_delta2[s]) * h_in[s] + h_loc[s];
//   * step:      the single-token recurrent update (decode), state in place;
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

cudaError_t launch_prep_bc(int tin, int64_t Bt, int N, int NP, int64_t L, const void* B,
                           const void* C, float* out, int* status, cudaStream_t st) {
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
__global__ void carry_kernel(int64_t Bt, int64_t D, int N, int NP, int nseg, const float* __restrict__ A,
                             const float* __restrict__ h0, const float* __restrict__ hloc,
                             const float* __restrict__ sumd, float* __restrict__ hin) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;   // (b, d, n)
    if (i >= Bt * D * NP) return;
    const int n = (int)(i % NP);
    const int64_t row = i / NP;
    const int64_t d = row % D;
    const int64_t seg_stride = Bt * D;
    const float a = n < N ? A[d * N + n] : 0.0f;
    float h = (h0 && n < N) ? h0[row * N + n] : 0.0f;
    for (int s = 0; s < nseg; ++s) {
        hin[(s * seg_stride + row) * NP + n] = h;
        if (s + 1 < nseg)
            h = ex2(a * sumd[s * seg_stride + row]) * h + hloc[(s * seg_stride + row) * NP + n];
    }
}

cudaError_t launch_carry(int64_t Bt, int64_t D, int N, int NP, int nseg, const float* A,
                         const float* h0, const float* hloc, const float* sumd, float* hin,
                         cudaStream_t st) {
    const int64_t total = Bt * D * NP;
    carry_kernel<<<(unsigned)((total + 255) / 256), 256, 0, st>>>(Bt, D, N, NP, nseg, A, h0, hloc,
                                                                  sumd, hin);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- step ---
// One thread per (b, d, group of S states); GT = ceil(N / S) threads per
// channel.  The step reads the state once and writes it once, so it is bound
// by the state's HBM traffic: each thread keeps S * 4 bytes of state loads in
// flight (S = 16 at N = 16, 64 bytes), issued before any arithmetic.
template <typename TIN>
__device__ __forceinline__ void load_vec4_in(const TIN* p, float (&v)[4]) {
    if constexpr (sizeof(TIN) == 2) {
        const uint2 w = *reinterpret_cast<const uint2*>(p);
        v[0] = bf_lo(w.x); v[1] = bf_hi(w.x); v[2] = bf_lo(w.y); v[3] = bf_hi(w.y);
    } else {
        const float4 w = *reinterpret_cast<const float4*>(p);
        v[0] = w.x; v[1] = w.y; v[2] = w.z; v[3] = w.w;
    }
}

template <typename TIN, typename TOUT, int S, int GT>
__global__ void __launch_bounds__(256) step_kernel(const StepParams p) {
    const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t row = gid / GT;   // b * D + d
    const int g = (int)(gid % GT);
    const bool ok = row < p.Bt * p.D;
    const int64_t r = ok ? row : 0;
    const int64_t b = r / p.D, d = r % p.D;
    const int N = p.N;
    const int n0 = g * S;
    const TIN* u = static_cast<const TIN*>(p.u);
    const TIN* dr = static_cast<const TIN*>(p.dr);
    const TIN* Bv = static_cast<const TIN*>(p.B) + b * N;
    const TIN* Cv = static_cast<const TIN*>(p.C) + b * N;
    const float* Ad = p.A + d * N;
    float* st = p.state + r * N;
    // vector loads need 16-byte (state, A) and 8/16-byte (B, C) aligned rows
    const bool vec = (N % 4) == 0 && n0 + S <= N;

    float hv[S], av[S], bv[S], cv[S];
    if (vec) {
#pragma unroll
        for (int q = 0; q < S; q += 4) {
            const float4 h4 = *reinterpret_cast<const float4*>(st + n0 + q);
            hv[q] = h4.x; hv[q + 1] = h4.y; hv[q + 2] = h4.z; hv[q + 3] = h4.w;
        }
#pragma unroll
        for (int q = 0; q < S; q += 4) {
            const float4 a4 = *reinterpret_cast<const float4*>(Ad + n0 + q);
            av[q] = a4.x; av[q + 1] = a4.y; av[q + 2] = a4.z; av[q + 3] = a4.w;
            float t4[4];
            load_vec4_in<TIN>(Bv + n0 + q, t4);
            bv[q] = t4[0]; bv[q + 1] = t4[1]; bv[q + 2] = t4[2]; bv[q + 3] = t4[3];
            load_vec4_in<TIN>(Cv + n0 + q, t4);
            cv[q] = t4[0]; cv[q + 1] = t4[1]; cv[q + 2] = t4[2]; cv[q + 3] = t4[3];
        }
    } else {
#pragma unroll
        for (int q = 0; q < S; ++q) {
            const bool in = ok && n0 + q < N;
            hv[q] = in ? st[n0 + q] : 0.0f;
            av[q] = in ? Ad[n0 + q] : 0.0f;
            bv[q] = in ? Elem<TIN>::to_f(Bv[n0 + q]) : 0.0f;
            cv[q] = in ? Elem<TIN>::to_f(Cv[n0 + q]) : 0.0f;
        }
    }
    const float uu = Elem<TIN>::to_f(u[r]);
    const float x = fmaf(Elem<TIN>::to_f(dr[r]), kLog2e, p.bias ? p.bias[d] * kLog2e : 0.0f);
    float d2;
    if (sizeof(TIN) == 4) {
        const float e = ex2(-fabsf(x));
        float q = fmaf(e, 0.2f, -0.25f);
        q = fmaf(e, q, 0.33333334f);
        q = fmaf(e, q, -0.5f);
        q = fmaf(e, q, 1.0f);
        d2 = fmaxf(x, 0.0f) + (e < 0.0625f ? e * q * kLog2e : lg2(1.0f + e));
    } else {
        d2 = fmaxf(x, lg2(1.0f + ex2(fminf(x, 64.0f))));
    }
    const float du = d2 * uu * kLn2;   // delta * u

    float acc = 0.0f;
#pragma unroll
    for (int q = 0; q < S; ++q) {
        const float a = sizeof(TIN) == 4 ? exp2_accurate(d2 * av[q]) : ex2(d2 * av[q]);
        hv[q] = fmaf(a, hv[q], du * bv[q]);
        acc = fmaf(cv[q], hv[q], acc);
    }
    if (ok) {
        if (vec) {
#pragma unroll
            for (int q = 0; q < S; q += 4)
                *reinterpret_cast<float4*>(st + n0 + q) =
                    make_float4(hv[q], hv[q + 1], hv[q + 2], hv[q + 3]);
        } else {
#pragma unroll
            for (int q = 0; q < S; ++q)
                if (n0 + q < N) st[n0 + q] = hv[q];
        }
    }
#pragma unroll
    for (int o = 1; o < GT; o <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (ok && g == 0) {
        float v = acc + (p.Dv ? p.Dv[d] * uu : 0.0f);
        if (p.z) {
            const float zq = Elem<TIN>::to_f(static_cast<const TIN*>(p.z)[r]);
            v *= zq * rcp(1.0f + ex2(-kLog2e * zq));
        }
        if (sizeof(TOUT) == 2)
            static_cast<__nv_bfloat16*>(p.y)[r] = __float2bfloat16_rn(v);
        else
            static_cast<float*>(p.y)[r] = v;
    }
}

template <typename TIN, typename TOUT, int S, int GT>
static cudaError_t launch_step_s(const StepParams& p, cudaStream_t st) {
    const int64_t threads = p.Bt * p.D * GT;
    const unsigned blocks = (unsigned)((threads + 255) / 256);
    step_kernel<TIN, TOUT, S, GT><<<blocks, 256, 0, st>>>(p);
    return cudaGetLastError();
}

template <typename TIN, typename TOUT>
static cudaError_t launch_step_t(const StepParams& p, cudaStream_t st) {
    // S states per thread (a multiple of 4 when N allows vector loads), GT
    // threads per channel (a power of two, for the shuffle reduction)
    if (p.N <= 4) return launch_step_s<TIN, TOUT, 4, 1>(p, st);
    if (p.N <= 8) return launch_step_s<TIN, TOUT, 8, 1>(p, st);
    if (p.N <= 16) return launch_step_s<TIN, TOUT, 16, 1>(p, st);
    if (p.N <= 32) return launch_step_s<TIN, TOUT, 16, 2>(p, st);
    return launch_step_s<TIN, TOUT, 16, 4>(p, st);
}

cudaError_t launch_step(int tin, int tout, const StepParams& p, cudaStream_t st) {
    if (tin == SSM_BF16)
        return tout == SSM_BF16 ? launch_step_t<__nv_bfloat16, __nv_bfloat16>(p, st)
                                : launch_step_t<__nv_bfloat16, float>(p, st);
    return tout == SSM_BF16 ? launch_step_t<float, __nv_bfloat16>(p, st)
                            : launch_step_t<float, float>(p, st);
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
