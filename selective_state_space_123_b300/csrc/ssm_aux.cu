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
// One thread per (b, d, group of 4 states); GT threads per channel (power of
// two, GT * 4 >= N).  Reads the state once and writes it once: the step is
// bound by the state's HBM traffic.
template <typename TIN, typename TOUT, int GT>
__global__ void __launch_bounds__(256) step_kernel(const StepParams p) {
    const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t row = gid / GT;   // b * D + d
    const int g = (int)(gid % GT);
    const bool ok = row < p.Bt * p.D;
    const int64_t r = ok ? row : 0;
    const int64_t b = r / p.D, d = r % p.D;
    const int N = p.N;
    const TIN* u = static_cast<const TIN*>(p.u);
    const TIN* dr = static_cast<const TIN*>(p.dr);
    const TIN* Bv = static_cast<const TIN*>(p.B);
    const TIN* Cv = static_cast<const TIN*>(p.C);

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

    const int n0 = g * 4;
    float* st = p.state + r * N;
    float hv[4];
    const bool vec = ok && (N % 4 == 0) && (n0 + 4 <= N);
    if (vec) {
        const float4 v = *reinterpret_cast<const float4*>(st + n0);
        hv[0] = v.x; hv[1] = v.y; hv[2] = v.z; hv[3] = v.w;
    } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) hv[q] = (ok && n0 + q < N) ? st[n0 + q] : 0.0f;
    }
    float acc = 0.0f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int n = n0 + q;
        if (n < N) {
            const float a = ex2(d2 * p.A[d * N + n]);
            const float Bn = Elem<TIN>::to_f(Bv[b * N + n]);
            const float Cn = Elem<TIN>::to_f(Cv[b * N + n]);
            hv[q] = fmaf(a, hv[q], du * Bn);
            acc = fmaf(Cn, hv[q], acc);
        }
    }
    if (vec) {
        *reinterpret_cast<float4*>(st + n0) = make_float4(hv[0], hv[1], hv[2], hv[3]);
    } else if (ok) {
#pragma unroll
        for (int q = 0; q < 4; ++q)
            if (n0 + q < N) st[n0 + q] = hv[q];
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

template <typename TIN, typename TOUT>
static cudaError_t launch_step_t(const StepParams& p, cudaStream_t st) {
    const int groups = (p.N + 3) / 4;
    int GT = 1;
    while (GT < groups) GT <<= 1;
    const int64_t threads = p.Bt * p.D * GT;
    const unsigned blocks = (unsigned)((threads + 255) / 256);
    switch (GT) {
        case 1: step_kernel<TIN, TOUT, 1><<<blocks, 256, 0, st>>>(p); break;
        case 2: step_kernel<TIN, TOUT, 2><<<blocks, 256, 0, st>>>(p); break;
        case 4: step_kernel<TIN, TOUT, 4><<<blocks, 256, 0, st>>>(p); break;
        case 8: step_kernel<TIN, TOUT, 8><<<blocks, 256, 0, st>>>(p); break;
        default: step_kernel<TIN, TOUT, 16><<<blocks, 256, 0, st>>>(p); break;
    }
    return cudaGetLastError();
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
