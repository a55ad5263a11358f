// ssm_fwd_launch.cuh -- host-side launch of one forward-kernel instantiation
// (included by the per-state-size translation units ssm_fwd_np*.cu).
#pragma once

#include "ssm_fwd.cuh"
#include "ssm_internal.h"

namespace ssm {

template <int NP, int NT, typename TIN, typename TOUT, bool SUMMARY, bool TMA, bool CONV = false,
          bool VARLEN = false, int DIR = 0>
cudaError_t launch_fwd_one(const FwdParams& p, const FwdMaps& m, dim3 grid, int warps,
                           size_t smem, cudaStream_t st) {
    auto kern = fwd_kernel<NP, NT, TIN, TOUT, SUMMARY, TMA, CONV, VARLEN, DIR>;
    // raise the kernel's dynamic shared-memory limit when a launch needs more
    // than any earlier one on this device
    static size_t attr_val[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || attr_val[dev] < smem) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_val[dev] = smem;
    }
    kern<<<grid, 32 * (warps + 1), smem, st>>>(p, m.u, m.dr, m.z, m.bc, m.ya);
    return cudaGetLastError();
}

template <int NP, int NT, typename TIN>
cudaError_t launch_fwd_tin(int tout, bool summary, bool tma, const FwdParams& p, const FwdMaps& m,
                           dim3 grid, int warps, size_t smem, cudaStream_t st) {
    if (summary)
        return tma ? launch_fwd_one<NP, NT, TIN, float, true, true>(p, m, grid, warps, smem, st)
                   : launch_fwd_one<NP, NT, TIN, float, true, false>(p, m, grid, warps, smem, st);
    if (tout == SSM_BF16)
        return tma ? launch_fwd_one<NP, NT, TIN, __nv_bfloat16, false, true>(p, m, grid, warps, smem, st)
                   : launch_fwd_one<NP, NT, TIN, __nv_bfloat16, false, false>(p, m, grid, warps, smem, st);
    return tma ? launch_fwd_one<NP, NT, TIN, float, false, true>(p, m, grid, warps, smem, st)
               : launch_fwd_one<NP, NT, TIN, float, false, false>(p, m, grid, warps, smem, st);
}

template <int NP, int NT>
cudaError_t launch_fwd_nt(int tin, int tout, bool summary, bool tma, const FwdParams& p,
                          const FwdMaps& m, dim3 grid, int warps, size_t smem, cudaStream_t st) {
    if (tin == SSM_BF16)
        return launch_fwd_tin<NP, NT, __nv_bfloat16>(tout, summary, tma, p, m, grid, warps, smem, st);
    return launch_fwd_tin<NP, NT, float>(tout, summary, tma, p, m, grid, warps, smem, st);
}

}  // namespace ssm
