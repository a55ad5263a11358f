// ssm_fwd_launch.cuh -- host-side launch of one forward-kernel instantiation
// (included by the per-state-size translation units ssm_fwd_np*.cu).
#pragma once

#include "ssm_fwd.cuh"
#include "ssm_internal.h"

namespace ssm {

template <int NP, int NT, typename TIN, typename TOUT, bool SUMMARY, bool TMA>
cudaError_t launch_fwd_one(const FwdParams& p, const FwdMaps& m, dim3 grid, cudaStream_t st) {
    auto kern = fwd_kernel<NP, NT, TIN, TOUT, SUMMARY, TMA>;
    constexpr int smem = fwd_smem_bytes<NT, (int)sizeof(TIN), NP, SUMMARY>();
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !attr_set[dev]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_set[dev] = true;
    }
    kern<<<grid, kThreads, smem, st>>>(p, m.u, m.dr, m.z, m.bc);
    return cudaGetLastError();
}

template <int NP, int NT, typename TIN>
cudaError_t launch_fwd_tin(int tout, bool summary, bool tma, const FwdParams& p, const FwdMaps& m,
                           dim3 grid, cudaStream_t st) {
    if (summary)
        return tma ? launch_fwd_one<NP, NT, TIN, float, true, true>(p, m, grid, st)
                   : launch_fwd_one<NP, NT, TIN, float, true, false>(p, m, grid, st);
    if (tout == SSM_BF16)
        return tma ? launch_fwd_one<NP, NT, TIN, __nv_bfloat16, false, true>(p, m, grid, st)
                   : launch_fwd_one<NP, NT, TIN, __nv_bfloat16, false, false>(p, m, grid, st);
    return tma ? launch_fwd_one<NP, NT, TIN, float, false, true>(p, m, grid, st)
               : launch_fwd_one<NP, NT, TIN, float, false, false>(p, m, grid, st);
}

template <int NP, int NT>
cudaError_t launch_fwd_nt(int tin, int tout, bool summary, bool tma, const FwdParams& p,
                          const FwdMaps& m, dim3 grid, cudaStream_t st) {
    if (tin == SSM_BF16) return launch_fwd_tin<NP, NT, __nv_bfloat16>(tout, summary, tma, p, m, grid, st);
    return launch_fwd_tin<NP, NT, float>(tout, summary, tma, p, m, grid, st);
}

}  // namespace ssm
