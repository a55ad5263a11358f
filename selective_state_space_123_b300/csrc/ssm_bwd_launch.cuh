// ssm_bwd_launch.cuh -- host-side launch of one backward instantiation (the
// forward sweep followed by the reverse sweep on the same stream); included
// by the per-state-size translation units ssm_bwd_np*.cu.
#pragma once

#include "ssm_bwd.cuh"
#include "ssm_internal.h"

namespace ssm {

template <int NP, int NT, typename TIN, typename TOUT, bool TMA>
cudaError_t launch_bwd_one(const BwdParams& p, const BwdMaps& m, dim3 grid, cudaStream_t st) {
    auto kf = bwd_fwd_kernel<NP, NT, TIN, TOUT, TMA>;
    auto kr = bwd_rev_kernel<NP, NT, TIN, TOUT, TMA>;
    constexpr int sf = bwd_smem_bytes<NT, (int)sizeof(TIN), NP, false>();
    constexpr int sr = bwd_smem_bytes<NT, (int)sizeof(TIN), NP, true>();
    static_assert(sf <= 227 * 1024 && sr <= 227 * 1024, "shared memory per CTA");
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !attr_set[dev]) {
        e = cudaFuncSetAttribute(kf, cudaFuncAttributeMaxDynamicSharedMemorySize, sf);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(kr, cudaFuncAttributeMaxDynamicSharedMemorySize, sr);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_set[dev] = true;
    }
    kf<<<grid, kThreads, sf, st>>>(p, m.u, m.dr, m.z, m.dy, m.bc);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    kr<<<grid, kThreads, sr, st>>>(p, m.u, m.dr, m.z, m.dy, m.phi, m.bc);
    return cudaGetLastError();
}

template <int NP, int NT, typename TIN>
cudaError_t launch_bwd_tin(int tout, bool tma, const BwdParams& p, const BwdMaps& m, dim3 grid,
                           cudaStream_t st) {
    if (tout == SSM_BF16)
        return tma ? launch_bwd_one<NP, NT, TIN, __nv_bfloat16, true>(p, m, grid, st)
                   : launch_bwd_one<NP, NT, TIN, __nv_bfloat16, false>(p, m, grid, st);
    return tma ? launch_bwd_one<NP, NT, TIN, float, true>(p, m, grid, st)
               : launch_bwd_one<NP, NT, TIN, float, false>(p, m, grid, st);
}

template <int NP, int NT>
cudaError_t launch_bwd_nt(int tin, int tout, bool tma, const BwdParams& p, const BwdMaps& m,
                          dim3 grid, cudaStream_t st) {
    if (tin == SSM_BF16) return launch_bwd_tin<NP, NT, __nv_bfloat16>(tout, tma, p, m, grid, st);
    return launch_bwd_tin<NP, NT, float>(tout, tma, p, m, grid, st);
}

}  // namespace ssm
