// ssm_bwd_launch.cuh -- host-side launch of one backward instantiation (the
// forward sweep followed by the reverse sweep on the same stream); included
// by the per-state-size translation units ssm_bwd_np*.cu.
#pragma once

#include "ssm_bwd.cuh"
#include "ssm_internal.h"

namespace ssm {

template <int NP, int NT, typename TIN, typename TOUT, bool TMA, bool VARLEN = false, bool CONV = false>
cudaError_t launch_bwd_one(const BwdParams& p, const BwdMaps& m, const BwdLaunch& lc, cudaStream_t st) {
    auto kf = bwd_fwd_kernel<NP, NT, TIN, TOUT, TMA, VARLEN, false, CONV>;
    auto kr = bwd_rev_kernel<NP, NT, TIN, TOUT, TMA, VARLEN, CONV>;
    // raise the kernels' dynamic shared-memory limits when a launch needs more
    // than any earlier one on this device
    static size_t attr_f[64] = {}, attr_r[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || attr_f[dev] < lc.smem_f) {
        e = cudaFuncSetAttribute(kf, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)lc.smem_f);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_f[dev] = lc.smem_f;
    }
    if (dev < 0 || dev >= 64 || attr_r[dev] < lc.smem_r) {
        e = cudaFuncSetAttribute(kr, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)lc.smem_r);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_r[dev] = lc.smem_r;
    }
    BwdParams pf = p;
    pf.stages = lc.stages_f;
    kf<<<lc.grid, 32 * (lc.warps + 1), lc.smem_f, st>>>(pf, m.u, m.dr, m.z, m.dy, m.bc);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    BwdParams pr = p;
    pr.stages = lc.stages_r;
    kr<<<lc.grid, 32 * (lc.warps + 1), lc.smem_r, st>>>(pr, m.u, m.dr, m.z, m.dy, m.phi, m.bc);
    return cudaGetLastError();
}

template <int NP, int NT, typename TIN>
cudaError_t launch_bwd_tin(int tout, bool tma, const BwdParams& p, const BwdMaps& m,
                           const BwdLaunch& lc, cudaStream_t st) {
    if (tout == SSM_BF16)
        return tma ? launch_bwd_one<NP, NT, TIN, __nv_bfloat16, true>(p, m, lc, st)
                   : launch_bwd_one<NP, NT, TIN, __nv_bfloat16, false>(p, m, lc, st);
    return tma ? launch_bwd_one<NP, NT, TIN, float, true>(p, m, lc, st)
               : launch_bwd_one<NP, NT, TIN, float, false>(p, m, lc, st);
}

template <int NP, int NT>
cudaError_t launch_bwd_nt(int tin, int tout, bool tma, const BwdParams& p, const BwdMaps& m,
                          const BwdLaunch& lc, cudaStream_t st) {
    if (tin == SSM_BF16) return launch_bwd_tin<NP, NT, __nv_bfloat16>(tout, tma, p, m, lc, st);
    return launch_bwd_tin<NP, NT, float>(tout, tma, p, m, lc, st);
}

}  // namespace ssm
