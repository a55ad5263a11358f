// ssm_bwd_seg.cuh -- launch of the backward's segmented plan (long
// sequences with few channels) for padded state size 16 and 16-byte token
// rows: the adjoint summary, the forward sweep with the tangent sums, the
// reverse sweep, each over (channel tile, batch row, segment); included by
// ssm_bwd_seg.cu (whole rows) and ssm_bwd_seg_varlen.cu (packed sequences).
#pragma once

#include "ssm_bwd_launch.cuh"

namespace ssm {

namespace {

// raise a kernel's dynamic shared-memory limit when a launch needs more than
// any earlier one on this device
template <typename K>
cudaError_t raise_smem(K kernel, size_t bytes, size_t (&seen)[64]) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64 && seen[dev] >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e == cudaSuccess && dev >= 0 && dev < 64) seen[dev] = bytes;
    return e;
}

template <int NT, typename TIN, typename TOUT, bool VARLEN>
cudaError_t seg_part(int part, const BwdParams& p, const BwdMaps& m, const BwdLaunch& lc,
                     cudaStream_t st) {
    const unsigned threads = 32u * (unsigned)(lc.warps + 1);
    cudaError_t e = cudaSuccess;
    BwdParams q = p;
    if (part == 0) {
        static size_t seen[64] = {};
        auto k = bwd_lam_kernel<16, NT, TIN, true, VARLEN>;
        if ((e = raise_smem(k, lc.smem_l, seen)) != cudaSuccess) return e;
        q.stages = lc.stages_l;
        const dim3 grid(lc.grid.x, lc.grid.y, lc.grid.z - 1);
        k<<<grid, threads, lc.smem_l, st>>>(q, m.u, m.dr, m.z, m.dy, m.bc);
    } else if (part == 1) {
        static size_t seen[64] = {};
        auto k = bwd_fwd_kernel<16, NT, TIN, TOUT, true, VARLEN, true>;
        if ((e = raise_smem(k, lc.smem_f, seen)) != cudaSuccess) return e;
        q.stages = lc.stages_f;
        k<<<lc.grid, threads, lc.smem_f, st>>>(q, m.u, m.dr, m.z, m.dy, m.bc);
    } else {
        static size_t seen[64] = {};
        auto k = bwd_rev_kernel<16, NT, TIN, TOUT, true, VARLEN>;
        if ((e = raise_smem(k, lc.smem_r, seen)) != cudaSuccess) return e;
        q.stages = lc.stages_r;
        k<<<lc.grid, threads, lc.smem_r, st>>>(q, m.u, m.dr, m.z, m.dy, m.phi, m.bc);
    }
    return cudaGetLastError();
}

template <int NT, typename TIN, bool VARLEN>
cudaError_t seg_tin(int tout, int part, const BwdParams& p, const BwdMaps& m, const BwdLaunch& lc,
                    cudaStream_t st) {
    return tout == SSM_BF16 ? seg_part<NT, TIN, __nv_bfloat16, VARLEN>(part, p, m, lc, st)
                            : seg_part<NT, TIN, float, VARLEN>(part, p, m, lc, st);
}

template <int NT, bool VARLEN>
cudaError_t seg_nt(int tin, int tout, int part, const BwdParams& p, const BwdMaps& m,
                   const BwdLaunch& lc, cudaStream_t st) {
    return tin == SSM_BF16 ? seg_tin<NT, __nv_bfloat16, VARLEN>(tout, part, p, m, lc, st)
                           : seg_tin<NT, float, VARLEN>(tout, part, p, m, lc, st);
}

template <bool VARLEN>
cudaError_t launch_seg(int NT, int tin, int tout, int part, const BwdParams& p, const BwdMaps& m,
                       const BwdLaunch& lc, cudaStream_t st) {
    switch (NT) {
        case 2: return seg_nt<2, VARLEN>(tin, tout, part, p, m, lc, st);
        case 4: return seg_nt<4, VARLEN>(tin, tout, part, p, m, lc, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

}  // namespace ssm
