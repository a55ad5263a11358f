// ssm_fwd_varlen.cu -- forward-kernel instantiations for packed sequences
// (padded state size 16, TMA tiles), with and without the conv prologue.
#include "ssm_fwd_launch.cuh"

namespace ssm {

template <int NT, typename TIN, bool CONV>
static cudaError_t launch_varlen_conv(int tout, bool summary, const FwdParams& p, const FwdMaps& m,
                                      dim3 grid, int warps, size_t smem, cudaStream_t st) {
    if (summary)
        return launch_fwd_one<16, NT, TIN, float, true, true, CONV, true>(p, m, grid, warps, smem, st);
    return tout == SSM_BF16
               ? launch_fwd_one<16, NT, TIN, __nv_bfloat16, false, true, CONV, true>(p, m, grid, warps, smem, st)
               : launch_fwd_one<16, NT, TIN, float, false, true, CONV, true>(p, m, grid, warps, smem, st);
}

template <int NT, typename TIN>
static cudaError_t launch_varlen_tin(int tout, bool summary, bool conv, const FwdParams& p,
                                     const FwdMaps& m, dim3 grid, int warps, size_t smem,
                                     cudaStream_t st) {
    return conv ? launch_varlen_conv<NT, TIN, true>(tout, summary, p, m, grid, warps, smem, st)
                : launch_varlen_conv<NT, TIN, false>(tout, summary, p, m, grid, warps, smem, st);
}

template <int NT>
static cudaError_t launch_varlen_nt(int tin, int tout, bool summary, bool conv, const FwdParams& p,
                                    const FwdMaps& m, dim3 grid, int warps, size_t smem,
                                    cudaStream_t st) {
    return tin == SSM_BF16
               ? launch_varlen_tin<NT, __nv_bfloat16>(tout, summary, conv, p, m, grid, warps, smem, st)
               : launch_varlen_tin<NT, float>(tout, summary, conv, p, m, grid, warps, smem, st);
}

cudaError_t launch_fwd_varlen_np16(int NT, int tin, int tout, bool summary, bool conv,
                                   const FwdParams& p, const FwdMaps& m, dim3 grid, int warps,
                                   size_t smem, cudaStream_t st) {
    switch (NT) {
        case 2: return launch_varlen_nt<2>(tin, tout, summary, conv, p, m, grid, warps, smem, st);
        case 4: return launch_varlen_nt<4>(tin, tout, summary, conv, p, m, grid, warps, smem, st);
        case 1: return launch_varlen_nt<1>(tin, tout, summary, conv, p, m, grid, warps, smem, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace ssm
