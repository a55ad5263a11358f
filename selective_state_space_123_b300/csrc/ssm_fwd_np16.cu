// ssm_fwd_np16.cu -- forward-kernel instantiations for padded state size 16.
#include "ssm_fwd_launch.cuh"

namespace ssm {

cudaError_t launch_fwd_np16(int NT, int tin, int tout, bool summary, bool tma_raw,
                             const FwdParams& p, const FwdMaps& m, dim3 grid, int warps,
                             size_t smem, cudaStream_t st) {
    switch (NT) {
        case 2: return launch_fwd_nt<16, 2>(tin, tout, summary, tma_raw, p, m, grid, warps, smem, st);
        case 4: return launch_fwd_nt<16, 4>(tin, tout, summary, tma_raw, p, m, grid, warps, smem, st);
        case 1: return launch_fwd_nt<16, 1>(tin, tout, summary, tma_raw, p, m, grid, warps, smem, st);
        default: return cudaErrorInvalidValue;
    }
}

// The forward with the conv prologue (TMA tiles only).
template <int NT, typename TIN>
static cudaError_t launch_conv_tin(int tout, bool summary, const FwdParams& p, const FwdMaps& m,
                                   dim3 grid, int warps, size_t smem, cudaStream_t st) {
    if (summary) return launch_fwd_one<16, NT, TIN, float, true, true, true>(p, m, grid, warps, smem, st);
    return tout == SSM_BF16
               ? launch_fwd_one<16, NT, TIN, __nv_bfloat16, false, true, true>(p, m, grid, warps, smem, st)
               : launch_fwd_one<16, NT, TIN, float, false, true, true>(p, m, grid, warps, smem, st);
}

template <int NT>
static cudaError_t launch_conv_nt(int tin, int tout, bool summary, const FwdParams& p, const FwdMaps& m,
                                  dim3 grid, int warps, size_t smem, cudaStream_t st) {
    return tin == SSM_BF16 ? launch_conv_tin<NT, __nv_bfloat16>(tout, summary, p, m, grid, warps, smem, st)
                           : launch_conv_tin<NT, float>(tout, summary, p, m, grid, warps, smem, st);
}

cudaError_t launch_fwd_conv_np16(int NT, int tin, int tout, bool summary, const FwdParams& p,
                                 const FwdMaps& m, dim3 grid, int warps, size_t smem, cudaStream_t st) {
    switch (NT) {
        case 2: return launch_conv_nt<2>(tin, tout, summary, p, m, grid, warps, smem, st);
        case 4: return launch_conv_nt<4>(tin, tout, summary, p, m, grid, warps, smem, st);
        case 1: return launch_conv_nt<1>(tin, tout, summary, p, m, grid, warps, smem, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace ssm
