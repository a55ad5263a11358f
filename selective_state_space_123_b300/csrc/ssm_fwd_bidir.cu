// ssm_fwd_bidir.cu -- forward-kernel instantiations of the bidirectional scan
// (padded state size 16, TMA tiles): dir 1 is the right-to-left pass writing
// its gated output in fp32 (and, for the segmented plan, its segment
// summaries), dir 2 the left-to-right pass adding it to its own.
#include "ssm_fwd_launch.cuh"

namespace ssm {

template <int NT, typename TIN>
static cudaError_t launch_bidir_tin(int tout, int dir, bool summary, const FwdParams& p,
                                    const FwdMaps& m, dim3 grid, int warps, size_t smem,
                                    cudaStream_t st) {
    if (dir == 1 && summary)
        return launch_fwd_one<16, NT, TIN, float, true, true, false, false, 1>(p, m, grid, warps, smem, st);
    if (dir == 1)
        return launch_fwd_one<16, NT, TIN, float, false, true, false, false, 1>(p, m, grid, warps, smem, st);
    return tout == SSM_BF16
               ? launch_fwd_one<16, NT, TIN, __nv_bfloat16, false, true, false, false, 2>(p, m, grid, warps, smem, st)
               : launch_fwd_one<16, NT, TIN, float, false, true, false, false, 2>(p, m, grid, warps, smem, st);
}

template <int NT>
static cudaError_t launch_bidir_nt(int tin, int tout, int dir, bool summary, const FwdParams& p,
                                   const FwdMaps& m, dim3 grid, int warps, size_t smem,
                                   cudaStream_t st) {
    return tin == SSM_BF16
               ? launch_bidir_tin<NT, __nv_bfloat16>(tout, dir, summary, p, m, grid, warps, smem, st)
               : launch_bidir_tin<NT, float>(tout, dir, summary, p, m, grid, warps, smem, st);
}

cudaError_t launch_fwd_bidir_np16(int NT, int tin, int tout, int dir, bool summary,
                                  const FwdParams& p, const FwdMaps& m, dim3 grid, int warps,
                                  size_t smem, cudaStream_t st) {
    if (dir != 1 && dir != 2) return cudaErrorInvalidValue;
    if (summary && dir != 1) return cudaErrorInvalidValue;
    switch (NT) {
        case 2: return launch_bidir_nt<2>(tin, tout, dir, summary, p, m, grid, warps, smem, st);
        case 4: return launch_bidir_nt<4>(tin, tout, dir, summary, p, m, grid, warps, smem, st);
        case 1: return launch_bidir_nt<1>(tin, tout, dir, summary, p, m, grid, warps, smem, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace ssm
