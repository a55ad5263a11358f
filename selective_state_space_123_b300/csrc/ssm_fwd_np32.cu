// ssm_fwd_np32.cu -- forward-kernel instantiations for padded state size 32.
#include "ssm_fwd_launch.cuh"

namespace ssm {

cudaError_t launch_fwd_np32(int NT, int tin, int tout, bool summary, bool tma_raw,
                             const FwdParams& p, const FwdMaps& m, dim3 grid, int warps,
                             size_t smem, cudaStream_t st) {
    switch (NT) {
        case 4: return launch_fwd_nt<32, 4>(tin, tout, summary, tma_raw, p, m, grid, warps, smem, st);
        case 2: return launch_fwd_nt<32, 2>(tin, tout, summary, tma_raw, p, m, grid, warps, smem, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace ssm
