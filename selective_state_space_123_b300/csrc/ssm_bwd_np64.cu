// ssm_bwd_np64.cu -- backward instantiations for padded state size 64.
#include "ssm_bwd_launch.cuh"

namespace ssm {

cudaError_t launch_bwd_np64(int NT, int tin, int tout, bool tma, const BwdParams& p,
                             const BwdMaps& m, const BwdLaunch& lc, cudaStream_t st) {
    switch (NT) {
        case 4: return launch_bwd_nt<64, 4>(tin, tout, tma, p, m, lc, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace ssm
