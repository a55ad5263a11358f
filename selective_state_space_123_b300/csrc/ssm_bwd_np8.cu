// ssm_bwd_np8.cu -- backward instantiations for padded state size 8.
#include "ssm_bwd_launch.cuh"

namespace ssm {

cudaError_t launch_bwd_np8(int NT, int tin, int tout, bool tma, const BwdParams& p,
                             const BwdMaps& m, const BwdLaunch& lc, cudaStream_t st) {
    switch (NT) {
        case 2: return launch_bwd_nt<8, 2>(tin, tout, tma, p, m, lc, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace ssm
