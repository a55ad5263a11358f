// ssm_bwd_varlen.cu -- backward instantiations over packed sequences ("Mamba
// Architecture Explained", section "Problem 3: Ecosystem maturity": sequence
// packing): padded state size 16, two threads per channel, TMA tiles.
#include "ssm_bwd_launch.cuh"

namespace ssm {

cudaError_t launch_bwd_varlen_np16(int tin, int tout, const BwdParams& p, const BwdMaps& m,
                                   const BwdLaunch& lc, cudaStream_t st) {
    if (tin == SSM_BF16) {
        if (tout == SSM_BF16)
            return launch_bwd_one<16, 2, __nv_bfloat16, __nv_bfloat16, true, true>(p, m, lc, st);
        return launch_bwd_one<16, 2, __nv_bfloat16, float, true, true>(p, m, lc, st);
    }
    if (tout == SSM_BF16) return launch_bwd_one<16, 2, float, __nv_bfloat16, true, true>(p, m, lc, st);
    return launch_bwd_one<16, 2, float, float, true, true>(p, m, lc, st);
}

}  // namespace ssm
