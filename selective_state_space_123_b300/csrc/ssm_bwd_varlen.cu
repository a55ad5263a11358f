// ssm_bwd_varlen.cu -- backward instantiations over packed sequences ("Mamba
// Architecture Explained", section "Problem 3: Ecosystem maturity": sequence
// packing): padded state size 16, two or four threads per channel, TMA tiles.
#include "ssm_bwd_launch.cuh"

namespace ssm {

template <int NT>
static cudaError_t launch_bwd_varlen_nt(int tin, int tout, const BwdParams& p, const BwdMaps& m,
                                        const BwdLaunch& lc, cudaStream_t st) {
    using bf = __nv_bfloat16;
    if (tin == SSM_BF16) {
        if (tout == SSM_BF16) return launch_bwd_one<16, NT, bf, bf, true, true>(p, m, lc, st);
        return launch_bwd_one<16, NT, bf, float, true, true>(p, m, lc, st);
    }
    if (tout == SSM_BF16) return launch_bwd_one<16, NT, float, bf, true, true>(p, m, lc, st);
    return launch_bwd_one<16, NT, float, float, true, true>(p, m, lc, st);
}

cudaError_t launch_bwd_varlen_np16(int NT, int tin, int tout, const BwdParams& p,
                                   const BwdMaps& m, const BwdLaunch& lc, cudaStream_t st) {
    switch (NT) {
        case 2: return launch_bwd_varlen_nt<2>(tin, tout, p, m, lc, st);
        case 4: return launch_bwd_varlen_nt<4>(tin, tout, p, m, lc, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace ssm
