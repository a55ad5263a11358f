// ssm_bwd_seg_varlen.cu -- the backward's segmented plan over packed
// sequences (see ssm_bwd_seg.cuh).
#include "ssm_bwd_seg.cuh"

namespace ssm {

cudaError_t launch_bwd_seg_varlen_np16(int NT, int tin, int tout, int part, const BwdParams& p,
                                       const BwdMaps& m, const BwdLaunch& lc, cudaStream_t st) {
    return launch_seg<true>(NT, tin, tout, part, p, m, lc, st);
}

}  // namespace ssm
