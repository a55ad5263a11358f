// ssm_bwd_seg.cu -- the backward's segmented plan over whole rows (see
// ssm_bwd_seg.cuh).
#include "ssm_bwd_seg.cuh"

namespace ssm {

cudaError_t launch_bwd_seg_np16(int NT, int tin, int tout, int part, const BwdParams& p,
                                const BwdMaps& m, const BwdLaunch& lc, cudaStream_t st) {
    return launch_seg<false>(NT, tin, tout, part, p, m, lc, st);
}

}  // namespace ssm
