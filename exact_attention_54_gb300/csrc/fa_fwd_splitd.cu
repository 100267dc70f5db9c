// Split-D instantiations of the 256-column forward kernel: head dimensions
// 512 and 1024, one 256-column output slice per work item (dense and varlen).
#include "fa_fwd_d256.cuh"

namespace fa {

cudaError_t launch_fwd_splitd(int D, bool bf16, bool causal, bool varlen, const CUtensorMap *maps,
                              const FwdParams &p, int grid, cudaStream_t stream) {
#define FA_SPLITD(DD, BB, CC, VV)                                    \
    if (D == DD && bf16 == BB && causal == CC && varlen == VV) \
        return d256::launch<DD, BB, CC, VV>(maps, p, grid, stream);
#define FA_SPLITD_D(DD)                                                                                  \
    FA_SPLITD(DD, false, false, false) FA_SPLITD(DD, false, true, false) FA_SPLITD(DD, true, false, false) \
    FA_SPLITD(DD, true, true, false) FA_SPLITD(DD, false, false, true) FA_SPLITD(DD, false, true, true)    \
    FA_SPLITD(DD, true, false, true) FA_SPLITD(DD, true, true, true)
    FA_SPLITD_D(512)
    FA_SPLITD_D(1024)
#undef FA_SPLITD_D
#undef FA_SPLITD
    return cudaErrorInvalidValue;
}

}  // namespace fa
