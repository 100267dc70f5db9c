// Head-dimension-256 instantiations of the forward kernel (dense and varlen).
#include "fa_fwd_d256.cuh"

namespace fa {

cudaError_t launch_fwd_d256(bool bf16, bool causal, bool varlen, const CUtensorMap *maps, const FwdParams &p,
                            int grid, cudaStream_t stream) {
#define FA_D256(BB, CC, VV) \
    if (bf16 == BB && causal == CC && varlen == VV) return d256::launch<256, BB, CC, VV>(maps, p, grid, stream);
    FA_D256(false, false, false) FA_D256(false, true, false) FA_D256(true, false, false) FA_D256(true, true, false)
    FA_D256(false, false, true) FA_D256(false, true, true) FA_D256(true, false, true) FA_D256(true, true, true)
#undef FA_D256
    return cudaErrorInvalidValue;
}

}  // namespace fa
