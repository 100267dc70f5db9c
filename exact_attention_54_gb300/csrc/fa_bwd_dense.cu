// Dense [B,H,S,D] instantiations of the backward pass (preprocess, main kernel,
// dQ conversion).
#include "fa_bwd.cuh"

namespace fa {

cudaError_t launch_bwd_dense(int D, bool bf16, bool causal, const CUtensorMap *maps, const void *o,
                             const void *dout, const float *lse, void *dq, const BwdParams &p, cudaStream_t stream) {
#define FA_BWD(DD, BB, CC) \
    if (D == DD && bf16 == BB && causal == CC) \
        return bwd::launch_t<DD, BB, CC, false>(maps, o, dout, lse, dq, p, stream);
    FA_BWD(64, false, false) FA_BWD(64, false, true) FA_BWD(64, true, false) FA_BWD(64, true, true)
    FA_BWD(128, false, false) FA_BWD(128, false, true) FA_BWD(128, true, false) FA_BWD(128, true, true)
#undef FA_BWD
    return cudaErrorInvalidValue;
}

}  // namespace fa
