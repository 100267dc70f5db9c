// Packed variable-length [total,H,D] instantiations of the forward kernel.
#include "fa_fwd_kernel.cuh"

namespace fa {

cudaError_t launch_fwd_varlen(int D, bool bf16, bool causal, const CUtensorMap *maps, const FwdParams &p,
                              int grid, cudaStream_t stream) {
#define FA_VARLEN(DD, BB, CC) \
    if (D == DD && bf16 == BB && causal == CC) return launch_fwd_t<DD, BB, CC, true>(maps, p, grid, stream);
    FA_VARLEN(64, false, false) FA_VARLEN(64, false, true) FA_VARLEN(64, true, false) FA_VARLEN(64, true, true)
    FA_VARLEN(128, false, false) FA_VARLEN(128, false, true) FA_VARLEN(128, true, false) FA_VARLEN(128, true, true)
#undef FA_VARLEN
    return cudaErrorInvalidValue;
}

}  // namespace fa
