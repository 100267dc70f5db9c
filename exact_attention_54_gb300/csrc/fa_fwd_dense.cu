// Dense [B,H,S,D] instantiations of the forward kernel.
#include "fa_fwd_kernel.cuh"

namespace fa {

int fwd_smem_bytes(int D) { return D == 64 ? FwdShape<64>::kSmemBytes : FwdShape<128>::kSmemBytes; }

cudaError_t launch_fwd_dense(int D, bool bf16, bool causal, const CUtensorMap *maps, const FwdParams &p,
                             int grid, cudaStream_t stream) {
#define FA_DENSE(DD, BB, CC) \
    if (D == DD && bf16 == BB && causal == CC) return launch_fwd_t<DD, BB, CC, false>(maps, p, grid, stream);
    FA_DENSE(64, false, false) FA_DENSE(64, false, true) FA_DENSE(64, true, false) FA_DENSE(64, true, true)
    FA_DENSE(128, false, false) FA_DENSE(128, false, true) FA_DENSE(128, true, false) FA_DENSE(128, true, true)
#undef FA_DENSE
    return cudaErrorInvalidValue;
}

}  // namespace fa

