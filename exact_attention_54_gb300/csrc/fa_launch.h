// Internal interface between the C ABI (fa_api.cu) and the kernel translation
// units. Not installed, not part of the public header.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace fa {

// Value written to the device error word when a kernel abandons a wait.
constexpr int kDeviceErrTimeout = 1;

// Default bound on any single wait on an on-chip barrier.
constexpr unsigned long long kWaitTimeoutNs = 1000000000ull;  // 1 s

// Parameters of the forward kernel (dense and packed-varlen layouts).
struct FwdParams {
    void *o;               // [B,H,Sq,D] dense | [total_q,H,D] varlen
    float *lse;            // [B,H,Sq]   dense | [H,total_q]   varlen
    const int *cu_q;       // varlen only: int32[B+1]
    const int *cu_k;       // varlen only: int32[B+1]
    int B;                 // batch size (dense) or number of sequences (varlen)
    int H;                 // heads
    int Sq;                // query length (dense) or max query length (varlen)
    int Sk;                // key length (dense only)
    int total_q;           // varlen: LSE row stride of one head
    int n_pairs;           // query-tile pairs per (sequence, head): ceil(ceil(Sq/128)/2)
    int num_work;          // n_pairs * B * H
    float scale_log2;      // scale * log2(e)
    int *err;              // device error word
    unsigned long long timeout_ns;
};

int fwd_smem_bytes(int D);

// maps: {Q, K, V} tensor maps (see fa_api.cu for their geometry).
cudaError_t launch_fwd_dense(int D, bool bf16, bool causal, const CUtensorMap *maps,
                             const FwdParams &p, int grid, cudaStream_t stream);
cudaError_t launch_fwd_varlen(int D, bool bf16, bool causal, const CUtensorMap *maps,
                              const FwdParams &p, int grid, cudaStream_t stream);

cudaError_t launch_decode_split(int D, bool bf16, const void *q, const void *k, const void *v,
                                float *o_part, float *m_part, float *l_part, int BH, int Sk,
                                int num_splits, int keys_per_split, float scale_log2,
                                cudaStream_t stream);

cudaError_t launch_splitkv_merge(int D, bool bf16, const float *o_part, const float *m_part,
                                 const float *l_part, void *o, float *lse, int BH,
                                 int num_splits, cudaStream_t stream);

}  // namespace fa
