// Internal interface between the C ABI (fa_api.cu) and the kernel translation
// units. Not installed, not part of the public header.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace fa {

// Values written to the device error word: a kernel abandoned a wait, met an
// out-of-range device-side index (a page number in a block table), or found
// packed-sequence offsets that do not describe sequences inside the tensors
// (or a query sequence longer than the launch was sized for).
constexpr int kDeviceErrTimeout = 1;
constexpr int kDeviceErrBadIndex = 2;
constexpr int kDeviceErrSeqLens = 3;

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
    int total_k;           // varlen: key tokens (bound of cu_k)
    int n_pairs;           // query-tile pairs per (sequence, head): ceil(ceil(Sq/128)/2)
    int n_qtiles;          // 128-row query tiles per (sequence, head): ceil(Sq/128)
    int num_work;          // work items: n_pairs * B * H (D <= 128), n_qtiles * B * H * D / 256 (D >= 256)
    float scale_log2;      // scale * log2(e)
    int *err;              // device error word
    unsigned long long timeout_ns;
    int withhold;          // test support, 0 = off: CTA 0 never issues its V tile load number withhold - 1
};

int fwd_smem_bytes(int D);

// A packed sequence whose offsets [q0, q1) and [k0, k1) do not lie inside the
// tensors (0 <= begin <= end <= total), or whose query length exceeds p.Sq
// (the max_seqlen_q the launch was sized for).
__device__ __forceinline__ bool varlen_seq_bad(const FwdParams &p, int q0, int q1, int k0, int k1) {
    return q0 < 0 || q1 < q0 || q1 > p.total_q || q1 - q0 > p.Sq || k0 < 0 || k1 < k0 || k1 > p.total_k;
}

// Packed-sequence offsets check, run by every thread of a CTA (all must call
// it): true when no sequence is bad. Every CTA reaches the same answer;
// thread 0 of each CTA that finds a fault records it in the device error word.
__device__ __forceinline__ bool varlen_offsets_ok(const FwdParams &p) {
    bool bad = false;
    for (int b = static_cast<int>(threadIdx.x); b < p.B; b += static_cast<int>(blockDim.x))
        bad |= varlen_seq_bad(p, p.cu_q[b], p.cu_q[b + 1], p.cu_k[b], p.cu_k[b + 1]);
    bad = __syncthreads_or(bad) != 0;
    if (bad && threadIdx.x == 0) atomicExch(p.err, kDeviceErrSeqLens);
    return !bad;
}

// Parameters of the split-KV decode kernel (dense and paged K/V).
struct DecodeParams {
    const uint16_t *q, *k, *v;   // q [B*H, D]; k, v dense [B*H, Sk, D] or pages [num_blocks, H, bs, D]
    float *o_part, *m_part, *l_part;
    int H;                       // heads (paged: to locate the head inside a page)
    int Sk;                      // dense: keys per head
    int num_splits;
    int keys_per_split;          // dense: ceil(Sk / num_splits)
    float scale_log2;
    const int *block_table;      // paged: [B, max_blocks] page numbers
    const int *seq_lens;         // paged: [B] keys per sequence
    int max_blocks;              // paged: row length of block_table
    int log2_bs;                 // paged: log2(block_size)
    int num_blocks;              // paged: pages in the cache
    int *err;                    // paged: device error word
    void *o;                     // fused: [B*H, D] output (input dtype)
    float *lse;                  // fused: [B*H] log-sum-exp
    int *counters;               // fused: [B*H] finished partitions per head, zero between calls
};

// Parameters of the backward pass: dense [B,H,S,D] or packed [T,H,D] layout.
// A work unit is a head (dense) or a (sequence, head) pair (packed).
struct BwdParams {
    float *lse2;           // dense [B*H][Sq_pad], +inf past Sq | packed [H][total_q]: forward LSE * log2(e)
    float *delta;          // same layout: D_i = sum_d dO_id O_id (0 past Sq, dense)
    float *dq_acc;         // dense [B*H][Sq][D] | packed [total_q][H][D]: fp32 accumulator of dS K
    void *dk, *dv;         // dense [B*H][Sk][D] | packed [total_k][H][D] outputs (input dtype)
    int BH;                // work units: B*H (dense), num_seqs*H (packed)
    int Sq, Sk;            // dense: lengths; packed: max_seqlen_q, max_seqlen_k
    int Sq_pad;            // dense: Sq rounded up to whole 128-row tiles
    int n_qtiles, n_ktiles;
    int heads_per_group;   // CTAs run work units group by group (see bwd_work)
    const int *cu_q;       // packed: int32[num_seqs + 1]
    const int *cu_k;       // packed: int32[num_seqs + 1]
    int H;                 // packed: heads
    int total_q, total_k;  // packed: tokens
    float scale, scale_log2;
    int *err;              // device error word
    unsigned long long timeout_ns;
    int withhold;          // test support, 0 = off: CTA 0 never issues its Q/dO load number withhold - 1
    int *work_counter;     // D = 128: next work unit to hand out (in the workspace, zeroed by the prep kernel)
    int total_units;       // D = 128: work units of the launch (BH * n_ktiles)
    int grid;              // D = 128: persistent CTAs (at most one per SM)
};

// Test support: a launch that withholds one load (see FwdParams::withhold)
// leaves a wait that nothing completes, so the kernel's bounded wait runs
// out and its abort path (drain, TMEM release, error word) runs.
__device__ __forceinline__ bool withheld(int withhold, uint32_t load) {
    return withhold > 0 && blockIdx.x == 0 && load + 1 == static_cast<uint32_t>(withhold);
}

// maps: {Q, K, V, dO, dQ accumulator (fp32)}; lse dense [B*H][Sq] | packed
// [H][total_q]; dq output (input dtype). Dense maps are 3-D {D, S, B*H},
// packed maps {D, H, tokens}.
cudaError_t launch_bwd_dense(int D, bool bf16, bool causal, const CUtensorMap *maps, const void *o,
                             const void *dout, const float *lse, void *dq, const BwdParams &p, cudaStream_t stream);
cudaError_t launch_bwd_varlen(int D, bool bf16, bool causal, const CUtensorMap *maps, const void *o,
                              const void *dout, const float *lse, void *dq, const BwdParams &p, cudaStream_t stream);

// maps: {Q, K, V} tensor maps (see fa_api.cu for their geometry).
cudaError_t launch_fwd_dense(int D, bool bf16, bool causal, const CUtensorMap *maps,
                             const FwdParams &p, int grid, cudaStream_t stream);
cudaError_t launch_fwd_varlen(int D, bool bf16, bool causal, const CUtensorMap *maps,
                              const FwdParams &p, int grid, cudaStream_t stream);
// D = 256: one query tile per work item; maps: Q boxes of 128 rows, K/V boxes of 64.
cudaError_t launch_fwd_d256(bool bf16, bool causal, bool varlen, const CUtensorMap *maps, const FwdParams &p,
                            int grid, cudaStream_t stream);
// D = 512, 1024 (Split-D): one query tile and one 256-column output slice per
// work item; same maps (boxes of 64 columns; 128 rows for Q, 64 for K/V).
cudaError_t launch_fwd_splitd(int D, bool bf16, bool causal, bool varlen, const CUtensorMap *maps,
                              const FwdParams &p, int grid, cudaStream_t stream);

cudaError_t launch_decode_split(int D, bool bf16, const void *q, const void *k, const void *v,
                                float *o_part, float *m_part, float *l_part, int BH, int Sk,
                                int num_splits, int keys_per_split, float scale_log2,
                                cudaStream_t stream);

cudaError_t launch_decode_split_paged(int D, bool bf16, const DecodeParams &p, int BH, cudaStream_t stream);

// Phase 1 and phase 2 in one launch: the last partition of each head to
// finish merges that head (p.o, p.lse, p.counters must be set).
cudaError_t launch_decode_fused(int D, bool bf16, bool paged, const DecodeParams &p, int BH, cudaStream_t stream);

cudaError_t launch_splitkv_merge(int D, bool bf16, const float *o_part, const float *m_part,
                                 const float *l_part, void *o, float *lse, int BH,
                                 int num_splits, cudaStream_t stream);

}  // namespace fa
