// Split-KV decoding for one query per head (S_q = 1).
//
// Phase 1 ("Adaptive High-Performance Attention Kernels in CUDA", Advanced
// Production Features 1; "FlashAttention-2 MMA", Split-KV strategy): the Sk
// keys of a head are cut into num_splits partitions of P = ceil(Sk/num_splits)
// keys and one CTA computes the partial result of each partition:
//   m_s = max_j scale q.k_j,  l_s = sum_j e^{scale q.k_j - m_s},
//   O_s = sum_j e^{scale q.k_j - m_s} v_j   (not normalised).
// The work is a stream over K and V that are read exactly once, so the kernel
// is bound by HBM bandwidth: every lane moves 16-byte vectors, a warp reads
// whole 256-byte key rows back to back (512 contiguous bytes per instruction at
// D = 128), and each thread keeps 8 K rows and 8 V rows in flight.
//
// Phase 2 (same passage): O = sum_s e^{m_s - m_g} / l_g * O_s with
// m_g = max_s m_s, l_g = sum_s e^{m_s - m_g} l_s, and LSE = m_g + ln l_g.
// It runs either as its own launch (one CTA per head) or fused into phase 1:
// every partition CTA counts itself done on a per-head counter after its
// partials are out, and the CTA that finishes last merges the head with the
// same routine, then resets the counter for the next call.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include <cstdint>

#include "fa.h"
#include "fa_launch.h"
#include "sm103_ptx.cuh"

namespace fa {

constexpr int kDecodeThreads = 128;
constexpr int kDecodeUnroll = 8;  // keys in flight per lane group
// Four CTAs per SM: up to 128 registers a thread, no spills, and 4,096
// partitions fill 6.7 waves (five CTAs at 96 registers spilled and left the
// last of 5.4 waves 39 % full; three or two CTAs keep too few bytes in flight).
constexpr int kDecodeCtasPerSm = 4;

template <bool BF16>
__device__ __forceinline__ void unpack8(const uint4 &u, float (&f)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if constexpr (BF16) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        } else {
            const __half2 h = *reinterpret_cast<const __half2 *>(&w[i]);
            const float2 x = __half22float2(h);
            f[2 * i] = x.x;
            f[2 * i + 1] = x.y;
        }
    }
}

__device__ __forceinline__ uint4 ldg_stream(const void *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// Phase 2 for one head, run by a whole CTA of THREADS threads = kGroups groups
// of D (one output element per thread and group). The weights e^{m_s - m_g}
// are computed once per partition in parallel and kept in shared memory; each
// group then sums every kGroups-th partition with eight independent loads in
// flight, and the group sums are added through shared memory. Partials are
// read through L2 (ld.global.cg): in the fused path other CTAs wrote them
// during this launch.
template <int THREADS>
__device__ __forceinline__ float block_reduce(float v, bool is_max, float *red) {
    constexpr int kWarps = THREADS / 32;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float o = __shfl_xor_sync(0xffffffffu, v, off);
        v = is_max ? fmaxf(v, o) : v + o;
    }
    if (threadIdx.x % 32 == 0) red[threadIdx.x / 32] = v;
    __syncthreads();
    float r = red[0];
#pragma unroll
    for (int i = 1; i < kWarps; ++i) r = is_max ? fmaxf(r, red[i]) : r + red[i];
    __syncthreads();
    return r;
}

template <int D, bool BF16, int THREADS>
__device__ __forceinline__ void merge_head(const float *o_part, const float *m_part, const float *l_part,
                                           uint16_t *o, float *lse, int bh, int num_splits) {
    constexpr int kGroups = THREADS / D;
    constexpr int U = 8;
    __shared__ float w[FA_MAX_SPLITS];
    __shared__ float red[THREADS / 32];
    __shared__ float part[kGroups][D];
    const int tid = threadIdx.x;
    const int g = tid / D, d = tid % D;
    const float *mp = m_part + static_cast<size_t>(bh) * num_splits;
    const float *lp = l_part + static_cast<size_t>(bh) * num_splits;
    const float *op = o_part + static_cast<size_t>(bh) * num_splits * D + d;

    float mx = -CUDART_INF_F;
    for (int s = tid; s < num_splits; s += THREADS) mx = fmaxf(mx, __ldcg(mp + s));
    const float mg = block_reduce<THREADS>(mx, true, red);
    float lsum = 0.f;
    for (int s = tid; s < num_splits; s += THREADS) {
        const float ws = (mg == -CUDART_INF_F) ? 0.f : expf(__ldcg(mp + s) - mg);
        w[s] = ws;
        lsum = fmaf(ws, __ldcg(lp + s), lsum);
    }
    const float lg = block_reduce<THREADS>(lsum, false, red);  // its barriers also publish w[]

    float acc[U];
#pragma unroll
    for (int u = 0; u < U; ++u) acc[u] = 0.f;
    int s = g;
    for (; s + (U - 1) * kGroups < num_splits; s += U * kGroups) {
        float x[U];
#pragma unroll
        for (int u = 0; u < U; ++u) x[u] = __ldcg(op + static_cast<size_t>(s + u * kGroups) * D);
#pragma unroll
        for (int u = 0; u < U; ++u) acc[u] = fmaf(w[s + u * kGroups], x[u], acc[u]);
    }
    for (; s < num_splits; s += kGroups) acc[0] = fmaf(w[s], __ldcg(op + static_cast<size_t>(s) * D), acc[0]);
    float total = 0.f;
#pragma unroll
    for (int u = 0; u < U; ++u) total += acc[u];
    if constexpr (kGroups > 1) {
        part[g][d] = total;
        __syncthreads();
    }
    if (g == 0) {
#pragma unroll
        for (int i = 1; i < kGroups; ++i) total += part[i][d];
        const float out = lg > 0.f ? total / lg : 0.f;
        if constexpr (BF16) {
            const __nv_bfloat16 h = __float2bfloat16_rn(out);
            o[static_cast<size_t>(bh) * D + d] = *reinterpret_cast<const uint16_t *>(&h);
        } else {
            const __half h = __float2half_rn(out);
            o[static_cast<size_t>(bh) * D + d] = *reinterpret_cast<const uint16_t *>(&h);
        }
        if (d == 0) lse[bh] = lg > 0.f ? mg + logf(lg) : -CUDART_INF_F;
    }
}

// grid: one CTA per (head, partition), x = bh * num_splits + s.
// PAGED: K and V live in pages [num_blocks, H, block_size, D]; key position p
// of sequence b is row p % block_size of page block_table[b][p / block_size],
// and the sequence holds seq_lens[b] keys ("Adaptive High-Performance
// Attention Kernels in CUDA", Advanced Production Features 4). A page index
// outside [0, num_blocks) is never dereferenced: its keys are skipped and the
// device error word records kDeviceErrBadIndex.
template <int D, bool BF16, bool PAGED, bool FUSED>
__global__ void __launch_bounds__(kDecodeThreads, kDecodeCtasPerSm)
    fa_decode_split_kernel(const DecodeParams p) {
    constexpr int kLanesPerKey = D / 8;                  // 16-byte pieces per key row
    constexpr int kKeysPerWarp = 32 / kLanesPerKey;      // key rows one warp load covers
    constexpr int kWarps = kDecodeThreads / 32;
    constexpr int kGroups = kWarps * kKeysPerWarp;       // lane groups per CTA, one key each per step
    constexpr int U = kDecodeUnroll;

    __shared__ float sm_m[kGroups];
    __shared__ float sm_l[kGroups];
    __shared__ __align__(16) float sm_acc[kGroups][D];

    const int num_splits = p.num_splits;
    const int bh = blockIdx.x / num_splits;
    const int s = blockIdx.x % num_splits;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int sub = lane % kLanesPerKey;                  // which 8 elements of the row
    const int gw = lane / kLanesPerKey;                   // lane group within the warp
    const int g = warp * kKeysPerWarp + gw;
    int seq_len, part;
    if constexpr (PAGED) {
        const int cap = p.max_blocks << p.log2_bs;
        seq_len = p.seq_lens[bh / p.H];
        seq_len = seq_len < 0 ? 0 : (seq_len > cap ? cap : seq_len);
        part = (seq_len + num_splits - 1) / num_splits;
    } else {
        seq_len = p.Sk;
        part = p.keys_per_split;
    }
    const int k_lo = s * part;
    const int k_hi = min(k_lo + part, seq_len);

    float qf[8];
    unpack8<BF16>(*reinterpret_cast<const uint4 *>(p.q + static_cast<size_t>(bh) * D + sub * 8), qf);
#pragma unroll
    for (int e = 0; e < 8; ++e) qf[e] *= p.scale_log2;  // scores in base-2 units

    // address of row `key` of this head (dense), or nullptr offset semantics for a bad page (paged)
    const int b = bh / p.H, h = bh % p.H;
    const int *bt = PAGED ? p.block_table + static_cast<size_t>(b) * p.max_blocks : nullptr;
    // Paged: the partition's slice of the block table is staged in shared
    // memory once, so no key waits for a dependent table load before its K
    // and V loads; a slice longer than the buffer is read from global memory.
    constexpr int kTableSlots = PAGED ? 512 : 1;
    __shared__ int sm_table[kTableSlots];
    int blk_lo = 0;
    bool staged = false;
    if constexpr (PAGED) {
        if (k_lo < k_hi) {
            blk_lo = k_lo >> p.log2_bs;
            const int n_ent = ((k_hi - 1) >> p.log2_bs) - blk_lo + 1;
            staged = n_ent <= kTableSlots;  // uniform across the CTA
            if (staged)
                for (int i = threadIdx.x; i < n_ent; i += kDecodeThreads) sm_table[i] = bt[blk_lo + i];
        }
        __syncthreads();
    }
    auto row_offset = [&](int key, bool &ok) -> size_t {
        if constexpr (PAGED) {
            const int blk = staged ? sm_table[(key >> p.log2_bs) - blk_lo] : bt[key >> p.log2_bs];
            ok = static_cast<unsigned>(blk) < static_cast<unsigned>(p.num_blocks);
            const int blk_safe = ok ? blk : 0;
            return ((static_cast<size_t>(blk_safe) * p.H + h) << p.log2_bs | (key & ((1 << p.log2_bs) - 1))) * D;
        } else {
            ok = true;
            return (static_cast<size_t>(bh) * p.Sk + key) * D;
        }
    };
    const uint16_t *kb = p.k + sub * 8;
    const uint16_t *vb = p.v + sub * 8;
    float m = -CUDART_INF_F, l = 0.f;
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
    bool bad_page = false;

    // The trip count depends on the warp only (never on the lane group), so every
    // lane reaches every shuffle below; keys past k_hi are predicated off.
    for (int base = k_lo + warp * kKeysPerWarp; base < k_hi; base += kGroups * U) {
        const int key0 = base + gw;
        uint4 kr[U], vr[U];
        bool valid[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int key = key0 + u * kGroups;
            bool ok = false;
            size_t off = 0;
            if (key < k_hi) {
                off = row_offset(key, ok);
                bad_page |= !ok;
            }
            valid[u] = ok;
            if (ok) {
                kr[u] = ldg_stream(kb + off);
                vr[u] = ldg_stream(vb + off);
            } else {
                kr[u] = make_uint4(0, 0, 0, 0);
                vr[u] = make_uint4(0, 0, 0, 0);
            }
        }
        float sc[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            float kf[8];
            unpack8<BF16>(kr[u], kf);
            float d = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) d = fmaf(qf[e], kf[e], d);
            // butterfly over the lanes of one key row: every lane ends with the same bits
#pragma unroll
            for (int off = kLanesPerKey / 2; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
            sc[u] = valid[u] ? d : -CUDART_INF_F;
        }
        float mx = sc[0];
#pragma unroll
        for (int u = 1; u < U; ++u) mx = fmaxf(mx, sc[u]);
        const float m_new = fmaxf(m, mx);
        const float m_sub = (m_new == -CUDART_INF_F) ? 0.f : m_new;
        const float alpha = ptx::ex2(m - m_sub);
        l *= alpha;
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] *= alpha;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const float pu = ptx::ex2(sc[u] - m_sub);
            l += pu;
            float vf[8];
            unpack8<BF16>(vr[u], vf);
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = fmaf(pu, vf[e], acc[e]);
        }
        m = m_new;
    }
    if (PAGED && bad_page) atomicExch(p.err, kDeviceErrBadIndex);

    // merge the lane groups of this CTA (same log-sum-exp rule as phase 2)
    if (sub == 0) {
        sm_m[g] = m;
        sm_l[g] = l;
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) sm_acc[g][sub * 8 + e] = acc[e];
    __syncthreads();
    for (int d = threadIdx.x; d < D; d += kDecodeThreads) {
        float M = -CUDART_INF_F;
#pragma unroll
        for (int i = 0; i < kGroups; ++i) M = fmaxf(M, sm_m[i]);
        float L = 0.f, O = 0.f;
        if (M != -CUDART_INF_F) {
#pragma unroll
            for (int i = 0; i < kGroups; ++i) {
                const float w = ptx::ex2(sm_m[i] - M);
                L = fmaf(w, sm_l[i], L);
                O = fmaf(w, sm_acc[i][d], O);
            }
        }
        const size_t ps = static_cast<size_t>(bh) * num_splits + s;
        p.o_part[ps * D + d] = O;
        if (d == 0) {
            p.m_part[ps] = (M == -CUDART_INF_F) ? -CUDART_INF_F : M * 0.69314718055994531f;
            p.l_part[ps] = L;
        }
    }
    if constexpr (FUSED) {
        // Count this partition done once its partials are visible device-wide;
        // the last one of the head merges it and re-arms the counter.
        __shared__ int is_last;
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0) is_last = atomicAdd(p.counters + bh, 1) == num_splits - 1;
        __syncthreads();
        if (is_last) {
            __threadfence();
            merge_head<D, BF16, kDecodeThreads>(p.o_part, p.m_part, p.l_part, static_cast<uint16_t *>(p.o), p.lse,
                                                bh, num_splits);
            if (threadIdx.x == 0) p.counters[bh] = 0;
        }
    }
}

// Phase 2 as its own launch: one CTA per head.
constexpr int kMergeThreads = 256;

template <int D, bool BF16>
__global__ void __launch_bounds__(kMergeThreads)
    fa_splitkv_merge_kernel(const float *__restrict__ o_part, const float *__restrict__ m_part,
                            const float *__restrict__ l_part, uint16_t *__restrict__ o, float *__restrict__ lse,
                            int num_splits) {
    merge_head<D, BF16, kMergeThreads>(o_part, m_part, l_part, o, lse, static_cast<int>(blockIdx.x), num_splits);
}

template <int D, bool BF16, bool PAGED, bool FUSED>
static cudaError_t launch_split_t(const DecodeParams &p, int BH, cudaStream_t st) {
    const long long grid = static_cast<long long>(BH) * p.num_splits;
    fa_decode_split_kernel<D, BF16, PAGED, FUSED><<<static_cast<unsigned>(grid), kDecodeThreads, 0, st>>>(p);
    return cudaGetLastError();
}

template <bool PAGED, bool FUSED = false>
static cudaError_t launch_split_any(int D, bool bf16, const DecodeParams &p, int BH, cudaStream_t st) {
    if (D == 64 && !bf16) return launch_split_t<64, false, PAGED, FUSED>(p, BH, st);
    if (D == 64 && bf16) return launch_split_t<64, true, PAGED, FUSED>(p, BH, st);
    if (D == 128 && !bf16) return launch_split_t<128, false, PAGED, FUSED>(p, BH, st);
    if (D == 128 && bf16) return launch_split_t<128, true, PAGED, FUSED>(p, BH, st);
    return cudaErrorInvalidValue;
}

template <int D, bool BF16>
static cudaError_t launch_merge_t(const float *op, const float *mp, const float *lp, void *o, float *lse, int BH,
                                  int S, cudaStream_t st) {
    fa_splitkv_merge_kernel<D, BF16><<<BH, kMergeThreads, 0, st>>>(op, mp, lp, static_cast<uint16_t *>(o), lse, S);
    return cudaGetLastError();
}

cudaError_t launch_decode_split(int D, bool bf16, const void *q, const void *k, const void *v, float *o_part,
                                float *m_part, float *l_part, int BH, int Sk, int num_splits, int keys_per_split,
                                float scale_log2, cudaStream_t stream) {
    DecodeParams p{};
    p.q = static_cast<const uint16_t *>(q);
    p.k = static_cast<const uint16_t *>(k);
    p.v = static_cast<const uint16_t *>(v);
    p.o_part = o_part;
    p.m_part = m_part;
    p.l_part = l_part;
    p.H = 1;
    p.Sk = Sk;
    p.num_splits = num_splits;
    p.keys_per_split = keys_per_split;
    p.scale_log2 = scale_log2;
    return launch_split_any<false>(D, bf16, p, BH, stream);
}

cudaError_t launch_decode_split_paged(int D, bool bf16, const DecodeParams &p, int BH, cudaStream_t stream) {
    return launch_split_any<true>(D, bf16, p, BH, stream);
}

cudaError_t launch_decode_fused(int D, bool bf16, bool paged, const DecodeParams &p, int BH, cudaStream_t stream) {
    return paged ? launch_split_any<true, true>(D, bf16, p, BH, stream)
                 : launch_split_any<false, true>(D, bf16, p, BH, stream);
}

cudaError_t launch_splitkv_merge(int D, bool bf16, const float *o_part, const float *m_part, const float *l_part,
                                 void *o, float *lse, int BH, int num_splits, cudaStream_t stream) {
    if (D == 64 && !bf16) return launch_merge_t<64, false>(o_part, m_part, l_part, o, lse, BH, num_splits, stream);
    if (D == 64 && bf16) return launch_merge_t<64, true>(o_part, m_part, l_part, o, lse, BH, num_splits, stream);
    if (D == 128 && !bf16) return launch_merge_t<128, false>(o_part, m_part, l_part, o, lse, BH, num_splits, stream);
    if (D == 128 && bf16) return launch_merge_t<128, true>(o_part, m_part, l_part, o, lse, BH, num_splits, stream);
    return cudaErrorInvalidValue;
}

}  // namespace fa
