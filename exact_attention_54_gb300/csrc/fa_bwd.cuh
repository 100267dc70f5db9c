// FlashAttention-2 backward pass on sm_103a.
//
// Method ("Adaptive High-Performance Attention Kernels in CUDA", Advanced
// Production Features 2, Custom CUDA Backward Pass): the N x N probability
// matrix is never stored. S = scale Q K^T and P = exp(S - LSE) are recomputed
// tile by tile from the forward pass's per-row LSE, D_i = sum_k dO_ik O_ik is
// precomputed, and dS = P (dP - D_i) with dP = dO V^T. The gradients follow by
// the chain rule: dV = P^T dO, dK = scale dS^T Q, dQ = scale dS K.
//
// Three launches:
//   fa_bwd_prep_kernel  per query row: D_i, the LSE in base 2 (padded to whole
//                       128-row tiles with +inf, which zeroes P there), and a
//                       zeroed fp32 dQ accumulator row.
//   fa_bwd_d64_kernel   (D = 64) one CTA per (head, 128-key tile), looping
//                       over the query tiles that see those keys (causal:
//                       from the diagonal on). Per query tile, on the tensor
//                       core:
//                         S^T  = K Q^T     (TMEM, lanes = keys)
//                         dP^T = V dO^T    (TMEM)
//                       the key-row warps turn them into P^T (16-bit, back into
//                       TMEM over S^T) and dS^T (16-bit, shared memory, in the
//                       128-byte-swizzled layout a TMA load would produce), then
//                         dV  += P^T dO    (P^T from TMEM, dO MN-major)
//                         dK  += dS^T Q    (dS^T K-major, Q MN-major)
//                         dQ_t = dS K      (dS^T read as an MN-major A operand)
//                       dV and dK run chunk by chunk (32 queries) as the key-row
//                       work publishes them; dQ_t follows; the query-row warps move it to
//                       registers (releasing its TMEM columns), then into the
//                       step's Q/dO stage once dV and dK are done with it, and
//                       warp 3 adds the staged tile to the fp32 accumulator
//                       with TMA bulk tensor reductions. dK and dV stay in
//                       TMEM for the whole loop and are written once.
//   fa_bwd_kernel       (D = 128) the same products on 64-query sub-steps with
//                       two TMEM buffers, so that the key-row work of one
//                       sub-step overlaps the tensor core's products of the
//                       next; described where it is defined below.
//   fa_bwd_dq_kernel    dQ = scale * accumulator, in the input dtype.
//
// Roles of fa_bwd_d64_kernel (384 threads): warp 0 TMA producer (K, V once; Q and
// dO double-buffered), warp 1 MMA issuer and TMEM owner, warp 3 bulk
// reductions of dQ_t, warps 4..11 two warpgroups that split every step by
// halves: warpgroup h computes P^T and dS^T for queries [64h, 64h+64) of each
// key row, then stages dQ_t columns [h D/2, (h+1) D/2) of each query row, and
// writes that column half of dK and dV at the end. P^T of half h sits in S^T
// columns [64h, 64h+32). TMEM columns: S^T [0,128), dP^T and then dQ_t
// [128,256), dV [256, 256+D), dK [256+D, 256+2D).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include <cstdint>

#include "fa_launch.h"
#include "sm103_ptx.cuh"

namespace fa {
namespace bwd {

constexpr int kBlock = 128;  // keys per work item and queries per inner step
constexpr int kThreads = 384;

template <int D>
struct Shape {
    static_assert(D == 64 || D == 128, "head dim");
    static constexpr int kColBlocks = D / 64;
    static constexpr int kBoxBytes = 128 * 128;         // 128 rows x 64 columns of 16-bit values
    static constexpr int kTileBytes = kBlock * D * 2;   // one 128-row tile of Q, K, V or dO
    static constexpr int kOffK = 0;
    static constexpr int kOffV = kOffK + kTileBytes;
    static constexpr int kOffQ = kOffV + kTileBytes;    // + s * tile, s = 0, 1
    static constexpr int kOffDO = kOffQ + 2 * kTileBytes;
    static constexpr int kOffDS = kOffDO + 2 * kTileBytes;  // dS^T [128 keys][128 queries], 2 boxes
    static constexpr int kTilesBytes = kOffDS + 2 * kBoxBytes;
    // The small region (barriers, TMEM base, abort flag, the step's base-2 LSE
    // and D values) sits at the start of the allocation, in front of the
    // 1024-aligned tiles, so it reuses the alignment slack.
    static constexpr int kOffBar = 0;
    static constexpr int kKVFull = 0;
    static constexpr int kQFull = 1;    // +s
    static constexpr int kQEmpty = 3;   // +s
    static constexpr int kSFull = 5;    // S^T and dP^T written (MMA commit)
    static constexpr int kPChunk = 6;   // +c: P^T and dS^T of queries [32c, 32c+32) written (4 warps)
    static constexpr int kDQFull = 10;  // dQ_t in TMEM (MMA commit)
    static constexpr int kDQFree = 11;  // dQ_t read out (8 warps)
    static constexpr int kDSFree = 12;  // dS^T no longer read (MMA commit after dQ_t)
    static constexpr int kStageReady = 13;  // dQ_t staged in the step's Q/dO buffers (8 warps)
    static constexpr int kStageFree = 14;   // +s: the bulk reduction has read stage s (1 thread)
    static constexpr int kLFull = 16;       // the step's LSE and D values are in shared memory (bulk copy)
    static constexpr int kTeardown = 17;
    static constexpr int kNumBars = 18;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kOffRows = 256;                     // float lse2[128], delta[128]
    static constexpr int kSmallBytes = kOffRows + 2 * 128 * 4;
    static_assert(kOffMisc + 16 <= kOffRows, "small region layout");
    // small region + worst-case padding to the next 1024-byte boundary + tiles
    static constexpr int kSmemBytes = kSmallBytes + 1024 + kTilesBytes;
    static constexpr uint32_t kTmemS = 0;
    static constexpr uint32_t kTmemDP = 128;
    static constexpr uint32_t kTmemDV = 256;
    static constexpr uint32_t kTmemDK = 256 + D;
    static constexpr uint32_t kTmemCols = 512;
    static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

template <bool BF16>
__device__ __forceinline__ float to_f32(uint16_t x) {
    if constexpr (BF16) return __uint_as_float(static_cast<uint32_t>(x) << 16);
    else return __half2float(__ushort_as_half(x));
}

// ------------------------------------------------------------- preprocess --

// Per query row of every head: D_i = sum_d dO_id O_id, the LSE in base 2 and
// a zeroed dQ accumulator row. Grid: x = chunks of kPrepRows rows, y and z =
// the head (dense: B*H index over [B*H][Sq_pad] row arrays; packed: head h
// over [H][total_q] row arrays, with O, dO and the accumulator laid out
// [total_q][H][D]). Dense rows past Sq get D = 0 and LSE = +inf. Each warp
// takes kPrepPasses groups of rows, all of its 16-byte loads in flight
// before the first sum; the D/8 lanes of a row reduce among themselves.
constexpr int kPrepPasses = 4;
template <int D>
constexpr int kPrepRows = 8 * (32 / (D / 8)) * kPrepPasses;  // rows per 256-thread block

template <int D, bool BF16, bool VARLEN>
__global__ void __launch_bounds__(256)
    fa_bwd_prep_kernel(const uint16_t *__restrict__ o, const uint16_t *__restrict__ dout,
                       const float *__restrict__ lse, const BwdParams p) {
    constexpr int kLanesPerRow = D / 8;              // 16-byte pieces of a 16-bit row
    constexpr int kRowsPerPass = 32 / kLanesPerRow;  // rows one warp instruction covers
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    // the main kernel may be launched now: it sets up its barriers and TMEM
    // and then waits for this grid to complete
    ptx::grid_launch_dependents();
    // the main kernel's work counter starts every call at zero
    if (blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && threadIdx.x == 0 && p.work_counter != nullptr)
        *p.work_counter = 0;
    const int z = static_cast<int>(blockIdx.z * gridDim.y + blockIdx.y);
    if (z >= (VARLEN ? p.H : p.BH)) return;
    const int rows = VARLEN ? p.total_q : p.Sq_pad;   // rows of one head's row arrays
    const int valid = VARLEN ? p.total_q : p.Sq;       // rows with O and dO
    const int sub = lane % kLanesPerRow, grp = lane / kLanesPerRow;
    const int r0 = static_cast<int>(blockIdx.x) * kPrepRows<D> + warp * kRowsPerPass * kPrepPasses + grp;
    uint4 ov[kPrepPasses], gv[kPrepPasses];
    size_t off[kPrepPasses];
#pragma unroll
    for (int i = 0; i < kPrepPasses; ++i) {
        const int r = r0 + i * kRowsPerPass;
        off[i] = (VARLEN ? static_cast<size_t>(r) * p.H + z : static_cast<size_t>(z) * p.Sq + r) * D + sub * 8;
        if (r < valid) {
            ov[i] = __ldcs(reinterpret_cast<const uint4 *>(o + off[i]));
            gv[i] = __ldcs(reinterpret_cast<const uint4 *>(dout + off[i]));
        } else {
            ov[i] = gv[i] = make_uint4(0u, 0u, 0u, 0u);
        }
    }
#pragma unroll
    for (int i = 0; i < kPrepPasses; ++i) {
        const int r = r0 + i * kRowsPerPass;
        const uint32_t a[4] = {ov[i].x, ov[i].y, ov[i].z, ov[i].w}, c[4] = {gv[i].x, gv[i].y, gv[i].z, gv[i].w};
        float acc = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            acc = fmaf(to_f32<BF16>(static_cast<uint16_t>(a[e] & 0xffffu)), to_f32<BF16>(static_cast<uint16_t>(c[e] & 0xffffu)), acc);
            acc = fmaf(to_f32<BF16>(static_cast<uint16_t>(a[e] >> 16)), to_f32<BF16>(static_cast<uint16_t>(c[e] >> 16)), acc);
        }
#pragma unroll
        for (int s = kLanesPerRow / 2; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
        if (r < valid) {
            float4 *acc_row = reinterpret_cast<float4 *>(p.dq_acc + off[i]);
            acc_row[0] = make_float4(0.f, 0.f, 0.f, 0.f);
            acc_row[1] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        if (sub == 0 && r < rows) {
            const size_t srow = static_cast<size_t>(z) * rows + r;
            if (r < valid) {
                p.delta[srow] = acc;
                p.lse2[srow] = lse[VARLEN ? srow : static_cast<size_t>(z) * p.Sq + r] * 1.4426950408889634f;
            } else {
                p.delta[srow] = 0.f;
                p.lse2[srow] = CUDART_INF_F;
            }
        }
    }
}

// ------------------------------------------------------------ postprocess --

template <bool BF16>
__global__ void __launch_bounds__(256) fa_bwd_dq_kernel(const float *__restrict__ acc, uint16_t *__restrict__ dq,
                                                        long long n8, float scale) {
    // launched as a dependent of the main kernel: its reductions must be complete
    ptx::grid_dependency_wait();
    const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= n8) return;
    const float4 a = reinterpret_cast<const float4 *>(acc)[2 * i];
    const float4 b = reinterpret_cast<const float4 *>(acc)[2 * i + 1];
    uint4 out;
    out.x = ptx::pack2<BF16>(a.x * scale, a.y * scale);
    out.y = ptx::pack2<BF16>(a.z * scale, a.w * scale);
    out.z = ptx::pack2<BF16>(b.x * scale, b.y * scale);
    out.w = ptx::pack2<BF16>(b.z * scale, b.w * scale);
    reinterpret_cast<uint4 *>(dq)[i] = out;
}

// ------------------------------------------------------------ main kernel --

// Work item of this CTA: key tile kt of head bh. Heads are taken a group at a
// time, and within a group the heavy causal key tiles (low kt) come first.
// Every CTA of a head re-reads its Q and dO and adds into its dQ accumulator,
// so running a few heads at once keeps that set (8 Sq D bytes per head)
// within L2 instead of streaming every head's through it at once.
__device__ __forceinline__ void bwd_work_at(const BwdParams &p, int w, int &kt, int &bh) {
    const int per_group = p.heads_per_group * p.n_ktiles;
    const int g = w / per_group;
    const int i = w % per_group;
    const int rest = p.BH - g * p.heads_per_group;
    const int g_heads = rest < p.heads_per_group ? rest : p.heads_per_group;
    kt = i / g_heads;
    bh = g * p.heads_per_group + i % g_heads;
}

// The unit of this CTA (one unit per CTA, in block order).
__device__ __forceinline__ void bwd_work(const BwdParams &p, int &kt, int &bh) {
    bwd_work_at(p, static_cast<int>(blockIdx.x), kt, bh);
}

// This CTA's key tile and what it needs of its unit: the unit's index (dense
// tensor maps), head, first query and key token and lengths (packed). A packed
// unit whose offsets do not lie inside the tensors, or whose lengths exceed
// the launch's maxima, is not ok.
struct BwdUnit {
    int kt;
    int z;         // dense: B*H index of the unit
    int hh;        // packed: head
    int tq0, tk0;  // packed: first query and key token of the sequence
    int Lq, Lk;
    bool ok;
};

template <bool VARLEN>
__device__ __forceinline__ BwdUnit bwd_unit_at(const BwdParams &p, int w) {
    BwdUnit u;
    int unit;
    bwd_work_at(p, w, u.kt, unit);
    if constexpr (VARLEN) {
        const int b = unit / p.H;
        u.z = 0;
        u.hh = unit % p.H;
        const int q0 = p.cu_q[b], q1 = p.cu_q[b + 1], k0 = p.cu_k[b], k1 = p.cu_k[b + 1];
        u.ok = !(q0 < 0 || q1 < q0 || q1 > p.total_q || q1 - q0 > p.Sq || k0 < 0 || k1 < k0 || k1 > p.total_k ||
                 k1 - k0 > p.Sk);
        u.tq0 = q0;
        u.tk0 = k0;
        u.Lq = u.ok ? q1 - q0 : 0;
        u.Lk = u.ok ? k1 - k0 : 0;
    } else {
        u.z = unit;
        u.hh = 0;
        u.tq0 = u.tk0 = 0;
        u.Lq = p.Sq;
        u.Lk = p.Sk;
        u.ok = true;
    }
    return u;
}

template <bool VARLEN>
__device__ __forceinline__ BwdUnit bwd_unit(const BwdParams &p) {
    return bwd_unit_at<VARLEN>(p, static_cast<int>(blockIdx.x));
}

// Tensor-map coordinates (y, z) of row `row` of the unit's queries or keys:
// dense maps are {D, S, B*H}, packed maps {D, H, tokens}.
template <bool VARLEN>
__device__ __forceinline__ void unit_coords(const BwdUnit &u, bool keys, int row, int &y, int &z) {
    if constexpr (VARLEN) {
        y = u.hh;
        z = (keys ? u.tk0 : u.tq0) + row;
    } else {
        y = row;
        z = u.z;
    }
}

// Packed sequences: the per-row values (base-2 LSE, D_i) of query rows
// [q0, q0 + n) of the unit, read by the calling warp into shared memory at
// `dst` (LSE at dst, D_i at dst + n floats); rows past the sequence get
// LSE = +inf and D_i = 0, which zero P and dS there. Then one arrival on `bar`.
template <int n>
__device__ __forceinline__ void load_rows_packed(const BwdParams &p, const BwdUnit &u, int q0, float *dst,
                                                 uint32_t bar, bool leader) {
    const float *l = p.lse2 + static_cast<size_t>(u.hh) * p.total_q + u.tq0;
    const float *d = p.delta + static_cast<size_t>(u.hh) * p.total_q + u.tq0;
#pragma unroll
    for (int i = threadIdx.x % 32; i < n; i += 32) {
        const int r = q0 + i;
        dst[i] = r < u.Lq ? l[r] : CUDART_INF_F;
        dst[n + i] = r < u.Lq ? d[r] : 0.f;
    }
    __syncwarp();
    if (leader) ptx::bar_arrive(bar);
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr)
                 : "memory");
    return v;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// 128 rows starting at `row0` of head `bh`, all 64-column boxes, into `dst`.
template <int D>
__device__ __forceinline__ void load_tile(const CUtensorMap *tm, uint32_t dst, uint32_t bar, int row0, int bh) {
#pragma unroll
    for (int c = 0; c < D / 64; ++c) ptx::tma_load_3d(dst + c * Shape<D>::kBoxBytes, tm, bar, c * 64, row0, bh);
}

template <int D, bool BF16, bool CAUSAL, bool VARLEN>
__global__ void __launch_bounds__(kThreads, 1)
    fa_bwd_d64_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                  const __grid_constant__ CUtensorMap tm_dq, const BwdParams p) {
    using S = Shape<D>;
    extern __shared__ __align__(16) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + S::kSmallBytes + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = ptx::smem_addr(smem);     // 1024-aligned tiles
    const uint32_t ssmall = ptx::smem_addr(smem_raw);  // barriers, misc, row values
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem_raw + S::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem_raw + S::kOffMisc + 4);
    const float *rows_lse = reinterpret_cast<const float *>(smem_raw + S::kOffRows);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t bars = ssmall + S::kOffBar;
    auto bar = [&](int i) { return bars + 8u * static_cast<uint32_t>(i); };
    auto wait = [&](int i, uint32_t parity) {
        return __all_sync(0xffffffffu, ptx::bar_wait(bar(i), parity, abort_flag, p.timeout_ns));
    };

    // work item: key tile kt of a head (dense) or of a sequence's head (packed)
    const BwdUnit u = bwd_unit<VARLEN>(p);
    if constexpr (VARLEN) {
        // packed: offsets outside the tensors are reported and skipped; a
        // key tile past the sequence's keys has nothing to compute or write
        if (!u.ok) {
            if (threadIdx.x == 0) atomicExch(p.err, kDeviceErrSeqLens);
            return;
        }
        if (u.kt * kBlock >= u.Lk) return;
    }
    const int kt = u.kt;
    const int k0 = kt * kBlock;
    const int qt0 = CAUSAL ? kt : 0;  // first query tile that sees any of these keys
    const int n_qt = (u.Lq + kBlock - 1) / kBlock;
    const int n = n_qt > qt0 ? n_qt - qt0 : 0;
    // 128 rows of the unit's queries (keys = false) or keys, every 64-column box
    auto load_rows = [&](const CUtensorMap *tm, uint32_t dst, uint32_t bar_addr, int row0, bool keys) {
        int y, z;
        unit_coords<VARLEN>(u, keys, row0, y, z);
#pragma unroll
        for (int c = 0; c < D / 64; ++c) ptx::tma_load_3d(dst + c * S::kBoxBytes, tm, bar_addr, c * 64, y, z);
    };

    if (threadIdx.x == 0) {
        for (int i = 0; i < S::kNumBars; ++i) {
            uint32_t count = 1;                                              // MMA commits, TMA
            if (i >= S::kPChunk && i < S::kPChunk + 4) count = kBlock / 32;  // the owning warpgroup
            if (i == S::kDQFree || i == S::kStageReady) count = 2 * kBlock / 32;
            ptx::bar_init(bar(i), count);
        }
        *abort_flag = 0;
        ptx::bar_init_fence();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&tm_q);
        ptx::prefetch_tmap(&tm_k);
        ptx::prefetch_tmap(&tm_v);
        ptx::prefetch_tmap(&tm_do);
        ptx::prefetch_tmap(&tm_dq);
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_addr(tmem_slot), S::kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0 && n > 0) {
        // ---- TMA producer ----
        const bool leader = ptx::elect_one();
        if (leader) {
            ptx::bar_arrive_expect_tx(bar(S::kKVFull), 2 * S::kTileBytes);
            load_rows(&tm_k, sbase + S::kOffK, bar(S::kKVFull), k0, true);
            load_rows(&tm_v, sbase + S::kOffV, bar(S::kKVFull), k0, true);
        }
        int nq = 0, nl = 0;  // Q/dO steps and row-value steps loaded
        for (int it = 0; it < n; ++it) {
            const int s = it & 1;
            // stage s is free once the bulk reduction of step it-2 has read it
            if (it >= 2 && !wait(S::kStageFree + s, ((it >> 1) - 1) & 1)) break;
            const int q0 = (qt0 + it) * kBlock;
            if (leader && !withheld(p.withhold, static_cast<uint32_t>(it))) {
                ptx::bar_arrive_expect_tx(bar(S::kQFull + s), 2 * S::kTileBytes);
                load_rows(&tm_q, sbase + S::kOffQ + s * S::kTileBytes, bar(S::kQFull + s), q0, false);
                load_rows(&tm_do, sbase + S::kOffDO + s * S::kTileBytes, bar(S::kQFull + s), q0, false);
            }
            ++nq;
            // the single row-value buffer is free once every compute warp has
            // finished the previous step's P^T and dS^T (its four chunks)
            if (it >= 1) {
                bool got = true;
                for (int c = 0; c < 4 && got; ++c) got = wait(S::kPChunk + c, (it - 1) & 1);
                if (!got) break;
            }
            if constexpr (VARLEN) {
                load_rows_packed<128>(p, u, q0, reinterpret_cast<float *>(smem_raw + S::kOffRows), bar(S::kLFull),
                                      leader);
            } else if (leader) {
                const size_t ro = static_cast<size_t>(u.z) * p.Sq_pad + q0;
                ptx::bar_arrive_expect_tx(bar(S::kLFull), 2 * 128 * 4);
                ptx::bulk_load(ssmall + S::kOffRows, p.lse2 + ro, 128 * 4, bar(S::kLFull));
                ptx::bulk_load(ssmall + S::kOffRows + 128 * 4, p.delta + ro, 128 * 4, bar(S::kLFull));
            }
            ++nl;
        }
        // never leave with copies in flight
        ptx::bar_wait(bar(S::kKVFull), 0, nullptr, p.timeout_ns);
        if (nl > 0) ptx::bar_wait(bar(S::kLFull), (nl - 1) & 1, nullptr, p.timeout_ns);
        for (int s = 0; s < 2 && s < nq; ++s) {
            const int last = (nq - 1) - ((nq - 1 - s) % 2);
            ptx::bar_wait(bar(S::kQFull + s), (last >> 1) & 1, nullptr, p.timeout_ns);
        }
    } else if (warp == 1 && n > 0) {
        // ---- MMA issuer ----
        const bool leader = ptx::elect_one();
        constexpr uint32_t kIdS = ptx::idesc_f16(BF16, kBlock, kBlock, false);    // S^T, dP^T
        constexpr uint32_t kIdKV = ptx::idesc_f16(BF16, kBlock, D, true);         // dV, dK: B MN-major
        constexpr uint32_t kIdQ = ptx::idesc_f16(BF16, kBlock, D, true, true);    // dQ: A and B MN-major
        constexpr uint64_t kBox16 = S::kBoxBytes >> 4, kTile16 = S::kTileBytes >> 4, kRows16 = 2048 >> 4;
        const uint64_t k_kmaj = ptx::smem_desc_sw128(sbase + S::kOffK, 16, 1024);
        const uint64_t v_kmaj = ptx::smem_desc_sw128(sbase + S::kOffV, 16, 1024);
        const uint64_t q_kmaj = ptx::smem_desc_sw128(sbase + S::kOffQ, 16, 1024);
        const uint64_t do_kmaj = ptx::smem_desc_sw128(sbase + S::kOffDO, 16, 1024);
        const uint64_t q_mn = ptx::smem_desc_sw128(sbase + S::kOffQ, S::kBoxBytes, 1024);
        const uint64_t do_mn = ptx::smem_desc_sw128(sbase + S::kOffDO, S::kBoxBytes, 1024);
        const uint64_t k_mn = ptx::smem_desc_sw128(sbase + S::kOffK, S::kBoxBytes, 1024);
        const uint64_t ds_kmaj = ptx::smem_desc_sw128(sbase + S::kOffDS, 16, 1024);
        const uint64_t ds_mn = ptx::smem_desc_sw128(sbase + S::kOffDS, S::kBoxBytes, 1024);
        bool ok = wait(S::kKVFull, 0);
        for (int it = 0; it < n && ok; ++it) {
            const int s = it & 1;
            if (!(ok = wait(S::kQFull + s, (it >> 1) & 1))) break;
            const uint64_t st = static_cast<uint64_t>(s) * kTile16;
            // S^T = K Q^T into [0,128): the previous P^T was consumed by the
            // dV MMA issued before this one.
            if (leader) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t off = (kk / 4) * kBox16 + (kk % 4) * 2;
                    ptx::mma_ss(tmem + S::kTmemS, k_kmaj + off, q_kmaj + st + off, kIdS, kk > 0);
                }
            }
            // dP^T = V dO^T into [128,256), once the last dQ_t there is read
            if (it > 0 && !(ok = wait(S::kDQFree, (it - 1) & 1))) break;
            ptx::tc_fence_after();
            if (leader) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t off = (kk / 4) * kBox16 + (kk % 4) * 2;
                    ptx::mma_ss(tmem + S::kTmemDP, v_kmaj + off, do_kmaj + st + off, kIdS, kk > 0);
                }
                ptx::mma_commit(bar(S::kSFull));
            }
            // dV += P^T dO and dK += dS^T Q contract over the queries: each
            // 32-query chunk goes to the tensor core as soon as its warps have
            // published it, overlapping the rest of the key-row work. P^T of
            // queries [0,64) sits in columns [0,32), of [64,128) in [64,96).
            for (int c = 0; c < 4 && ok; ++c) {
                if (!(ok = wait(S::kPChunk + c, it & 1))) break;
                ptx::tc_fence_after();
                if (leader) {
#pragma unroll
                    for (int k2 = 0; k2 < 2; ++k2) {
                        const int kk = 2 * c + k2;
                        ptx::mma_ts(tmem + S::kTmemDV, tmem + S::kTmemS + kk * 8 + (kk >= 4 ? 32 : 0),
                                    do_mn + st + kk * kRows16, kIdKV, (it > 0 || kk > 0) ? 1u : 0u);
                        const uint64_t off = (kk / 4) * kBox16 + (kk % 4) * 2;
                        ptx::mma_ss(tmem + S::kTmemDK, ds_kmaj + off, q_mn + st + kk * kRows16, kIdKV,
                                    (it > 0 || kk > 0) ? 1u : 0u);
                    }
                }
            }
            if (!ok) break;
            if (leader) {
                ptx::mma_commit(bar(S::kQEmpty + s));  // Q and dO of this step have all their readers
                // dQ_t = dS K (over the keys: needs every chunk) into [128,256),
                // where dP^T was consumed by the key-row warps
#pragma unroll
                for (int kk = 0; kk < kBlock / 16; ++kk)
                    ptx::mma_ss(tmem + S::kTmemDP, ds_mn + kk * kRows16, k_mn + kk * kRows16, kIdQ, kk > 0);
                ptx::mma_commit(bar(S::kDQFull));
                ptx::mma_commit(bar(S::kDSFree));
            }
        }
        if (leader) ptx::mma_commit(bar(S::kTeardown));
        __syncwarp();
        ptx::bar_wait(bar(S::kTeardown), 0, nullptr, p.timeout_ns);
    } else if (warp >= 4) {
        // ---- compute warps: warpgroup h = 0, 1 owns queries [64h, 64h+64)
        // of every key row (P^T, dS^T), then dQ_t columns [h D/2, (h+1) D/2)
        // of every query row (to registers, releasing the TMEM columns, then
        // staged into the step's Q/dO buffers for warp 3's bulk reductions),
        // and at the end columns [h D/2, (h+1) D/2) of dK and dV. ----
        const int wq = warp % 4;       // TMEM lane quarter
        const int h = (warp - 4) / 4;
        const int r = wq * 32 + lane;  // key row (P^T, dS^T, epilogue) or query row (dQ_t)
        const int key = k0 + r;
        const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
        const uint32_t ds_row = sbase + S::kOffDS + (r >> 3) * 1024 + (r & 7) * 128;
        const uint32_t row_off = (r >> 3) * 1024 + (r & 7) * 128;
        bool ok = true;
        for (int it = 0; it < n; ++it) {
            const int s = it & 1;
            const int q0 = (qt0 + it) * kBlock;
            // the step's LSE and D values and the free dS^T buffer are ready
            // well before S^T and dP^T: wait for them first, so that only one
            // wait separates the tensor core's commit from the key-row work
            if (!(ok = wait(S::kLFull, it & 1))) break;
            if (it > 0 && !(ok = wait(S::kDSFree, (it - 1) & 1))) break;
            if (!(ok = wait(S::kSFull, it & 1))) break;
            ptx::tc_fence_after();
#pragma unroll 1
            for (int cl = 0; cl < 2; ++cl) {
                const int c = 2 * h + cl;  // 32-query chunk of the tile
                uint32_t sv[32], dpv[32];
                ptx::tmem_ld32(tmem + lane_base + S::kTmemS + 32 * c, sv);
                ptx::tmem_ld32(tmem + lane_base + S::kTmemDP + 32 * c, dpv);
                ptx::tmem_ld_wait();
                ptx::reg_fence(sv);
                ptx::reg_fence(dpv);
                const int qc = q0 + 32 * c;
                const bool need_mask = (CAUSAL && key > qc) || key >= u.Lk;
                // queries j < lo of the chunk do not see this key (causal: a
                // key is seen from its own position on; a key past Lk by none)
                const int lo = key >= u.Lk ? 32 : (CAUSAL ? key - qc : 0);
                uint32_t pp[16], dd[16];
                const float4 *lq = reinterpret_cast<const float4 *>(rows_lse + 32 * c);
                const float4 *dq4 = reinterpret_cast<const float4 *>(rows_lse + 128 + 32 * c);
#pragma unroll
                for (int j = 0; j < 32; j += 2) {
                    // queries 32c + j, +1 of the tile (every lane reads the same address)
                    const float4 lv = lq[j / 4], dv4 = dq4[j / 4];
                    const float l0 = (j % 4 == 0) ? lv.x : lv.z, l1 = (j % 4 == 0) ? lv.y : lv.w;
                    const float d0 = (j % 4 == 0) ? dv4.x : dv4.z, d1 = (j % 4 == 0) ? dv4.y : dv4.w;
                    float e0 = ptx::ex2(fmaf(__uint_as_float(sv[j]), p.scale_log2, -l0));
                    float e1 = ptx::ex2(fmaf(__uint_as_float(sv[j + 1]), p.scale_log2, -l1));
                    if (need_mask) {
                        if (j < lo) e0 = 0.f;
                        if (j + 1 < lo) e1 = 0.f;
                    }
                    pp[j / 2] = ptx::pack2<BF16>(e0, e1);
                    dd[j / 2] = ptx::pack2<BF16>(e0 * (__uint_as_float(dpv[j]) - d0),
                                                 e1 * (__uint_as_float(dpv[j + 1]) - d1));
                }
                // P^T for queries [32c, 32c+32) goes to columns 64h + 16 cl: inside
                // this half's own S^T columns, which it has already read
                ptx::tmem_st16(tmem + lane_base + S::kTmemS + 64 * h + 16 * cl, pp);
                // dS^T row r, queries [32c, 32c+32): box c/2, 16-byte chunks 4(c%2)..+3, 128-byte swizzle
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const uint32_t chunk = static_cast<uint32_t>(((c & 1) * 4 + m) ^ (r & 7));
                    st_shared_v4(ds_row + (c >> 1) * S::kBoxBytes + chunk * 16, dd[4 * m], dd[4 * m + 1],
                                 dd[4 * m + 2], dd[4 * m + 3]);
                }
                // publish the chunk: the tensor core reads P^T (TMEM) and dS^T (smem) next
                ptx::tmem_st_wait();
                ptx::tc_fence_before();
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) ptx::bar_arrive(bar(S::kPChunk + c));
            }

            // dQ_t, this half's columns of query row r
            if (!(ok = wait(S::kDQFull, it & 1))) break;
            ptx::tc_fence_after();
            uint32_t v[D / 64][32];
#pragma unroll
            for (int c = 0; c < D / 64; ++c)
                ptx::tmem_ld32(tmem + lane_base + S::kTmemDP + h * (D / 2) + 32 * c, v[c]);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < D / 64; ++c) ptx::reg_fence(v[c]);
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::bar_arrive(bar(S::kDQFree));
            if (!(ok = wait(S::kQEmpty + s, (it >> 1) & 1))) break;  // Q and dO of this step have all their readers
#pragma unroll
            for (int c = 0; c < D / 64; ++c) {
                const int box_i = h * (D / 64) + c;  // 32-column box of the dQ_t tile
                // boxes [0, D/64) in the Q stage, the rest in the dO stage
                const uint32_t box =
                    sbase + (box_i < D / 64 ? S::kOffQ + s * S::kTileBytes + box_i * S::kBoxBytes
                                            : S::kOffDO + s * S::kTileBytes + (box_i - D / 64) * S::kBoxBytes);
#pragma unroll
                for (int m = 0; m < 8; ++m)
                    st_shared_v4(box + row_off + ((m ^ (r & 7)) * 16), v[c][4 * m], v[c][4 * m + 1], v[c][4 * m + 2],
                                 v[c][4 * m + 3]);
            }
            ptx::fence_proxy_async_smem();  // the bulk reduction reads the stage next
            __syncwarp();
            if (lane == 0) ptx::bar_arrive(bar(S::kStageReady));
        }
        // epilogue: columns [h D/2, (h+1) D/2) of dV and scale * dK for this key row
        if (ok && n > 0) {
            ok = wait(S::kDSFree, (n - 1) & 1);  // the last dV and dK of the loop are done
            ptx::tc_fence_after();
        }
        // The TMEM loads are warp-collective (.sync.aligned): every lane runs
        // them; only the global stores are limited to keys that exist.
        if (ok) {
            const bool row_valid = key < u.Lk;
            const size_t row_g = (VARLEN ? (static_cast<size_t>(u.tk0) + key) * p.H + u.hh
                                         : static_cast<size_t>(u.z) * p.Sk + key) * D + h * (D / 2);
            const uint64_t once = ptx::l2_policy_evict_first();
            // 32-byte stores when both outputs are 32-byte aligned
            const bool v8 = ((reinterpret_cast<uintptr_t>(p.dk) | reinterpret_cast<uintptr_t>(p.dv)) & 31) == 0;
#pragma unroll 1
            for (int t = 0; t < 2; ++t) {
                const float f = t == 0 ? 1.f : p.scale;
                uint16_t *dst = static_cast<uint16_t *>(t == 0 ? p.dv : p.dk) + row_g;
#pragma unroll 1
                for (int c = 0; c < D / 64; ++c) {
                    uint32_t w[32];
                    if (n > 0) {
                        ptx::tmem_ld32(tmem + lane_base + (t == 0 ? S::kTmemDV : S::kTmemDK) + h * (D / 2) + 32 * c,
                                       w);
                        ptx::tmem_ld_wait();
                        ptx::reg_fence(w);
                    } else {
#pragma unroll
                        for (int k = 0; k < 32; ++k) w[k] = 0u;
                    }
                    uint32_t pk[16];
#pragma unroll
                    for (int k = 0; k < 16; ++k)
                        pk[k] = ptx::pack2<BF16>(__uint_as_float(w[2 * k]) * f, __uint_as_float(w[2 * k + 1]) * f);
                    if (row_valid) {
                        // written once: evict first
                        uint4 *d4 = reinterpret_cast<uint4 *>(dst + 32 * c);
                        if (v8) {
                            ptx::st_global_v8_hint(d4, pk, once);
                            ptx::st_global_v8_hint(d4 + 2, pk + 8, once);
                        } else {
#pragma unroll
                            for (int k = 0; k < 4; ++k)
                                ptx::st_global_v4_hint(d4 + k, pk[4 * k], pk[4 * k + 1], pk[4 * k + 2],
                                                       pk[4 * k + 3], once);
                        }
                    }
                }
            }
        }
    } else if (warp == 3 && n > 0) {
        // ---- bulk reductions of the staged dQ_t into the accumulator ----
        const bool leader = ptx::elect_one();
        for (int it = 0; it < n; ++it) {
            const int s = it & 1;
            if (!wait(S::kStageReady, it & 1)) break;
            if (leader) {
                const int q0 = (qt0 + it) * kBlock;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    const uint32_t box = sbase + (c < D / 64 ? S::kOffQ + s * S::kTileBytes + c * S::kBoxBytes
                                                             : S::kOffDO + s * S::kTileBytes + (c - D / 64) * S::kBoxBytes);
                    int y, z;
                    unit_coords<VARLEN>(u, false, q0, y, z);
                    ptx::tma_reduce_add_3d(&tm_dq, box, 32 * c, y, z);  // rows past the tensor are clipped
                }
                ptx::bulk_commit();
                ptx::bulk_wait_read_all();  // the stage may be refilled now
                ptx::bar_arrive(bar(S::kStageFree + s));
            }
            __syncwarp();
        }
        if (leader) ptx::bulk_wait_all();  // the reductions themselves are complete
        __syncwarp();
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, S::kTmemCols);
    }
    if (threadIdx.x == 0 && *abort_flag) atomicExch(p.err, kDeviceErrTimeout);
}


// ------------------------------------------- main kernel, head dimension 128 --
//
// D = 128 runs the same products on 64-query sub-steps so that the tensor
// core and the key-row warps overlap: TMEM holds dV [0,128) and dK [128,256)
// plus two sub-step buffers b = 0, 1 at 256 + 128 b, each S^T (64 columns;
// P^T of queries [32h, 32h+32) packed over its own first 16) and dP^T (64
// columns, then dQ_t^T). While the key-row warps turn buffer b into P^T and
// dS^T, the tensor core already forms S^T and dP^T of the next sub-step in
// the other buffer. dQ_t is produced transposed, dQ_t^T = K^T dS^T (K read
// as an MN-major A operand, dS^T as an MN-major B operand), so its M side is
// the 128 head columns and no 64-row MMA is needed; each compute thread then
// owns one head column and stages it into the fp32 tile that warp 2 adds to
// the accumulator with TMA bulk tensor reductions.
//
// Roles (512 threads): warp 0 TMA producer (K, V once; Q and dO in a ring of
// 4 stages, the sub-step's LSE/D rows double-buffered), warps 1 and 3 MMA
// issuers (warp 1 also owns TMEM), warp 2 bulk reductions, warps 4..11 two
// warpgroups: warpgroup h handles queries [32h, 32h+32) of every sub-step
// (P^T, dS^T) and, at the end, head columns
// [64h, 64h+64) of dK and dV; warps 12..15 move each dQ_t^T out of TMEM
// (releasing the buffer for the next S^T/dP^T) and stage it, off the key-row
// warps' path, into the sub-step's own Q/dO stage once dV and dK are done with
// it; the stage is refilled only after the bulk reductions have read it.
constexpr int kThreadsQ64 = 512;

struct ShapeQ64 {
    static constexpr int D = 128;
    static constexpr int kQ = 64;                        // queries per sub-step
    static constexpr int kKTileBytes = kBlock * D * 2;   // K or V: 32 KB (2 boxes of 128 rows x 64 columns)
    static constexpr int kKBoxBytes = kBlock * 128;
    static constexpr int kQTileBytes = kQ * D * 2;       // Q_j or dO_j: 16 KB (2 boxes of 64 rows x 64 columns)
    static constexpr int kQBoxBytes = kQ * 128;
    static constexpr int kStages = 4;
    static constexpr int kStageBytes = 2 * kQTileBytes;  // Q_j then dO_j; later the sub-step's fp32 dQ_t tile
    static constexpr int kDSBytes = kBlock * kQ * 2;     // dS^T [128 keys][64 queries]: one 16 KB box
    static constexpr int kDQBoxBytes = kQ * 128;         // 64 query rows x 32 fp32 head columns
    static_assert(4 * kDQBoxBytes == kStageBytes, "the dQ_t tile fills its sub-step's stage");
    static constexpr int kOffK = 0;
    static constexpr int kOffV = kOffK + kKTileBytes;
    static constexpr int kOffQ = kOffV + kKTileBytes;    // + stage * kStageBytes
    static constexpr int kOffDS = kOffQ + kStages * kStageBytes;  // + b * kDSBytes
    static constexpr int kTilesBytes = kOffDS + 2 * kDSBytes;
    // small region: barriers, TMEM base and abort flag, then for sub-steps
    // j mod 2 the 64 base-2 LSE values and 64 D values
    static constexpr int kKVFull = 0;
    static constexpr int kQFull = 1;       // +stage: Q_j landed (TMA)
    static constexpr int kQEmpty = 5;      // +stage: dV_j and dK_j done with them (MMA commit)
    static constexpr int kSFull = 9;       // +b: S^T of the buffer written (MMA commit)
    static constexpr int kPFull = 11;      // +b: dS^T written (8 warps; P^T came earlier, on kPTFull)
    static constexpr int kDQFull = 13;     // +b: dQ_t^T written (MMA commit)
    static constexpr int kBufFree = 15;    // +b: dQ_t^T read out, the buffer's dP^T columns free (4 warps)
    static constexpr int kDSFree = 17;     // +b: products of the buffer done: dS^T no longer read (MMA commit)
    // The dQ warps may run up to a ring's length ahead of the reductions, so
    // the hand-off between them is per stage (a single barrier waited by
    // parity would alias phases two or more apart).
    static constexpr int kStageReady = 19; // +stage: dQ_t staged in its sub-step's stage (4 warps)
    // The fp32 dQ_t tile's boxes 0, 1 lie over Q_j and boxes 2, 3 over dO_j;
    // each half of the stage is refilled once the boxes over it are read.
    static constexpr int kStageFree = 23;  // +stage: the boxes over dO_j read (1 thread)
    static constexpr int kTeardown = 27;
    static constexpr int kPTFree = 28;     // +b: dV of the buffer done, its S^T columns free (MMA commit)
    static constexpr int kLFull = 30;      // +b: the sub-step's LSE and D values landed (bulk copy)
    static constexpr int kKVEmpty = 32;    // the unit's last products done: K and V may be replaced (MMA commit)
    static constexpr int kRing = 4;        // unit slots
    static constexpr int kUnitReady = 33;  // +slot: a unit published (warp 0)
    static constexpr int kUnitFree = 37;   // +slot: every role has read it (15 warps)
    // a unit's dK/dV written out of every key-row warp's staging block (8 warps)
    static constexpr int kStagingFree = 41;
    static constexpr int kPTFull = 42;     // +b: P^T written (8 warps): dV may start before dS^T is
    static constexpr int kDPFull = 44;     // +b: dP^T of the buffer written (MMA commit)
    static constexpr int kDOFull = 46;     // +stage: dO_j landed (TMA)
    static constexpr int kStageFreeQ = 50; // +stage: the boxes over Q_j read (1 thread)
    static constexpr int kNumBars = 54;
    static constexpr int kOffMisc = kNumBars * 8;
    static constexpr int kOffRows = 448;   // + b * 512: float lse2[64], delta[64]
    // + slot * 32: int {live, kt, z, hh, tq0, tk0, Lq, Lk} of a published unit
    static constexpr int kOffUnits = kOffRows + 2 * 2 * kQ * 4;
    static constexpr int kSmallBytes = kOffUnits + kRing * 32;
    static_assert(kOffMisc + 16 <= kOffRows, "small region layout");
    static constexpr int kSmemBytes = kSmallBytes + 1024 + kTilesBytes;
    static constexpr uint32_t kTmemDV = 0;
    static constexpr uint32_t kTmemDK = 128;
    static constexpr uint32_t kTmemBuf = 256;  // + 128 b: S^T [0,64), dP^T / dQ_t^T [64,128)
    static constexpr uint32_t kTmemCols = 512;
    static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

template <bool BF16, bool CAUSAL, bool VARLEN>
__global__ void __launch_bounds__(kThreadsQ64, 1)
    fa_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                  const __grid_constant__ CUtensorMap tm_dq, const BwdParams p) {
    using S = ShapeQ64;
    constexpr int D = S::D;
    extern __shared__ __align__(16) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + S::kSmallBytes + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = ptx::smem_addr(smem);
    const uint32_t ssmall = ptx::smem_addr(smem_raw);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem_raw + S::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem_raw + S::kOffMisc + 4);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    auto bar = [&](int i) { return ssmall + 8u * static_cast<uint32_t>(i); };
    auto wait = [&](int i, uint32_t parity) {
        return __all_sync(0xffffffffu, ptx::bar_wait(bar(i), parity, abort_flag, p.timeout_ns));
    };

    // Persistent: each CTA takes work units (key tile kt of a head, dense, or
    // of a sequence's head, packed; heavy causal tiles first) from a counter
    // until none is left. Warp 0 fetches a unit and publishes it in a ring of
    // unit slots that every role reads in turn; ring stages and buffers keep
    // their phases across units through one running sub-step count J, and
    // the next unit's K and V are loaded while the current unit's dK and dV
    // are written out. tests/test_bwd_barrier_protocol.py models this
    // protocol.
    if (threadIdx.x == 0) {
        for (int i = 0; i < S::kNumBars; ++i) {
            uint32_t count = 1;  // MMA commits, TMA, the reduction thread, warp 0
            if (i >= S::kPFull && i < S::kPFull + 2) count = 2 * kBlock / 32;  // the key-row warps
            if ((i >= S::kBufFree && i < S::kBufFree + 2) || (i >= S::kStageReady && i < S::kStageReady + S::kStages))
                count = kBlock / 32;  // dQ warps
            if (i == S::kTeardown) count = 2;  // one commit per MMA-issuing warp
            if (i >= S::kUnitFree && i < S::kUnitFree + S::kRing) count = kThreadsQ64 / 32 - 1;  // every warp but 0
            if (i == S::kStagingFree) count = 2 * kBlock / 32;  // the key-row warps
            if (i >= S::kPTFull && i < S::kPTFull + 2) count = 2 * kBlock / 32;  // the key-row warps
            ptx::bar_init(bar(i), count);
        }
        *abort_flag = 0;
        ptx::bar_init_fence();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&tm_q);
        ptx::prefetch_tmap(&tm_k);
        ptx::prefetch_tmap(&tm_v);
        ptx::prefetch_tmap(&tm_do);
        ptx::prefetch_tmap(&tm_dq);
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_addr(tmem_slot), S::kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // Launched as a dependent of the prep kernel: everything above overlaps
    // its tail; the work counter, row values and zeroed accumulator it writes
    // are read only after this wait. The dQ conversion launch may start.
    ptx::grid_dependency_wait();
    ptx::grid_launch_dependents();

    // A published unit as every role sees it; n: its 64-query sub-steps from
    // the first query that sees any of its keys.
    struct UnitView {
        bool live;  // false: no unit is left
        BwdUnit u;
        int k0, qs0, n;
    };
    // Unit slot i of this CTA: waits until warp 0 has published it, copies it
    // and releases the slot. False when the wait gave up.
    auto read_unit = [&](int i, UnitView &uv) -> bool {
        const int s = i % S::kRing;
        if (!wait(S::kUnitReady + s, (i / S::kRing) & 1)) return false;
        const volatile int *e = reinterpret_cast<const volatile int *>(smem_raw + S::kOffUnits + s * 32);
        uv.live = e[0] != 0;
        uv.u.kt = e[1];
        uv.u.z = e[2];
        uv.u.hh = e[3];
        uv.u.tq0 = e[4];
        uv.u.tk0 = e[5];
        uv.u.Lq = e[6];
        uv.u.Lk = e[7];
        uv.u.ok = true;
        uv.k0 = uv.u.kt * kBlock;
        uv.qs0 = CAUSAL ? uv.k0 : 0;
        uv.n = uv.u.Lq > uv.qs0 ? (uv.u.Lq - uv.qs0 + S::kQ - 1) / S::kQ : 0;
        __syncwarp();
        if (lane == 0) ptx::bar_arrive(bar(S::kUnitFree + s));
        return true;
    };

    if (warp == 0) {
        // ---- unit fetch and TMA producer ----
        const bool leader = ptx::elect_one();
        // K and V are read by this CTA only: evict them first, keep L2 for
        // the Q, dO and dQ accumulator rows the head's other CTAs reuse
        const uint64_t once = ptx::l2_policy_evict_first();
        int J = 0, wi = 0;   // sub-steps and units with work so far
        int nq = 0, nl = 0;  // Q/dO and row-value loads issued
        bool ok = true;
        for (int i = 0; ok; ++i) {
            const int s = i % S::kRing;
            // slot s held unit i - kRing until every role had read it
            if (i >= S::kRing && !(ok = wait(S::kUnitFree + s, ((i / S::kRing) - 1) & 1))) break;
            // the next unit with keys to handle; offsets outside the tensors
            // (packed) are reported and skipped
            BwdUnit u{};
            int w;
            for (;;) {
                int got = 0;
                if (lane == 0) got = atomicAdd(p.work_counter, 1);
                w = __shfl_sync(0xffffffffu, got, 0);
                if (w >= p.total_units) break;
                u = bwd_unit_at<VARLEN>(p, w);
                if constexpr (VARLEN) {
                    if (!u.ok) {
                        if (lane == 0) atomicExch(p.err, kDeviceErrSeqLens);
                        continue;
                    }
                    if (u.kt * kBlock >= u.Lk) continue;  // a key tile past the sequence's keys
                }
                break;
            }
            const bool live = w < p.total_units;
            if (lane == 0) {
                volatile int *e = reinterpret_cast<volatile int *>(smem_raw + S::kOffUnits + s * 32);
                e[0] = live ? 1 : 0;
                e[1] = u.kt;
                e[2] = u.z;
                e[3] = u.hh;
                e[4] = u.tq0;
                e[5] = u.tk0;
                e[6] = u.Lq;
                e[7] = u.Lk;
                ptx::bar_arrive(bar(S::kUnitReady + s));
            }
            __syncwarp();
            if (!live) break;
            const int k0 = u.kt * kBlock, qs0 = CAUSAL ? k0 : 0;
            const int n = u.Lq > qs0 ? (u.Lq - qs0 + S::kQ - 1) / S::kQ : 0;
            if (n == 0) continue;  // no query sees these keys: zero dK and dV only
            // K and V of the unit once the previous unit's products are done with theirs
            if (wi >= 1 && !(ok = wait(S::kKVEmpty, (wi - 1) & 1))) break;
            if (leader) {
                ptx::bar_arrive_expect_tx(bar(S::kKVFull), 2 * S::kKTileBytes);
                int ky, kz;
                unit_coords<VARLEN>(u, true, k0, ky, kz);
                for (int c = 0; c < 2; ++c) {
                    ptx::tma_load_3d_hint(sbase + S::kOffK + c * S::kKBoxBytes, &tm_k, bar(S::kKVFull), c * 64, ky,
                                          kz, once);
                    ptx::tma_load_3d_hint(sbase + S::kOffV + c * S::kKBoxBytes, &tm_v, bar(S::kKVFull), c * 64, ky,
                                          kz, once);
                }
            }
            ++wi;
            for (int j = 0; j < n; ++j, ++J) {
                const int st = J % S::kStages, b = J & 1;
                // each half of the stage held part of sub-step J-4's staged dQ_t
                // until its reductions read it: Q_J first (S^T needs it), then dO_J
                const int q0 = qs0 + j * S::kQ;
                const uint32_t qb = sbase + S::kOffQ + st * S::kStageBytes;
                int qy, qz;
                unit_coords<VARLEN>(u, false, q0, qy, qz);
                if (J >= S::kStages && !(ok = wait(S::kStageFreeQ + st, ((J / S::kStages) - 1) & 1))) break;
                if (leader && !withheld(p.withhold, static_cast<uint32_t>(J))) {
                    ptx::bar_arrive_expect_tx(bar(S::kQFull + st), S::kQTileBytes);
                    for (int c = 0; c < 2; ++c)
                        ptx::tma_load_3d(qb + c * S::kQBoxBytes, &tm_q, bar(S::kQFull + st), c * 64, qy, qz);
                }
                if (J >= S::kStages && !(ok = wait(S::kStageFree + st, ((J / S::kStages) - 1) & 1))) break;
                if (leader) {
                    ptx::bar_arrive_expect_tx(bar(S::kDOFull + st), S::kQTileBytes);
                    for (int c = 0; c < 2; ++c)
                        ptx::tma_load_3d(qb + S::kQTileBytes + c * S::kQBoxBytes, &tm_do, bar(S::kDOFull + st),
                                         c * 64, qy, qz);
                }
                ++nq;
                // row buffer b is free once the key-row warps are done with sub-step J-2
                if (J >= 2 && !(ok = wait(S::kPFull + b, ((J - 2) >> 1) & 1))) break;
                if constexpr (VARLEN) {
                    load_rows_packed<S::kQ>(p, u, q0,
                                            reinterpret_cast<float *>(smem_raw + S::kOffRows + b * 2 * S::kQ * 4),
                                            bar(S::kLFull + b), leader);
                } else if (leader) {
                    const uint32_t rows = ssmall + S::kOffRows + b * 2 * S::kQ * 4;
                    const size_t ro = static_cast<size_t>(u.z) * p.Sq_pad + q0;
                    ptx::bar_arrive_expect_tx(bar(S::kLFull + b), 2 * S::kQ * 4);
                    ptx::bulk_load(rows, p.lse2 + ro, S::kQ * 4, bar(S::kLFull + b));
                    ptx::bulk_load(rows + S::kQ * 4, p.delta + ro, S::kQ * 4, bar(S::kLFull + b));
                }
                ++nl;
            }
        }
        // never leave with copies in flight
        if (wi > 0) ptx::bar_wait(bar(S::kKVFull), (wi - 1) & 1, nullptr, p.timeout_ns);
        for (int st = 0; st < S::kStages && st < nq; ++st) {
            const int last = (nq - 1) - ((nq - 1 - st) % S::kStages);
            ptx::bar_wait(bar(S::kQFull + st), (last / S::kStages) & 1, nullptr, p.timeout_ns);
            ptx::bar_wait(bar(S::kDOFull + st), (last / S::kStages) & 1, nullptr, p.timeout_ns);
        }
        for (int b = 0; b < 2 && b < nl; ++b) {
            const int last = (nl - 1) - ((nl - 1 - b) % 2);
            ptx::bar_wait(bar(S::kLFull + b), (last >> 1) & 1, nullptr, p.timeout_ns);
        }
    } else if (warp == 1 || warp == 3) {
        // ---- MMA issuers: warp 1 forms S^T and dP^T of each sub-step, warp 3
        // the products of the sub-step before it. A warp blocks in
        // tcgen05.mma while the tensor core's queue (a few MMAs) is full, so
        // one issuer alone starves the pipe at every barrier wait; with two,
        // one keeps the queue filled while the other waits. ----
        const bool leader = ptx::elect_one();
        constexpr uint32_t kIdS = ptx::idesc_f16(BF16, kBlock, S::kQ, false);        // S^T, dP^T: N = 64 queries
        constexpr uint32_t kIdKV = ptx::idesc_f16(BF16, kBlock, D, true);            // dV, dK: B MN-major
        constexpr uint32_t kIdQ = ptx::idesc_f16(BF16, D, S::kQ, true, true);       // dQ_t^T: A, B MN-major
        constexpr uint64_t kKBox16 = S::kKBoxBytes >> 4, kQBox16 = S::kQBoxBytes >> 4;
        constexpr uint64_t kStage16 = S::kStageBytes >> 4, kDS16 = S::kDSBytes >> 4, kRows16 = 2048 >> 4;
        int J = 0, wi = 0;  // sub-steps and units with work so far
        bool ok = true;
        if (warp == 1) {
            const uint64_t k_kmaj = ptx::smem_desc_sw128(sbase + S::kOffK, 16, 1024);
            const uint64_t v_kmaj = ptx::smem_desc_sw128(sbase + S::kOffV, 16, 1024);
            const uint64_t q_kmaj = ptx::smem_desc_sw128(sbase + S::kOffQ, 16, 1024);
            const uint64_t do_kmaj = ptx::smem_desc_sw128(sbase + S::kOffQ + S::kQTileBytes, 16, 1024);
            for (int i = 0; ok; ++i) {
              UnitView uv;
              if (!(ok = read_unit(i, uv)) || !uv.live) break;
              if (uv.n == 0) continue;
              if (!(ok = wait(S::kKVFull, wi & 1))) break;
              ++wi;
              for (int j = 0; j < uv.n && ok; ++j, ++J) {
                const int st = J % S::kStages, b = J & 1;
                // S^T: Q_J landed and the buffer's P^T of sub-step J-2 consumed by its dV
                const bool ready = ptx::bar_try_wait(bar(S::kQFull + st), (J / S::kStages) & 1) &&
                                   (J < 2 || ptx::bar_try_wait(bar(S::kPTFree + b), ((J - 2) >> 1) & 1));
                if (!__all_sync(0xffffffffu, ready)) {
                    if (!(ok = wait(S::kQFull + st, (J / S::kStages) & 1))) break;
                    if (J >= 2 && !(ok = wait(S::kPTFree + b, ((J - 2) >> 1) & 1))) break;
                }
                ptx::tc_fence_after();
                const uint64_t so = static_cast<uint64_t>(st) * kStage16;
                const uint32_t tb = tmem + S::kTmemBuf + 128 * b;
                if (leader) {
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint64_t ka = (kk / 4) * kKBox16 + (kk % 4) * 2;
                        const uint64_t qa = (kk / 4) * kQBox16 + (kk % 4) * 2;
                        ptx::mma_ss(tb, k_kmaj + ka, q_kmaj + so + qa, kIdS, kk > 0);
                    }
                    // the key-row warps exponentiate S^T while dP^T is formed
                    ptx::mma_commit(bar(S::kSFull + b));
                }
                // dP^T: dO_J landed and the buffer's dQ_t^T of sub-step J-2 read out
                if (!(ok = wait(S::kDOFull + st, (J / S::kStages) & 1))) break;
                if (J >= 2 && !(ok = wait(S::kBufFree + b, ((J - 2) >> 1) & 1))) break;
                ptx::tc_fence_after();
                if (leader) {
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint64_t ka = (kk / 4) * kKBox16 + (kk % 4) * 2;
                        const uint64_t qa = (kk / 4) * kQBox16 + (kk % 4) * 2;
                        ptx::mma_ss(tb + 64, v_kmaj + ka, do_kmaj + so + qa, kIdS, kk > 0);
                    }
                    ptx::mma_commit(bar(S::kDPFull + b));
                }
                __syncwarp();
              }
            }
        } else {
            const uint64_t k_mn = ptx::smem_desc_sw128(sbase + S::kOffK, S::kKBoxBytes, 1024);
            const uint64_t q_mn = ptx::smem_desc_sw128(sbase + S::kOffQ, S::kQBoxBytes, 1024);
            const uint64_t do_mn = ptx::smem_desc_sw128(sbase + S::kOffQ + S::kQTileBytes, S::kQBoxBytes, 1024);
            const uint64_t ds_kmaj = ptx::smem_desc_sw128(sbase + S::kOffDS, 16, 1024);
            const uint64_t ds_mn = ptx::smem_desc_sw128(sbase + S::kOffDS, S::kDSBytes, 1024);
            for (int i = 0; ok; ++i) {
              UnitView uv;
              if (!(ok = read_unit(i, uv)) || !uv.live) break;
              if (uv.n == 0) continue;
              // dQ_t^T reads K: the unit's K and V must have landed
              if (!(ok = wait(S::kKVFull, wi & 1))) break;
              ++wi;
              for (int j = 0; j < uv.n && ok; ++j, ++J) {
                const int st = J % S::kStages, b = J & 1;
                const uint64_t so = static_cast<uint64_t>(st) * kStage16;
                const uint32_t tb = tmem + S::kTmemBuf + 128 * b;
                // dV += P^T dO over the 64 queries (P^T of queries [32h, 32h+32)
                // in columns [32h, 32h+16) of the buffer) as soon as P^T is in:
                // it frees the buffer's S^T columns for sub-step J+2
                if (!(ok = wait(S::kPTFull + b, (J >> 1) & 1))) break;
                if (!(ok = wait(S::kDOFull + st, (J / S::kStages) & 1))) break;  // dV reads dO_J
                ptx::tc_fence_after();
                if (leader) {
#pragma unroll
                    for (int kk = 0; kk < S::kQ / 16; ++kk)
                        ptx::mma_ts(tmem + S::kTmemDV, tb + kk * 8 + (kk >= 2 ? 16 : 0), do_mn + so + kk * kRows16,
                                    kIdKV, (j > 0 || kk > 0) ? 1u : 0u);
                    ptx::mma_commit(bar(S::kPTFree + b));
                }
                __syncwarp();
                if (!(ok = wait(S::kPFull + b, (J >> 1) & 1))) break;
                ptx::tc_fence_after();
                if (leader) {
                    // dQ_t^T = K^T dS^T over the 128 keys, into the buffer's dP^T
                    // columns: its read-out frees them for sub-step J+2
#pragma unroll
                    for (int kk = 0; kk < kBlock / 16; ++kk)
                        ptx::mma_ss(tb + 64, k_mn + kk * kRows16, ds_mn + b * kDS16 + kk * kRows16, kIdQ, kk > 0);
                    ptx::mma_commit(bar(S::kDQFull + b));
                    // dK += dS^T Q
#pragma unroll
                    for (int kk = 0; kk < S::kQ / 16; ++kk)
                        ptx::mma_ss(tmem + S::kTmemDK, ds_kmaj + b * kDS16 + kk * 2, q_mn + so + kk * kRows16, kIdKV,
                                    (j > 0 || kk > 0) ? 1u : 0u);
                    ptx::mma_commit(bar(S::kQEmpty + st));  // Q_J and dO_J have all their readers
                    ptx::mma_commit(bar(S::kDSFree + b));   // and so has dS^T of buffer b
                }
                __syncwarp();
              }
              // the unit's last products (and, before them, every S^T and
              // dP^T) have read K and V: the next unit's may be loaded
              if (ok && leader) ptx::mma_commit(bar(S::kKVEmpty));
              __syncwarp();
            }
        }
        // each issuer waits for its own MMAs before the CTA may free TMEM
        if (leader) ptx::mma_commit(bar(S::kTeardown));
        __syncwarp();
        ptx::bar_wait(bar(S::kTeardown), 0, nullptr, p.timeout_ns);
    } else if (warp >= 4 && warp < 12) {
        // ---- key-row warps ----
        const int wq = warp % 4;       // TMEM lane quarter
        const int h = (warp - 4) / 4;  // query half of every sub-step
        const int r = wq * 32 + lane;  // key row
        const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
        const uint32_t ds_row = sbase + S::kOffDS + (r >> 3) * 1024 + (r & 7) * 128;
        int J = 0;  // sub-steps so far
        bool ok = true;
        for (int iu = 0; ok; ++iu) {
          UnitView uv;
          if (!(ok = read_unit(iu, uv)) || !uv.live) break;
          const BwdUnit &u = uv.u;
          const int k0 = uv.k0, qs0 = uv.qs0, n = uv.n;
          const int key = k0 + r;
          for (int j = 0; j < n; ++j, ++J) {
            const int b = J & 1;
            const int qc = qs0 + j * S::kQ + 32 * h;  // first query of this warp's chunk
            const uint32_t tb = tmem + lane_base + S::kTmemBuf + 128 * b;
            // the sub-step's rows, then S^T: one test of both first, the
            // bounded waits only when one is open
            const bool ready = ptx::bar_try_wait(bar(S::kSFull + b), (J >> 1) & 1) &&
                               ptx::bar_try_wait(bar(S::kLFull + b), (J >> 1) & 1);
            if (!__all_sync(0xffffffffu, ready)) {
                if (!(ok = wait(S::kLFull + b, (J >> 1) & 1))) break;
                if (!(ok = wait(S::kSFull + b, (J >> 1) & 1))) break;
            }
            ptx::tc_fence_after();
            uint32_t sv[32], dpv[32];
            ptx::tmem_ld32(tb + 32 * h, sv);
            ptx::tmem_ld_wait();
            ptx::reg_fence(sv);
            const bool need_mask = (CAUSAL && key > qc) || key >= u.Lk;
            const int lo = key >= u.Lk ? 32 : (CAUSAL ? key - qc : 0);  // queries i < lo do not see the key
            const float *rows = reinterpret_cast<const float *>(smem_raw + S::kOffRows + b * 2 * S::kQ * 4);
            const float4 *lq = reinterpret_cast<const float4 *>(rows + 32 * h);
            const float4 *dq4 = reinterpret_cast<const float4 *>(rows + S::kQ + 32 * h);
            uint32_t pp[16], dd[16];
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
                const float4 lv = lq[i / 4];
                const float l0 = (i % 4 == 0) ? lv.x : lv.z, l1 = (i % 4 == 0) ? lv.y : lv.w;
                float e0 = ptx::ex2(fmaf(__uint_as_float(sv[i]), p.scale_log2, -l0));
                float e1 = ptx::ex2(fmaf(__uint_as_float(sv[i + 1]), p.scale_log2, -l1));
                if (need_mask) {
                    if (i < lo) e0 = 0.f;
                    if (i + 1 < lo) e1 = 0.f;
                }
                pp[i / 2] = ptx::pack2<BF16>(e0, e1);
            }
            // P^T over the first 16 of this half's own S^T columns, published
            // at once: dV starts while dS^T is formed
            ptx::tmem_st16(tb + 32 * h, pp);
            ptx::tmem_st_wait();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::bar_arrive(bar(S::kPTFull + b));
            // dP^T, formed on the tensor core meanwhile
            if (!(ok = wait(S::kDPFull + b, (J >> 1) & 1))) break;
            ptx::tc_fence_after();
            ptx::tmem_ld32(tb + 64 + 32 * h, dpv);
            ptx::tmem_ld_wait();
            ptx::reg_fence(dpv);
            // dS = P (dP - D_i), with P as rounded for dV
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
                const float4 dv4 = dq4[i / 4];
                const float d0 = (i % 4 == 0) ? dv4.x : dv4.z, d1 = (i % 4 == 0) ? dv4.y : dv4.w;
                const float e0 = ptx::unpack_lo<BF16>(pp[i / 2]), e1 = ptx::unpack_hi<BF16>(pp[i / 2]);
                dd[i / 2] = ptx::pack2<BF16>(e0 * (__uint_as_float(dpv[i]) - d0),
                                             e1 * (__uint_as_float(dpv[i + 1]) - d1));
            }
            // dS^T buffer b is free once sub-step J-2's dQ_t^T and dK have read it
            if (J >= 2 && !(ok = wait(S::kDSFree + b, ((J - 2) >> 1) & 1))) break;
            // the dS^T buffers hold the key-row warps' staging blocks during a
            // unit's epilogue: every warp must have written out the previous unit's
            if (j == 0 && iu > 0 && !(ok = wait(S::kStagingFree, (iu - 1) & 1))) break;
            // dS^T row r, queries [32h, 32h+32): 16-byte chunks 4h..4h+3, 128-byte swizzle
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const uint32_t chunk = static_cast<uint32_t>((4 * h + m) ^ (r & 7));
                st_shared_v4(ds_row + b * S::kDSBytes + chunk * 16, dd[4 * m], dd[4 * m + 1], dd[4 * m + 2],
                             dd[4 * m + 3]);
            }
            ptx::tc_fence_before();         // the dP^T loads precede dQ_t^T over those columns
            ptx::fence_proxy_async_smem();  // dS^T is read by the tensor core next
            __syncwarp();
            if (lane == 0) ptx::bar_arrive(bar(S::kPFull + b));
          }
          if (!ok) break;
        // epilogue: head columns [64h, 64h+64) of dV and scale * dK for this key
        // row. The dV/dK accumulators are read out before this warp publishes
        // the next unit's first P^T, which the next unit's first dV/dK wait for.
        if (n > 0) {
            ok = wait(S::kDSFree + ((J - 1) & 1), ((J - 1) >> 1) & 1);  // the last dV and dK are done
            ptx::tc_fence_after();
        }
        // The TMEM loads are warp-collective (.sync.aligned): every lane runs
        // them; only the global stores are limited to keys that exist.
        if (ok) {
            const uint64_t once = ptx::l2_policy_evict_first();
            // dV, then scale * dK. Each warp stages its 32 key rows (64 head
            // columns, 128 bytes a row) in its own 4 KB of the dS^T buffers,
            // free once the last products are done, and writes them back four
            // whole rows (full 128-byte lines) per store instruction instead
            // of pieces of 32 rows, which took the LSU ~8x the transactions.
            const uint32_t stage = sbase + S::kOffDS + static_cast<uint32_t>(warp - 4) * 4096u;
            const uint32_t my_row = stage + static_cast<uint32_t>(lane) * 128u;
#pragma unroll 1
            for (int t = 0; t < 2; ++t) {
                const float f = t == 0 ? 1.f : p.scale;
                uint32_t w[D / 64][32];
                if (n > 0) {
#pragma unroll
                    for (int c = 0; c < D / 64; ++c)
                        ptx::tmem_ld32(tmem + lane_base + (t == 0 ? S::kTmemDV : S::kTmemDK) + h * (D / 2) + 32 * c,
                                       w[c]);
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int c = 0; c < D / 64; ++c) ptx::reg_fence(w[c]);
                } else {
#pragma unroll
                    for (int c = 0; c < D / 64; ++c)
#pragma unroll
                        for (int k = 0; k < 32; ++k) w[c][k] = 0u;
                }
                // row `lane` of the block: 16-byte chunk q at (q ^ (row & 7)) * 16
#pragma unroll
                for (int c = 0; c < D / 64; ++c) {
                    uint32_t pk[16];
#pragma unroll
                    for (int k = 0; k < 16; ++k)
                        pk[k] = ptx::pack2<BF16>(__uint_as_float(w[c][2 * k]) * f, __uint_as_float(w[c][2 * k + 1]) * f);
#pragma unroll
                    for (int m = 0; m < 4; ++m)
                        st_shared_v4(my_row + static_cast<uint32_t>(((4 * c + m) ^ (lane & 7)) * 16), pk[4 * m],
                                     pk[4 * m + 1], pk[4 * m + 2], pk[4 * m + 3]);
                }
                __syncwarp();
                uint16_t *out = static_cast<uint16_t *>(t == 0 ? p.dv : p.dk);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int rr = 4 * k + (lane >> 3), q = lane & 7;  // row of the block, 16-byte chunk
                    const uint4 val = ld_shared_v4(stage + static_cast<uint32_t>(rr * 128 + ((q ^ (rr & 7)) * 16)));
                    const int key_r = k0 + wq * 32 + rr;
                    if (key_r < u.Lk) {
                        // written once: evict first
                        const size_t row_g = (VARLEN ? (static_cast<size_t>(u.tk0) + key_r) * p.H + u.hh
                                                     : static_cast<size_t>(u.z) * p.Sk + key_r) * D + h * (D / 2);
                        ptx::st_global_v4_hint(reinterpret_cast<uint4 *>(out + row_g) + q, val.x, val.y, val.z,
                                               val.w, once);
                    }
                }
                __syncwarp();  // the block is rewritten for the next tensor
            }
            if (lane == 0) ptx::bar_arrive(bar(S::kStagingFree));
        }
        }
    } else if (warp >= 12) {
        // ---- dQ_t^T warps: head column r, all 64 queries of the sub-step ----
        const int wq = warp % 4;
        const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
        // head column r = 32 wq + lane of the staging tile: box wq, 4-byte word lane
        const uint32_t dq_col = sbase + S::kOffQ + wq * S::kDQBoxBytes + (lane & 3) * 4;
        int J = 0;  // sub-steps so far
        bool ok = true;
        for (int iu = 0; ok; ++iu) {
          UnitView uv;
          if (!(ok = read_unit(iu, uv)) || !uv.live) break;
          for (int j = 0; j < uv.n; ++j, ++J) {
            const int b = J & 1, st = J % S::kStages;
            if (!(ok = wait(S::kDQFull + b, (J >> 1) & 1))) break;
            ptx::tc_fence_after();
            uint32_t v0[32], v1[32];
            const uint32_t tb = tmem + lane_base + S::kTmemBuf + 128 * b + 64;
            ptx::tmem_ld32(tb, v0);
            ptx::tmem_ld32(tb + 32, v1);
            ptx::tmem_ld_wait();
            ptx::reg_fence(v0);
            ptx::reg_fence(v1);
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::bar_arrive(bar(S::kBufFree + b));
            // the sub-step's stage takes the tile once dV and dK are done with Q_J, dO_J
            if (!(ok = wait(S::kQEmpty + st, (J / S::kStages) & 1))) break;
            const uint32_t col = dq_col + st * S::kStageBytes;
#pragma unroll
            for (int i = 0; i < 64; ++i) {
                const uint32_t chunk = static_cast<uint32_t>((lane >> 2) ^ (i & 7));
                asm volatile("st.shared.b32 [%0], %1;" ::"r"(col + i * 128 + chunk * 16),
                             "r"(i < 32 ? v0[i] : v1[i - 32])
                             : "memory");
            }
            ptx::fence_proxy_async_smem();  // the bulk reduction reads the tile next
            __syncwarp();
            if (lane == 0) ptx::bar_arrive(bar(S::kStageReady + st));
          }
        }
    } else if (warp == 2) {
        // ---- bulk reductions of the staged dQ_t into the accumulator ----
        const bool leader = ptx::elect_one();
        int J = 0;  // sub-steps so far
        bool ok = true;
        for (int iu = 0; ok; ++iu) {
          UnitView uv;
          if (!(ok = read_unit(iu, uv)) || !uv.live) break;
          const BwdUnit &u = uv.u;
          for (int j = 0; j < uv.n; ++j, ++J) {
            const int st = J % S::kStages;
            if (!(ok = wait(S::kStageReady + st, (J / S::kStages) & 1))) break;
            if (leader) {
                const int q0 = uv.qs0 + j * S::kQ;
                const uint32_t tile = sbase + S::kOffQ + st * S::kStageBytes;
                int y, z;
                unit_coords<VARLEN>(u, false, q0, y, z);
                // boxes 0, 1 (over Q_J), then 2, 3 (over dO_J), as two groups
                for (int c = 0; c < D / 32; ++c) {
                    ptx::tma_reduce_add_3d(&tm_dq, tile + c * S::kDQBoxBytes, 32 * c, y, z);
                    if (c == 1 || c == D / 32 - 1) ptx::bulk_commit();
                }
                ptx::bulk_wait_read_all_but_newest();  // Q's half may be refilled now
                ptx::bar_arrive(bar(S::kStageFreeQ + st));
                ptx::bulk_wait_read_all();              // and dO's
                ptx::bar_arrive(bar(S::kStageFree + st));
            }
            __syncwarp();
          }
        }
        if (leader) ptx::bulk_wait_all();  // the reductions themselves are complete
        __syncwarp();
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, S::kTmemCols);
    }
    if (threadIdx.x == 0 && *abort_flag) atomicExch(p.err, kDeviceErrTimeout);
}

template <int D, bool BF16, bool CAUSAL, bool VARLEN>
cudaError_t launch_t(const CUtensorMap *maps, const void *o, const void *dout, const float *lse, void *dq,
                     const BwdParams &p, cudaStream_t st) {
    // prep grid: row chunks x heads (heads split over y and z: at most 65535 each)
    const int heads = VARLEN ? p.H : p.BH;
    const int head_rows = VARLEN ? p.total_q : p.Sq_pad;
    const unsigned hy = static_cast<unsigned>(heads < 65535 ? heads : 65535);
    const dim3 prep_grid(static_cast<unsigned>((head_rows + kPrepRows<D> - 1) / kPrepRows<D>), hy,
                         static_cast<unsigned>((heads + hy - 1) / hy));
    fa_bwd_prep_kernel<D, BF16, VARLEN><<<prep_grid, 256, 0, st>>>(static_cast<const uint16_t *>(o),
                                                                   static_cast<const uint16_t *>(dout), lse, p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // D = 64: 128-query steps; D = 128: 64-query sub-steps, double-buffered in TMEM
    auto kern = D == 64 ? fa_bwd_d64_kernel<64, BF16, CAUSAL, VARLEN> : fa_bwd_kernel<BF16, CAUSAL, VARLEN>;
    constexpr int kSmem = D == 64 ? Shape<64>::kSmemBytes : ShapeQ64::kSmemBytes;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    // D = 64: one CTA per work unit; D = 128: persistent CTAs take units from a counter
    const long long units = static_cast<long long>(p.BH) * p.n_ktiles;
    const long long grid = D == 64 ? units : (units < p.grid ? units : p.grid);
    // D = 128: the main and the conversion kernels are launched as programmatic
    // dependents (each waits for its predecessor in the kernel itself)
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(D == 64 ? kThreads : kThreadsQ64);
    cfg.dynamicSmemBytes = kSmem;
    cfg.stream = st;
    cfg.attrs = pdl;
    cfg.numAttrs = D == 64 ? 0 : 1;
    e = cudaLaunchKernelEx(&cfg, kern, maps[0], maps[1], maps[2], maps[3], maps[4], p);
    if (e != cudaSuccess) return e;
    const long long n8 = (VARLEN ? static_cast<long long>(p.total_q) * p.H : static_cast<long long>(p.BH) * p.Sq) * D / 8;
    cudaLaunchConfig_t cfg2 = {};
    cfg2.gridDim = dim3(static_cast<unsigned>((n8 + 255) / 256));
    cfg2.blockDim = dim3(256);
    cfg2.stream = st;
    cfg2.attrs = pdl;
    cfg2.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg2, fa_bwd_dq_kernel<BF16>, static_cast<const float *>(p.dq_acc),
                              static_cast<uint16_t *>(dq), n8, p.scale);
}

}  // namespace bwd

}  // namespace fa
