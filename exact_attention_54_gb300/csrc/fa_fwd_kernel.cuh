// FlashAttention-2 forward on sm_103a: TMA-staged tiles, tcgen05 MMAs with
// TMEM accumulators, online softmax in registers.
//
// Method ("FlashAttention-2 MMA", Technical Details; "Adaptive
// High-Performance Attention Kernels in CUDA", Architectural Progression
// stages 2-4): the outer loop runs over 128-row query tiles, the inner loop
// over 128-key K/V tiles; each step forms S = Q K^T, updates the running row
// maximum m and running sum l, rescales the output accumulator by
// alpha = exp(m_old - m_new) and adds P V. The output stays on chip for the
// whole inner loop and one log-sum-exp per row is written at the end. Causal
// tiles that lie entirely above the diagonal are never visited; only tiles
// that straddle it are masked (k_idx <= q_idx, top-left aligned).
//
// GB300 mapping (one CTA per SM, persistent):
//   warp 0        TMA producer of Q (a tile pair once per work item) and of
//                 the K ring (128-byte swizzle, 128 rows x 64 columns per box)
//   warp 2        TMA producer of the V ring (K and V rings are separate, so K
//                 tiles, needed first, are released and refilled earlier)
//   warp 1        MMA issuer (one thread): S_t = Q_t K^T into TMEM, then
//                 O_t += P_t V with P_t read from TMEM (A operand) and V
//                 MN-major from shared memory. Also owns the TMEM allocation.
//   warps 4..7    softmax warpgroup for query tile 0 (one row per thread)
//   warps 8..11   softmax warpgroup for query tile 1
// The two query tiles of a work item share every K/V stage and alternate on
// the tensor core: while one warpgroup exponentiates its S tile, the MMAs of
// the other tile run. TMEM columns: S0 [0,128) S1 [128,256) O0 and O1 after;
// P_t (16-bit) overwrites the first 64 columns of S_t.
//
// The running maximum is only moved when it grows by more than 2^8 (in the
// exponent's base-2 units); until then P may exceed 1 by up to 256x. O and l
// carry the same stale maximum, so O / l is unchanged; this only saves
// rescaling work.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include "fa_launch.h"
#include "sm103_ptx.cuh"

namespace fa {

constexpr int kBlockM = 128;      // query rows per tile
constexpr int kBlockN = 128;      // keys per K/V tile
constexpr int kFwdThreads = 384;  // 12 warps
constexpr float kRescaleThreshold = 8.0f;

// Size of the packed-sequence schedule table (see VarlenSched).
constexpr int kSchedSeqs = 256;
constexpr int kSchedPairs = 64;
constexpr int kSchedInts = 4 + 2 * kSchedPairs + kSchedSeqs;

template <int D>
struct FwdShape {
    static_assert(D == 64 || D == 128, "head dim");
    static constexpr int kColBlocks = D / 64;            // 128-byte column blocks per row
    static constexpr int kBlockBytes = kBlockM * 128;    // one 128-row x 64-column box
    static constexpr int kTileBytes = kBlockM * D * 2;   // one 128-row tile of Q, K or V
    // D = 128: a K tile is free once both Q K^T of its round are issued, a V
    // tile only after both P V, so V gets the deeper ring
    static constexpr int kKStages = (D == 128) ? 2 : 4;  // K ring depth
    static constexpr int kVStages = (D == 128) ? 3 : 4;  // V ring depth
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kOffQ + 2 * kTileBytes;
    static constexpr int kOffV = kOffK + kKStages * kTileBytes;
    static constexpr int kOffBar = kOffV + kVStages * kTileBytes;
    // barrier indices
    static constexpr int kQFull = 0, kQEmpty = 1, kTeardown = 2;
    static constexpr int kKFull = 3;
    static constexpr int kKEmpty = kKFull + kKStages;
    static constexpr int kVFull = kKEmpty + kKStages;
    static constexpr int kVEmpty = kVFull + kVStages;
    static constexpr int kSFull = kVEmpty + kVStages;    // +t
    static constexpr int kPFull = kSFull + 2;            // +t: P keys [0,64) written, O corrected
    static constexpr int kPFull2 = kPFull + 2;           // +t: P keys [64,128) written
    static constexpr int kODone = kPFull2 + 2;           // +t
    static constexpr int kFirstQ = kODone + 2;           // the CTA's first Q pair has landed (one phase only)
    static constexpr int kNumBars = kFirstQ + 1;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    // packed-sequence schedule (varlen): see VarlenSched
    static constexpr int kOffSched = (kOffMisc + 16 + 15) & ~15;
    static constexpr int kSmemBytes = kOffSched + kSchedInts * 4 + 1024;  // + slack to align the base to 1024
    static constexpr uint32_t kTmemS = 0;                     // + t * 128
    static constexpr uint32_t kTmemO = 256;                   // + t * D
    static constexpr uint32_t kTmemCols = 512;
    static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

// Packed-sequence schedule, built by every CTA from cu_seqlens_q at launch
// (no host synchronisation, no workspace): only the work items that exist are
// handed out, heaviest first. Item order: query-tile pair index descending;
// within a pair index, sequences ascending (those long enough to have that
// pair), then heads. In shared memory, as ints: [0] 1 when the table is in
// use, [1] the number of items, [2] the number of cached item records (see
// below), then for each pair index p the first item of its bucket and the
// number of sequences in it, then each sequence's pair count. Batches beyond
// the table's size use the plain enumeration (every (pair, sequence, head) up
// to the longest sequence; missing tiles inactive).
//
// Looking an item up in the table walks the pair buckets and the sequences
// and reads the item's offsets from cu_seqlens in global memory, which cost
// more than a microsecond per item on every role. So once the table is
// built, the CTA resolves all of its own items at once (one thread per
// round) and keeps them as 32-byte records {b, h, pair, q0, k0, Lq, Lk} in
// place of the table, when they fit; every role then reads its item with two
// shared-memory loads.
struct VarlenSched {
    static constexpr int kOn = 0, kItems = 1, kRecs = 2;
    static constexpr int kStart = 4, kCount = kStart + kSchedPairs, kPairs = kCount + kSchedPairs;
    static constexpr int kRec0 = 4, kRecInts = 8;
    static constexpr int kMaxRecs = (kSchedInts - kRec0) / kRecInts;
};

__device__ __forceinline__ int lds_int(uint32_t addr) {
    int v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ int4 lds_int4(uint32_t addr) {
    int4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

// Work items of this launch: the packed-sequence table's count when it is in use.
template <bool VARLEN>
__device__ __forceinline__ int num_items(const FwdParams &p, uint32_t sched) {
    if constexpr (VARLEN) {
        if (lds_int(sched + 4 * VarlenSched::kOn)) return lds_int(sched + 4 * VarlenSched::kItems);
    }
    return p.num_work;
}

// One unit of work: a pair of consecutive 128-row query tiles of one
// (sequence, head). Tiles past the end of the sequence are inactive.
struct Work {
    int b, h;
    int seq_q0, seq_k0;  // token offsets of the sequence (varlen), else 0
    int Lq, Lk;          // query and key lengths of the sequence
    int q_start[2];      // first query row of each tile (relative to the sequence)
    int rows[2];         // valid rows of each tile (0 = inactive)
    int n_kv[2];         // K/V tiles each query tile visits
    int n_kv_max;
};

// Query tiles, rows and key-tile counts of a work item from its sequence
// lengths and pair index.
template <bool CAUSAL>
__device__ __forceinline__ void finish_work(Work &k, int pair) {
    const int nk_all = (k.Lk + kBlockN - 1) / kBlockN;
    k.n_kv_max = 0;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        const int qs = (2 * pair + t) * kBlockM;
        k.q_start[t] = qs;
        const int rows = k.Lq - qs;
        k.rows[t] = rows <= 0 ? 0 : (rows < kBlockM ? rows : kBlockM);
        int nkv = 0;
        if (k.rows[t] > 0) {
            nkv = nk_all;
            if (CAUSAL) {
                const int last = (qs + k.rows[t] - 1) / kBlockN + 1;
                nkv = last < nk_all ? last : nk_all;
            }
        }
        k.n_kv[t] = nkv;
        k.n_kv_max = nkv > k.n_kv_max ? nkv : k.n_kv_max;
    }
}

// Work item w, resolved from the launch parameters (dense), the schedule
// table or the plain enumeration (packed sequences). `pair_out` receives its
// query-tile pair index.
template <bool CAUSAL, bool VARLEN>
__device__ __forceinline__ Work resolve_work(const FwdParams &p, int w, uint32_t sched, int *pair_out = nullptr) {
    Work k;
    const int BH = p.B * p.H;
    int pair = p.n_pairs - 1 - w / BH;  // longest causal work first
    const int bh = w % BH;
    k.b = bh / p.H;
    k.h = bh % p.H;
    if constexpr (VARLEN) {
        if (lds_int(sched + 4 * VarlenSched::kOn)) {
            // bucket of pair index `pair` holds items [start(pair), start(pair - 1))
            pair = p.n_pairs - 1;
            while (pair > 0 && w >= lds_int(sched + 4 * (VarlenSched::kStart + pair - 1))) --pair;
            const int wr = w - lds_int(sched + 4 * (VarlenSched::kStart + pair));
            int idx = wr / p.H;
            k.h = wr % p.H;
            int b = 0;
            for (; b < p.B; ++b)
                if (lds_int(sched + 4 * (VarlenSched::kPairs + b)) > pair && idx-- == 0) break;
            k.b = b;
        }
        k.seq_q0 = p.cu_q[k.b];
        k.Lq = p.cu_q[k.b + 1] - k.seq_q0;
        k.seq_k0 = p.cu_k[k.b];
        k.Lk = p.cu_k[k.b + 1] - k.seq_k0;
    } else {
        k.seq_q0 = 0;
        k.seq_k0 = 0;
        k.Lq = p.Sq;
        k.Lk = p.Sk;
    }
    if (pair_out != nullptr) *pair_out = pair;
    finish_work<CAUSAL>(k, pair);
    return k;
}

__device__ __forceinline__ int work_index(int r);

// The work item of this CTA's round r (an item of the launch: callers check
// work_index(r) < num_items first).
template <bool CAUSAL, bool VARLEN>
__device__ __forceinline__ Work get_work(const FwdParams &p, int r, uint32_t sched) {
    if constexpr (VARLEN) {
        if (r < lds_int(sched + 4 * VarlenSched::kRecs)) {
            const uint32_t rec = sched + 4 * (VarlenSched::kRec0 + VarlenSched::kRecInts * r);
            const int4 a = lds_int4(rec), c = lds_int4(rec + 16);
            Work k;
            k.b = a.x;
            k.h = a.y;
            k.seq_q0 = a.w;
            k.seq_k0 = c.x;
            k.Lq = c.y;
            k.Lk = c.z;
            finish_work<CAUSAL>(k, a.z);
            return k;
        }
    }
    return resolve_work<CAUSAL, VARLEN>(p, work_index(r), sched);
}

// Static persistent schedule: round r hands out work items [r*G, (r+1)*G),
// alternating direction each round so that the heavy early items and the light
// late items balance across CTAs.
__device__ __forceinline__ int work_index(int r) {
    const int G = static_cast<int>(gridDim.x);
    const int pos = (r & 1) ? (G - 1 - static_cast<int>(blockIdx.x)) : static_cast<int>(blockIdx.x);
    return r * G + pos;
}

// ------------------------------------------------------------------ roles --

// Loads one K or V tile (all 64-column boxes) of key tile j into `dst`.
template <int D, bool VARLEN>
__device__ __forceinline__ void load_kv_tile(const CUtensorMap *tm, uint32_t dst, uint32_t bar, const Work &wk,
                                             int j, int H) {
    using S = FwdShape<D>;
#pragma unroll
    for (int c = 0; c < S::kColBlocks; ++c) {
        if constexpr (VARLEN)
            ptx::tma_load_3d(dst + c * S::kBlockBytes, tm, bar, c * 64, wk.h, wk.seq_k0 + j * kBlockN);
        else
            ptx::tma_load_3d(dst + c * S::kBlockBytes, tm, bar, c * 64, j * kBlockN, wk.b * H + wk.h);
    }
}

// Q and K producer (one thread). It issues no L2 prefetches: asking L2 for
// the next item's Q while the current item ran cost 1.5 % (dense) and 4 %
// (packed sequences), and K/V tiles prefetched ahead of the ring cost more.
template <int D, bool CAUSAL, bool VARLEN>
__device__ void fwd_producer_qk(const CUtensorMap *tq, const CUtensorMap *tk, const FwdParams &p, uint32_t sbase,
                                volatile int *abort_flag) {
    using S = FwdShape<D>;
    const uint32_t sched = sbase + S::kOffSched;
    const uint32_t bars = sbase + S::kOffBar;
    auto bar = [&](int i) { return bars + 8u * static_cast<uint32_t>(i); };
    const bool leader = ptx::elect_one();
    const uint64_t stream_pol = ptx::l2_policy_evict_first();
    uint32_t it = 0;  // K tiles issued
    uint32_t wi = 0;  // work items loaded
    uint32_t nq = 0;  // Q pair loads issued
    bool ok = true;
    for (int r = 0; ok; ++r) {
        const int w = work_index(r);
        if (w >= num_items<VARLEN>(p, sched)) break;
        const Work wk = get_work<CAUSAL, VARLEN>(p, r, sched);
        if (wk.n_kv_max == 0) continue;
        // The item's Q pair, once the previous item's last Q K^T has read
        // the buffer.
        auto load_q = [&]() -> bool {
            if (nq > 0 &&
                !ptx::warp_all(ptx::bar_wait(bar(S::kQEmpty), (nq - 1) & 1, abort_flag, p.timeout_ns)))
                return false;
            uint32_t qbytes = 0;
#pragma unroll
            for (int t = 0; t < 2; ++t) qbytes += wk.n_kv[t] > 0 ? S::kTileBytes : 0;
            if (leader) ptx::bar_arrive_expect_tx(bar(S::kQFull), qbytes);
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                if (wk.n_kv[t] == 0 || !leader) continue;
#pragma unroll
                for (int c = 0; c < S::kColBlocks; ++c) {
                    // Q tiles are read once: evict them first, keep L2 for K and V
                    const uint32_t dst = sbase + S::kOffQ + t * S::kTileBytes + c * S::kBlockBytes;
                    if constexpr (VARLEN)
                        ptx::tma_load_3d_hint(dst, tq, bar(S::kQFull), c * 64, wk.h, wk.seq_q0 + wk.q_start[t],
                                              stream_pol);
                    else
                        ptx::tma_load_3d_hint(dst, tq, bar(S::kQFull), c * 64, wk.q_start[t], wk.b * p.H + wk.h,
                                              stream_pol);
                }
            }
            ++nq;
            return true;
        };
        // The first item loads Q before K; a later item loads its first K
        // tile first: that ring stage frees rounds before the Q buffer does
        // (at the previous item's last Q K^T), and the K tile would otherwise
        // wait behind the Q load.
        if (wi == 0 && !(ok = load_q())) break;
        for (int j = 0; j < wk.n_kv_max; ++j, ++it) {
            // All CTAs fill their rings at once when the kernel starts; the
            // first products need only Q and K tile 0, so the rest of the
            // first ring fill waits until this CTA's first Q pair has landed.
            if (wi == 0 && j == 1 &&
                !(ok = ptx::warp_all(ptx::bar_wait(bar(S::kQFull), 0, abort_flag, p.timeout_ns))))
                break;
            const uint32_t stage = it % S::kKStages;
            if (it >= S::kKStages &&
                !(ok = ptx::warp_all(ptx::bar_wait(bar(S::kKEmpty + stage), ((it / S::kKStages) - 1) & 1, abort_flag,
                                     p.timeout_ns))))
                break;
            if (leader) {
                ptx::bar_arrive_expect_tx(bar(S::kKFull + stage), S::kTileBytes);
                load_kv_tile<D, VARLEN>(tk, sbase + S::kOffK + stage * S::kTileBytes, bar(S::kKFull + stage), wk, j,
                                        p.H);
            }
            if (wi > 0 && j == 0 && !(ok = load_q())) break;
        }
        if (!ok) break;
        ++wi;
    }
    // Never leave with copies in flight: wait (bounded, even after an abort)
    // for the newest load into every stage and for the newest Q load.
    for (uint32_t s = 0; s < S::kKStages && s < it; ++s) {
        const uint32_t last = (it - 1) - ((it - 1 - s) % S::kKStages);
        ptx::bar_wait(bar(S::kKFull + s), (last / S::kKStages) & 1, nullptr, p.timeout_ns);
    }
    if (nq > 0) ptx::bar_wait(bar(S::kQFull), (nq - 1) & 1, nullptr, p.timeout_ns);
}

// V producer (one thread): runs ahead of the P V products as far as its ring allows.
template <int D, bool CAUSAL, bool VARLEN>
__device__ void fwd_producer_v(const CUtensorMap *tv, const FwdParams &p, uint32_t sbase, volatile int *abort_flag) {
    using S = FwdShape<D>;
    const uint32_t sched = sbase + S::kOffSched;
    const uint32_t bars = sbase + S::kOffBar;
    auto bar = [&](int i) { return bars + 8u * static_cast<uint32_t>(i); };
    const bool leader = ptx::elect_one();
    uint32_t it = 0;
    bool ok = true;
    for (int r = 0; ok; ++r) {
        const int w = work_index(r);
        if (w >= num_items<VARLEN>(p, sched)) break;
        const Work wk = get_work<CAUSAL, VARLEN>(p, r, sched);
        for (int j = 0; j < wk.n_kv_max; ++j, ++it) {
            // V tile 0 goes with the first Q and K tiles; later V tiles wait
            // until the first Q pair has landed (see the Q/K producer).
            if (it == 1 && !(ok = ptx::warp_all(ptx::bar_wait(bar(S::kFirstQ), 0, abort_flag, p.timeout_ns)))) break;
            const uint32_t stage = it % S::kVStages;
            if (it >= S::kVStages &&
                !(ok = ptx::warp_all(ptx::bar_wait(bar(S::kVEmpty + stage), ((it / S::kVStages) - 1) & 1, abort_flag,
                                     p.timeout_ns))))
                break;
            if (leader && !withheld(p.withhold, it)) {
                ptx::bar_arrive_expect_tx(bar(S::kVFull + stage), S::kTileBytes);
                load_kv_tile<D, VARLEN>(tv, sbase + S::kOffV + stage * S::kTileBytes, bar(S::kVFull + stage), wk, j,
                                        p.H);
            }
        }
    }
    for (uint32_t s = 0; s < S::kVStages && s < it; ++s) {
        const uint32_t last = (it - 1) - ((it - 1 - s) % S::kVStages);
        ptx::bar_wait(bar(S::kVFull + s), (last / S::kVStages) & 1, nullptr, p.timeout_ns);
    }
}

template <int D, bool BF16, bool CAUSAL, bool VARLEN>
__device__ void fwd_mma(const FwdParams &p, uint32_t sbase, uint32_t tmem, volatile int *abort_flag) {
    using S = FwdShape<D>;
    const uint32_t sched = sbase + S::kOffSched;
    constexpr uint32_t kIdescQK = ptx::idesc_f16(BF16, kBlockM, kBlockN, false);
    constexpr uint32_t kIdescPV = ptx::idesc_f16(BF16, kBlockM, D, true);
    const uint32_t bars = sbase + S::kOffBar;
    auto bar = [&](int i) { return bars + 8u * static_cast<uint32_t>(i); };

    const bool leader = ptx::elect_one();
    // Operand descriptors are built once; each MMA only advances the 14-bit
    // start-address field (16-byte units), so issuing stays a few instructions
    // per MMA. Stage buffers are contiguous, so stage s adds s * tile / 16.
    const uint64_t dq0 = ptx::smem_desc_sw128(sbase + S::kOffQ, 16, 1024);
    const uint64_t dk0 = ptx::smem_desc_sw128(sbase + S::kOffK, 16, 1024);
    const uint64_t dv0 = ptx::smem_desc_sw128(sbase + S::kOffV, S::kBlockBytes, 1024);
    constexpr uint64_t kTile16 = S::kTileBytes >> 4;

    // S_t = Q_t K^T: D/16 MMAs of K=16, both operands K-major, 128-byte swizzled.
    auto issue_qk = [&](int t, uint32_t stage) {
        const uint64_t qd = dq0 + static_cast<uint64_t>(t) * kTile16;
        const uint64_t kd = dk0 + static_cast<uint64_t>(stage) * kTile16;
        const uint32_t dst = tmem + S::kTmemS + t * 128;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            constexpr uint64_t kBlock16 = S::kBlockBytes >> 4;
            const uint64_t off = (kk / 4) * kBlock16 + (kk % 4) * 2;
            ptx::mma_ss(dst, qd + off, kd + off, kIdescQK, kk > 0);
        }
    };
    // O_t (+)= P_t V: 128/16 MMAs of K=16; P_t from TMEM (two 16-bit values per
    // column), V MN-major: 64-column boxes 16 KB apart, 8-key atoms 1 KB apart.
    // half 0: keys [0,64), half 1: keys [64,128) (each published separately)
    auto issue_pv = [&](int t, uint32_t stage, bool accumulate, int half) {
        const uint64_t vd = dv0 + static_cast<uint64_t>(stage) * kTile16;
        const uint32_t dst = tmem + S::kTmemO + t * D;
        const uint32_t pa = tmem + S::kTmemS + t * 128;
#pragma unroll
        for (int k4 = 0; k4 < kBlockN / 32; ++k4) {
            const int kk = half * (kBlockN / 32) + k4;
            ptx::mma_ts(dst, pa + kk * 8, vd + kk * (2048 >> 4), kIdescPV, (accumulate || kk > 0) ? 1u : 0u);
        }
    };

    uint32_t it = 0, wi = 0;   // K/V tiles consumed, work items consumed
    uint32_t cnt[2] = {0, 0};  // PV steps issued per query tile (= P_FULL phases consumed)
    bool ok = true;
    for (int r = 0; ok; ++r) {
        const int w = work_index(r);
        if (w >= num_items<VARLEN>(p, sched)) break;
        const Work wk = get_work<CAUSAL, VARLEN>(p, r, sched);
        if (wk.n_kv_max == 0) continue;
        if (!(ok = ptx::warp_all(ptx::bar_wait(bar(S::kQFull), wi & 1, abort_flag, p.timeout_ns)))) break;
        if (wi == 0 && leader) ptx::bar_arrive(bar(S::kFirstQ));  // releases the V producer's ring fill
        {
            const uint32_t ks = it % S::kKStages;
            if (!(ok = ptx::warp_all(ptx::bar_wait(bar(S::kKFull + ks), (it / S::kKStages) & 1, abort_flag, p.timeout_ns))))
                break;
            ptx::tc_fence_after();
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                if (wk.n_kv[t] == 0) continue;
                if (leader) {
                    issue_qk(t, ks);
                    ptx::mma_commit(bar(S::kSFull + t));
                }
            }
            if (leader) ptx::mma_commit(bar(S::kKEmpty + ks));  // K tile 0 has all its readers
            // Q is read by Q K^T only: once an item's last Q K^T is issued, the
            // producer may load the next item's Q pair, which then lands while
            // this item's last P V products run.
            if (wk.n_kv_max == 1 && leader) ptx::mma_commit(bar(S::kQEmpty));
        }
        for (int j = 0; j < wk.n_kv_max && ok; ++j) {
            const uint32_t itj = it + j;
            const uint32_t vs = itj % S::kVStages;
            const uint32_t kn = (itj + 1) % S::kKStages;
            bool v_ready = false, k_next_used = false;
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                if (j >= wk.n_kv[t]) continue;
                if (!(ok = ptx::warp_all(ptx::bar_wait(bar(S::kPFull + t), cnt[t] & 1, abort_flag, p.timeout_ns)))) break;
                if (!v_ready) {
                    if (!(ok = ptx::warp_all(ptx::bar_wait(bar(S::kVFull + vs), (itj / S::kVStages) & 1, abort_flag,
                                             p.timeout_ns))))
                        break;
                    v_ready = true;
                }
                ptx::tc_fence_after();
                if (leader) issue_pv(t, vs, j > 0, 0);
                // the second half of P V once the softmax has published keys [64,128)
                if (!(ok = ptx::warp_all(ptx::bar_wait(bar(S::kPFull2 + t), cnt[t] & 1, abort_flag, p.timeout_ns))))
                    break;
                ptx::tc_fence_after();
                if (leader) {
                    issue_pv(t, vs, true, 1);
                    // the epilogue needs the last product; earlier ones are covered by S_FULL
                    if (j + 1 == wk.n_kv[t]) ptx::mma_commit(bar(S::kODone + t));
                }
                ++cnt[t];
                if (j + 1 < wk.n_kv[t]) {
                    if (!k_next_used) {
                        if (!(ok = ptx::warp_all(ptx::bar_wait(bar(S::kKFull + kn), ((itj + 1) / S::kKStages) & 1, abort_flag,
                                                 p.timeout_ns))))
                            break;
                        k_next_used = true;
                    }
                    ptx::tc_fence_after();
                    if (leader) {
                        issue_qk(t, kn);
                        ptx::mma_commit(bar(S::kSFull + t));
                    }
                }
            }
            if (!ok) break;
            if (leader) {
                ptx::mma_commit(bar(S::kVEmpty + vs));                 // V tile j: both P V products issued
                if (k_next_used) ptx::mma_commit(bar(S::kKEmpty + kn));  // K tile j+1: both Q K^T issued
                if (j + 2 == wk.n_kv_max) ptx::mma_commit(bar(S::kQEmpty));  // the item's last Q K^T issued
            }
        }
        if (!ok) break;
        it += wk.n_kv_max;
        ++wi;
    }
    // Every MMA issued above must finish before TMEM is released.
    if (leader) ptx::mma_commit(bar(S::kTeardown));
    __syncwarp();
    ptx::bar_wait(bar(S::kTeardown), 0, nullptr, p.timeout_ns);
}

template <int D, bool BF16, bool CAUSAL, bool VARLEN>
__device__ void fwd_softmax(const FwdParams &p, uint32_t sbase, uint32_t tmem, int t, int wq, int lane,
                            volatile int *abort_flag) {
    using S = FwdShape<D>;
    using Elem = uint16_t;
    const uint32_t sched = sbase + S::kOffSched;
    const uint32_t bars = sbase + S::kOffBar;
    auto bar = [&](int i) { return bars + 8u * static_cast<uint32_t>(i); };
    const int row = wq * 32 + lane;                             // row within the query tile
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;  // this warp's TMEM lanes
    const uint32_t tS = tmem + lane_base + S::kTmemS + t * 128;
    const uint32_t tO = tmem + lane_base + S::kTmemO + t * D;
    const float scale_log2 = p.scale_log2;
    const uint64_t stream_pol = ptx::l2_policy_evict_first();
    constexpr unsigned kFull = 0xffffffffu;
    uint32_t cnt = 0;    // S tiles consumed by this warpgroup
    uint32_t items = 0;  // work items finished by this warpgroup
    bool ok = true;

    for (int r = 0; ok; ++r) {
        const int w = work_index(r);
        if (w >= num_items<VARLEN>(p, sched)) break;
        const Work wk = get_work<CAUSAL, VARLEN>(p, r, sched);
        if (wk.rows[t] == 0) continue;
        const int q_row = wk.q_start[t] + row;
        const bool row_valid = row < wk.rows[t];
        const int nkv = wk.n_kv[t];
        float m_used = -CUDART_INF_F;  // running max in base-2 units of the scaled score
        float l = 0.f;

        for (int j = 0; j < nkv; ++j) {
            ok = ptx::bar_wait(bar(S::kSFull + t), cnt & 1, abort_flag, p.timeout_ns);
            if (!__all_sync(kFull, ok)) { ok = false; break; }
            ptx::tc_fence_after();
            // The keys of this tile that the row sees are the columns c < lim:
            // the sequence ends at Lk and, causal, the row sees keys up to its
            // own position. Tiles inside both limits (need_mask false, the
            // same for the whole warpgroup) are not tested.
            const int k0 = j * kBlockN;
            const bool need_mask = (k0 + kBlockN > wk.Lk) || (CAUSAL && k0 + kBlockN - 1 > wk.q_start[t]);
            // The row maximum comes with the loads (one wait for all four).
            uint32_t s[4][32];
            float mx4[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) ptx::tmem_ld32_max(tS + 32 * c, s[c], mx4[c]);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                ptx::reg_fence(s[c]);
                asm volatile("" : "+f"(mx4[c]));
            }
            if (need_mask) {
                // masked tile: the maximum is taken again after the mask
                int lim = wk.Lk - k0;
                if (CAUSAL) lim = min(lim, q_row + 1 - k0);
#pragma unroll
                for (int c = 0; c < kBlockN; ++c)
                    if (c >= lim) s[c / 32][c % 32] = 0xff800000u;  // -inf
#pragma unroll
                for (int c = 0; c < 4; ++c) mx4[c] = -CUDART_INF_F;
#pragma unroll
                for (int c = 0; c < kBlockN; c += 2)
                    mx4[(c / 2) % 4] = ptx::fmax3(mx4[(c / 2) % 4], __uint_as_float(s[c / 32][c % 32]),
                                                  __uint_as_float(s[(c + 1) / 32][(c + 1) % 32]));
            }
            const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
            const float m_cand = mx * scale_log2;
            const bool need = m_cand > m_used + kRescaleThreshold;
            float alpha = 1.f;
            if (need) {
                alpha = ptx::ex2(m_used - m_cand);  // 0 on the first tile (m_used = -inf)
                m_used = m_cand;
            }
            l *= alpha;
            const float m_sub = (m_used == -CUDART_INF_F) ? 0.f : m_used;

            // P = 2^(s * scale_log2 - m), packed two per 32-bit TMEM column and
            // stored 32 columns (64 keys) at a time.
            const uint64_t scale2 = ptx::pk2(scale_log2, scale_log2);
            const uint64_t negm2 = ptx::pk2(-m_sub, -m_sub);
            uint64_t sum2[2] = {ptx::pk2(0.f, 0.f), ptx::pk2(0.f, 0.f)};
            // Each half is published on its own barrier, so the tensor core
            // starts P V on keys [0,64) while keys [64,128) are exponentiated.
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t pk[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int c = 64 * h + 2 * i;
                    const uint64_t x = ptx::ffma2(ptx::pk2(__uint_as_float(s[c / 32][c % 32]),
                                                           __uint_as_float(s[(c + 1) / 32][(c + 1) % 32])),
                                                  scale2, negm2);
                    float x0, x1;
                    ptx::upk2(x, x0, x1);
                    const float e0 = ptx::ex2(x0), e1 = ptx::ex2(x1);
                    sum2[i % 2] = ptx::fadd2(sum2[i % 2], ptx::pk2(e0, e1));
                    pk[i] = ptx::pack2<BF16>(e0, e1);
                }
                ptx::tmem_st32(tS + 32 * h, pk);
                // O *= alpha before the first half's P V accumulates into it
                // (only when a row of this warp moved its maximum). The previous
                // P V has landed: Q K^T j was issued after it, and S_FULL tracks
                // every MMA issued before that Q K^T.
                if (h == 0 && j > 0 && __any_sync(kFull, need)) {
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t o[32];
                        ptx::tmem_ld32(tO + c * 32, o);
                        ptx::tmem_ld_wait();
                        ptx::reg_fence(o);
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                        ptx::tmem_st32(tO + c * 32, o);
                    }
                }
                ptx::tmem_st_wait();
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::bar_arrive(bar((h == 0 ? S::kPFull : S::kPFull2) + t));
            }
            {
                float a0, a1, b0, b1;
                ptx::upk2(sum2[0], a0, a1);
                ptx::upk2(sum2[1], b0, b1);
                l += (a0 + a1) + (b0 + b1);
            }
            ++cnt;
        }
        if (!ok) break;

        // epilogue: O / l in the input dtype, LSE = (m + log2 l) * ln 2. O_DONE
        // completes once per work item of this tile, after its last P V.
        if (nkv > 0) {
            ok = ptx::bar_wait(bar(S::kODone + t), items & 1, abort_flag, p.timeout_ns);
            if (!__all_sync(kFull, ok)) { ok = false; break; }
            ptx::tc_fence_after();
            ++items;
        }
        const float inv_l = l > 0.f ? 1.f / l : 0.f;
        const float lse = l > 0.f ? (m_used + __log2f(l)) * 0.69314718055994531f : -CUDART_INF_F;
        Elem *orow;
        if constexpr (VARLEN)
            orow = static_cast<Elem *>(p.o) + (static_cast<size_t>(wk.seq_q0 + q_row) * p.H + wk.h) * D;
        else
            orow = static_cast<Elem *>(p.o) + (static_cast<size_t>(wk.b * p.H + wk.h) * p.Sq + q_row) * D;
        uint32_t o[D / 32][32];
        if (nkv > 0) {
#pragma unroll
            for (int c = 0; c < D / 32; ++c) ptx::tmem_ld32(tO + c * 32, o[c]);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < D / 32; ++c) ptx::reg_fence(o[c]);
        } else {
#pragma unroll
            for (int c = 0; c < D / 32; ++c)
#pragma unroll
                for (int i = 0; i < 32; ++i) o[c][i] = 0u;
        }
        // One wait for all of O's TMEM loads; rows go out in 32-byte stores
        // when O is 32-byte aligned (every row then is: a row is D * 2 bytes).
        const bool v8 = (reinterpret_cast<uintptr_t>(p.o) & 31) == 0;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
                pk[i] = ptx::pack2<BF16>(__uint_as_float(o[c][2 * i]) * inv_l, __uint_as_float(o[c][2 * i + 1]) * inv_l);
            if (row_valid) {
                // O and LSE are written once: evict them first, keep L2 for K and V
                uint4 *dst = reinterpret_cast<uint4 *>(orow + c * 32);
                if (v8) {
                    ptx::st_global_v8_hint(dst, pk, stream_pol);
                    ptx::st_global_v8_hint(dst + 2, pk + 8, stream_pol);
                } else {
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        ptx::st_global_v4_hint(dst + i, pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3], stream_pol);
                }
            }
        }
        if (row_valid) {
            if constexpr (VARLEN)
                ptx::st_global_f32_hint(p.lse + static_cast<size_t>(wk.h) * p.total_q + wk.seq_q0 + q_row, lse,
                                        stream_pol);
            else
                ptx::st_global_f32_hint(p.lse + static_cast<size_t>(wk.b * p.H + wk.h) * p.Sq + q_row, lse,
                                        stream_pol);
        }
    }
}

// ----------------------------------------------------------------- kernel --

template <int D, bool BF16, bool CAUSAL, bool VARLEN>
__global__ void __launch_bounds__(kFwdThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
    using S = FwdShape<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = ptx::smem_addr(smem);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + S::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + S::kOffMisc + 4);
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;

    if (threadIdx.x == 0) {
        const uint32_t bars = sbase + S::kOffBar;
        for (int i = 0; i < S::kNumBars; ++i) {
            const bool p_full = i >= S::kPFull && i < S::kODone;  // P_FULL and P_FULL2
            ptx::bar_init(bars + 8u * i, p_full ? kBlockM / 32 : 1u);  // one arrival per softmax warp
        }
        *abort_flag = 0;
        ptx::bar_init_fence();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&tm_q);
        ptx::prefetch_tmap(&tm_k);
        ptx::prefetch_tmap(&tm_v);
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_addr(tmem_slot), S::kTmemCols);
        ptx::tmem_relinquish();
    }
    if constexpr (VARLEN) {
        // the packed-sequence schedule (uniform decision across the CTA);
        // offsets that do not describe sequences inside the tensors leave it
        // empty (nothing is read or written, the error word says why)
        int *sch = reinterpret_cast<int *>(smem + S::kOffSched);
        const int nb = p.B, np = p.n_pairs;
        const bool table = nb <= kSchedSeqs && np <= kSchedPairs;
        // one pass over the offsets: checked, and (for the table) each
        // sequence's pair count
        bool bad = false;
        for (int b = threadIdx.x; b < nb; b += blockDim.x) {
            const int q0 = p.cu_q[b], q1 = p.cu_q[b + 1];
            bad |= varlen_seq_bad(p, q0, q1, p.cu_k[b], p.cu_k[b + 1]);
            if (table) {
                const int len = q1 - q0;
                const int tiles = len > 0 ? (len + kBlockM - 1) / kBlockM : 0;
                sch[VarlenSched::kPairs + b] = (tiles + 1) / 2;
            }
        }
        if (__syncthreads_or(bad)) {
            if (threadIdx.x == 0) {
                atomicExch(p.err, kDeviceErrSeqLens);
                sch[VarlenSched::kItems] = 0;
                sch[VarlenSched::kRecs] = 0;
                sch[VarlenSched::kOn] = 1;
            }
        } else if (table) {
            for (int q = threadIdx.x; q < np; q += blockDim.x) {
                int c = 0;
                for (int b = 0; b < nb; ++b) c += sch[VarlenSched::kPairs + b] > q ? 1 : 0;
                sch[VarlenSched::kCount + q] = c;
            }
            __syncthreads();
            if (threadIdx.x == 0) {
                int off = 0;
                for (int q = np - 1; q >= 0; --q) {
                    sch[VarlenSched::kStart + q] = off;
                    off += sch[VarlenSched::kCount + q] * p.H;
                }
                sch[VarlenSched::kItems] = off;
                sch[VarlenSched::kRecs] = 0;
                sch[VarlenSched::kOn] = 1;
            }
            __syncthreads();
            // This CTA's own items, one thread per round, resolved while the
            // table is intact; then written over it as records (when every
            // CTA's rounds fit: the decision is the same in every CTA).
            const int items = sch[VarlenSched::kItems];
            const int rounds = (items + static_cast<int>(gridDim.x) - 1) / static_cast<int>(gridDim.x);
            const int r = static_cast<int>(threadIdx.x);
            const bool mine = rounds <= VarlenSched::kMaxRecs && r < rounds && work_index(r) < items;
            int pair = 0;
            Work wk{};
            if (mine) wk = resolve_work<CAUSAL, VARLEN>(p, work_index(r), sbase + S::kOffSched, &pair);
            __syncthreads();
            if (mine) {
                int *rec = sch + VarlenSched::kRec0 + VarlenSched::kRecInts * r;
                rec[0] = wk.b;
                rec[1] = wk.h;
                rec[2] = pair;
                rec[3] = wk.seq_q0;
                rec[4] = wk.seq_k0;
                rec[5] = wk.Lq;
                rec[6] = wk.Lk;
            }
            if (threadIdx.x == 0 && rounds <= VarlenSched::kMaxRecs) sch[VarlenSched::kRecs] = rounds;
        } else if (threadIdx.x == 0) {
            sch[VarlenSched::kRecs] = 0;
            sch[VarlenSched::kOn] = 0;
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp < 4) {
        // Whole warps run the producer and MMA loops (uniform control flow and
        // operands); the TMA, MMA and commit instructions come from one elected lane.
        if (warp == 0) {
            fwd_producer_qk<D, CAUSAL, VARLEN>(&tm_q, &tm_k, p, sbase, abort_flag);
        } else if (warp == 1) {
            fwd_mma<D, BF16, CAUSAL, VARLEN>(p, sbase, tmem, abort_flag);
        } else if (warp == 2) {
            fwd_producer_v<D, CAUSAL, VARLEN>(&tm_v, p, sbase, abort_flag);
        }
    } else {
        fwd_softmax<D, BF16, CAUSAL, VARLEN>(p, sbase, tmem, (warp - 4) / 4, warp % 4, lane, abort_flag);
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
cudaError_t launch_fwd_t(const CUtensorMap *maps, const FwdParams &p, int grid, cudaStream_t stream) {
    auto kern = fa_fwd_kernel<D, BF16, CAUSAL, VARLEN>;
    constexpr int kSmem = FwdShape<D>::kSmemBytes;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    kern<<<grid, kFwdThreads, kSmem, stream>>>(maps[0], maps[1], maps[2], p);
    return cudaGetLastError();
}

}  // namespace fa
