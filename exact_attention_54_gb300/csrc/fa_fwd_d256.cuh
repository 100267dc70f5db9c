// FlashAttention-2 forward for head dimensions 256, 512 and 1024 on sm_103a.
//
// Same method as the D <= 128 kernel ("FlashAttention-2 MMA", Technical
// Details; "Adaptive High-Performance Attention Kernels in CUDA",
// Architectural Progression stages 2-4; large head dimensions are the pages'
// "GPT-4 style" (1, 16, 2048, 2048, 256) configuration): 128-row query tiles,
// online softmax over K/V tiles, O kept on chip, one LSE per row, causal tiles
// above the diagonal skipped and straddling tiles masked (k_idx <= q_idx).
//
// What changes at D = 256 is the on-chip budget. The output accumulator of
// one 128-row tile takes 256 of the 512 TMEM columns and a 128-key K or V tile
// 64 KB of shared memory, so:
//   - one query tile per work item (Q: 64 KB of shared memory),
//   - K/V tiles of 64 keys (32 KB each; K ring of 3, V ring of 2),
//   - S double-buffered in TMEM (two 64-column buffers), O in columns
//     [256, 512); P (16-bit) overwrites the first 32 columns of its S buffer.
// Because S is double-buffered, the MMA issue order per work item is
// QK(0), QK(1), PV(0), QK(2), PV(1), ...: Q K^T of tile j+1 runs while the
// softmax warps exponentiate tile j, and "S tile j is ready" also means that
// P V j-2 has finished (so P buffer j mod 2 is free again).
//
// Roles (256 threads): warp 0 TMA producer of Q and K, warp 1 MMA issuer and
// TMEM owner, warp 2 TMA producer of
// V, warps 4..7 softmax (one query row per thread). Q K^T is 16 MMAs of
// 128x64x16 per K tile; P V is 4 MMAs of 128x256x16 per V tile with P read
// from TMEM.
//
// Head dimensions above 256 (the pages' "Large Head" (1, 8, 1024, 1024, 512)
// and "Massive Head" (1, 4, 512, 512, 1024) rows) take the Split-D strategy
// ("FlashAttention-2 MMA", Supported Dispatch Strategies 3: the head
// dimension is partitioned across thread blocks). A work item is one query
// tile and one 256-column slice of the output: the
// CTA forms the full S = Q K^T (the contraction runs over all DQK columns)
// and accumulates only its slice O[:, 256 s : 256 s + 256] = P V[:, slice],
// so O still fits TMEM next to the two S buffers. Every slice of a tile sees
// the same S, the same masking and the same arithmetic, so the row statistics
// agree bit for bit; slice 0 writes the LSE. Q no longer fits shared memory
// (128 x 1024 x 2 B = 256 KB), so Q and K travel together through a 192 KB
// ring, 64 columns a stage at DQK = 512 and 128 at 1024 (a 48 KB stage: 32 KB
// of Q, 16 KB of K), with one V stage beside it; the Q re-reads per K tile
// are served by L2, which the slices of a tile share.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include "fa_launch.h"
#include "sm103_ptx.cuh"

namespace fa {
namespace d256 {

constexpr int D = 256;            // output columns per work item (the whole row at DQK = 256)
constexpr int kBlockM = 128;      // query rows per tile
constexpr int kBlockN = 64;       // keys per K/V tile
constexpr int kThreads = 256;     // 8 warps
constexpr float kRescaleThreshold = 8.0f;

template <int DQK>
struct Shape {
    static_assert(DQK % D == 0 && DQK >= D && DQK <= 1024, "head dimension");
    static constexpr bool kStream = DQK > D;              // Split-D: Q streams with K
    static constexpr int kSlices = DQK / D;               // 256-column output slices per query tile
    static constexpr int kColBlocks = D / 64;             // 64-column (128-byte) boxes per slice row
    static constexpr int kQBoxBytes = kBlockM * 128;      // 128 rows x 64 columns
    static constexpr int kKVBoxBytes = kBlockN * 128;     // 64 rows x 64 columns
    static constexpr int kQTileBytes = kStream ? 0 : kBlockM * D * 2;  // resident Q: 64 KB
    static constexpr int kKVTileBytes = kBlockN * D * 2;  // V tile of one slice: 32 KB
    // One ring stage: a K tile (resident Q), or kChunkCols columns of Q and of
    // K: 64 at DQK = 512 (24 KB stages), 128 at DQK = 1024 (48 KB; with 64 the
    // extra waits per K tile cost more than the earlier starts gain).
    static constexpr int kChunkCols = kStream ? (DQK <= 512 ? 64 : 128) : D;
    static constexpr int kChunks = DQK / kChunkCols;      // ring stages per S tile
    static constexpr int kStageK = kStream ? kBlockM * kChunkCols * 2 : 0;  // K's offset in a stage
    static constexpr int kStageBytes = kStageK + kBlockN * kChunkCols * 2;
    // Streaming (Split-D) keeps more of the Q/K ring in flight: each stage
    // is consumed in a few hundred cycles and the ring must cover an L2 round
    // trip; one V stage suffices, its next tile has a whole Q K^T and softmax
    // period to land.
    static constexpr int kKStages = kStream ? 192 * 1024 / kStageBytes : 3;
    static constexpr int kVStages = kStream ? 1 : 2;
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kOffQ + kQTileBytes;
    static constexpr int kOffV = kOffK + kKStages * kStageBytes;
    static constexpr int kOffBar = kOffV + kVStages * kKVTileBytes;
    static constexpr int kQFull = 0, kQEmpty = 1, kTeardown = 2;
    static constexpr int kKFull = 3;
    static constexpr int kKEmpty = kKFull + kKStages;
    static constexpr int kVFull = kKEmpty + kKStages;
    static constexpr int kVEmpty = kVFull + kVStages;
    static constexpr int kSFull = kVEmpty + kVStages;  // +b: S buffer b written (MMA commit)
    static constexpr int kPFull = kSFull + 2;          // +b: P in buffer b written, O corrected (4 warps)
    static constexpr int kPDone = kPFull + 2;          // +b: the P V product from buffer b finished (MMA commit)
    static constexpr int kNumBars = kPDone + 2;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + slack to align the base to 1024
    static constexpr uint32_t kTmemS = 0;                     // + b * 64
    static constexpr uint32_t kTmemO = 256;
    static constexpr uint32_t kTmemCols = 512;
    static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

// One unit of work: one 128-row query tile of one (sequence, head) and, for
// DQK > 256, one 256-column slice of its output.
struct Work {
    int b, h;
    int slice;           // output columns [256 slice, 256 slice + 256)
    int seq_q0, seq_k0;  // token offsets of the sequence (varlen), else 0
    int Lq, Lk;          // query and key lengths of the sequence
    int q_start;         // first query row of the tile (relative to the sequence)
    int rows;            // valid rows of the tile (0 = inactive)
    int n_kv;            // K/V tiles the tile visits
};

template <int DQK, bool CAUSAL, bool VARLEN>
__device__ __forceinline__ Work get_work(const FwdParams &p, int w) {
    constexpr int NS = Shape<DQK>::kSlices;
    Work k;
    const int units = p.B * p.H * NS;
    const int qt = p.n_qtiles - 1 - w / units;  // longest causal work first
    const int u = w % units;                    // the slices of a tile run side by side
    const int bh = u / NS;
    k.slice = u % NS;
    k.b = bh / p.H;
    k.h = bh % p.H;
    if constexpr (VARLEN) {
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
    const int nk_all = (k.Lk + kBlockN - 1) / kBlockN;
    k.q_start = qt * kBlockM;
    const int rows = k.Lq - k.q_start;
    k.rows = rows <= 0 ? 0 : (rows < kBlockM ? rows : kBlockM);
    int nkv = 0;
    if (k.rows > 0) {
        nkv = nk_all;
        if (CAUSAL) {
            const int last = (k.q_start + k.rows - 1) / kBlockN + 1;
            nkv = last < nk_all ? last : nk_all;
        }
    }
    k.n_kv = nkv;
    return k;
}

// Work items of this launch. Packed sequences: the count each CTA stored
// after checking the sequence offsets (0 when they are inconsistent).
template <int DQK, bool VARLEN>
__device__ __forceinline__ int num_items(const FwdParams &p, uint32_t sbase) {
    if constexpr (VARLEN) {
        int v;
        asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(sbase + Shape<DQK>::kOffMisc + 8));
        return v;
    }
    return p.num_work;
}

// Static persistent schedule: round r hands out items [r*G, (r+1)*G) in
// alternating direction, so heavy early items and light late items balance.
__device__ __forceinline__ int work_index(int r) {
    const int G = static_cast<int>(gridDim.x);
    const int pos = (r & 1) ? (G - 1 - static_cast<int>(blockIdx.x)) : static_cast<int>(blockIdx.x);
    return r * G + pos;
}

// Columns [col0, col0 + 64 NBOX) of rows [row0, row0 + box rows) of
// (sequence/head) into `dst`, one box per 64 columns.
template <int NBOX, bool VARLEN>
__device__ __forceinline__ void load_rows(const CUtensorMap *tm, uint32_t dst, uint32_t box_bytes, uint32_t bar,
                                          const Work &wk, int seq0, int row0, int H, int col0) {
#pragma unroll
    for (int c = 0; c < NBOX; ++c) {
        if constexpr (VARLEN)
            ptx::tma_load_3d(dst + c * box_bytes, tm, bar, col0 + c * 64, wk.h, seq0 + row0);
        else
            ptx::tma_load_3d(dst + c * box_bytes, tm, bar, col0 + c * 64, row0, wk.b * H + wk.h);
    }
}

// Waits (bounded) for the newest of `count` loads into a ring of `stages`
// buffers: nothing may leave with copies in flight, even after an abort.
__device__ __forceinline__ void drain_ring(uint32_t full0, uint32_t stages, uint32_t count, uint64_t timeout_ns) {
    for (uint32_t s = 0; s < stages && s < count; ++s) {
        const uint32_t last = (count - 1) - ((count - 1 - s) % stages);
        ptx::bar_wait(full0 + 8u * s, (last / stages) & 1, nullptr, timeout_ns);
    }
}

template <int DQK, bool CAUSAL, bool VARLEN>
__device__ void producer_qk(const CUtensorMap *tq, const CUtensorMap *tk, const FwdParams &p, uint32_t sbase,
                            volatile int *abort_flag) {
    using S = Shape<DQK>;
    constexpr int kBoxes = S::kChunkCols / 64;
    const uint32_t bars = sbase + S::kOffBar;
    auto bar = [&](int i) { return bars + 8u * static_cast<uint32_t>(i); };
    auto wait = [&](int i, uint32_t parity) {
        return ptx::warp_all(ptx::bar_wait(bar(i), parity, abort_flag, p.timeout_ns));
    };
    const bool leader = ptx::elect_one();
    uint32_t it = 0, wi = 0;
    bool ok = true;
    for (int r = 0; ok; ++r) {
        const int w = work_index(r);
        if (w >= num_items<DQK, VARLEN>(p, sbase)) break;
        const Work wk = get_work<DQK, CAUSAL, VARLEN>(p, w);
        if (wk.n_kv == 0) continue;
        if (!S::kStream && wi > 0 && !(ok = wait(S::kQEmpty, (wi - 1) & 1))) break;
        if (!S::kStream && leader) {
            ptx::bar_arrive_expect_tx(bar(S::kQFull), S::kQTileBytes);
            load_rows<S::kColBlocks, VARLEN>(tq, sbase + S::kOffQ, S::kQBoxBytes, bar(S::kQFull), wk, wk.seq_q0,
                                             wk.q_start, p.H, 0);
        }
        for (int j = 0; j < wk.n_kv && ok; ++j) {
            for (int c = 0; c < S::kChunks; ++c, ++it) {
                const uint32_t stage = it % S::kKStages;
                if (it >= S::kKStages && !(ok = wait(S::kKEmpty + stage, ((it / S::kKStages) - 1) & 1))) break;
                if (leader) {
                    const uint32_t dst = sbase + S::kOffK + stage * S::kStageBytes;
                    ptx::bar_arrive_expect_tx(bar(S::kKFull + stage), S::kStageBytes);
                    if constexpr (S::kStream)
                        load_rows<kBoxes, VARLEN>(tq, dst, S::kQBoxBytes, bar(S::kKFull + stage), wk, wk.seq_q0,
                                                  wk.q_start, p.H, c * S::kChunkCols);
                    load_rows<kBoxes, VARLEN>(tk, dst + S::kStageK, S::kKVBoxBytes, bar(S::kKFull + stage), wk,
                                              wk.seq_k0, j * kBlockN, p.H, c * S::kChunkCols);
                }
            }
        }
        ++wi;
    }
    drain_ring(bar(S::kKFull), S::kKStages, it, p.timeout_ns);
    if (!S::kStream) drain_ring(bar(S::kQFull), 1, wi, p.timeout_ns);
}

template <int DQK, bool CAUSAL, bool VARLEN>
__device__ void producer_v(const CUtensorMap *tv, const FwdParams &p, uint32_t sbase, volatile int *abort_flag) {
    using S = Shape<DQK>;
    const uint32_t bars = sbase + S::kOffBar;
    auto bar = [&](int i) { return bars + 8u * static_cast<uint32_t>(i); };
    const bool leader = ptx::elect_one();
    uint32_t it = 0;
    bool ok = true;
    for (int r = 0; ok; ++r) {
        const int w = work_index(r);
        if (w >= num_items<DQK, VARLEN>(p, sbase)) break;
        const Work wk = get_work<DQK, CAUSAL, VARLEN>(p, w);
        for (int j = 0; j < wk.n_kv; ++j, ++it) {
            const uint32_t stage = it % S::kVStages;
            if (it >= S::kVStages &&
                !(ok = ptx::warp_all(ptx::bar_wait(bar(S::kVEmpty + stage), ((it / S::kVStages) - 1) & 1, abort_flag,
                                     p.timeout_ns))))
                break;
            if (leader && !withheld(p.withhold, it)) {
                ptx::bar_arrive_expect_tx(bar(S::kVFull + stage), S::kKVTileBytes);
                load_rows<S::kColBlocks, VARLEN>(tv, sbase + S::kOffV + stage * S::kKVTileBytes, S::kKVBoxBytes,
                                                 bar(S::kVFull + stage), wk, wk.seq_k0, j * kBlockN, p.H,
                                                 wk.slice * D);
            }
        }
    }
    drain_ring(bar(S::kVFull), S::kVStages, it, p.timeout_ns);
}

template <int DQK, bool BF16, bool CAUSAL, bool VARLEN>
__device__ void mma_role(const FwdParams &p, uint32_t sbase, uint32_t tmem, volatile int *abort_flag) {
    using S = Shape<DQK>;
    constexpr uint32_t kIdescQK = ptx::idesc_f16(BF16, kBlockM, kBlockN, false);
    constexpr uint32_t kIdescPV = ptx::idesc_f16(BF16, kBlockM, D, true);
    const uint32_t bars = sbase + S::kOffBar;
    auto bar = [&](int i) { return bars + 8u * static_cast<uint32_t>(i); };
    auto wait = [&](int i, uint32_t parity) {
        return ptx::warp_all(ptx::bar_wait(bar(i), parity, abort_flag, p.timeout_ns));
    };
    const bool leader = ptx::elect_one();
    // Descriptors are built once; each MMA advances the start-address field
    // only. V is MN-major: its four 64-column boxes are one box (8 KB) apart,
    // 8-key atoms 1 KB apart.
    const uint64_t dq = ptx::smem_desc_sw128(sbase + S::kOffQ, 16, 1024);
    const uint64_t dk0 = ptx::smem_desc_sw128(sbase + S::kOffK, 16, 1024);
    const uint64_t dv0 = ptx::smem_desc_sw128(sbase + S::kOffV, S::kKVBoxBytes, 1024);
    constexpr uint64_t kKVTile16 = S::kKVTileBytes >> 4;
    constexpr uint64_t kStage16 = S::kStageBytes >> 4;

    // S = Q K^T for tile t into S buffer t mod 2: DQK / 16 MMAs of K = 16,
    // over kChunks ring stages (Q from the stage too when it streams).
    auto qk = [&](uint32_t t) -> bool {
        const uint32_t dst = tmem + S::kTmemS + (t & 1) * kBlockN;
        for (int c = 0; c < S::kChunks; ++c) {
            const uint32_t u = t * S::kChunks + c;
            const uint32_t ks = u % S::kKStages;
            if (!wait(S::kKFull + ks, (u / S::kKStages) & 1)) return false;
            if (leader) {
                const uint64_t sd = dk0 + static_cast<uint64_t>(ks) * kStage16;
                const uint64_t qd = S::kStream ? sd : dq;
                const uint64_t kd = sd + (S::kStageK >> 4);
#pragma unroll
                for (int kk = 0; kk < S::kChunkCols / 16; ++kk) {
                    const uint64_t qo = (kk / 4) * (S::kQBoxBytes >> 4) + (kk % 4) * 2;
                    const uint64_t ko = (kk / 4) * (S::kKVBoxBytes >> 4) + (kk % 4) * 2;
                    ptx::mma_ss(dst, qd + qo, kd + ko, kIdescQK, (c > 0 || kk > 0) ? 1u : 0u);
                }
                ptx::mma_commit(bar(S::kKEmpty + ks));
            }
        }
        if (leader) ptx::mma_commit(bar(S::kSFull + (t & 1)));
        return true;
    };
    // O (+)= P V for tile t (4 MMAs of K = 16 keys, N = 256).
    auto pv = [&](uint32_t t, bool accumulate) -> bool {
        const uint32_t b = t & 1;
        const uint32_t vs = t % S::kVStages;
        if (!wait(S::kVFull + vs, (t / S::kVStages) & 1)) return false;
        if (!wait(S::kPFull + b, (t >> 1) & 1)) return false;
        ptx::tc_fence_after();  // P was written by tcgen05.st in other threads
        if (leader) {
            const uint64_t vd = dv0 + static_cast<uint64_t>(vs) * kKVTile16;
            const uint32_t pa = tmem + S::kTmemS + b * kBlockN;
#pragma unroll
            for (int kk = 0; kk < kBlockN / 16; ++kk)
                ptx::mma_ts(tmem + S::kTmemO, pa + kk * 8, vd + kk * (2048 >> 4), kIdescPV,
                            (accumulate || kk > 0) ? 1u : 0u);
            ptx::mma_commit(bar(S::kPDone + b));
            ptx::mma_commit(bar(S::kVEmpty + vs));
        }
        return true;
    };

    uint32_t g = 0, wi = 0;
    bool ok = true;
    for (int r = 0; ok; ++r) {
        const int w = work_index(r);
        if (w >= num_items<DQK, VARLEN>(p, sbase)) break;
        const Work wk = get_work<DQK, CAUSAL, VARLEN>(p, w);
        const int n = wk.n_kv;
        if (n == 0) continue;
        if (!S::kStream && !(ok = wait(S::kQFull, wi & 1))) break;
        const uint32_t g0 = g;
        if (!(ok = qk(g0))) break;
        if (n > 1 && !(ok = qk(g0 + 1))) break;
        // every Q K^T of this tile issued: the resident Q may be replaced
        if (!S::kStream && n <= 2 && leader) ptx::mma_commit(bar(S::kQEmpty));
        for (int i = 0; i < n && ok; ++i) {
            const uint32_t t = g0 + i;
            if (!(ok = pv(t, i > 0))) break;
            if (i + 2 < n) {
                if (!(ok = qk(t + 2))) break;
                if (!S::kStream && i + 3 == n && leader) ptx::mma_commit(bar(S::kQEmpty));
            }
        }
        if (!ok) break;
        g += n;
        ++wi;
    }
    if (leader) ptx::mma_commit(bar(S::kTeardown));
    __syncwarp();
    ptx::bar_wait(bar(S::kTeardown), 0, nullptr, p.timeout_ns);
}

template <int DQK, bool BF16, bool CAUSAL, bool VARLEN>
__device__ void softmax_role(const FwdParams &p, uint32_t sbase, uint32_t tmem, int wq, int lane,
                             volatile int *abort_flag) {
    using S = Shape<DQK>;
    using Elem = uint16_t;
    const uint32_t bars = sbase + S::kOffBar;
    auto bar = [&](int i) { return bars + 8u * static_cast<uint32_t>(i); };
    constexpr unsigned kFull = 0xffffffffu;
    auto wait = [&](int i, uint32_t parity) {
        return __all_sync(kFull, ptx::bar_wait(bar(i), parity, abort_flag, p.timeout_ns));
    };
    const int row = wq * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tO = tmem + lane_base + S::kTmemO;
    const float scale_log2 = p.scale_log2;
    uint32_t g = 0;
    bool ok = true;

    for (int r = 0; ok; ++r) {
        const int w = work_index(r);
        if (w >= num_items<DQK, VARLEN>(p, sbase)) break;
        const Work wk = get_work<DQK, CAUSAL, VARLEN>(p, w);
        const int n = wk.n_kv;
        if (n == 0) continue;
        const int q_row = wk.q_start + row;
        const bool row_valid = row < wk.rows;
        float m_used = -CUDART_INF_F;
        float l = 0.f;

        for (int i = 0; i < n; ++i, ++g) {
            const uint32_t b = g & 1;
            if (!(ok = wait(S::kSFull + b, (g >> 1) & 1))) break;
            ptx::tc_fence_after();
            const uint32_t tS = tmem + lane_base + S::kTmemS + b * kBlockN;
            // the row maximum comes with the loads (tcgen05.ld.red); a masked
            // tile takes it again after the mask
            uint32_t s[2][32];
            float mr[2];
            ptx::tmem_ld32_max(tS, s[0], mr[0]);
            ptx::tmem_ld32_max(tS + 32, s[1], mr[1]);
            ptx::tmem_ld_wait();
            ptx::reg_fence(s[0]);
            ptx::reg_fence(s[1]);
            asm volatile("" : "+f"(mr[0]), "+f"(mr[1]));

            const int k0 = i * kBlockN;
            const bool need_mask = (k0 + kBlockN > wk.Lk) || (CAUSAL && k0 + kBlockN - 1 > wk.q_start);
            float mx = fmaxf(mr[0], mr[1]);
            if (need_mask) {
                // the row sees columns c < lim: the sequence's end and, causal, its own position
                int lim = wk.Lk - k0;
                if (CAUSAL) lim = min(lim, q_row + 1 - k0);
#pragma unroll
                for (int c = 0; c < kBlockN; ++c)
                    if (c >= lim) s[c / 32][c % 32] = 0xff800000u;  // -inf
                float mx4[4] = {-CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F};
#pragma unroll
                for (int c = 0; c < kBlockN; c += 2)
                    mx4[(c / 2) % 4] = ptx::fmax3(mx4[(c / 2) % 4], __uint_as_float(s[c / 32][c % 32]),
                                                  __uint_as_float(s[(c + 1) / 32][(c + 1) % 32]));
                mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
            }
            const float m_cand = mx * scale_log2;
            const bool need = m_cand > m_used + kRescaleThreshold;
            float alpha = 1.f;
            if (need) {
                alpha = ptx::ex2(m_used - m_cand);  // 0 on the first tile (m_used = -inf)
                m_used = m_cand;
            }
            l *= alpha;
            const float m_sub = (m_used == -CUDART_INF_F) ? 0.f : m_used;

            // P = 2^(s * scale_log2 - m): 32 columns of 16-bit pairs over the
            // start of this S buffer (free: S tile g ready => P V g-2 done).
            const uint64_t scale2 = ptx::pk2(scale_log2, scale_log2);
            const uint64_t negm2 = ptx::pk2(-m_sub, -m_sub);
            uint64_t sum2[2] = {ptx::pk2(0.f, 0.f), ptx::pk2(0.f, 0.f)};
            uint32_t pk[32];
#pragma unroll
            for (int k = 0; k < 32; ++k) {
                const int c = 2 * k;
                const uint64_t xx = ptx::ffma2(ptx::pk2(__uint_as_float(s[c / 32][c % 32]),
                                                        __uint_as_float(s[(c + 1) / 32][(c + 1) % 32])),
                                               scale2, negm2);
                float x0, x1;
                ptx::upk2(xx, x0, x1);
                const float e0 = ptx::ex2(x0), e1 = ptx::ex2(x1);
                sum2[k % 2] = ptx::fadd2(sum2[k % 2], ptx::pk2(e0, e1));
                pk[k] = ptx::pack2<BF16>(e0, e1);
            }
            ptx::tmem_st32(tS, pk);
            {
                float a0, a1, b0, b1;
                ptx::upk2(sum2[0], a0, a1);
                ptx::upk2(sum2[1], b0, b1);
                l += (a0 + a1) + (b0 + b1);
            }
            // O *= alpha once the previous P V has landed (only when a row of
            // this warp moved its maximum).
            if (i > 0 && __any_sync(kFull, need)) {
                const uint32_t t = g - 1;
                if (!(ok = wait(S::kPDone + (t & 1), (t >> 1) & 1))) break;
                ptx::tc_fence_after();
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t o[32];
                    ptx::tmem_ld32(tO + c * 32, o);
                    ptx::tmem_ld_wait();
                    ptx::reg_fence(o);
#pragma unroll
                    for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
                    ptx::tmem_st32(tO + c * 32, o);
                }
            }
            ptx::tmem_st_wait();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::bar_arrive(bar(S::kPFull + b));
        }
        if (!ok) break;

        // Epilogue: O / l in the input dtype, LSE = (m + log2 l) ln 2. The last
        // P V is the newest on its buffer; the one before it on that buffer
        // (tile g-3) is covered by S tile g-1 being ready.
        {
            const uint32_t t = g - 1;
            if (!(ok = wait(S::kPDone + (t & 1), (t >> 1) & 1))) break;
            ptx::tc_fence_after();
        }
        const float inv_l = l > 0.f ? 1.f / l : 0.f;
        Elem *orow;  // this slice's 256 columns of the output row
        if constexpr (VARLEN)
            orow = static_cast<Elem *>(p.o) + (static_cast<size_t>(wk.seq_q0 + q_row) * p.H + wk.h) * DQK;
        else
            orow = static_cast<Elem *>(p.o) + (static_cast<size_t>(wk.b * p.H + wk.h) * p.Sq + q_row) * DQK;
        orow += wk.slice * D;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            ptx::tmem_ld32(tO + c * 32, o);
            ptx::tmem_ld_wait();
            ptx::reg_fence(o);
            uint32_t pk[16];
#pragma unroll
            for (int k = 0; k < 16; ++k)
                pk[k] = ptx::pack2<BF16>(__uint_as_float(o[2 * k]) * inv_l, __uint_as_float(o[2 * k + 1]) * inv_l);
            if (row_valid) {
                uint4 *dst = reinterpret_cast<uint4 *>(orow + c * 32);
#pragma unroll
                for (int k = 0; k < 4; ++k) dst[k] = make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
            }
        }
        if (row_valid && wk.slice == 0) {
            const float lse = l > 0.f ? (m_used + __log2f(l)) * 0.69314718055994531f : -CUDART_INF_F;
            if constexpr (VARLEN)
                p.lse[static_cast<size_t>(wk.h) * p.total_q + wk.seq_q0 + q_row] = lse;
            else
                p.lse[static_cast<size_t>(wk.b * p.H + wk.h) * p.Sq + q_row] = lse;
        }
        // O is read: the next tile's first P V (issued only after this warp's
        // next P_FULL arrival) may overwrite it.
        ptx::tc_fence_before();
    }
}

template <int DQK, bool BF16, bool CAUSAL, bool VARLEN>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_d256_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
    using S = Shape<DQK>;
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
            const bool by_warps = i >= S::kPFull && i < S::kPDone;  // one arrival per softmax warp
            ptx::bar_init(bars + 8u * i, by_warps ? kBlockM / 32 : 1u);
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
        // offsets that do not describe sequences inside the tensors: no work
        // (nothing is read or written; the error word says why)
        const bool offsets_ok = varlen_offsets_ok(p);
        if (threadIdx.x == 0) *reinterpret_cast<int *>(smem + S::kOffMisc + 8) = offsets_ok ? p.num_work : 0;
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        producer_qk<DQK, CAUSAL, VARLEN>(&tm_q, &tm_k, p, sbase, abort_flag);
    } else if (warp == 1) {
        mma_role<DQK, BF16, CAUSAL, VARLEN>(p, sbase, tmem, abort_flag);
    } else if (warp == 2) {
        producer_v<DQK, CAUSAL, VARLEN>(&tm_v, p, sbase, abort_flag);
    } else if (warp >= 4) {
        softmax_role<DQK, BF16, CAUSAL, VARLEN>(p, sbase, tmem, warp - 4, lane, abort_flag);
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

template <int DQK, bool BF16, bool CAUSAL, bool VARLEN>
cudaError_t launch(const CUtensorMap *maps, const FwdParams &p, int grid, cudaStream_t stream) {
    auto kern = fa_fwd_d256_kernel<DQK, BF16, CAUSAL, VARLEN>;
    constexpr int kSmem = Shape<DQK>::kSmemBytes;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    kern<<<grid, kThreads, kSmem, stream>>>(maps[0], maps[1], maps[2], p);
    return cudaGetLastError();
}

}  // namespace d256
}  // namespace fa
