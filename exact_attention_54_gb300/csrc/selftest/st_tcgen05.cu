// Test-only kernels (libfa_selftest.so) that exercise the sm_103a building
// blocks of the forward kernel one at a time, with the same helpers and the
// same shared-memory / TMEM layouts:
//   fa_selftest_qk       C[128x128] = A[128xD] B[128xD]^T: TMA (128-byte
//                        swizzle) + tcgen05.mma with two K-major smem operands
//   fa_selftest_pv       C[128xD] = P[128x128] V[128xD]: P written to TMEM
//                        with tcgen05.st, V MN-major from smem (TS form)
//   fa_selftest_tn       C[128xD] = X^T Y for X [128x128], Y [128xD]: X is loaded
//                        like any 128-row tile and read by the MMA as an
//                        MN-major A operand (the backward pass's dQ = dS K
//                        reads dS^T this way), Y as an MN-major B operand
//   fa_selftest_ldmax    x[128x32] fp32 written to TMEM and read back with the
//                        reducing load (tcgen05.ld.red max): the values and
//                        each row's maximum, as the forward's softmax uses it
//   fa_selftest_watchdog a bounded wait on a barrier nobody arrives at; the
//                        kernel must give up, release TMEM and report it
// Each kernel writes 0 (done) or 1 (a wait timed out) to *status.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <mutex>

#include "sm103_ptx.cuh"

namespace {

using namespace fa;

template <int D>
struct StShape {
    static constexpr int kTile = 128 * D * 2;
    static constexpr int kBlock = 128 * 128;
    static constexpr int kOffA = 0;
    static constexpr int kOffB = kTile;
    static constexpr int kOffBar = 2 * kTile;
    static constexpr int kSmem = kOffBar + 64 + 1024;
};

__device__ uint8_t *align1024(uint8_t *p) {
    return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

template <int D, bool BF16>
__global__ void __launch_bounds__(128, 1)
    st_qk_kernel(const __grid_constant__ CUtensorMap ta, const __grid_constant__ CUtensorMap tb, float *c,
                 int *status, unsigned long long timeout_ns) {
    using S = StShape<D>;
    extern __shared__ uint8_t raw[];
    uint8_t *smem = align1024(raw);
    const uint32_t sb = ptx::smem_addr(smem);
    const uint32_t bar_load = sb + S::kOffBar, bar_mma = bar_load + 8;
    uint32_t *slot = reinterpret_cast<uint32_t *>(smem + S::kOffBar + 16);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + S::kOffBar + 20);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (threadIdx.x == 0) {
        ptx::bar_init(bar_load, 1);
        ptx::bar_init(bar_mma, 1);
        *abort_flag = 0;
        ptx::bar_init_fence();
    }
    if (warp == 0) {
        ptx::tmem_alloc(ptx::smem_addr(slot), 128);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *slot;
    if (threadIdx.x == 0) {
        ptx::bar_arrive_expect_tx(bar_load, 2 * S::kTile);
        for (int b = 0; b < D / 64; ++b) {
            ptx::tma_load_3d(sb + S::kOffA + b * S::kBlock, &ta, bar_load, b * 64, 0, 0);
            ptx::tma_load_3d(sb + S::kOffB + b * S::kBlock, &tb, bar_load, b * 64, 0, 0);
        }
        if (ptx::bar_wait(bar_load, 0, abort_flag, timeout_ns)) {
            ptx::tc_fence_after();
            constexpr uint32_t idesc = ptx::idesc_f16(BF16, 128, 128, false);
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = (kk / 4) * S::kBlock + (kk % 4) * 32;
                ptx::mma_ss(tmem, ptx::smem_desc_sw128(sb + S::kOffA + off, 16, 1024),
                            ptx::smem_desc_sw128(sb + S::kOffB + off, 16, 1024), idesc, kk > 0);
            }
            ptx::mma_commit(bar_mma);
            ptx::bar_wait(bar_mma, 0, nullptr, timeout_ns);
        } else {
            ptx::bar_wait(bar_load, 0, nullptr, timeout_ns);  // drain the copies
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (!*abort_flag) {
        const int row = warp * 32 + lane;
        for (int ch = 0; ch < 4; ++ch) {
            uint32_t r[32];
            ptx::tmem_ld32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + ch * 32, r);
            ptx::tmem_ld_wait();
            ptx::reg_fence(r);
            for (int i = 0; i < 32; ++i) c[row * 128 + ch * 32 + i] = __uint_as_float(r[i]);
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 128);
    }
    if (threadIdx.x == 0) *status = *abort_flag ? 1 : 0;
}

template <int D, bool BF16>
__global__ void __launch_bounds__(128, 1)
    st_pv_kernel(const uint16_t *p, const __grid_constant__ CUtensorMap tv, float *c, int *status,
                 unsigned long long timeout_ns) {
    using S = StShape<D>;
    extern __shared__ uint8_t raw[];
    uint8_t *smem = align1024(raw);
    const uint32_t sb = ptx::smem_addr(smem);
    const uint32_t bar_load = sb + S::kOffBar, bar_mma = bar_load + 8;
    uint32_t *slot = reinterpret_cast<uint32_t *>(smem + S::kOffBar + 16);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + S::kOffBar + 20);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int row = warp * 32 + lane;
    if (threadIdx.x == 0) {
        ptx::bar_init(bar_load, 1);
        ptx::bar_init(bar_mma, 1);
        *abort_flag = 0;
        ptx::bar_init_fence();
    }
    if (warp == 0) {
        ptx::tmem_alloc(ptx::smem_addr(slot), 256);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *slot;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    if (threadIdx.x == 0) {
        ptx::bar_arrive_expect_tx(bar_load, S::kTile);
        for (int b = 0; b < D / 64; ++b) ptx::tma_load_3d(sb + S::kOffA + b * S::kBlock, &tv, bar_load, b * 64, 0, 0);
    }
    // P row -> TMEM columns [0, 64) of this thread's lane, two 16-bit values per column
    {
        const uint32_t *prow = reinterpret_cast<const uint32_t *>(p + row * 128);
        uint32_t w0[32], w1[32];
        for (int i = 0; i < 32; ++i) {
            w0[i] = prow[i];
            w1[i] = prow[32 + i];
        }
        ptx::tmem_st32(tmem + lane_base, w0);
        ptx::tmem_st32(tmem + lane_base + 32, w1);
        ptx::tmem_st_wait();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (threadIdx.x == 0) {
        if (ptx::bar_wait(bar_load, 0, abort_flag, timeout_ns)) {
            constexpr uint32_t idesc = ptx::idesc_f16(BF16, 128, D, true);
            for (int kk = 0; kk < 8; ++kk)
                ptx::mma_ts(tmem + 128, tmem + kk * 8, ptx::smem_desc_sw128(sb + S::kOffA + kk * 2048, S::kBlock, 1024),
                            idesc, kk > 0);
            ptx::mma_commit(bar_mma);
            ptx::bar_wait(bar_mma, 0, nullptr, timeout_ns);
        } else {
            ptx::bar_wait(bar_load, 0, nullptr, timeout_ns);
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (!*abort_flag) {
        for (int ch = 0; ch < D / 32; ++ch) {
            uint32_t r[32];
            ptx::tmem_ld32(tmem + lane_base + 128 + ch * 32, r);
            ptx::tmem_ld_wait();
            ptx::reg_fence(r);
            for (int i = 0; i < 32; ++i) c[row * D + ch * 32 + i] = __uint_as_float(r[i]);
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 256);
    }
    if (threadIdx.x == 0) *status = *abort_flag ? 1 : 0;
}

// C = X^T Y: 8 MMAs of K = 16 (rows of X and Y), both operands MN-major.
template <int D, bool BF16>
__global__ void __launch_bounds__(128, 1)
    st_tn_kernel(const __grid_constant__ CUtensorMap tx, const __grid_constant__ CUtensorMap ty, float *c, int *status,
                 unsigned long long timeout_ns) {
    constexpr int kBox = 128 * 128;
    constexpr int kOffX = 0, kOffY = 2 * kBox, kOffBar = kOffY + (D / 64) * kBox;
    extern __shared__ uint8_t raw[];
    uint8_t *smem = align1024(raw);
    const uint32_t sb = ptx::smem_addr(smem);
    const uint32_t bar_load = sb + kOffBar, bar_mma = bar_load + 8;
    uint32_t *slot = reinterpret_cast<uint32_t *>(smem + kOffBar + 16);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kOffBar + 20);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (threadIdx.x == 0) {
        ptx::bar_init(bar_load, 1);
        ptx::bar_init(bar_mma, 1);
        *abort_flag = 0;
        ptx::bar_init_fence();
    }
    if (warp == 0) {
        ptx::tmem_alloc(ptx::smem_addr(slot), 128);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *slot;
    if (threadIdx.x == 0) {
        ptx::bar_arrive_expect_tx(bar_load, (2 + D / 64) * kBox);
        for (int b = 0; b < 2; ++b) ptx::tma_load_3d(sb + kOffX + b * kBox, &tx, bar_load, b * 64, 0, 0);
        for (int b = 0; b < D / 64; ++b) ptx::tma_load_3d(sb + kOffY + b * kBox, &ty, bar_load, b * 64, 0, 0);
        if (ptx::bar_wait(bar_load, 0, abort_flag, timeout_ns)) {
            constexpr uint32_t idesc = ptx::idesc_f16(BF16, 128, D, true, true);
            for (int kk = 0; kk < 8; ++kk)
                ptx::mma_ss(tmem, ptx::smem_desc_sw128(sb + kOffX + kk * 2048, kBox, 1024),
                            ptx::smem_desc_sw128(sb + kOffY + kk * 2048, kBox, 1024), idesc, kk > 0);
            ptx::mma_commit(bar_mma);
            ptx::bar_wait(bar_mma, 0, nullptr, timeout_ns);
        } else {
            ptx::bar_wait(bar_load, 0, nullptr, timeout_ns);
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (!*abort_flag) {
        const int row = warp * 32 + lane;
        for (int ch = 0; ch < D / 32; ++ch) {
            uint32_t r[32];
            ptx::tmem_ld32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + ch * 32, r);
            ptx::tmem_ld_wait();
            ptx::reg_fence(r);
            for (int i = 0; i < 32; ++i) c[row * D + ch * 32 + i] = __uint_as_float(r[i]);
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 128);
    }
    if (threadIdx.x == 0) *status = *abort_flag ? 1 : 0;
}

// Writes x[128][32] into 32 TMEM columns (row r in lane r) and reads it back
// with tmem_ld32_max: y gets the values, mx each row's maximum.
__global__ void __launch_bounds__(128, 1) st_ldmax_kernel(const float *x, float *y, float *mx) {
    __shared__ uint32_t slot;
    const int warp = threadIdx.x / 32;
    if (warp == 0) {
        ptx::tmem_alloc(ptx::smem_addr(&slot), 32);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t taddr = slot + (static_cast<uint32_t>(warp * 32) << 16);
    uint32_t w[32];
    for (int c = 0; c < 32; ++c) w[c] = __float_as_uint(x[threadIdx.x * 32 + c]);
    ptx::tmem_st32(taddr, w);
    ptx::tmem_st_wait();
    float m;
    ptx::tmem_ld32_max(taddr, w, m);
    ptx::tmem_ld_wait();
    ptx::reg_fence(w);
    for (int c = 0; c < 32; ++c) y[threadIdx.x * 32 + c] = __uint_as_float(w[c]);
    mx[threadIdx.x] = m;
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(slot, 32);
    }
}

// Waits on a barrier that never completes, while holding TMEM, and must come
// back on its own after timeout_ns with the TMEM released.
__global__ void __launch_bounds__(128, 1) st_watchdog_kernel(int *status, unsigned long long timeout_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t slot;
    __shared__ int abort_flag;
    const int warp = threadIdx.x / 32;
    if (threadIdx.x == 0) {
        ptx::bar_init(ptx::smem_addr(&bar), 1);
        abort_flag = 0;
        ptx::bar_init_fence();
    }
    if (warp == 0) {
        ptx::tmem_alloc(ptx::smem_addr(&slot), 32);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    // every thread waits; the first to time out raises the flag for the rest
    ptx::bar_wait(ptx::smem_addr(&bar), 0, &abort_flag, timeout_ns);
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(slot, 32);
    }
    if (threadIdx.x == 0) *status = abort_flag ? 1 : 0;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// A [rows, D] row-major 16-bit matrix as a 3-D map {D, rows, 1} with 64 x rows x 1 boxes.
bool encode_rows(CUtensorMap *m, const void *base, int rows, int D, bool bf16) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows), 1};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(D) * 2 * rows};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(rows), 1};
    const cuuint32_t es[3] = {1, 1, 1};
    return fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void *>(base),
              dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A [128, D] row-major 16-bit matrix as a 3-D map {D, 128, 1} with 64x128x1 boxes.
bool encode_128xD(CUtensorMap *m, const void *base, int D, bool bf16) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), 128, 1};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(D) * 2 * 128};
    const cuuint32_t box[3] = {64, 128, 1};
    const cuuint32_t es[3] = {1, 1, 1};
    return fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void *>(base),
              dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, bool BF16>
int run_qk(const void *a, const void *b, float *c, int *status, unsigned long long t, cudaStream_t st) {
    CUtensorMap ma, mb;
    if (!encode_128xD(&ma, a, D, BF16) || !encode_128xD(&mb, b, D, BF16)) return -2;
    auto k = st_qk_kernel<D, BF16>;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, StShape<D>::kSmem) != cudaSuccess) return -3;
    k<<<1, 128, StShape<D>::kSmem, st>>>(ma, mb, c, status, t);
    return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

template <int D, bool BF16>
int run_pv(const void *p, const void *v, float *c, int *status, unsigned long long t, cudaStream_t st) {
    CUtensorMap mv;
    if (!encode_128xD(&mv, v, D, BF16)) return -2;
    auto k = st_pv_kernel<D, BF16>;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, StShape<D>::kSmem) != cudaSuccess) return -3;
    k<<<1, 128, StShape<D>::kSmem, st>>>(static_cast<const uint16_t *>(p), mv, c, status, t);
    return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

template <int D, bool BF16>
int run_tn(const void *x, const void *y, float *c, int *status, unsigned long long t, cudaStream_t st) {
    CUtensorMap mx, my;
    if (!encode_rows(&mx, x, 128, 128, BF16) || !encode_rows(&my, y, 128, D, BF16)) return -2;
    auto k = st_tn_kernel<D, BF16>;
    constexpr int kSmem = (2 + D / 64) * 128 * 128 + 64 + 1024;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) != cudaSuccess) return -3;
    k<<<1, 128, kSmem, st>>>(mx, my, c, status, t);
    return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

// Does nothing: launched with a kernel's grid, block and dynamic shared
// memory, its event-timed duration is the fixed cost of such a launch (block
// scheduling, shared-memory carve-out, completion) with no work in it.
__global__ void st_empty_kernel() {}

}  // namespace

extern "C" {

__attribute__((visibility("default"))) int fa_selftest_qk(const void *a, const void *b, float *c, int D, int bf16,
                                                          int *status, unsigned long long timeout_ns, void *stream) {
    auto st = static_cast<cudaStream_t>(stream);
    if (D == 64) return bf16 ? run_qk<64, true>(a, b, c, status, timeout_ns, st) : run_qk<64, false>(a, b, c, status, timeout_ns, st);
    if (D == 128) return bf16 ? run_qk<128, true>(a, b, c, status, timeout_ns, st) : run_qk<128, false>(a, b, c, status, timeout_ns, st);
    return -1;
}

__attribute__((visibility("default"))) int fa_selftest_pv(const void *p, const void *v, float *c, int D, int bf16,
                                                          int *status, unsigned long long timeout_ns, void *stream) {
    auto st = static_cast<cudaStream_t>(stream);
    if (D == 64) return bf16 ? run_pv<64, true>(p, v, c, status, timeout_ns, st) : run_pv<64, false>(p, v, c, status, timeout_ns, st);
    if (D == 128) return bf16 ? run_pv<128, true>(p, v, c, status, timeout_ns, st) : run_pv<128, false>(p, v, c, status, timeout_ns, st);
    return -1;
}

// x [128,128], y [128,D] row-major 16-bit; c [128,D] fp32 = x^T y. D: 64 or 128.
__attribute__((visibility("default"))) int fa_selftest_tn(const void *x, const void *y, float *c, int D, int bf16,
                                                          int *status, unsigned long long timeout_ns, void *stream) {
    auto st = static_cast<cudaStream_t>(stream);
    if (D == 64) return bf16 ? run_tn<64, true>(x, y, c, status, timeout_ns, st) : run_tn<64, false>(x, y, c, status, timeout_ns, st);
    if (D == 128) return bf16 ? run_tn<128, true>(x, y, c, status, timeout_ns, st) : run_tn<128, false>(x, y, c, status, timeout_ns, st);
    return -1;
}

__attribute__((visibility("default"))) int fa_selftest_watchdog(int *status, unsigned long long timeout_ns,
                                                                void *stream) {
    st_watchdog_kernel<<<1, 128, 0, static_cast<cudaStream_t>(stream)>>>(status, timeout_ns);
    return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

__attribute__((visibility("default"))) int fa_selftest_ldmax(const float *x, float *y, float *mx, void *stream) {
    if (!x || !y || !mx) return -1;
    st_ldmax_kernel<<<1, 128, 0, static_cast<cudaStream_t>(stream)>>>(x, y, mx);
    return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

__attribute__((visibility("default"))) int fa_selftest_empty_launch(int grid, int block, int smem_bytes,
                                                                    void *stream) {
    if (grid < 1 || grid > 65535 || block < 1 || block > 1024 || smem_bytes < 0 || smem_bytes > 227 * 1024)
        return -1;
    if (cudaFuncSetAttribute(st_empty_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes) != cudaSuccess)
        return -3;
    st_empty_kernel<<<grid, block, smem_bytes, static_cast<cudaStream_t>(stream)>>>();
    return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

}  // extern "C"
