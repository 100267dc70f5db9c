// C ABI of libfa.so (declared in include/fa.h): argument validation, TMA tensor
// map encoding and kernel launches. Allocates no memory; the only state is one
// device-resident error word per GPU.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <atomic>
#include <mutex>

#include "fa.h"
#include "fa_launch.h"

namespace {

__device__ int g_device_error_word = 0;

constexpr int kMaxDevices = 64;

// Address of the error word on the current device (looked up once per device).
// Test support (fa_test_withhold_load): the load to withhold and the wait
// limit every launch uses.
std::atomic<int> g_withhold{0};
std::atomic<unsigned long long> g_wait_limit_ns{fa::kWaitTimeoutNs};

int *device_error_word() {
    static std::mutex mu;
    static int *cache[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_error_word) != cudaSuccess) return nullptr;
        cache[dev] = static_cast<int *>(p);
    }
    return cache[dev];
}

int num_sms() {
    static std::mutex mu;
    static int cache[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cache[dev] = n;
    }
    return cache[dev];
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

// 3-D map over a 16-bit tensor whose innermost dimension is D, with 64 x 1 x
// 128 or 64 x 128 x 1 boxes and 128-byte swizzle (rows of 128 bytes land in
// shared memory in the layout the MMA descriptors describe). Out-of-range
// rows read as zero.
bool encode_map(CUtensorMap *m, bool bf16, const void *base, uint64_t d0, uint64_t d1, uint64_t d2,
                uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box1, uint32_t box2) {
    auto fn = encode_fn();
    if (fn == nullptr) return false;
    const cuuint64_t dims[3] = {d0, d1, d2};
    const cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
    const cuuint32_t box[3] = {64, box1, box2};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                          const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 3-D map over an fp32 dQ accumulator with 32-column boxes and 128-byte
// swizzle: the target of the backward pass's bulk reductions. Dense
// [B*H][Sq][D]: dims {D, Sq, B*H}, boxes 32 x rows x 1; packed [T][H][D]:
// dims {D, H, T}, boxes 32 x 1 x rows.
bool encode_map_f32(CUtensorMap *m, void *base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t stride1_bytes,
                    uint64_t stride2_bytes, uint32_t box1, uint32_t box2) {
    auto fn = encode_fn();
    if (fn == nullptr) return false;
    const cuuint64_t dims[3] = {d0, d1, d2};
    const cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
    const cuuint32_t box[3] = {32, box1, box2};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Work units per group of the backward's CTA order: the group's Q, dO and fp32
// dQ accumulator rows (8 L D bytes per unit of L query rows) within 32 MB, a
// quarter of L2.
int bwd_units_per_group(long long units, long long rows, int D) {
    const long long per_unit = 8LL * (rows > 0 ? rows : 1) * D;
    const long long g = (32LL << 20) / per_unit;
    return static_cast<int>(g < 1 ? 1 : (g > units ? units : g));
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

bool scale_ok(float s) { return std::isfinite(s) && s > 0.f; }

constexpr float kLog2e = 1.4426950408889634f;

// Forward head dimensions: 64 and 128 (two query tiles per work item), 256
// (one), 512 and 1024 (Split-D: one query tile and 256 output columns).
bool fwd_head_dim_ok(int D) { return D == 64 || D == 128 || D == 256 || D == 512 || D == 1024; }

long long fwd_work_items(int D, long long heads, int Sq) {
    const long long n_qtiles = (Sq + 127) / 128;
    if (D >= 256) return heads * n_qtiles * (D / 256);
    return heads * ((n_qtiles + 1) / 2);
}
constexpr int kMaxLen = 1 << 30;

}  // namespace

extern "C" {

int fa_version(void) { return 200; }

const char *fa_status_string(fa_status_t s) {
    switch (s) {
        case FA_OK: return "ok";
        case FA_ERR_NULL: return "a required pointer is NULL";
        case FA_ERR_SHAPE: return "invalid or too large tensor shape";
        case FA_ERR_HEADDIM: return "unsupported head dimension (forward: 64, 128, 256, 512, 1024; decode and backward: 64, 128)";
        case FA_ERR_DTYPE: return "dtype must be FA_FP16 or FA_BF16";
        case FA_ERR_ALIGN: return "tensor pointer is not 16-byte aligned";
        case FA_ERR_SPLITS: return "num_splits must be in [1, min(Sk, FA_MAX_SPLITS)]";
        case FA_ERR_SCALE: return "scale must be finite and positive";
        case FA_ERR_CUDA: return "CUDA runtime error";
        case FA_ERR_DEVICE_TIMEOUT: return "a kernel abandoned a barrier wait (device timeout)";
        case FA_ERR_SCRATCH: return "problem larger than the built-in decode scratch";
        case FA_ERR_DEVICE_INDEX: return "a kernel met an out-of-range block-table entry";
        case FA_ERR_WORKSPACE: return "workspace smaller than fa_bwd_workspace_bytes()";
        case FA_ERR_DEVICE_SEQLENS:
            return "cu_seqlens do not describe sequences inside total_q/total_k, or a query sequence is longer "
                   "than max_seqlen_q (nothing was computed)";
    }
    return "unknown status";
}

fa_status_t fa_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H, int Sq, int Sk,
                   int D, int causal, float scale, fa_dtype_t dtype, void *stream) {
    if (!q || !k || !v || !o || !lse) return FA_ERR_NULL;
    if (dtype != FA_FP16 && dtype != FA_BF16) return FA_ERR_DTYPE;
    if (!fwd_head_dim_ok(D)) return FA_ERR_HEADDIM;
    if (B < 1 || H < 1 || Sq < 1 || Sk < 1 || Sq > kMaxLen || Sk > kMaxLen) return FA_ERR_SHAPE;
    const long long BH = static_cast<long long>(B) * H;
    const long long n_pairs = ((Sq + 127) / 128 + 1) / 2;
    const long long n_work = fwd_work_items(D, BH, Sq);
    if (BH > INT_MAX || n_work > INT_MAX) return FA_ERR_SHAPE;
    if (!scale_ok(scale)) return FA_ERR_SCALE;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned4(lse)) return FA_ERR_ALIGN;

    const bool bf16 = dtype == FA_BF16;
    CUtensorMap maps[3];
    const uint64_t row = static_cast<uint64_t>(D) * 2;
    const uint32_t kv_rows = D >= 256 ? 64 : 128;  // K/V tile height of the kernel that runs
    if (!encode_map(&maps[0], bf16, q, D, Sq, BH, row, row * Sq, 128, 1) ||
        !encode_map(&maps[1], bf16, k, D, Sk, BH, row, row * Sk, kv_rows, 1) ||
        !encode_map(&maps[2], bf16, v, D, Sk, BH, row, row * Sk, kv_rows, 1))
        return FA_ERR_CUDA;
    int *err = device_error_word();
    const int sms = num_sms();
    if (err == nullptr || sms <= 0) return FA_ERR_CUDA;

    fa::FwdParams p{};
    p.o = o;
    p.lse = lse;
    p.B = B;
    p.H = H;
    p.Sq = Sq;
    p.Sk = Sk;
    p.total_q = 0;
    p.n_pairs = static_cast<int>(n_pairs);
    p.n_qtiles = (Sq + 127) / 128;
    p.num_work = static_cast<int>(n_work);
    p.scale_log2 = scale * kLog2e;
    p.err = err;
    p.timeout_ns = g_wait_limit_ns.load();
    p.withhold = g_withhold.load();
    const int grid = p.num_work < sms ? p.num_work : sms;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    const cudaError_t e = D > 256    ? fa::launch_fwd_splitd(D, bf16, causal != 0, false, maps, p, grid, st)
                          : D == 256 ? fa::launch_fwd_d256(bf16, causal != 0, false, maps, p, grid, st)
                                     : fa::launch_fwd_dense(D, bf16, causal != 0, maps, p, grid, st);
    return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status_t fa_fwd_varlen(const void *q, const void *k, const void *v, void *o, float *lse,
                          const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k, int num_seqs, int total_q,
                          int total_k, int max_seqlen_q, int H, int D, int causal, float scale, fa_dtype_t dtype,
                          void *stream) {
    if (!q || !k || !v || !o || !lse || !cu_seqlens_q || !cu_seqlens_k) return FA_ERR_NULL;
    if (dtype != FA_FP16 && dtype != FA_BF16) return FA_ERR_DTYPE;
    if (!fwd_head_dim_ok(D)) return FA_ERR_HEADDIM;
    if (num_seqs < 1 || total_q < 1 || total_k < 1 || max_seqlen_q < 1 || H < 1 || max_seqlen_q > kMaxLen ||
        total_q > kMaxLen || total_k > kMaxLen)
        return FA_ERR_SHAPE;
    const long long SH = static_cast<long long>(num_seqs) * H;
    const long long n_pairs = ((max_seqlen_q + 127) / 128 + 1) / 2;
    const long long n_work = fwd_work_items(D, SH, max_seqlen_q);
    if (SH > INT_MAX || n_work > INT_MAX) return FA_ERR_SHAPE;
    if (!scale_ok(scale)) return FA_ERR_SCALE;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned4(lse)) return FA_ERR_ALIGN;

    const bool bf16 = dtype == FA_BF16;
    CUtensorMap maps[3];
    const uint64_t row = static_cast<uint64_t>(D) * 2;
    const uint64_t tok = row * H;
    const uint32_t kv_rows = D >= 256 ? 64 : 128;
    if (!encode_map(&maps[0], bf16, q, D, H, total_q, row, tok, 1, 128) ||
        !encode_map(&maps[1], bf16, k, D, H, total_k, row, tok, 1, kv_rows) ||
        !encode_map(&maps[2], bf16, v, D, H, total_k, row, tok, 1, kv_rows))
        return FA_ERR_CUDA;
    int *err = device_error_word();
    const int sms = num_sms();
    if (err == nullptr || sms <= 0) return FA_ERR_CUDA;

    fa::FwdParams p{};
    p.o = o;
    p.lse = lse;
    p.cu_q = cu_seqlens_q;
    p.cu_k = cu_seqlens_k;
    p.B = num_seqs;
    p.H = H;
    p.Sq = max_seqlen_q;
    p.Sk = 0;
    p.total_q = total_q;
    p.total_k = total_k;
    p.n_pairs = static_cast<int>(n_pairs);
    p.n_qtiles = (max_seqlen_q + 127) / 128;
    p.num_work = static_cast<int>(n_work);
    p.scale_log2 = scale * kLog2e;
    p.err = err;
    p.timeout_ns = g_wait_limit_ns.load();
    p.withhold = g_withhold.load();
    const int grid = p.num_work < sms ? p.num_work : sms;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    const cudaError_t e = D > 256    ? fa::launch_fwd_splitd(D, bf16, causal != 0, true, maps, p, grid, st)
                          : D == 256 ? fa::launch_fwd_d256(bf16, causal != 0, true, maps, p, grid, st)
                                     : fa::launch_fwd_varlen(D, bf16, causal != 0, maps, p, grid, st);
    return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status_t fa_decode_splitkv(const void *q, const void *k, const void *v, float *o_part, float *m_part,
                              float *l_part, int B, int H, int Sk, int D, int num_splits, float scale,
                              fa_dtype_t dtype, void *stream) {
    if (!q || !k || !v || !o_part || !m_part || !l_part) return FA_ERR_NULL;
    if (dtype != FA_FP16 && dtype != FA_BF16) return FA_ERR_DTYPE;
    if (D != 64 && D != 128) return FA_ERR_HEADDIM;
    if (B < 1 || H < 1 || Sk < 1 || Sk > kMaxLen) return FA_ERR_SHAPE;
    if (num_splits < 1 || num_splits > Sk || num_splits > FA_MAX_SPLITS) return FA_ERR_SPLITS;
    const long long BH = static_cast<long long>(B) * H;
    if (BH * num_splits > INT_MAX) return FA_ERR_SHAPE;
    if (!scale_ok(scale)) return FA_ERR_SCALE;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned4(o_part) || !aligned4(m_part) ||
        !aligned4(l_part))
        return FA_ERR_ALIGN;
    const int P = (Sk + num_splits - 1) / num_splits;
    const cudaError_t e = fa::launch_decode_split(D, dtype == FA_BF16, q, k, v, o_part, m_part, l_part,
                                                  static_cast<int>(BH), Sk, num_splits, P, scale * kLog2e,
                                                  static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status_t fa_decode_paged_splitkv(const void *q, const void *k_cache, const void *v_cache,
                                    const int32_t *block_table, const int32_t *seq_lens, float *o_part,
                                    float *m_part, float *l_part, int B, int H, int D, int num_blocks,
                                    int block_size, int max_blocks_per_seq, int num_splits, float scale,
                                    fa_dtype_t dtype, void *stream) {
    if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !o_part || !m_part || !l_part)
        return FA_ERR_NULL;
    if (dtype != FA_FP16 && dtype != FA_BF16) return FA_ERR_DTYPE;
    if (D != 64 && D != 128) return FA_ERR_HEADDIM;
    if (B < 1 || H < 1 || num_blocks < 1 || max_blocks_per_seq < 1) return FA_ERR_SHAPE;
    if (block_size < 1 || block_size > 1024 || (block_size & (block_size - 1)) != 0) return FA_ERR_SHAPE;
    if (static_cast<long long>(max_blocks_per_seq) * block_size > kMaxLen) return FA_ERR_SHAPE;
    if (num_splits < 1 || num_splits > FA_MAX_SPLITS) return FA_ERR_SPLITS;
    const long long BH = static_cast<long long>(B) * H;
    if (BH * num_splits > INT_MAX || static_cast<long long>(num_blocks) * H > INT_MAX) return FA_ERR_SHAPE;
    if (!scale_ok(scale)) return FA_ERR_SCALE;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned4(block_table) ||
        !aligned4(seq_lens) || !aligned4(o_part) || !aligned4(m_part) || !aligned4(l_part))
        return FA_ERR_ALIGN;
    int *err = device_error_word();
    if (err == nullptr) return FA_ERR_CUDA;
    int log2_bs = 0;
    while ((1 << log2_bs) < block_size) ++log2_bs;
    fa::DecodeParams p{};
    p.q = static_cast<const uint16_t *>(q);
    p.k = static_cast<const uint16_t *>(k_cache);
    p.v = static_cast<const uint16_t *>(v_cache);
    p.o_part = o_part;
    p.m_part = m_part;
    p.l_part = l_part;
    p.H = H;
    p.num_splits = num_splits;
    p.scale_log2 = scale * kLog2e;
    p.block_table = block_table;
    p.seq_lens = seq_lens;
    p.max_blocks = max_blocks_per_seq;
    p.log2_bs = log2_bs;
    p.num_blocks = num_blocks;
    p.err = err;
    const cudaError_t e =
        fa::launch_decode_split_paged(D, dtype == FA_BF16, p, static_cast<int>(BH), static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status_t fa_decode_splitkv_fused(const void *q, const void *k, const void *v, void *o, float *lse, float *o_part,
                                    float *m_part, float *l_part, int32_t *counters, int B, int H, int Sk, int D,
                                    int num_splits, float scale, fa_dtype_t dtype, void *stream) {
    if (!q || !k || !v || !o || !lse || !o_part || !m_part || !l_part || !counters) return FA_ERR_NULL;
    if (dtype != FA_FP16 && dtype != FA_BF16) return FA_ERR_DTYPE;
    if (D != 64 && D != 128) return FA_ERR_HEADDIM;
    if (B < 1 || H < 1 || Sk < 1 || Sk > kMaxLen) return FA_ERR_SHAPE;
    if (num_splits < 1 || num_splits > Sk || num_splits > FA_MAX_SPLITS) return FA_ERR_SPLITS;
    const long long BH = static_cast<long long>(B) * H;
    if (BH * num_splits > INT_MAX) return FA_ERR_SHAPE;
    if (!scale_ok(scale)) return FA_ERR_SCALE;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned4(lse) || !aligned4(o_part) ||
        !aligned4(m_part) || !aligned4(l_part) || !aligned4(counters))
        return FA_ERR_ALIGN;
    fa::DecodeParams p{};
    p.q = static_cast<const uint16_t *>(q);
    p.k = static_cast<const uint16_t *>(k);
    p.v = static_cast<const uint16_t *>(v);
    p.o_part = o_part;
    p.m_part = m_part;
    p.l_part = l_part;
    p.H = H;
    p.Sk = Sk;
    p.num_splits = num_splits;
    p.keys_per_split = (Sk + num_splits - 1) / num_splits;
    p.scale_log2 = scale * kLog2e;
    p.o = o;
    p.lse = lse;
    p.counters = counters;
    const cudaError_t e = fa::launch_decode_fused(D, dtype == FA_BF16, false, p, static_cast<int>(BH),
                                                  static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status_t fa_decode_paged_splitkv_fused(const void *q, const void *k_cache, const void *v_cache,
                                          const int32_t *block_table, const int32_t *seq_lens, void *o, float *lse,
                                          float *o_part, float *m_part, float *l_part, int32_t *counters, int B,
                                          int H, int D, int num_blocks, int block_size, int max_blocks_per_seq,
                                          int num_splits, float scale, fa_dtype_t dtype, void *stream) {
    if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !o || !lse || !o_part || !m_part || !l_part ||
        !counters)
        return FA_ERR_NULL;
    if (dtype != FA_FP16 && dtype != FA_BF16) return FA_ERR_DTYPE;
    if (D != 64 && D != 128) return FA_ERR_HEADDIM;
    if (B < 1 || H < 1 || num_blocks < 1 || max_blocks_per_seq < 1) return FA_ERR_SHAPE;
    if (block_size < 1 || block_size > 1024 || (block_size & (block_size - 1)) != 0) return FA_ERR_SHAPE;
    if (static_cast<long long>(max_blocks_per_seq) * block_size > kMaxLen) return FA_ERR_SHAPE;
    if (num_splits < 1 || num_splits > FA_MAX_SPLITS) return FA_ERR_SPLITS;
    const long long BH = static_cast<long long>(B) * H;
    if (BH * num_splits > INT_MAX || static_cast<long long>(num_blocks) * H > INT_MAX) return FA_ERR_SHAPE;
    if (!scale_ok(scale)) return FA_ERR_SCALE;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned4(block_table) ||
        !aligned4(seq_lens) || !aligned16(o) || !aligned4(lse) || !aligned4(o_part) || !aligned4(m_part) ||
        !aligned4(l_part) || !aligned4(counters))
        return FA_ERR_ALIGN;
    int *err = device_error_word();
    if (err == nullptr) return FA_ERR_CUDA;
    int log2_bs = 0;
    while ((1 << log2_bs) < block_size) ++log2_bs;
    fa::DecodeParams p{};
    p.q = static_cast<const uint16_t *>(q);
    p.k = static_cast<const uint16_t *>(k_cache);
    p.v = static_cast<const uint16_t *>(v_cache);
    p.o_part = o_part;
    p.m_part = m_part;
    p.l_part = l_part;
    p.H = H;
    p.num_splits = num_splits;
    p.scale_log2 = scale * kLog2e;
    p.block_table = block_table;
    p.seq_lens = seq_lens;
    p.max_blocks = max_blocks_per_seq;
    p.log2_bs = log2_bs;
    p.num_blocks = num_blocks;
    p.err = err;
    p.o = o;
    p.lse = lse;
    p.counters = counters;
    const cudaError_t e = fa::launch_decode_fused(D, dtype == FA_BF16, true, p, static_cast<int>(BH),
                                                  static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

size_t fa_bwd_workspace_bytes(int B, int H, int Sq, int D) {
    if (B < 1 || H < 1 || Sq < 1 || Sq > kMaxLen || (D != 64 && D != 128)) return 0;
    const long long BH = static_cast<long long>(B) * H;
    if (BH > INT_MAX) return 0;
    const long long pad = (static_cast<long long>(Sq) + 127) / 128 * 128;
    // + 16 bytes: the main kernel's work counter
    return static_cast<size_t>(BH * Sq * D + 2 * BH * pad) * sizeof(float) + 16;
}

fa_status_t fa_bwd(const void *q, const void *k, const void *v, const void *o, const void *dout, const float *lse,
                   void *dq, void *dk, void *dv, float *workspace, size_t workspace_bytes, int B, int H, int Sq,
                   int Sk, int D, int causal, float scale, fa_dtype_t dtype, void *stream) {
    if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv || !workspace) return FA_ERR_NULL;
    if (dtype != FA_FP16 && dtype != FA_BF16) return FA_ERR_DTYPE;
    if (D != 64 && D != 128) return FA_ERR_HEADDIM;
    if (B < 1 || H < 1 || Sq < 1 || Sk < 1 || Sq > kMaxLen || Sk > kMaxLen) return FA_ERR_SHAPE;
    const long long BH = static_cast<long long>(B) * H;
    const long long n_kt = (Sk + 127) / 128;
    if (BH > INT_MAX || BH * n_kt > INT_MAX) return FA_ERR_SHAPE;
    if (!scale_ok(scale)) return FA_ERR_SCALE;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) || !aligned4(lse) ||
        !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(workspace))
        return FA_ERR_ALIGN;
    const size_t need = fa_bwd_workspace_bytes(B, H, Sq, D);
    if (need == 0) return FA_ERR_SHAPE;
    if (workspace_bytes < need) return FA_ERR_WORKSPACE;

    const bool bf16 = dtype == FA_BF16;
    CUtensorMap maps[5];
    const uint64_t row = static_cast<uint64_t>(D) * 2;
    const uint32_t q_rows = D == 128 ? 64 : 128;  // query rows per step of the kernel that runs
    if (!encode_map(&maps[0], bf16, q, D, Sq, BH, row, row * Sq, q_rows, 1) ||
        !encode_map(&maps[1], bf16, k, D, Sk, BH, row, row * Sk, 128, 1) ||
        !encode_map(&maps[2], bf16, v, D, Sk, BH, row, row * Sk, 128, 1) ||
        !encode_map(&maps[3], bf16, dout, D, Sq, BH, row, row * Sq, q_rows, 1) ||
        !encode_map_f32(&maps[4], workspace, D, Sq, BH, D * 4, D * 4 * static_cast<uint64_t>(Sq), q_rows, 1))
        return FA_ERR_CUDA;
    int *err = device_error_word();
    if (err == nullptr) return FA_ERR_CUDA;

    fa::BwdParams p{};
    p.BH = static_cast<int>(BH);
    p.Sq = Sq;
    p.Sk = Sk;
    p.n_qtiles = (Sq + 127) / 128;
    p.n_ktiles = static_cast<int>(n_kt);
    p.Sq_pad = p.n_qtiles * 128;
    p.heads_per_group = bwd_units_per_group(BH, Sq, D);
    p.dq_acc = workspace;
    p.lse2 = workspace + static_cast<size_t>(BH) * Sq * D;
    p.delta = p.lse2 + static_cast<size_t>(BH) * p.Sq_pad;
    p.work_counter = reinterpret_cast<int *>(p.delta + static_cast<size_t>(BH) * p.Sq_pad);
    p.total_units = static_cast<int>(BH * n_kt);
    p.grid = num_sms();
    if (p.grid <= 0) return FA_ERR_CUDA;
    p.dk = dk;
    p.dv = dv;
    p.scale = scale;
    p.scale_log2 = scale * kLog2e;
    p.err = err;
    p.timeout_ns = g_wait_limit_ns.load();
    p.withhold = g_withhold.load();
    const cudaError_t e = fa::launch_bwd_dense(D, bf16, causal != 0, maps, o, dout, lse, dq, p,
                                         static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

size_t fa_bwd_varlen_workspace_bytes(int total_q, int H, int D) {
    if (total_q < 1 || H < 1 || total_q > kMaxLen || (D != 64 && D != 128)) return 0;
    const long long TH = static_cast<long long>(total_q) * H;
    if (TH > INT_MAX) return 0;
    return static_cast<size_t>(TH * D + 2 * TH) * sizeof(float) + 16;  // + the work counter
}

fa_status_t fa_bwd_varlen(const void *q, const void *k, const void *v, const void *o, const void *dout,
                          const float *lse, void *dq, void *dk, void *dv, float *workspace, size_t workspace_bytes,
                          const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k, int num_seqs, int total_q,
                          int total_k, int max_seqlen_q, int max_seqlen_k, int H, int D, int causal, float scale,
                          fa_dtype_t dtype, void *stream) {
    if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv || !workspace || !cu_seqlens_q || !cu_seqlens_k)
        return FA_ERR_NULL;
    if (dtype != FA_FP16 && dtype != FA_BF16) return FA_ERR_DTYPE;
    if (D != 64 && D != 128) return FA_ERR_HEADDIM;
    if (num_seqs < 1 || total_q < 1 || total_k < 1 || max_seqlen_q < 1 || max_seqlen_k < 1 || H < 1 ||
        total_q > kMaxLen || total_k > kMaxLen || max_seqlen_q > kMaxLen || max_seqlen_k > kMaxLen)
        return FA_ERR_SHAPE;
    const long long units = static_cast<long long>(num_seqs) * H;
    const long long n_kt = (max_seqlen_k + 127) / 128;
    if (units > INT_MAX || units * n_kt > INT_MAX || static_cast<long long>(total_q) * H > INT_MAX ||
        static_cast<long long>(total_k) * H > INT_MAX)
        return FA_ERR_SHAPE;
    if (!scale_ok(scale)) return FA_ERR_SCALE;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) || !aligned4(lse) ||
        !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(workspace) || !aligned4(cu_seqlens_q) ||
        !aligned4(cu_seqlens_k))
        return FA_ERR_ALIGN;
    const size_t need = fa_bwd_varlen_workspace_bytes(total_q, H, D);
    if (need == 0) return FA_ERR_SHAPE;
    if (workspace_bytes < need) return FA_ERR_WORKSPACE;

    const bool bf16 = dtype == FA_BF16;
    CUtensorMap maps[5];
    const uint64_t row = static_cast<uint64_t>(D) * 2;
    const uint64_t tok = row * H;
    const uint32_t q_rows = D == 128 ? 64 : 128;  // query rows per step of the kernel that runs
    if (!encode_map(&maps[0], bf16, q, D, H, total_q, row, tok, 1, q_rows) ||
        !encode_map(&maps[1], bf16, k, D, H, total_k, row, tok, 1, 128) ||
        !encode_map(&maps[2], bf16, v, D, H, total_k, row, tok, 1, 128) ||
        !encode_map(&maps[3], bf16, dout, D, H, total_q, row, tok, 1, q_rows) ||
        !encode_map_f32(&maps[4], workspace, D, H, total_q, D * 4, D * 4 * static_cast<uint64_t>(H), 1, q_rows))
        return FA_ERR_CUDA;
    int *err = device_error_word();
    if (err == nullptr) return FA_ERR_CUDA;

    fa::BwdParams p{};
    p.BH = static_cast<int>(units);
    p.Sq = max_seqlen_q;
    p.Sk = max_seqlen_k;
    p.n_qtiles = (max_seqlen_q + 127) / 128;
    p.n_ktiles = static_cast<int>(n_kt);
    p.Sq_pad = 0;
    p.heads_per_group = bwd_units_per_group(units, max_seqlen_q, D);
    p.cu_q = cu_seqlens_q;
    p.cu_k = cu_seqlens_k;
    p.H = H;
    p.total_q = total_q;
    p.total_k = total_k;
    p.dq_acc = workspace;
    p.lse2 = workspace + static_cast<size_t>(total_q) * H * D;
    p.delta = p.lse2 + static_cast<size_t>(total_q) * H;
    p.work_counter = reinterpret_cast<int *>(p.delta + static_cast<size_t>(total_q) * H);
    p.total_units = p.BH * p.n_ktiles;
    p.grid = num_sms();
    if (p.grid <= 0) return FA_ERR_CUDA;
    p.dk = dk;
    p.dv = dv;
    p.scale = scale;
    p.scale_log2 = scale * kLog2e;
    p.err = err;
    p.timeout_ns = g_wait_limit_ns.load();
    p.withhold = g_withhold.load();
    const cudaError_t e = fa::launch_bwd_varlen(D, bf16, causal != 0, maps, o, dout, lse, dq, p,
                                                static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status_t fa_splitkv_merge(const float *o_part, const float *m_part, const float *l_part, void *o, float *lse,
                             int B, int H, int D, int num_splits, fa_dtype_t dtype, void *stream) {
    if (!o_part || !m_part || !l_part || !o || !lse) return FA_ERR_NULL;
    if (dtype != FA_FP16 && dtype != FA_BF16) return FA_ERR_DTYPE;
    if (D != 64 && D != 128) return FA_ERR_HEADDIM;
    if (B < 1 || H < 1) return FA_ERR_SHAPE;
    if (num_splits < 1 || num_splits > FA_MAX_SPLITS) return FA_ERR_SPLITS;
    const long long BH = static_cast<long long>(B) * H;
    if (BH > INT_MAX) return FA_ERR_SHAPE;
    if (!aligned4(o_part) || !aligned4(m_part) || !aligned4(l_part) || !aligned16(o) || !aligned4(lse))
        return FA_ERR_ALIGN;
    const cudaError_t e = fa::launch_splitkv_merge(D, dtype == FA_BF16, o_part, m_part, l_part, o, lse,
                                                   static_cast<int>(BH), num_splits,
                                                   static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status_t fa_test_withhold_load(int load, unsigned long long wait_limit_ns) {
    if (load < 0) return FA_ERR_SHAPE;
    g_withhold.store(load);
    g_wait_limit_ns.store(wait_limit_ns == 0 ? fa::kWaitTimeoutNs : wait_limit_ns);
    return FA_OK;
}

fa_status_t fa_check_device_error(void *stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_CUDA;
    int *err = device_error_word();
    if (err == nullptr) return FA_ERR_CUDA;
    int host = 0;
    if (cudaMemcpy(&host, err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return FA_ERR_CUDA;
    if (host == 0) return FA_OK;
    const int zero = 0;
    if (cudaMemcpy(err, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return FA_ERR_CUDA;
    if (host == fa::kDeviceErrBadIndex) return FA_ERR_DEVICE_INDEX;
    if (host == fa::kDeviceErrSeqLens) return FA_ERR_DEVICE_SEQLENS;
    return FA_ERR_DEVICE_TIMEOUT;
}

}  // extern "C"
