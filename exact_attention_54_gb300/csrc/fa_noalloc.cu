// fa_decode_noalloc: split-KV decoding (both phases) for callers that cannot
// allocate device memory when they call in, e.g. an inference engine whose
// enqueue hook may not allocate, a latency-critical loop that cannot afford
// the device-wide synchronisation a cudaMalloc may bring, or a process whose
// device memory is already fully reserved by a pool allocator.
//
// The partial results live in a file-scope device array of fixed size that
// every GPU loading the library holds until the process exits. Host code
// cannot pass the array's name to a kernel (on the host it names a host-side
// stand-in, not device memory), so its device address is looked up once per
// device with cudaGetSymbolAddress, with that device current, on the first
// call made on that device; make that first call before any stream capture.
// Every call reuses the same array: calls whose work overlaps on the GPU (on
// different streams, or from several host threads) race on it and must be
// serialised by the caller. Nothing in it needs clearing between calls: phase
// 1 writes every partial that phase 2 reads.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "fa.h"
#include "fa_launch.h"

namespace {

static __device__ __align__(256) float g_decode_scratch[FA_NOALLOC_SCRATCH_FLOATS];

constexpr int kMaxDevices = 64;

float *scratch_address() {
    static std::mutex mu;
    static float *cache[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev] == nullptr) {
        float *p = nullptr;
        if (cudaGetSymbolAddress(reinterpret_cast<void **>(&p), g_decode_scratch) != cudaSuccess) return nullptr;
        cache[dev] = p;
    }
    return cache[dev];
}

// Rounds a float count up to a multiple of 4 floats (16 bytes), so that each
// part of the scratch starts 16-byte aligned.
long long round_up_4_floats(long long nfloats) { return (nfloats + 3) / 4 * 4; }

}  // namespace

extern "C" {

fa_status_t fa_decode_noalloc(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H,
                              int Sk, int D, int num_splits, float scale, fa_dtype_t dtype, void *stream) {
    if (!q || !k || !v || !o || !lse) return FA_ERR_NULL;
    if (dtype != FA_FP16 && dtype != FA_BF16) return FA_ERR_DTYPE;
    if (D != 64 && D != 128) return FA_ERR_HEADDIM;
    if (B < 1 || H < 1 || Sk < 1 || Sk > (1 << 30)) return FA_ERR_SHAPE;
    if (num_splits < 1 || num_splits > Sk || num_splits > FA_MAX_SPLITS) return FA_ERR_SPLITS;
    // B*H*num_splits*D may not fit 64 bits for absurd B and H: bound the head
    // count by the scratch size first (num_splits >= 1 here), then form sizes.
    if (static_cast<long long>(B) * H > FA_NOALLOC_SCRATCH_FLOATS / num_splits) return FA_ERR_SCRATCH;
    const long long parts = static_cast<long long>(B) * H * num_splits;
    const long long o_floats = round_up_4_floats(parts * D);
    const long long ml_floats = round_up_4_floats(parts);
    if (o_floats + 2 * ml_floats > FA_NOALLOC_SCRATCH_FLOATS) return FA_ERR_SCRATCH;
    if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_SCALE;
    if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v) |
         reinterpret_cast<uintptr_t>(o)) & 15u)
        return FA_ERR_ALIGN;
    if (reinterpret_cast<uintptr_t>(lse) & 3u) return FA_ERR_ALIGN;
    float *scratch = scratch_address();
    if (scratch == nullptr) return FA_ERR_CUDA;
    float *o_part = scratch;
    float *m_part = scratch + o_floats;
    float *l_part = m_part + ml_floats;
    const int BH = B * H;
    const int P = (Sk + num_splits - 1) / num_splits;
    const bool bf16 = dtype == FA_BF16;
    auto st = static_cast<cudaStream_t>(stream);
    if (fa::launch_decode_split(D, bf16, q, k, v, o_part, m_part, l_part, BH, Sk, num_splits, P,
                                scale * 1.4426950408889634f, st) != cudaSuccess)
        return FA_ERR_CUDA;
    if (fa::launch_splitkv_merge(D, bf16, o_part, m_part, l_part, o, lse, BH, num_splits, st) != cudaSuccess)
        return FA_ERR_CUDA;
    return FA_OK;
}

}  // extern "C"
