// kda_common.cuh -- helpers shared by libkda's kernels and its C entry points.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "kda.h"

namespace kda {

constexpr int kChunk = 64;  // chunk length of the chunked forward ([RFC-0026] chunk_size=64)

__host__ __device__ inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

inline kda_status_t launch_status() {
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

// Raises kernel `Func`'s dynamic shared-memory limit to `bytes` on the current device, once
// per device (the attribute belongs to the device; a process may drive several).
constexpr int kMaxDevices = 64;
template <auto Func>
cudaError_t dynamic_smem_attr(int bytes) {
    static std::once_flag once[kMaxDevices];
    static cudaError_t err[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::call_once(once[dev], [dev, bytes] {
        err[dev] = cudaFuncSetAttribute(Func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    });
    return err[dev];
}

inline int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

// ---- device helpers ----------------------------------------------------------

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// Exact test "p is a multiple of T" for 0 <= p < 2^63 without a division:
// write T = 2^s d with d odd; p is a multiple of T iff its low s bits are zero
// and (p >> s) * d^-1 mod 2^64 <= (2^64 - 1) / d (divisibility by an odd
// invariant integer through its inverse modulo 2^64: Granlund and Montgomery,
// "Division by invariant integers using multiplication", PLDI 1994, sec. 9).
struct RowStartTest {
    uint64_t inv;    // d^-1 mod 2^64
    uint64_t lim;    // (2^64 - 1) / d
    uint64_t low;    // 2^s - 1
    int shift;       // s

    static RowStartTest make(int64_t T) {   // host side, T >= 1
        RowStartTest r;
        uint64_t t = uint64_t(T);
        r.shift = 0;
        while ((t & 1u) == 0) { t >>= 1; ++r.shift; }
        uint64_t x = t;                       // Newton's iteration for the inverse
        for (int i = 0; i < 6; ++i) x *= 2u - t * x;   // correct bits: 3, 6, 12, ... >= 64
        r.inv = x;
        r.lim = ~uint64_t(0) / t;
        r.low = (uint64_t(1) << r.shift) - 1u;
        return r;
    }
    __host__ __device__ __forceinline__ bool operator()(int64_t p) const {
        const uint64_t u = uint64_t(p);
        return (u & low) == 0 && (u >> shift) * inv <= lim;
    }
};

// The short conv fused into the chunked forward: the weights ([k_conv, H*D], the forward's
// dtype) of the convs that produce q, k and v, and the conv width.
struct ConvIn {
    const void* w[3];
    int32_t k_conv;
};

// A token starts a segment when it is real (id != 0) and is the first token
// of its row or its id differs from the previous token's ([RFC-0026] §3.1.1).
// With no ids, each row is one segment: only row starts are starts.
__device__ __forceinline__ bool is_segment_start(const int32_t* seg, int64_t p,
                                                 const RowStartTest& row_start) {
    if (seg == nullptr) return row_start(p);
    const int32_t s = seg[p];
    if (s == 0) return false;
    return row_start(p) || seg[p - 1] != s;
}

__device__ __forceinline__ bool is_real(const int32_t* seg, int64_t p) {
    return seg == nullptr || seg[p] != 0;
}

}  // namespace kda

// Launchers implemented in the kernel files, called from kda_api.cu.
kda_status_t kda_launch_segids_to_cu_seqlens(const int32_t* seg, int64_t B, int64_t T,
                                             int32_t max_segs, int32_t* cu, int32_t* n_segs,
                                             cudaStream_t stream);
kda_status_t kda_launch_short_conv(const void* x, const void* w, const int32_t* seg, void* y,
                                   int64_t B, int64_t T, int64_t F, int32_t K, kda_dtype_t dtype,
                                   cudaStream_t stream);
size_t kda_chunk_workspace_bytes(int64_t B, int64_t T, int32_t H, int32_t dk, int32_t dv,
                                 kda_dtype_t dtype);
kda_status_t kda_launch_chunk_fwd(const void* q, const void* k, const void* v, const void* g,
                                  const void* beta, const int32_t* seg, int64_t B, int64_t T,
                                  int32_t H, int32_t dk, int32_t dv, float scale,
                                  kda_dtype_t dtype, void* o, void* ws, size_t ws_bytes,
                                  uint32_t* status_dev, cudaStream_t stream);
