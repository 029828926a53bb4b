// kda_common.cuh -- helpers shared by libkda's kernels and its C entry points.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda.h"

namespace kda {

constexpr int kChunk = 64;  // chunk length of the chunked forward ([RFC-0026] chunk_size=64)

__host__ __device__ inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

inline kda_status_t launch_status() {
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
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

// A token starts a segment when it is real (id != 0) and is the first token
// of its row or its id differs from the previous token's ([RFC-0026] §3.1.1).
// With no ids, each row is one segment: only row starts are starts.
__device__ __forceinline__ bool is_segment_start(const int32_t* seg, int64_t p, int64_t T) {
    if (seg == nullptr) return (p % T) == 0;
    const int32_t s = seg[p];
    if (s == 0) return false;
    return (p % T) == 0 || seg[p - 1] != s;
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
