// kda_noalloc.cu -- kda_chunk_fwd_varlen_noalloc: the packed KDA forward for
// callers that cannot allocate device memory.
//
// Such callers hold no device allocator of their own: a plain C host program
// that only receives device buffers from another runtime, or a serving loop
// whose memory pool already owns all free device memory and forbids further
// cudaMalloc/cudaFree on its hot path (those calls can also synchronise the
// device). They cannot provide the scratch workspace kda_chunk_fwd_varlen asks
// for, so this variant takes its scratch from a fixed array compiled into the
// library instead.
#include <mutex>

#include "kda_common.cuh"

namespace {

// The scratch array. Every GPU that loads the library holds it until the process
// exits. In host code its name is only a host-side stand-in, never a device
// address: the device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) uint8_t g_noalloc_scratch[KDA_NOALLOC_SCRATCH_BYTES];

using kda::kMaxDevices;
std::once_flag g_once[kMaxDevices];
void* g_addr[kMaxDevices];
cudaError_t g_err[kMaxDevices];

// Device address of the scratch array on the current device, looked up once per
// device (with that device current) and cached.
kda_status_t scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return KDA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return KDA_ERR_UNSUPPORTED;
    std::call_once(g_once[dev], [dev] {
        void* p = nullptr;
        g_err[dev] = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        g_addr[dev] = p;
    });
    if (g_err[dev] != cudaSuccess || g_addr[dev] == nullptr) return KDA_ERR_CUDA;
    *out = g_addr[dev];
    return KDA_OK;
}

}  // namespace

extern "C" kda_status_t kda_chunk_fwd_varlen_noalloc(
    const void* q, const void* k, const void* v, const void* g, const void* beta,
    const int32_t* segment_ids, int64_t B, int64_t T, int32_t H, int32_t d_qk, int32_t d_v,
    float scale, kda_dtype_t dtype, kda_dtype_t out_dtype, void* o, uint32_t* status_dev,
    kda_stream_t stream) {
    // Same size rule as the allocating entry point; larger problems do not fit the
    // built-in array and are refused before anything is launched.
    const size_t need = kda_chunk_fwd_varlen_workspace_size(B, T, H, d_qk, d_v, dtype);
    if (need == 0) return KDA_ERR_INVALID_ARG;
    if (need > size_t(KDA_NOALLOC_SCRATCH_BYTES)) return KDA_ERR_WORKSPACE;
    void* scratch = nullptr;
    const kda_status_t s = scratch_address(&scratch);
    if (s != KDA_OK) return s;
    // The kernels write every scratch word they later read on each call (the
    // planner resets its counters and rewrites all chunk metadata), so what an
    // earlier call left in the array does not matter and nothing is cleared here.
    return kda_chunk_fwd_varlen(q, k, v, g, beta, segment_ids, B, T, H, d_qk, d_v, scale, dtype,
                                out_dtype, o, scratch, size_t(KDA_NOALLOC_SCRATCH_BYTES),
                                status_dev, stream);
}
