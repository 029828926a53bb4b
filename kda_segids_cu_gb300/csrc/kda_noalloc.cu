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
std::mutex g_mutex[kMaxDevices];
void* g_addr[kMaxDevices];

// Device address of the scratch array on the current device, looked up with that
// device current. Only a successful lookup is cached: after a failure (for instance a
// first call made during stream capture, or a transient context error) the next call
// on that device tries again.
kda_status_t scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return KDA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return KDA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mutex[dev]);
    if (g_addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
            (void)cudaGetLastError();        // leave no sticky error for the caller's next call
            return KDA_ERR_CUDA;
        }
        g_addr[dev] = p;
    }
    *out = g_addr[dev];
    return KDA_OK;
}

}  // namespace

namespace kda {
kda_status_t check_fwd_inputs(const void* q, const void* k, const void* v, const void* g,
                              const void* beta, const int32_t* segment_ids, int64_t B, int64_t T,
                              int32_t H, int32_t d_qk, int32_t d_v, kda_dtype_t dtype,
                              kda_dtype_t out_dtype, const void* o, const uint32_t* status_dev);
}

extern "C" kda_status_t kda_chunk_fwd_varlen_noalloc(
    const void* q, const void* k, const void* v, const void* g, const void* beta,
    const int32_t* segment_ids, int64_t B, int64_t T, int32_t H, int32_t d_qk, int32_t d_v,
    float scale, kda_dtype_t dtype, kda_dtype_t out_dtype, void* o, uint32_t* status_dev,
    kda_stream_t stream) {
    // The inputs are checked as kda_chunk_fwd_varlen checks them, and first; then the
    // size rule: a problem whose workspace would exceed the built-in array is refused
    // before anything is launched.
    const kda_status_t chk = kda::check_fwd_inputs(q, k, v, g, beta, segment_ids, B, T, H, d_qk,
                                                   d_v, dtype, out_dtype, o, status_dev);
    if (chk != KDA_OK) return chk;
    const size_t need = kda_chunk_fwd_varlen_workspace_min(B, T, H, d_qk, d_v, dtype);
    if (need == 0) return KDA_ERR_INVALID_ARG;
    if (need > size_t(KDA_NOALLOC_SCRATCH_BYTES)) return KDA_ERR_WORKSPACE;
    void* scratch = nullptr;
    const kda_status_t s = scratch_address(&scratch);
    if (s != KDA_OK) return s;
    // Nothing is cleared here: on every call the kernels write each scratch word before
    // they read it, so what an earlier call left in the array does not matter. That rests
    // on two places. The bf16, 128-wide path: plan_units_kernel (kda_chunk_tc.cu) resets
    // the work counters and the planner rewrites every chunk's metadata, unit and order
    // entry; the chunk kernel's last CTA rewinds the counters it advanced. The token-
    // recurrence path (fp32, or 64-wide heads): its segment-list pass rewrites the list
    // and its counters. A change to either that reads a word it did not write on the same
    // call would break this entry point.
    return kda_chunk_fwd_varlen(q, k, v, g, beta, segment_ids, B, T, H, d_qk, d_v, scale, dtype,
                                out_dtype, o, scratch, size_t(KDA_NOALLOC_SCRATCH_BYTES),
                                status_dev, stream);
}
