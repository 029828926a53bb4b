// kda_selftest.cu -- a check of the bounded waits behind KDA_DEV_TIMEOUT.
//
// The chunk kernels wait on mbarriers (TMA and tensor-core completions, their own
// roles' hand-offs) with a limit of wall time, after which a waiting warp gives up, the
// kernel ORs KDA_DEV_TIMEOUT into the caller's status word and every role leaves, so that
// the context stays usable. In a correct run no wait comes near the limit. This entry
// point makes one give up on purpose: one CTA waits, through the same bounded wait, on a
// barrier that nothing arrives on.
#include "kda_common.cuh"
#include "kda_sm100.cuh"

namespace kda {
namespace {

using namespace kda::sm100;

__global__ void wait_timeout_kernel(uint64_t timeout_ns, uint32_t* status) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    // phase 0 of a fresh barrier completes only when its one arrival comes: never here
    const bool ok = mbar_wait(&bar, 0, timeout_ns);
    if (!__all_sync(0xffffffffu, ok) && threadIdx.x == 0) atomicOr(status, KDA_DEV_TIMEOUT);
}

}  // namespace
}  // namespace kda

kda_status_t kda_selftest_wait_timeout(uint64_t timeout_ns, uint32_t* status_dev,
                                       kda_stream_t stream) {
    if (!status_dev || !kda::aligned(status_dev, 4)) return KDA_ERR_INVALID_ARG;
    if (timeout_ns < 1000000ull || timeout_ns > 10000000000ull) return KDA_ERR_INVALID_ARG;
    kda::wait_timeout_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(timeout_ns,
                                                                                   status_dev);
    return kda::launch_status();
}
