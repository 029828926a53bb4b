// kda_segids.cu -- segment-boundary scan and the padded cu_seqlens conversion.
//
// [RFC-0025] "RFC-0025: 支持 Attention Varlen 功能并对齐 Loss", 方案 §1
// "segment_ids → cu_seqlens 转换": boundaries are where a non-zero id differs
// from the previous token's (padding never starts a segment); cu_seqlens holds
// the cumulative segment ends, padded with zero-length phantom segments to
// max_segs+1 entries. Row starts are forced boundaries ([RFC-0026] §3.1.1:
// t = 0 always starts a segment), and the last real segment ends one past the
// last non-padding token.
//
// Design: one CTA of 1024 threads streams the ids in tiles of 16384 tokens
// (16 independent loads in flight per thread). Start flags are ranked with
// warp ballots + popc and a 512-entry scan of per-(item, warp) counts, so the
// k-th start lands in cu_seqlens[k] by a direct scatter: no scratch memory and
// no second pass. The tile order is item-major, so the ranks are the global
// order of the flattened sequence.
#include "kda_common.cuh"

namespace kda {
namespace {

constexpr int kThreads = 1024;
constexpr int kItems = 16;
constexpr int kWarps = kThreads / 32;
constexpr int64_t kTile = int64_t(kThreads) * kItems;

__global__ void __launch_bounds__(kThreads, 1)
segids_to_cu_seqlens_kernel(const int32_t* __restrict__ seg, int64_t N, int64_t T,
                            int32_t max_segs, int32_t* __restrict__ cu,
                            int32_t* __restrict__ n_segs_out) {
    __shared__ int counts[kItems][kWarps];
    __shared__ int offsets[kItems][kWarps];
    __shared__ int tile_total;
    __shared__ int warp_last[kWarps];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const unsigned lt_mask = (1u << lane) - 1u;

    int64_t running = 0;      // starts in earlier tiles (same value in every thread)
    int last_real_end = 0;    // max over real tokens of p + 1 (thread-local)

    for (int64_t base = 0; base < N; base += kTile) {
        bool st[kItems];
#pragma unroll
        for (int i = 0; i < kItems; ++i) {
            const int64_t p = base + int64_t(i) * kThreads + threadIdx.x;
            bool s = false;
            if (p < N) {
                const int32_t id = seg[p];
                if (id != 0) {
                    last_real_end = max(last_real_end, int(p + 1));
                    s = (p % T) == 0 || seg[p - 1] != id;
                }
            }
            st[i] = s;
        }
        unsigned m[kItems];
#pragma unroll
        for (int i = 0; i < kItems; ++i) {
            m[i] = __ballot_sync(0xffffffffu, st[i]);
            if (lane == 0) counts[i][warp] = __popc(m[i]);
        }
        __syncthreads();
        if (warp == 0) {
            // lane l scans flattened entries [16 l, 16 l + 16) of counts (item-major)
            int vals[16];
            int sum = 0;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int idx = lane * 16 + j;
                vals[j] = counts[idx / kWarps][idx % kWarps];
                sum += vals[j];
            }
            int incl = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int n = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += n;
            }
            int excl = incl - sum;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int idx = lane * 16 + j;
                offsets[idx / kWarps][idx % kWarps] = excl;
                excl += vals[j];
            }
            if (lane == 31) tile_total = incl;
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < kItems; ++i) {
            if (st[i]) {
                const int64_t p = base + int64_t(i) * kThreads + threadIdx.x;
                const int64_t rank = running + offsets[i][warp] + __popc(m[i] & lt_mask);
                // cu[r] = start of the (r+1)-th segment, for 1 <= r < max_segs
                if (rank >= 1 && rank < max_segs) cu[rank] = int32_t(p);
            }
        }
        running += tile_total;
        __syncthreads();   // counts/offsets are rewritten by the next tile
    }

    // block max of the end of the last real token
    int v = __reduce_max_sync(0xffffffffu, last_real_end);
    if (lane == 0) warp_last[warp] = v;
    __syncthreads();
    if (warp == 0) {
        v = __reduce_max_sync(0xffffffffu, warp_last[lane]);
        if (lane == 0) warp_last[0] = v;
    }
    __syncthreads();
    const int64_t n_end = warp_last[0];
    const int64_t n = running;
    for (int64_t i = threadIdx.x; i <= max_segs; i += kThreads) {
        if (i == 0) {
            cu[0] = 0;
        } else if (i >= n) {
            cu[i] = int32_t(n_end);               // last real segment, then phantoms
        } else if (i == max_segs) {
            cu[i] = int32_t(N);                   // overflow: the last slot takes the rest
        }
    }
    if (threadIdx.x == 0 && n_segs_out) *n_segs_out = int32_t(n);
}

}  // namespace
}  // namespace kda

kda_status_t kda_launch_segids_to_cu_seqlens(const int32_t* seg, int64_t B, int64_t T,
                                             int32_t max_segs, int32_t* cu, int32_t* n_segs,
                                             cudaStream_t stream) {
    kda::segids_to_cu_seqlens_kernel<<<1, kda::kThreads, 0, stream>>>(seg, B * T, T, max_segs,
                                                                      cu, n_segs);
    return kda::launch_status();
}
