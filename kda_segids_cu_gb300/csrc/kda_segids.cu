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
// Design: one CTA of 1024 threads walks the ids in tiles of 32768 tokens; each
// thread owns a contiguous run of 32 ids, read with eight 16-byte loads (one
// round trip per tile), and takes the previous token's id from its own run or,
// for its first token, from the neighbouring thread (a shuffle, or shared memory
// across warps and tiles). Starts are found as bitmasks over the run (real tokens,
// id changes, and the run's one possible row start when T >= 32). Each thread ranks
// its starts with a block-wide exclusive scan of per-thread counts, so the k-th start
// lands in cu_seqlens[k] by a direct scatter in token order: no scratch memory and no
// second pass.
#include "kda_common.cuh"

namespace kda {
namespace {

constexpr int kThreads = 1024;
constexpr int kRun = 32;                           // ids per thread per tile
constexpr int kWarps = kThreads / 32;
constexpr int64_t kTile = int64_t(kThreads) * kRun;

__global__ void __launch_bounds__(kThreads, 1)
segids_to_cu_seqlens_kernel(const int32_t* __restrict__ seg, int64_t N, int64_t T,
                            RowStartTest row_start, int32_t max_segs, int32_t* __restrict__ cu,
                            int32_t* __restrict__ n_segs_out) {
    __shared__ int warp_sum[kWarps];
    __shared__ int32_t warp_last_id[kWarps];       // last id of each warp's last thread
    __shared__ int tile_total;
    __shared__ int32_t carry_id;                   // last id of the previous tile
    __shared__ int red[kWarps];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;

    int64_t running = 0;      // starts in earlier tiles (same value in every thread)
    int64_t last_real_end = 0;
    const bool vec = (reinterpret_cast<uintptr_t>(seg) & 15u) == 0;   // 16-byte loads allowed
    if (threadIdx.x == 0) carry_id = 0;

    for (int64_t base = 0; base < N; base += kTile) {
        const int64_t p0 = base + int64_t(threadIdx.x) * kRun;
        int32_t id[kRun];
        if (vec && p0 + kRun <= N) {
            const int4* src = reinterpret_cast<const int4*>(seg + p0);
#pragma unroll
            for (int i = 0; i < kRun / 4; ++i) {
                const int4 v = src[i];
                id[4 * i] = v.x; id[4 * i + 1] = v.y; id[4 * i + 2] = v.z; id[4 * i + 3] = v.w;
            }
        } else {
#pragma unroll
            for (int i = 0; i < kRun; ++i) id[i] = (p0 + i < N) ? seg[p0 + i] : 0;
        }
        // id of the token before this run
        int32_t prev = __shfl_up_sync(0xffffffffu, id[kRun - 1], 1);
        if (lane == 31) warp_last_id[warp] = id[kRun - 1];
        __syncthreads();                            // also orders carry_id from the last tile
        if (lane == 0) prev = (warp == 0) ? carry_id : warp_last_id[warp - 1];
        // bit i: token p0 + i is real / differs from its predecessor / starts a row (ids
        // past N were read as 0, so they are not real)
        unsigned realm = 0, diffm = 0, rowm = 0;
#pragma unroll
        for (int i = 0; i < kRun; ++i) {
            const int32_t before = (i == 0) ? prev : id[i - 1];
            realm |= unsigned(id[i] != 0) << i;
            diffm |= unsigned(before != id[i]) << i;
        }
        if (T >= kRun) {                            // at most one row start in the run
            const int64_t rem = p0 % T;
            const int64_t o = rem ? T - rem : 0;
            if (o < kRun) rowm = 1u << o;
        } else {
#pragma unroll
            for (int i = 0; i < kRun; ++i) rowm |= unsigned(row_start(p0 + i)) << i;
        }
        unsigned mask = realm & (diffm | rowm);
        if (realm) {
            const int64_t e = p0 + kRun - __clz(realm);   // one past the run's last real token
            last_real_end = e > last_real_end ? e : last_real_end;
        }
        // block exclusive scan of the per-thread start counts
        const int cnt = __popc(mask);
        int incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += n;
        }
        if (lane == 31) warp_sum[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            const int ws = warp_sum[lane];
            int wi = ws;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int n = __shfl_up_sync(0xffffffffu, wi, o);
                if (lane >= o) wi += n;
            }
            warp_sum[lane] = wi - ws;
            if (lane == 31) tile_total = wi;
        }
        __syncthreads();
        int64_t rank = running + warp_sum[warp] + (incl - cnt);
        while (mask) {
            const int i = __ffs(mask) - 1;
            mask &= mask - 1;
            // cu[r] = start of the (r+1)-th segment, for 1 <= r < max_segs
            if (rank >= 1 && rank < max_segs) cu[rank] = int32_t(p0 + i);
            ++rank;
        }
        running += tile_total;
        if (threadIdx.x == kThreads - 1) carry_id = id[kRun - 1];
        __syncthreads();   // warp_sum / tile_total / carry_id are rewritten by the next tile
    }

    // block max of the end of the last real token
    int64_t v = last_real_end;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const int64_t n = __shfl_xor_sync(0xffffffffu, v, o);
        v = n > v ? n : v;
    }
    if (lane == 0) red[warp] = int(v);
    __syncthreads();
    if (warp == 0) {
        int m = red[lane];
        m = __reduce_max_sync(0xffffffffu, m);
        if (lane == 0) red[0] = m;
    }
    __syncthreads();
    const int64_t n_end = red[0];
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
    kda::segids_to_cu_seqlens_kernel<<<1, kda::kThreads, 0, stream>>>(
        seg, B * T, T, kda::RowStartTest::make(T), max_segs, cu, n_segs);
    return kda::launch_status();
}
