// kda_recurrent.cu -- the fp32 path of kda_chunk_fwd_varlen: the KDA token
// recurrence, one independent walk per (segment, head).
//
// [RFC-0026] "RFC-0026: Ling3 KDA Varlen 支持（packing 文档间隔离）", 背景
// "KDA 状态泄漏问题": S'_t = S_{t-1} exp(g_t) (rows = key channels),
// S_t = S'_t + beta_t k_t v_t^T, o_t = scale S_t^T q_t; §3.1.1: S = 0 at every
// segment start; padding (id 0) outputs 0.
//
// Why not tensor cores here: fp32 inputs are held to 1e-4 of the output RMS,
// which TF32 operands (10-bit mantissa) cannot meet. The token recurrence
// costs 4 d_qk d_v flops per token and head -- fewer than the chunked form --
// and keeps every step in fp32 with an exact per-token decay.
//
// Work split: a segment-list pass (one CTA, ballot/scan over the ids) writes
// each segment's [start, end) to the workspace; a persistent grid then walks
// (segment, head) units. In a unit, 2*D threads hold the D x D state: thread
// (half, c) keeps rows half*D/2 .. half*D/2 + D/2 - 1 of column c. Tokens are
// staged kWin at a time in shared memory as fp32 (exp(g) and beta*k
// precomputed there), and the two half-column partial read-outs are summed
// once per window.
//
// Per-segment state (the initial_state / output_final_state kwargs that [RFC-0026]
// passes to the chunked call): a unit of segment r starts from init[r] instead of
// zero and stores its state after the last token to fin[r] (both [n_state, H, D, D]
// fp32, row = key channel), when given and r < n_state; r is the segment's rank in
// flattened token order, as in cu_seqlens.
#include "kda_common.cuh"

namespace kda {
namespace {

constexpr int kListThreads = 1024;
constexpr int kListItems = 8;
constexpr int kListWarps = kListThreads / 32;

// Writes seg_start[r], seg_end[r] for every segment r (in flat-token order) and
// the segment count to counters[0]. A token p is the last of its segment when
// it is real and p+1 is the end of the array, a row start, or carries another id.
__global__ void __launch_bounds__(kListThreads, 1)
list_segments_kernel(const int32_t* __restrict__ seg, int64_t N, RowStartTest row_start,
                     int32_t* __restrict__ seg_start, int32_t* __restrict__ seg_end,
                     int32_t* __restrict__ counters) {
    __shared__ int counts[kListItems][kListWarps];
    __shared__ int offsets[kListItems][kListWarps];
    __shared__ int tile_total;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const unsigned lt_mask = (1u << lane) - 1u;
    const int64_t tile = int64_t(kListThreads) * kListItems;
    int64_t running = 0;
    for (int64_t base = 0; base < N; base += tile) {
        bool st[kListItems], last[kListItems];
#pragma unroll
        for (int i = 0; i < kListItems; ++i) {
            const int64_t p = base + int64_t(i) * kListThreads + threadIdx.x;
            st[i] = false;
            last[i] = false;
            if (p < N && is_real(seg, p)) {
                st[i] = is_segment_start(seg, p, row_start);
                const int64_t nx = p + 1;
                last[i] = nx == N || row_start(nx) || (seg != nullptr && seg[nx] != seg[p]);
            }
        }
        unsigned m[kListItems];
#pragma unroll
        for (int i = 0; i < kListItems; ++i) {
            m[i] = __ballot_sync(0xffffffffu, st[i]);
            if (lane == 0) counts[i][warp] = __popc(m[i]);
        }
        __syncthreads();
        if (warp == 0) {
            constexpr int per_lane = kListItems * kListWarps / 32;
            int vals[per_lane];
            int sum = 0;
#pragma unroll
            for (int j = 0; j < per_lane; ++j) {
                const int idx = lane * per_lane + j;
                vals[j] = counts[idx / kListWarps][idx % kListWarps];
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
            for (int j = 0; j < per_lane; ++j) {
                const int idx = lane * per_lane + j;
                offsets[idx / kListWarps][idx % kListWarps] = excl;
                excl += vals[j];
            }
            if (lane == 31) tile_total = incl;
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < kListItems; ++i) {
            const int64_t p = base + int64_t(i) * kListThreads + threadIdx.x;
            // inclusive count of starts up to p, minus one, is p's segment rank
            const int64_t incl = running + offsets[i][warp] + __popc(m[i] & lt_mask) + (st[i] ? 1 : 0);
            if (st[i]) seg_start[incl - 1] = int32_t(p);
            if (last[i]) seg_end[incl - 1] = int32_t(p + 1);
        }
        running += tile_total;
        __syncthreads();
    }
    if (threadIdx.x == 0) counters[0] = int32_t(running);
}

// Writes zeros to the outputs of padding tokens (all heads).
template <typename T>
__global__ void zero_padding_kernel(const int32_t* __restrict__ seg, int64_t N, int64_t row_elems,
                                    T* __restrict__ o) {
    const int64_t p = blockIdx.x;
    if (p >= N || seg[p] != 0) return;
    for (int64_t e = threadIdx.x; e < row_elems; e += blockDim.x)
        o[p * row_elems + e] = from_f32<T>(0.f);
}

template <int D> struct Win { static constexpr int value = D == 64 ? 16 : 8; };

template <typename T, typename To, int D>
__global__ void __launch_bounds__(2 * D)
recurrent_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                 const T* __restrict__ g, const T* __restrict__ beta, int32_t H, float scale,
                 const int32_t* __restrict__ seg_start, const int32_t* __restrict__ seg_end,
                 const int32_t* __restrict__ counters, To* __restrict__ o,
                 const float* __restrict__ init, float* __restrict__ fin, int64_t n_state) {
    constexpr int R = D / 2;              // state rows per thread
    constexpr int kWin = Win<D>::value;   // tokens staged per window (48 KB of smem)
    __shared__ float sq[kWin][D];
    __shared__ float sbk[kWin][D];
    __shared__ float se[kWin][D];
    __shared__ float sv[kWin][D];
    __shared__ float part[2][kWin][D];

    const int tid = threadIdx.x;
    const int c = tid % D;
    const int half = tid / D;
    const int64_t n_units = int64_t(counters[0]) * H;

    for (int64_t u = blockIdx.x; u < n_units; u += gridDim.x) {
        const int64_t s_idx = u / H;
        const int h = int(u % H);
        const int64_t p0 = seg_start[s_idx];
        const int64_t p1 = seg_end[s_idx];
        float S[R];
        // this thread's rows half*R .. +R-1 of column c in the segment's state slot
        const int64_t slot = ((s_idx * H + h) * D + half * R) * D + c;
        const bool has_slot = s_idx < n_state;
#pragma unroll
        for (int r = 0; r < R; ++r) S[r] = (init && has_slot) ? init[slot + int64_t(r) * D] : 0.f;

        for (int64_t pw = p0; pw < p1; pw += kWin) {
            const int nw = int((p1 - pw < kWin) ? p1 - pw : int64_t(kWin));
            __syncthreads();   // previous window fully consumed
            for (int e = tid; e < nw * D; e += 2 * D) {
                const int w = e / D, i = e % D;
                const int64_t row = (pw + w) * H + h;
                const float bt = to_f32(beta[row]);
                sq[w][i] = to_f32(q[row * D + i]);
                sbk[w][i] = bt * to_f32(k[row * D + i]);
                se[w][i] = expf(to_f32(g[row * D + i]));
                sv[w][i] = to_f32(v[row * D + i]);
            }
            __syncthreads();
            for (int w = 0; w < nw; ++w) {
                const float vc = sv[w][c];
                float acc = 0.f;
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const int i = half * R + r;
                    S[r] = fmaf(S[r], se[w][i], sbk[w][i] * vc);
                    acc = fmaf(sq[w][i], S[r], acc);
                }
                part[half][w][c] = acc;
            }
            __syncthreads();
            for (int e = tid; e < nw * D; e += 2 * D) {
                const int w = e / D, j = e % D;
                const int64_t row = (pw + w) * H + h;
                o[row * D + j] = from_f32<To>(scale * (part[0][w][j] + part[1][w][j]));
            }
        }
        if (fin && has_slot) {
#pragma unroll
            for (int r = 0; r < R; ++r) fin[slot + int64_t(r) * D] = S[r];
        }
    }
}

}  // namespace

size_t recurrent_workspace_bytes(int64_t N) {
    // seg_start[N], seg_end[N], counters[64]
    return size_t(N) * 8 + 256;
}

template <typename T, typename To>
static kda_status_t launch_recurrent_typed(const void* q, const void* k, const void* v,
                                           const void* g, const void* beta, const int32_t* seg,
                                           int64_t B, int64_t T_len, int32_t H, int32_t D,
                                           float scale, void* o, void* ws, const float* init,
                                           float* fin, int64_t n_state, cudaStream_t stream) {
    const int64_t N = B * T_len;
    int32_t* seg_start = static_cast<int32_t*>(ws);
    int32_t* seg_end = seg_start + N;
    int32_t* counters = seg_end + N;
    list_segments_kernel<<<1, kListThreads, 0, stream>>>(seg, N, RowStartTest::make(T_len),
                                                         seg_start, seg_end,
                                                         counters);
    if (cudaGetLastError() != cudaSuccess) return KDA_ERR_CUDA;
    if (seg != nullptr) {
        zero_padding_kernel<To><<<unsigned(N), 128, 0, stream>>>(seg, N, int64_t(H) * D,
                                                                 static_cast<To*>(o));
        if (cudaGetLastError() != cudaSuccess) return KDA_ERR_CUDA;
    }
    const int blocks = max(1, sm_count()) * (D == 64 ? 8 : 4);
    const T* qp = static_cast<const T*>(q);
    const T* kp = static_cast<const T*>(k);
    const T* vp = static_cast<const T*>(v);
    const T* gp = static_cast<const T*>(g);
    const T* bp = static_cast<const T*>(beta);
    To* op = static_cast<To*>(o);
    if (D == 64)
        recurrent_kernel<T, To, 64><<<blocks, 128, 0, stream>>>(qp, kp, vp, gp, bp, H, scale,
                                                                seg_start, seg_end, counters, op,
                                                                init, fin, n_state);
    else
        recurrent_kernel<T, To, 128><<<blocks, 256, 0, stream>>>(qp, kp, vp, gp, bp, H, scale,
                                                                 seg_start, seg_end, counters, op,
                                                                 init, fin, n_state);
    return launch_status();
}

kda_status_t launch_recurrent_state(const void* q, const void* k, const void* v, const void* g,
                                    const void* beta, const int32_t* seg, int64_t B, int64_t T_len,
                                    int32_t H, int32_t D, float scale, kda_dtype_t dtype,
                                    kda_dtype_t out_dtype, void* o, void* ws, const float* init,
                                    float* fin, int64_t n_state, cudaStream_t stream) {
    if (dtype == KDA_BF16) {
        if (out_dtype == KDA_F32)
            return launch_recurrent_typed<__nv_bfloat16, float>(q, k, v, g, beta, seg, B, T_len,
                                                                H, D, scale, o, ws, init, fin,
                                                                n_state, stream);
        return launch_recurrent_typed<__nv_bfloat16, __nv_bfloat16>(q, k, v, g, beta, seg, B,
                                                                    T_len, H, D, scale, o, ws,
                                                                    init, fin, n_state, stream);
    }
    return launch_recurrent_typed<float, float>(q, k, v, g, beta, seg, B, T_len, H, D, scale, o,
                                                ws, init, fin, n_state, stream);
}

kda_status_t launch_recurrent(const void* q, const void* k, const void* v, const void* g,
                              const void* beta, const int32_t* seg, int64_t B, int64_t T_len,
                              int32_t H, int32_t D, float scale, kda_dtype_t dtype,
                              kda_dtype_t out_dtype, void* o, void* ws, cudaStream_t stream) {
    return launch_recurrent_state(q, k, v, g, beta, seg, B, T_len, H, D, scale, dtype, out_dtype,
                                  o, ws, nullptr, nullptr, 0, stream);
}

}  // namespace kda
