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
// (segment, head) units. In a unit, (D/8)^2 threads hold the D x D state, each an
// 8 x 8 block (key rows 8 rg .., value columns 8 cg ..) updated with packed fp32x2
// arithmetic. Tokens are staged kWin at a time in shared memory as fp32 (exp(g)
// and beta*k precomputed there), the next window's inputs being loaded into
// registers while the current one is computed. Each token's partial read-outs are
// summed across the warp's row blocks by shuffles and across warps once per window.
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

// Packed fp32 pairs (one f32x2 instruction for two lanes of arithmetic).
__device__ __forceinline__ float2 rmul2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 u, v, w;\n\tmov.b64 u, {%2, %3};\n\tmov.b64 v, {%4, %5};\n\t"
        "mul.rn.f32x2 w, u, v;\n\tmov.b64 {%0, %1}, w;\n\t}"
        : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 rfma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 u, v, w, z;\n\tmov.b64 u, {%2, %3};\n\tmov.b64 v, {%4, %5};\n\t"
        "mov.b64 w, {%6, %7};\n\tfma.rn.f32x2 z, u, v, w;\n\tmov.b64 {%0, %1}, z;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

constexpr int kTile = 8;                  // each thread holds an 8 x 8 block of S
constexpr int kWin = 8;                   // tokens staged per window

template <int D> constexpr int rec_threads() { return (D / kTile) * (D / kTile); }
template <int D, bool kDelta = false> constexpr int rec_smem_bytes() {
    // staged q, beta*k, exp(g), v per token, and per-warp partial read-outs; the delta rule
    // also stages k and exchanges per-warp partial sums of S'^T k (two buffers)
    return 4 * kWin * D * 4 + (rec_threads<D>() / 32) * kWin * D * 4 +
           (kDelta ? kWin * D * 4 + 2 * (rec_threads<D>() / 32) * D * 4 : 0);
}

// kDelta: the delta rule, the reading of the method's name (the pages state only the
// additive update above): S'_t = S_{t-1} exp(g_t), S_t = S'_t + beta_t k_t (v_t - S'_t^T k_t)^T.
// Each token's u = S'^T k sums over all key rows, so the CTA meets once per token: the
// warps' partial sums go through shared memory (two buffers, by token parity).
template <typename T, typename To, int D, bool kDelta>
__global__ void __launch_bounds__(rec_threads<D>(), D == 64 ? 8 : 2)
recurrent_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                 const T* __restrict__ g, const T* __restrict__ beta, int32_t H, float scale,
                 const int32_t* __restrict__ seg_start, const int32_t* __restrict__ seg_end,
                 const int32_t* __restrict__ counters, To* __restrict__ o,
                 const float* __restrict__ init, float* __restrict__ fin, int64_t n_state) {
    constexpr int NG = D / kTile;         // row groups = column groups
    constexpr int NT = NG * NG;
    constexpr int NW = NT / 32;
    extern __shared__ __align__(16) float smem[];
    float* sq = smem;                     // [kWin][D]
    float* sbk = sq + kWin * D;
    float* se = sbk + kWin * D;
    float* sv = se + kWin * D;
    float* part = sv + kWin * D;          // [NW][kWin][D]
    float* sk = part + NW * kWin * D;     // delta rule: [kWin][D] k
    float* upart = sk + kWin * D;         // delta rule: [2][NW][D] partial S'^T k

    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int rg = tid / NG, cg = tid % NG;          // key rows 8 rg .., value columns 8 cg ..
    const int64_t n_units = int64_t(counters[0]) * H;

    for (int64_t u = blockIdx.x; u < n_units; u += gridDim.x) {
        const int64_t s_idx = u / H;
        const int h = int(u % H);
        const int64_t p0 = seg_start[s_idx];
        const int64_t p1 = seg_end[s_idx];
        // S[i][jp]: key row 8 rg + i, value columns 8 cg + 2 jp, +1
        float2 S[kTile][kTile / 2];
        const int64_t slot = (s_idx * H + h) * int64_t(D) * D;
        const bool has_slot = s_idx < n_state;
#pragma unroll
        for (int i = 0; i < kTile; ++i) {
            float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
            if (init && has_slot) {
                const float* src = init + slot + int64_t(kTile * rg + i) * D + kTile * cg;
                a = *reinterpret_cast<const float4*>(src);
                b = *reinterpret_cast<const float4*>(src + 4);
            }
            S[i][0] = make_float2(a.x, a.y); S[i][1] = make_float2(a.z, a.w);
            S[i][2] = make_float2(b.x, b.y); S[i][3] = make_float2(b.z, b.w);
        }

        // the window's inputs, loaded one window ahead into registers (element
        // e = tid + m * NT of the window: token e / D, channel e % D)
        constexpr int PER = kWin * D / NT;
        float rq[PER], rk[PER], rg_[PER], rv[PER], rb[PER];
        auto load_window = [&](int64_t pw) {
            const int nw = int((p1 - pw < kWin) ? p1 - pw : int64_t(kWin));
#pragma unroll
            for (int m = 0; m < PER; ++m) {
                const int e = tid + m * NT, w = e / D, i = e % D;
                if (pw < p1 && w < nw) {
                    const int64_t row = (pw + w) * H + h;
                    rb[m] = to_f32(beta[row]);
                    rq[m] = to_f32(q[row * D + i]);
                    rk[m] = to_f32(k[row * D + i]);
                    rg_[m] = to_f32(g[row * D + i]);
                    rv[m] = to_f32(v[row * D + i]);
                }
            }
        };
        load_window(p0);
        for (int64_t pw = p0; pw < p1; pw += kWin) {
            const int nw = int((p1 - pw < kWin) ? p1 - pw : int64_t(kWin));
            __syncthreads();   // previous window fully consumed
#pragma unroll
            for (int m = 0; m < PER; ++m) {
                const int e = tid + m * NT;
                if (e < nw * D) {
                    sq[e] = rq[m];
                    sbk[e] = rb[m] * rk[m];
                    se[e] = expf(rg_[m]);
                    sv[e] = rv[m];
                    if constexpr (kDelta) sk[e] = rk[m];
                }
            }
            load_window(pw + kWin);   // in flight while this window is computed
            __syncthreads();
            for (int w = 0; w < nw; ++w) {
                const float4* r4 = reinterpret_cast<const float4*>(sq + w * D + kTile * rg);
                const float4 q0 = r4[0], q1 = r4[1];
                const float4* k4 = reinterpret_cast<const float4*>(sbk + w * D + kTile * rg);
                const float4 b0 = k4[0], b1 = k4[1];
                const float4* e4 = reinterpret_cast<const float4*>(se + w * D + kTile * rg);
                const float4 e0 = e4[0], e1 = e4[1];
                const float4* v4 = reinterpret_cast<const float4*>(sv + w * D + kTile * cg);
                const float4 v0 = v4[0], v1 = v4[1];
                const float qi[kTile] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
                const float bi[kTile] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
                const float ei[kTile] = {e0.x, e0.y, e0.z, e0.w, e1.x, e1.y, e1.z, e1.w};
                const float2 vj[kTile / 2] = {make_float2(v0.x, v0.y), make_float2(v0.z, v0.w),
                                              make_float2(v1.x, v1.y), make_float2(v1.z, v1.w)};
                float2 acc[kTile / 2];
#pragma unroll
                for (int jp = 0; jp < kTile / 2; ++jp) acc[jp] = make_float2(0.f, 0.f);
                if constexpr (!kDelta) {
#pragma unroll
                    for (int i = 0; i < kTile; ++i) {
                        const float2 e2 = make_float2(ei[i], ei[i]);
                        const float2 b2 = make_float2(bi[i], bi[i]);
                        const float2 q2 = make_float2(qi[i], qi[i]);
#pragma unroll
                        for (int jp = 0; jp < kTile / 2; ++jp) {
                            S[i][jp] = rfma2(S[i][jp], e2, rmul2(b2, vj[jp]));   // decay, then add
                            acc[jp] = rfma2(q2, S[i][jp], acc[jp]);              // read-out after
                        }
                    }
                } else {
                    // decay, and this thread's part of u = S'^T k (its 8 key rows)
                    const float4* kr4 = reinterpret_cast<const float4*>(sk + w * D + kTile * rg);
                    const float4 k0 = kr4[0], k1 = kr4[1];
                    const float ki[kTile] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
                    float2 pu[kTile / 2];
#pragma unroll
                    for (int jp = 0; jp < kTile / 2; ++jp) pu[jp] = make_float2(0.f, 0.f);
#pragma unroll
                    for (int i = 0; i < kTile; ++i) {
                        const float2 e2 = make_float2(ei[i], ei[i]);
                        const float2 k2 = make_float2(ki[i], ki[i]);
#pragma unroll
                        for (int jp = 0; jp < kTile / 2; ++jp) {
                            S[i][jp] = rmul2(S[i][jp], e2);
                            pu[jp] = rfma2(k2, S[i][jp], pu[jp]);
                        }
                    }
                    // sum over the warp's row groups, then over the warps through shared memory
#pragma unroll
                    for (int m = NG; m < 32; m <<= 1) {
#pragma unroll
                        for (int jp = 0; jp < kTile / 2; ++jp) {
                            pu[jp].x += __shfl_xor_sync(0xffffffffu, pu[jp].x, m);
                            pu[jp].y += __shfl_xor_sync(0xffffffffu, pu[jp].y, m);
                        }
                    }
                    float* ub = upart + (w & 1) * NW * D;
                    if (lane < NG) {
                        float4* dst = reinterpret_cast<float4*>(ub + warp * D + kTile * cg);
                        dst[0] = make_float4(pu[0].x, pu[0].y, pu[1].x, pu[1].y);
                        dst[1] = make_float4(pu[2].x, pu[2].y, pu[3].x, pu[3].y);
                    }
                    __syncthreads();
                    float2 dv[kTile / 2];
#pragma unroll
                    for (int jp = 0; jp < kTile / 2; ++jp) dv[jp] = vj[jp];
#pragma unroll
                    for (int wp = 0; wp < NW; ++wp) {
                        const float4* src = reinterpret_cast<const float4*>(ub + wp * D + kTile * cg);
                        const float4 a = src[0], b = src[1];
                        dv[0].x -= a.x; dv[0].y -= a.y; dv[1].x -= a.z; dv[1].y -= a.w;
                        dv[2].x -= b.x; dv[2].y -= b.y; dv[3].x -= b.z; dv[3].y -= b.w;
                    }
                    // S = S' + beta k (v - u)^T, then the read-out
#pragma unroll
                    for (int i = 0; i < kTile; ++i) {
                        const float2 b2 = make_float2(bi[i], bi[i]);
                        const float2 q2 = make_float2(qi[i], qi[i]);
#pragma unroll
                        for (int jp = 0; jp < kTile / 2; ++jp) {
                            S[i][jp] = rfma2(b2, dv[jp], S[i][jp]);
                            acc[jp] = rfma2(q2, S[i][jp], acc[jp]);
                        }
                    }
                }
                // sum the partial read-outs of the warp's row groups, then one store per column
#pragma unroll
                for (int m = NG; m < 32; m <<= 1) {
#pragma unroll
                    for (int jp = 0; jp < kTile / 2; ++jp) {
                        acc[jp].x += __shfl_xor_sync(0xffffffffu, acc[jp].x, m);
                        acc[jp].y += __shfl_xor_sync(0xffffffffu, acc[jp].y, m);
                    }
                }
                if (lane < NG) {
                    float4* dst = reinterpret_cast<float4*>(part + (warp * kWin + w) * D + kTile * cg);
                    dst[0] = make_float4(acc[0].x, acc[0].y, acc[1].x, acc[1].y);
                    dst[1] = make_float4(acc[2].x, acc[2].y, acc[3].x, acc[3].y);
                }
            }
            __syncthreads();
            for (int e = tid; e < nw * D; e += NT) {
                const int w = e / D, j = e % D;
                float sum = 0.f;
#pragma unroll
                for (int wp = 0; wp < NW; ++wp) sum += part[(wp * kWin + w) * D + j];
                const int64_t row = (pw + w) * H + h;
                o[row * D + j] = from_f32<To>(scale * sum);
            }
        }
        if (fin && has_slot) {
#pragma unroll
            for (int i = 0; i < kTile; ++i) {
                float* dst = fin + slot + int64_t(kTile * rg + i) * D + kTile * cg;
                *reinterpret_cast<float4*>(dst) = make_float4(S[i][0].x, S[i][0].y, S[i][1].x, S[i][1].y);
                *reinterpret_cast<float4*>(dst + 4) = make_float4(S[i][2].x, S[i][2].y, S[i][3].x, S[i][3].y);
            }
        }
    }
}

}  // namespace

size_t recurrent_workspace_bytes(int64_t N) {
    // seg_start[N], seg_end[N], counters[64]
    return size_t(N) * 8 + 256;
}

// The segment list in the first 8 N + 256 bytes of ws: seg_start[N], seg_end[N], counters.
kda_status_t launch_segment_list(const int32_t* seg, int64_t B, int64_t T_len, void* ws,
                                 cudaStream_t stream) {
    const int64_t N = B * T_len;
    int32_t* seg_start = static_cast<int32_t*>(ws);
    int32_t* seg_end = seg_start + N;
    int32_t* counters = seg_end + N;
    list_segments_kernel<<<1, kListThreads, 0, stream>>>(seg, N, RowStartTest::make(T_len),
                                                         seg_start, seg_end, counters);
    return launch_status();
}

template <typename T, typename To, bool kDelta>
static kda_status_t launch_recurrent_typed(const void* q, const void* k, const void* v,
                                           const void* g, const void* beta, const int32_t* seg,
                                           int64_t B, int64_t T_len, int32_t H, int32_t D,
                                           float scale, void* o, void* ws, const float* init,
                                           float* fin, int64_t n_state, cudaStream_t stream) {
    const int64_t N = B * T_len;
    int32_t* seg_start = static_cast<int32_t*>(ws);
    int32_t* seg_end = seg_start + N;
    int32_t* counters = seg_end + N;
    if (launch_segment_list(seg, B, T_len, ws, stream) != KDA_OK) return KDA_ERR_CUDA;
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
    if (D == 64) {
        constexpr int smem = rec_smem_bytes<64, kDelta>();
        if (dynamic_smem_attr<recurrent_kernel<T, To, 64, kDelta>>(smem) != cudaSuccess)
            return KDA_ERR_CUDA;
        recurrent_kernel<T, To, 64, kDelta><<<blocks, rec_threads<64>(), smem, stream>>>(
            qp, kp, vp, gp, bp, H, scale, seg_start, seg_end, counters, op, init, fin, n_state);
    } else {
        constexpr int smem = rec_smem_bytes<128, kDelta>();
        if (dynamic_smem_attr<recurrent_kernel<T, To, 128, kDelta>>(smem) != cudaSuccess)
            return KDA_ERR_CUDA;
        recurrent_kernel<T, To, 128, kDelta><<<blocks, rec_threads<128>(), smem, stream>>>(
            qp, kp, vp, gp, bp, H, scale, seg_start, seg_end, counters, op, init, fin, n_state);
    }
    return launch_status();
}

template <bool kDelta>
static kda_status_t launch_recurrent_dtypes(const void* q, const void* k, const void* v,
                                            const void* g, const void* beta, const int32_t* seg,
                                            int64_t B, int64_t T_len, int32_t H, int32_t D,
                                            float scale, kda_dtype_t dtype, kda_dtype_t out_dtype,
                                            void* o, void* ws, const float* init, float* fin,
                                            int64_t n_state, cudaStream_t stream) {
    if (dtype == KDA_BF16) {
        if (out_dtype == KDA_F32)
            return launch_recurrent_typed<__nv_bfloat16, float, kDelta>(
                q, k, v, g, beta, seg, B, T_len, H, D, scale, o, ws, init, fin, n_state, stream);
        return launch_recurrent_typed<__nv_bfloat16, __nv_bfloat16, kDelta>(
            q, k, v, g, beta, seg, B, T_len, H, D, scale, o, ws, init, fin, n_state, stream);
    }
    return launch_recurrent_typed<float, float, kDelta>(q, k, v, g, beta, seg, B, T_len, H, D,
                                                        scale, o, ws, init, fin, n_state, stream);
}

kda_status_t launch_recurrent_state(const void* q, const void* k, const void* v, const void* g,
                                    const void* beta, const int32_t* seg, int64_t B, int64_t T_len,
                                    int32_t H, int32_t D, float scale, kda_dtype_t dtype,
                                    kda_dtype_t out_dtype, void* o, void* ws, const float* init,
                                    float* fin, int64_t n_state, cudaStream_t stream) {
    return launch_recurrent_dtypes<false>(q, k, v, g, beta, seg, B, T_len, H, D, scale, dtype,
                                          out_dtype, o, ws, init, fin, n_state, stream);
}

// The delta-rule recurrence (the reading of the method's name), every segment from zero.
kda_status_t launch_recurrent_delta(const void* q, const void* k, const void* v, const void* g,
                                    const void* beta, const int32_t* seg, int64_t B, int64_t T_len,
                                    int32_t H, int32_t D, float scale, kda_dtype_t dtype,
                                    kda_dtype_t out_dtype, void* o, void* ws, cudaStream_t stream) {
    return launch_recurrent_dtypes<true>(q, k, v, g, beta, seg, B, T_len, H, D, scale, dtype,
                                         out_dtype, o, ws, nullptr, nullptr, 0, stream);
}

kda_status_t launch_recurrent(const void* q, const void* k, const void* v, const void* g,
                              const void* beta, const int32_t* seg, int64_t B, int64_t T_len,
                              int32_t H, int32_t D, float scale, kda_dtype_t dtype,
                              kda_dtype_t out_dtype, void* o, void* ws, cudaStream_t stream) {
    return launch_recurrent_state(q, k, v, g, beta, seg, B, T_len, H, D, scale, dtype, out_dtype,
                                  o, ws, nullptr, nullptr, 0, stream);
}

}  // namespace kda
