// kda_bwd.cu -- kda_chunk_bwd_varlen: gradients of the packed KDA forward.
//
// [RFC-0026] "RFC-0026: Ling3 KDA Varlen 支持（packing 文档间隔离）", 背景 "KDA 状态泄漏问题":
// S_t = S_{t-1} exp(g_t) + beta_t k_t v_t^T (rows = key channels), o_t = scale S_t^T q_t,
// S = 0 at every segment start (§3.1.1); the pages give no backward, so this is the
// derivative of that recurrence. With do_t = dL/do_t and, per segment, the adjoint
// state A_t = dL/dS_t = scale q_t do_t^T + exp(g_{t+1}) * A_{t+1} (row scaling; zero past
// the segment's last token):
//   dq_t    = scale S_t do_t                  (a forward walk of S)
//   dk_t    = beta_t A_t v_t,   dv_t = beta_t A_t^T k_t,   dbeta_t = k_t^T A_t v_t
//                                             (a backward walk of A)
//   dg_t    = sum_{u >= t in the segment} (q_u * dq_u - k_u * dk_u)      (per channel)
// The last line holds because o depends on g only through G_t - G_j (G the cumulative
// log-decay), entering as q_t exp(G_t) and k_j exp(-G_j): dL/dG_u = q_u dq_u - k_u dk_u,
// and g_t enters every G_u with u >= t. It lets the backward walk take dg as a running
// sum, without the forward states. But the sum cancels (its total over a segment is zero),
// so its rounding error grows with the segment's length. The walk therefore restarts it
// at every 64-token chunk start t from the direct form
//   dg_t[i] = exp(g_t[i]) sum_j A_t[i][j] S_{t-1}[i][j] = sum_j X[i][j] S_{t-1}[i][j],
// X = exp(g_t) A_t being the adjoint it carries to t - 1. The forward walk leaves
// S_{t-1} there (a checkpoint per chunk and head), and dq in fp32; at a segment's first
// token dg is 0.
//
// Two launches after the segment list: the forward walk (dq, checkpoints), then the
// backward walk (dk, dv, dbeta and dg, reading dq and the checkpoints back). Each walks one (segment, head) per CTA with
// the layout of the fp32 recurrence: (D/8)^2 threads, each holding an 8 x 8 block of S
// or A (key rows 8 rg .., value columns 8 cg ..) in packed fp32x2 registers, tokens staged
// 8 at a time in shared memory with the next window's inputs prefetched into registers.
// fp32 arithmetic throughout; padding tokens get zero gradients.
#include "kda_common.cuh"

namespace kda {
kda_status_t launch_segment_list(const int32_t* seg, int64_t B, int64_t T_len, void* ws,
                                 cudaStream_t stream);

namespace {

constexpr int kTile = 8;                  // each thread holds an 8 x 8 block
constexpr int kWin = 8;                   // tokens staged per window

// workspace: the segment list (seg_start, seg_end, counters), the segments' order
// (longest first), then dq in fp32 [N, H, D], then the checkpoints S_{t-1} at chunk starts
// [ceil(N/64), H, D, D] fp32
inline size_t bwd_list_bytes(int64_t N) { return (size_t(N) * 12 + 256 + 255) & ~size_t(255); }

// Orders the segments longest first (a counting sort on 1024 buckets of log2 length,
// 1/48 octave wide), so that the longest serial walks start at once rather than when
// their turn in token order comes. One CTA of 1024 threads.
constexpr int kOrderThreads = 1024;
__global__ void __launch_bounds__(kOrderThreads, 1)
order_segments_kernel(const int32_t* __restrict__ seg_start, const int32_t* __restrict__ seg_end,
                      const int32_t* __restrict__ counters, int32_t* __restrict__ order) {
    __shared__ int hist[kOrderThreads];
    __shared__ int warp_sum[32];
    const int n = counters[0];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    auto bucket = [&](int s) {          // 0 = longest
        const float len = float(seg_end[s] - seg_start[s]);
        const int b = int(__log2f(len) * 48.f);
        return kOrderThreads - 1 - (b < kOrderThreads - 1 ? b : kOrderThreads - 1);
    };
    hist[tid] = 0;
    __syncthreads();
    for (int s = tid; s < n; s += kOrderThreads) atomicAdd(&hist[bucket(s)], 1);
    __syncthreads();
    // exclusive scan of hist, one bucket per thread
    const int v = hist[tid];
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += x;
    }
    if (lane == 31) warp_sum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int w = warp_sum[lane];
        int wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int x = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += x;
        }
        warp_sum[lane] = wi - w;
    }
    __syncthreads();
    hist[tid] = warp_sum[warp] + incl - v;
    __syncthreads();
    for (int s = tid; s < n; s += kOrderThreads) order[atomicAdd(&hist[bucket(s)], 1)] = s;
}

template <int D> constexpr int bwd_threads() { return (D / kTile) * (D / kTile); }

__device__ __forceinline__ float2 bmul2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 u, v, w;\n\tmov.b64 u, {%2, %3};\n\tmov.b64 v, {%4, %5};\n\t"
        "mul.rn.f32x2 w, u, v;\n\tmov.b64 {%0, %1}, w;\n\t}"
        : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 bfma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 u, v, w, z;\n\tmov.b64 u, {%2, %3};\n\tmov.b64 v, {%4, %5};\n\t"
        "mov.b64 w, {%6, %7};\n\tfma.rn.f32x2 z, u, v, w;\n\tmov.b64 {%0, %1}, z;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

__device__ __forceinline__ void ld8(const float* p, float* x) {
    const float4 a = reinterpret_cast<const float4*>(p)[0];
    const float4 b = reinterpret_cast<const float4*>(p)[1];
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

// value i of x[0..7] for a lane-dependent i, without local memory
__device__ __forceinline__ float pick8(const float* x, int i) {
    float r = x[0];
#pragma unroll
    for (int j = 1; j < 8; ++j) r = (i == j) ? x[j] : r;
    return r;
}

// Zero gradients of padding tokens (all heads).
template <typename To>
__global__ void zero_padding_grads(const int32_t* __restrict__ seg, int64_t N, int64_t row_elems,
                                   int32_t H, To* dq, To* dk, To* dv, To* dg, To* dbeta) {
    const int64_t p = blockIdx.x;
    if (p >= N || seg[p] != 0) return;
    const To z = from_f32<To>(0.f);
    for (int64_t e = threadIdx.x; e < row_elems; e += blockDim.x) {
        dq[p * row_elems + e] = z;
        dk[p * row_elems + e] = z;
        dv[p * row_elems + e] = z;
        dg[p * row_elems + e] = z;
    }
    for (int e = threadIdx.x; e < H; e += blockDim.x) dbeta[p * H + e] = z;
}

// ---- forward walk: dq_t = scale S_t do_t --------------------------------------------------
template <int D> constexpr int dq_smem_bytes() { return 5 * kWin * D * 4; }

template <typename T, typename To, int D>
__global__ void __launch_bounds__(bwd_threads<D>(), D == 64 ? 8 : 2)
bwd_dq_kernel(const T* __restrict__ k, const T* __restrict__ v, const T* __restrict__ g,
              const T* __restrict__ beta, const T* __restrict__ d_o, int32_t H, float scale,
              const int32_t* __restrict__ seg_start, const int32_t* __restrict__ seg_end,
              const int32_t* __restrict__ counters, const int32_t* __restrict__ order,
              To* __restrict__ dq, float* __restrict__ dq32, float* __restrict__ ckpt) {
    constexpr int NG = D / kTile;
    constexpr int NT = NG * NG;
    extern __shared__ __align__(16) float smem[];
    float* sbk = smem;                    // [kWin][D] beta k
    float* se = sbk + kWin * D;           // exp(g)
    float* sv = se + kWin * D;
    float* sdo = sv + kWin * D;
    float* sdq = sdo + kWin * D;          // [kWin][D] read-outs

    const int tid = threadIdx.x;
    const int rg = tid / NG, cg = tid % NG;
    const int64_t n_units = int64_t(counters[0]) * H;
    for (int64_t u = blockIdx.x; u < n_units; u += gridDim.x) {
        const int64_t s_idx = order[u / H];
        const int h = int(u % H);
        const int64_t p0 = seg_start[s_idx], p1 = seg_end[s_idx];
        float2 S[kTile][kTile / 2];
#pragma unroll
        for (int i = 0; i < kTile; ++i)
#pragma unroll
            for (int jp = 0; jp < kTile / 2; ++jp) S[i][jp] = make_float2(0.f, 0.f);

        constexpr int PER = kWin * D / NT;
        float rk[PER], rg_[PER], rv[PER], rb[PER], rd[PER];
        auto load_window = [&](int64_t pw) {
            const int nw = int((p1 - pw < kWin) ? p1 - pw : int64_t(kWin));
#pragma unroll
            for (int m = 0; m < PER; ++m) {
                const int e = tid + m * NT, w = e / D, i = e % D;
                if (pw < p1 && w < nw) {
                    const int64_t row = (pw + w) * H + h;
                    rb[m] = to_f32(beta[row]);
                    rk[m] = to_f32(k[row * D + i]);
                    rg_[m] = to_f32(g[row * D + i]);
                    rv[m] = to_f32(v[row * D + i]);
                    rd[m] = to_f32(d_o[row * D + i]);
                }
            }
        };
        load_window(p0);
        for (int64_t pw = p0; pw < p1; pw += kWin) {
            const int nw = int((p1 - pw < kWin) ? p1 - pw : int64_t(kWin));
            __syncthreads();              // the previous window is consumed
#pragma unroll
            for (int m = 0; m < PER; ++m) {
                const int e = tid + m * NT;
                if (e < nw * D) {
                    sbk[e] = rb[m] * rk[m];
                    se[e] = expf(rg_[m]);
                    sv[e] = rv[m];
                    sdo[e] = rd[m];
                }
            }
            load_window(pw + kWin);
            __syncthreads();
            for (int w = 0; w < nw; ++w) {
                const int64_t pos = pw + w;
                if ((pos & (kChunk - 1)) == 0 && pos > p0) {
                    // checkpoint S_{pos-1} for the backward walk's restart of dg at pos
                    float* dst = ckpt + ((pos / kChunk) * H + h) * int64_t(D) * D;
#pragma unroll
                    for (int i = 0; i < kTile; ++i) {
                        float4* d4 = reinterpret_cast<float4*>(dst + (kTile * rg + i) * D + kTile * cg);
                        d4[0] = make_float4(S[i][0].x, S[i][0].y, S[i][1].x, S[i][1].y);
                        d4[1] = make_float4(S[i][2].x, S[i][2].y, S[i][3].x, S[i][3].y);
                    }
                }
                float bi[kTile], ei[kTile], vv[kTile], dd[kTile];
                ld8(sbk + w * D + kTile * rg, bi);
                ld8(se + w * D + kTile * rg, ei);
                ld8(sv + w * D + kTile * cg, vv);
                ld8(sdo + w * D + kTile * cg, dd);
                float part[kTile];
#pragma unroll
                for (int i = 0; i < kTile; ++i) {
                    const float2 e2 = make_float2(ei[i], ei[i]);
                    const float2 b2 = make_float2(bi[i], bi[i]);
                    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
                    for (int jp = 0; jp < kTile / 2; ++jp) {
                        const float2 vj = make_float2(vv[2 * jp], vv[2 * jp + 1]);
                        S[i][jp] = bfma2(S[i][jp], e2, bmul2(b2, vj));      // decay, then add
                        acc = bfma2(S[i][jp], make_float2(dd[2 * jp], dd[2 * jp + 1]), acc);
                    }
                    part[i] = acc.x + acc.y;
                }
                // sum over the NG column blocks of each row block (lanes cg of one group)
#pragma unroll
                for (int m = 1; m < NG; m <<= 1)
#pragma unroll
                    for (int i = 0; i < kTile; ++i) part[i] += __shfl_xor_sync(0xffffffffu, part[i], m);
                if (cg < kTile) sdq[w * D + kTile * rg + cg] = pick8(part, cg);
            }
            __syncthreads();
            for (int e = tid; e < nw * D; e += NT) {
                const int w = e / D, c = e % D;
                const int64_t at = ((pw + w) * H + h) * D + c;
                const float x = scale * sdq[e];
                dq[at] = from_f32<To>(x);
                dq32[at] = x;
            }
        }
    }
}

// ---- backward walk: dk, dv, dbeta, dg ------------------------------------------------------
constexpr int kWinR = 16;                 // tokens staged per window of the backward walk
template <int D> constexpr int dkv_smem_bytes() {
    // staged q, do, k, v, exp(g), dq; out dk, dg, k u; per-warp dv partials; beta; the
    // restart values of dg
    return 9 * kWinR * D * 4 + (bwd_threads<D>() / 32) * kWinR * D * 4 + kWinR * 4 + D * 4;
}

// CTAs per SM of the backward walk: the full register file (no spills) for 128-wide heads
template <int D> constexpr int dkv_ctas_per_sm() { return D == 64 ? 4 : 1; }

template <typename T, typename To, int D>
__global__ void __launch_bounds__(bwd_threads<D>(), dkv_ctas_per_sm<D>())
bwd_dkv_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
               const T* __restrict__ g, const T* __restrict__ beta, const T* __restrict__ d_o,
               const float* __restrict__ dq, const float* __restrict__ ckpt, int32_t H,
               float scale,
               const int32_t* __restrict__ seg_start, const int32_t* __restrict__ seg_end,
               const int32_t* __restrict__ counters, const int32_t* __restrict__ order,
               To* __restrict__ dk, To* __restrict__ dv,
               To* __restrict__ dg, To* __restrict__ dbeta) {
    constexpr int NG = D / kTile;
    constexpr int NT = NG * NG;
    constexpr int NW = NT / 32;
    extern __shared__ __align__(16) float smem[];
    float* sq = smem;                     // [kWinR][D]
    float* sdo = sq + kWinR * D;
    float* sk = sdo + kWinR * D;
    float* sv = sk + kWinR * D;
    float* se = sv + kWinR * D;
    float* sdq = se + kWinR * D;
    float* sdk = sdq + kWinR * D;          // outputs of the window
    float* sdg = sdk + kWinR * D;
    float* sku = sdg + kWinR * D;          // k_c u_c, summed into dbeta
    float* part = sku + kWinR * D;         // [NW][kWinR][D] partial A^T k
    float* sb = part + NW * kWinR * D;     // [kWinR] beta
    float* sdir = sb + kWinR;              // [D] dg from its direct form at a chunk start

    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int rg = tid / NG, cg = tid % NG;
    const int64_t n_units = int64_t(counters[0]) * H;
    for (int64_t u = blockIdx.x; u < n_units; u += gridDim.x) {
        const int64_t s_idx = order[u / H];
        const int h = int(u % H);
        const int64_t p0 = seg_start[s_idx], p1 = seg_end[s_idx];
        float2 X[kTile][kTile / 2];       // exp(g_{t+1}) * A_{t+1}: the carried adjoint
#pragma unroll
        for (int i = 0; i < kTile; ++i)
#pragma unroll
            for (int jp = 0; jp < kTile / 2; ++jp) X[i][jp] = make_float2(0.f, 0.f);
        float run = 0.f;                  // threads tid < D: dg running sum of channel tid

        constexpr int PER = kWinR * D / NT;
        float rq[PER], rd[PER], rk[PER], rv[PER], rg_[PER], rdq[PER], rb[PER];
        // window [pw, pw + nw), the last window first
        auto load_window = [&](int64_t pw, int nw) {
#pragma unroll
            for (int m = 0; m < PER; ++m) {
                const int e = tid + m * NT, w = e / D, i = e % D;
                if (nw > 0 && w < nw) {
                    const int64_t row = (pw + w) * H + h;
                    rb[m] = to_f32(beta[row]);
                    rq[m] = to_f32(q[row * D + i]);
                    rd[m] = to_f32(d_o[row * D + i]);
                    rk[m] = to_f32(k[row * D + i]);
                    rv[m] = to_f32(v[row * D + i]);
                    rg_[m] = to_f32(g[row * D + i]);
                    rdq[m] = dq[row * D + i];
                }
            }
        };
        int64_t hi = p1;
        int64_t lo = (hi - p0 > kWinR) ? hi - kWinR : p0;
        load_window(lo, int(hi - lo));
        while (hi > p0) {
            const int nw = int(hi - lo);
            __syncthreads();              // the previous window is consumed
#pragma unroll
            for (int m = 0; m < PER; ++m) {
                const int e = tid + m * NT;
                if (e < nw * D) {
                    sq[e] = rq[m];
                    sdo[e] = rd[m];
                    sk[e] = rk[m];
                    sv[e] = rv[m];
                    se[e] = expf(rg_[m]);
                    sdq[e] = rdq[m];
                    if (e % D == 0) sb[e / D] = rb[m];
                }
            }
            const int64_t nhi = lo;
            const int64_t nlo = (nhi - p0 > kWinR) ? nhi - kWinR : p0;
            load_window(nlo, int(nhi - nlo));
            __syncthreads();
            for (int w = nw - 1; w >= 0; --w) {
                float qi[kTile], ki[kTile], ei[kTile], vv[kTile], dd[kTile];
                ld8(sq + w * D + kTile * rg, qi);
                ld8(sk + w * D + kTile * rg, ki);
                ld8(se + w * D + kTile * rg, ei);
                ld8(sv + w * D + kTile * cg, vv);
                ld8(sdo + w * D + kTile * cg, dd);
                float uo[kTile];                          // (A v) on this thread's rows, partial
                float2 wk[kTile / 2];                     // (A^T k) on its columns, partial
#pragma unroll
                for (int jp = 0; jp < kTile / 2; ++jp) wk[jp] = make_float2(0.f, 0.f);
#pragma unroll
                for (int i = 0; i < kTile; ++i) {
                    const float2 q2 = make_float2(scale * qi[i], scale * qi[i]);
                    const float2 k2 = make_float2(ki[i], ki[i]);
                    const float2 e2 = make_float2(ei[i], ei[i]);
                    float2 au = make_float2(0.f, 0.f);
#pragma unroll
                    for (int jp = 0; jp < kTile / 2; ++jp) {
                        // A_t = exp(g_{t+1}) A_{t+1} + scale q_t do_t^T
                        const float2 a = bfma2(q2, make_float2(dd[2 * jp], dd[2 * jp + 1]), X[i][jp]);
                        au = bfma2(a, make_float2(vv[2 * jp], vv[2 * jp + 1]), au);
                        wk[jp] = bfma2(a, k2, wk[jp]);
                        X[i][jp] = bmul2(a, e2);             // carried to token t - 1
                    }
                    uo[i] = au.x + au.y;
                }
                const int64_t pos = lo + w;
                float direct[kTile];                      // restart of dg at a chunk start
                const bool restart = (pos & (kChunk - 1)) == 0 && pos > p0;
                if (restart) {
                    const float* src = ckpt + ((pos / kChunk) * H + h) * int64_t(D) * D;
#pragma unroll
                    for (int i = 0; i < kTile; ++i) {
                        float sp[kTile];
                        ld8(src + (kTile * rg + i) * D + kTile * cg, sp);
                        float acc = 0.f;
#pragma unroll
                        for (int jp = 0; jp < kTile / 2; ++jp)
                            acc += X[i][jp].x * sp[2 * jp] + X[i][jp].y * sp[2 * jp + 1];
                        direct[i] = acc;
                    }
#pragma unroll
                    for (int m = 1; m < NG; m <<= 1)
#pragma unroll
                        for (int i = 0; i < kTile; ++i)
                            direct[i] += __shfl_xor_sync(0xffffffffu, direct[i], m);
                }
#pragma unroll
                for (int m = 1; m < NG; m <<= 1)
#pragma unroll
                    for (int i = 0; i < kTile; ++i) uo[i] += __shfl_xor_sync(0xffffffffu, uo[i], m);
#pragma unroll
                for (int m = NG; m < 32; m <<= 1)
#pragma unroll
                    for (int jp = 0; jp < kTile / 2; ++jp) {
                        wk[jp].x += __shfl_xor_sync(0xffffffffu, wk[jp].x, m);
                        wk[jp].y += __shfl_xor_sync(0xffffffffu, wk[jp].y, m);
                    }
                if (lane < NG) {                          // the warp's first row block
                    float4* dst = reinterpret_cast<float4*>(part + (warp * kWinR + w) * D + kTile * cg);
                    dst[0] = make_float4(wk[0].x, wk[0].y, wk[1].x, wk[1].y);
                    dst[1] = make_float4(wk[2].x, wk[2].y, wk[3].x, wk[3].y);
                }
                if (cg < kTile) {                         // channel c = 8 rg + cg
                    const int c = kTile * rg + cg;
                    const float uc = pick8(uo, cg);
                    const float kc = pick8(ki, cg);
                    const float dkc = sb[w] * uc;
                    sdk[w * D + c] = dkc;
                    sdg[w * D + c] = pick8(qi, cg) * sdq[w * D + c] - kc * dkc;   // dL/dG_t
                    sku[w * D + c] = kc * uc;
                    if (restart) sdir[c] = pick8(direct, cg);
                }
            }
            __syncthreads();
            if (tid < D) {                                // dg: the running sums, last token first
                for (int w = nw - 1; w >= 0; --w) {
                    const int64_t pos = lo + w;
                    run += sdg[w * D + tid];
                    if ((pos & (kChunk - 1)) == 0 && pos > p0) run = sdir[tid];
                    if (pos == p0) run = 0.f;             // S_{t-1} = 0 at a segment's start
                    sdg[w * D + tid] = run;
                }
            }
            __syncthreads();
            for (int e = tid; e < nw * D; e += NT) {
                const int w = e / D, c = e % D;
                const int64_t row = (lo + w) * H + h;
                dk[row * D + c] = from_f32<To>(sdk[e]);
                dg[row * D + c] = from_f32<To>(sdg[e]);
                float acc = 0.f;
#pragma unroll
                for (int wp = 0; wp < NW; ++wp) acc += part[(wp * kWinR + w) * D + c];
                dv[row * D + c] = from_f32<To>(sb[w] * acc);
            }
            for (int w = warp; w < nw; w += NW) {         // dbeta_t = sum_c k_c (A v)_c
                float acc = 0.f;
                for (int c = lane; c < D; c += 32) acc += sku[w * D + c];
#pragma unroll
                for (int m = 16; m > 0; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
                if (lane == 0) dbeta[(lo + w) * H + h] = from_f32<To>(acc);
            }
            hi = nhi;
            lo = nlo;
        }
    }
}

template <typename T, typename To, int D>
kda_status_t launch_bwd_typed(const void* q, const void* k, const void* v, const void* g,
                              const void* beta, const void* d_o, const int32_t* seg, int64_t B,
                              int64_t T_len, int32_t H, float scale, void* dq, void* dk, void* dv,
                              void* dg, void* dbeta, void* ws, cudaStream_t stream) {
    const int64_t N = B * T_len;
    int32_t* seg_start = static_cast<int32_t*>(ws);
    int32_t* seg_end = seg_start + N;
    int32_t* counters = seg_end + N;
    int32_t* order = counters + 64;
    float* dq32 = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + bwd_list_bytes(N));
    float* ckpt = dq32 + N * H * D;
    if (launch_segment_list(seg, B, T_len, ws, stream) != KDA_OK) return KDA_ERR_CUDA;
    order_segments_kernel<<<1, kOrderThreads, 0, stream>>>(seg_start, seg_end, counters, order);
    if (cudaGetLastError() != cudaSuccess) return KDA_ERR_CUDA;
    if (seg != nullptr) {
        zero_padding_grads<To><<<unsigned(N), 128, 0, stream>>>(
            seg, N, int64_t(H) * D, H, static_cast<To*>(dq), static_cast<To*>(dk),
            static_cast<To*>(dv), static_cast<To*>(dg), static_cast<To*>(dbeta));
        if (cudaGetLastError() != cudaSuccess) return KDA_ERR_CUDA;
    }
    if (dynamic_smem_attr<bwd_dq_kernel<T, To, D>>(dq_smem_bytes<D>()) != cudaSuccess ||
        dynamic_smem_attr<bwd_dkv_kernel<T, To, D>>(dkv_smem_bytes<D>()) != cudaSuccess)
        return KDA_ERR_CUDA;
    const int blocks = max(1, sm_count()) * (D == 64 ? 8 : 2);
    bwd_dq_kernel<T, To, D><<<blocks, bwd_threads<D>(), dq_smem_bytes<D>(), stream>>>(
        static_cast<const T*>(k), static_cast<const T*>(v), static_cast<const T*>(g),
        static_cast<const T*>(beta), static_cast<const T*>(d_o), H, scale, seg_start, seg_end,
        counters, order, static_cast<To*>(dq), dq32, ckpt);
    if (cudaGetLastError() != cudaSuccess) return KDA_ERR_CUDA;
    const int dkv_blocks = max(1, sm_count()) * dkv_ctas_per_sm<D>();
    bwd_dkv_kernel<T, To, D><<<dkv_blocks, bwd_threads<D>(), dkv_smem_bytes<D>(), stream>>>(
        static_cast<const T*>(q), static_cast<const T*>(k), static_cast<const T*>(v),
        static_cast<const T*>(g), static_cast<const T*>(beta), static_cast<const T*>(d_o),
        dq32, ckpt, H, scale, seg_start, seg_end, counters, order, static_cast<To*>(dk),
        static_cast<To*>(dv), static_cast<To*>(dg), static_cast<To*>(dbeta));
    return launch_status();
}

template <typename T, typename To>
kda_status_t launch_bwd_width(const void* q, const void* k, const void* v, const void* g,
                              const void* beta, const void* d_o, const int32_t* seg, int64_t B,
                              int64_t T_len, int32_t H, int32_t D, float scale, void* dq,
                              void* dk, void* dv, void* dg, void* dbeta, void* ws,
                              cudaStream_t stream) {
    if (D == 64)
        return launch_bwd_typed<T, To, 64>(q, k, v, g, beta, d_o, seg, B, T_len, H, scale, dq, dk,
                                           dv, dg, dbeta, ws, stream);
    return launch_bwd_typed<T, To, 128>(q, k, v, g, beta, d_o, seg, B, T_len, H, scale, dq, dk,
                                        dv, dg, dbeta, ws, stream);
}

}  // namespace

size_t bwd_workspace_bytes(int64_t N, int32_t H, int32_t D) {
    return bwd_list_bytes(N) + size_t(N) * H * D * 4 + size_t(ceil_div(N, kChunk)) * H * D * D * 4;
}

kda_status_t launch_bwd(const void* q, const void* k, const void* v, const void* g,
                        const void* beta, const void* d_o, const int32_t* seg, int64_t B,
                        int64_t T_len, int32_t H, int32_t D, float scale, kda_dtype_t dtype,
                        kda_dtype_t grad_dtype, void* dq, void* dk, void* dv, void* dg,
                        void* dbeta, void* ws, cudaStream_t stream) {
    if (dtype == KDA_BF16) {
        if (grad_dtype == KDA_F32)
            return launch_bwd_width<__nv_bfloat16, float>(q, k, v, g, beta, d_o, seg, B, T_len, H,
                                                          D, scale, dq, dk, dv, dg, dbeta, ws,
                                                          stream);
        return launch_bwd_width<__nv_bfloat16, __nv_bfloat16>(q, k, v, g, beta, d_o, seg, B, T_len,
                                                              H, D, scale, dq, dk, dv, dg, dbeta,
                                                              ws, stream);
    }
    return launch_bwd_width<float, float>(q, k, v, g, beta, d_o, seg, B, T_len, H, D, scale, dq,
                                          dk, dv, dg, dbeta, ws, stream);
}

}  // namespace kda
