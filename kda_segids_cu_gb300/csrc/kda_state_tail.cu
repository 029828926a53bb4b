// kda_state_tail.cu -- the state pass of kda_chunk_fwd_varlen_state on the bf16 path.
//
// [RFC-0026] "RFC-0026: Ling3 KDA Varlen 支持（packing 文档间隔离）" hands the chunked
// KDA call an initial_state and asks for output_final_state, one state per packed
// sequence; the recurrence is that of 背景 "KDA 状态泄漏问题" with the state reset at
// every segment start (§3.1.1).
//
// The chunk kernel does the bulk of it on the tensor cores. At the chunk where a segment
// starts and carries on, it seeds the carried state with the segment's initial state
// decayed to that chunk's end, so the segment's rows in later chunks read the initial
// state through the carried state. At the chunk where a segment ends, having come in
// carried, it stores the state carried into that chunk. What is left is local to single
// chunks (per head; G_i = sum of g over the chunk's real rows up to i, G_{-1} = 0):
//   - the rows t of a segment in the chunk where it starts (row r) see its initial state
//     S0 through the decay since the start, a term the chunk kernel leaves out; this pass
//     writes their outputs whole, in fp32 (one rounding to the output type):
//         Qd_t = q_t * exp(G_t - G_{r-1}),   Kd_j = beta_j k_j * exp(G_{r-1} - G_j)
//         o_t  = scale (Qd_t^T S0 + sum_{j=r..t} (Qd_t . Kd_j) v_j)
//   - a segment that ends at row e of a chunk, with state S_a before its first row a in
//     that chunk (S0 or zero at its start row, or the stored carried state at row 0), has
//     the final state
//         S_e = exp(G_e - G_{a-1}) * S_a + sum_{j=a..e} (beta_j k_j * exp(G_e - G_j)) v_j^T
//     where the products with exp(...) scale the key rows.
// One CTA takes one (chunk, head) at a time and passes over those with nothing to do.
// fp32 arithmetic with exact exponentials (expf).
#include "kda_common.cuh"
#include "kda_plan.cuh"

namespace kda {
namespace tc {
namespace {

constexpr int kTD = 128;                  // head width of the bf16 path
constexpr int kTR = kChunk;               // rows per chunk
constexpr int kTailThreads = 256;
// shared memory (bytes): q, k, v as stored (bf16 [64][128], row-major), the cumulative
// log-decay G [64][128] and work arrays W [128][64] or [64][128] and X [128][64] (fp32; W
// holds g as bf16 while G is formed), a score tile A [64][64] and beta [64] (fp32)
constexpr uint32_t kSq = 0;
constexpr uint32_t kSk = kSq + kTR * kTD * 2;
constexpr uint32_t kSv = kSk + kTR * kTD * 2;
constexpr uint32_t kSG = kSv + kTR * kTD * 2;
constexpr uint32_t kSW = kSG + kTR * kTD * 4;
constexpr uint32_t kSX = kSW + kTR * kTD * 4;
constexpr uint32_t kSA = kSX + kTR * kTD * 4;
constexpr uint32_t kSB = kSA + kTR * kTR * 4;
constexpr uint32_t kTailSmem = kSB + kTR * 4;   // 164,096 B: one CTA per SM

__device__ __forceinline__ float2 pfma(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 u, v, w, z;\n\tmov.b64 u, {%2, %3};\n\tmov.b64 v, {%4, %5};\n\t"
        "mov.b64 w, {%6, %7};\n\tfma.rn.f32x2 z, u, v, w;\n\tmov.b64 {%0, %1}, z;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

// 8 bf16 (one 16-byte word) -> 8 floats; exact (bf16 is the top half of an fp32 word)
__device__ __forceinline__ void unpack8(uint4 w, float* x) {
    const uint32_t a[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        x[2 * i] = __uint_as_float(a[i] << 16);
        x[2 * i + 1] = __uint_as_float(a[i] & 0xffff0000u);
    }
}

__device__ __forceinline__ uint32_t pack2(float a, float b) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
}

// dst[0..7] = scale * acc (one 16- or 32-byte group of an output row), rounded once
__device__ __forceinline__ void store_out(__nv_bfloat16* dst, const float2* acc, float scale) {
    *reinterpret_cast<uint4*>(dst) =
        make_uint4(pack2(scale * acc[0].x, scale * acc[0].y), pack2(scale * acc[1].x, scale * acc[1].y),
                   pack2(scale * acc[2].x, scale * acc[2].y), pack2(scale * acc[3].x, scale * acc[3].y));
}
__device__ __forceinline__ void store_out(float* dst, const float2* acc, float scale) {
    float4* p = reinterpret_cast<float4*>(dst);
    p[0] = make_float4(scale * acc[0].x, scale * acc[0].y, scale * acc[1].x, scale * acc[1].y);
    p[1] = make_float4(scale * acc[2].x, scale * acc[2].y, scale * acc[3].x, scale * acc[3].y);
}

struct Tile {                              // shared-memory views of the current (chunk, head)
    const __nv_bfloat16* q;
    const __nv_bfloat16* k;
    const __nv_bfloat16* v;
    const float* G;
    float* W;
    float* X;
    float* A;
    const float* beta;
};

// Final state of rows a..e (one segment): out = exp(G_e - G_{a-1}) * base + sum_j Kf_j v_j^T,
// Kf_j = beta_j k_j * exp(G_e - G_j). base may be null (zero) or equal to out (in place:
// each thread reads its own 8 x 8 block before writing it).
__device__ void final_state(const Tile& t, int a, int e, const float* base, float* out) {
    const int tid = threadIdx.x;
    const float* Ge = t.G + e * kTD;
    for (int idx = tid; idx < (e - a + 1) * kTD; idx += kTailThreads) {
        const int j = a + idx / kTD, c = idx % kTD;
        t.W[j * kTD + c] = t.beta[j] * __bfloat162float(t.k[j * kTD + c]) *
                           expf(Ge[c] - t.G[j * kTD + c]);
    }
    __syncthreads();
    const int rg = tid >> 4, cg = tid & 15;        // key rows 8 rg .., value columns 8 cg ..
    float2 acc[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int c = 8 * rg + i;
        const float dec = expf(Ge[c] - (a > 0 ? t.G[(a - 1) * kTD + c] : 0.f));
        if (base) {
            const float4* b4 = reinterpret_cast<const float4*>(base + c * kTD + 8 * cg);
            const float4 x = b4[0], y = b4[1];
            acc[i][0] = make_float2(dec * x.x, dec * x.y);
            acc[i][1] = make_float2(dec * x.z, dec * x.w);
            acc[i][2] = make_float2(dec * y.x, dec * y.y);
            acc[i][3] = make_float2(dec * y.z, dec * y.w);
        } else {
#pragma unroll
            for (int jp = 0; jp < 4; ++jp) acc[i][jp] = make_float2(0.f, 0.f);
        }
    }
#pragma unroll 2
    for (int j = a; j <= e; ++j) {
        const float4* w4 = reinterpret_cast<const float4*>(t.W + j * kTD + 8 * rg);
        const float4 w0 = w4[0], w1 = w4[1];
        const float w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
        float vv[8];
        unpack8(*reinterpret_cast<const uint4*>(t.v + j * kTD + 8 * cg), vv);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float2 wi = make_float2(w[i], w[i]);
#pragma unroll
            for (int jp = 0; jp < 4; ++jp)
                acc[i][jp] = pfma(wi, make_float2(vv[2 * jp], vv[2 * jp + 1]), acc[i][jp]);
        }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        float4* d4 = reinterpret_cast<float4*>(out + (8 * rg + i) * kTD + 8 * cg);
        d4[0] = make_float4(acc[i][0].x, acc[i][0].y, acc[i][1].x, acc[i][1].y);
        d4[1] = make_float4(acc[i][2].x, acc[i][2].y, acc[i][3].x, acc[i][3].y);
    }
    __syncthreads();                              // W is free again
}

// Outputs of rows r..end-1, the rows of a segment (with initial state S0) in the chunk
// where it starts: o_t = scale (Qd_t^T S0 + sum_{j=r..t} (Qd_t . Kd_j) v_j). Qd and Kd are
// kept transposed (W, X: [key channel][row]) and so is the score tile (A: [j][t]), so that
// the loops below read 16-byte groups without bank conflicts.
template <typename To>
__device__ void head_output(const Tile& t, int r, int end, const float* __restrict__ S0,
                            To* o, int64_t p0, int32_t H, int h, float scale) {
    const int tid = threadIdx.x;
    {
        // transposing writes: a warp takes 32 rows x 32 key channels along a diagonal
        // (lane l: row 32 rt + l, channel 32 ct + (l + d) % 32), so that both the row-major
        // reads and the column-major writes fall in 32 different banks
        const int lane = tid & 31, warp = tid >> 5;
        const int n_units = ((end - r + 31) / 32) * (kTD / 32) * 32;
        for (int wu = warp; wu < n_units; wu += kTailThreads / 32) {
            const int rt = wu / (kTD / 32 * 32), ct = (wu / 32) % (kTD / 32), d = wu % 32;
            const int i = r + rt * 32 + lane;
            const int c = ct * 32 + ((lane + d) & 31);
            if (i < end) {
                const float gr = r > 0 ? t.G[(r - 1) * kTD + c] : 0.f;
                const float gi = t.G[i * kTD + c];
                t.W[c * kTR + i] = __bfloat162float(t.q[i * kTD + c]) * expf(gi - gr);
                t.X[c * kTR + i] = t.beta[i] * __bfloat162float(t.k[i * kTD + c]) * expf(gr - gi);
            }
        }
    }
    __syncthreads();
    {                                             // A[j][t] = Qd_t . Kd_j for r <= j <= t < end
        const int ta = tid >> 4, jb = tid & 15;   // rows t 4 ta .. +3, columns j 4 jb .. +3
        float acc[4][4] = {};
        if (4 * ta + 3 >= r && 4 * ta < end && 4 * jb < end && 4 * jb <= 4 * ta + 3) {
#pragma unroll 4
            for (int c = 0; c < kTD; ++c) {
                const float4 w = *reinterpret_cast<const float4*>(t.W + c * kTR + 4 * ta);
                const float4 x = *reinterpret_cast<const float4*>(t.X + c * kTR + 4 * jb);
                const float wv[4] = {w.x, w.y, w.z, w.w}, xv[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(wv[i], xv[j], acc[i][j]);
            }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int jj = 4 * jb + j;
            float out[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int ti = 4 * ta + i;
                out[i] = (jj >= r && jj <= ti && ti < end) ? acc[i][j] : 0.f;
            }
            *reinterpret_cast<float4*>(t.A + jj * kTR + 4 * ta) = make_float4(out[0], out[1], out[2], out[3]);
        }
    }
    __syncthreads();
    const int tr = tid >> 4, cg = tid & 15;        // rows 4 tr .. +3, value columns 8 cg ..
    const int i0 = 4 * tr;
    if (i0 + 3 >= r && i0 < end) {
        float2 acc[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int jp = 0; jp < 4; ++jp) acc[i][jp] = make_float2(0.f, 0.f);
#pragma unroll 4
        for (int c = 0; c < kTD; ++c) {           // Qd^T S0
            const float4 s0 = __ldg(reinterpret_cast<const float4*>(S0 + c * kTD + 8 * cg));
            const float4 s1 = __ldg(reinterpret_cast<const float4*>(S0 + c * kTD + 8 * cg + 4));
            const float2 sv[4] = {make_float2(s0.x, s0.y), make_float2(s0.z, s0.w),
                                  make_float2(s1.x, s1.y), make_float2(s1.z, s1.w)};
            const float4 w = *reinterpret_cast<const float4*>(t.W + c * kTR + i0);
            const float wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 w2 = make_float2(wv[i], wv[i]);
#pragma unroll
                for (int jp = 0; jp < 4; ++jp) acc[i][jp] = pfma(w2, sv[jp], acc[i][jp]);
            }
        }
        const int j_hi = (i0 + 4 < end) ? i0 + 4 : end;
        for (int j = r; j < j_hi; ++j) {          // + A V (A is zero outside the segment)
            const float4 a = *reinterpret_cast<const float4*>(t.A + j * kTR + i0);
            const float av[4] = {a.x, a.y, a.z, a.w};
            float vv[8];
            unpack8(*reinterpret_cast<const uint4*>(t.v + j * kTD + 8 * cg), vv);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 a2 = make_float2(av[i], av[i]);
#pragma unroll
                for (int jp = 0; jp < 4; ++jp)
                    acc[i][jp] = pfma(a2, make_float2(vv[2 * jp], vv[2 * jp + 1]), acc[i][jp]);
            }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int row = i0 + i;
            if (row < r || row >= end) continue;
            To* dst = o + ((p0 + row) * H + h) * kTD + 8 * cg;
            store_out(dst, acc[i], scale);
        }
    }
    __syncthreads();                              // W, X and A are free again
}

template <typename To>
__global__ void __launch_bounds__(kTailThreads, 1)
state_tail_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                  const __nv_bfloat16* __restrict__ v, const __nv_bfloat16* __restrict__ g,
                  const __nv_bfloat16* __restrict__ beta, int64_t N, int32_t H, float scale,
                  void* ws, const float* __restrict__ init, float* fin, int64_t n_state,
                  To* o) {
    extern __shared__ __align__(16) uint8_t sm[];
    Tile t;
    t.q = reinterpret_cast<const __nv_bfloat16*>(sm + kSq);
    t.k = reinterpret_cast<const __nv_bfloat16*>(sm + kSk);
    t.v = reinterpret_cast<const __nv_bfloat16*>(sm + kSv);
    t.G = reinterpret_cast<const float*>(sm + kSG);
    t.W = reinterpret_cast<float*>(sm + kSW);
    t.X = reinterpret_cast<float*>(sm + kSX);
    t.A = reinterpret_cast<float*>(sm + kSA);
    t.beta = reinterpret_cast<const float*>(sm + kSB);
    const int64_t n_chunks = ceil_div(N, kTR);
    const Plan pl = plan_view(ws, n_chunks);
    const int tid = threadIdx.x;
    const int64_t slot_elems = int64_t(kTD) * kTD;

    for (int64_t u = blockIdx.x; u < n_chunks * H; u += gridDim.x) {
        const int64_t c = u / H;
        const int h = int(u % H);
        const ChunkMeta m = pl.meta[c];
        const int fc = pl.first_cut[c];
        // the next chunk opens with a start or padding (or there is none): a segment that
        // reaches this chunk's last row ends there
        const bool next_cut = c + 1 >= n_chunks || pl.first_cut[c + 1] == 0;
        const int rb = pl.rank_base[c];
        const unsigned long long cut = m.start | ~m.valid;
        // the carried segment (rank rb - 1) ends here: the chunk kernel stored its state
        const bool tail = fin != nullptr && fc > 0 && (fc < kTR || next_cut) && rb - 1 < n_state;
        // segments starting here with a slot: a read-out of their initial state, and their
        // final state if they end here
        unsigned long long work = 0;
        {
            unsigned long long st = m.start;
            int64_t rank = rb;
            while (st != 0ull && rank < n_state) {
                const int r = __ffsll((long long)st) - 1;
                st &= st - 1ull;
                const unsigned long long after = (r >= 63) ? 0ull : (cut & (~0ull << (r + 1)));
                if (init != nullptr || (fin != nullptr && (after != 0ull || next_cut)))
                    work |= 1ull << r;
                ++rank;
            }
        }
        if (!tail && work == 0ull) continue;

        __syncthreads();                          // the previous unit's reads are done
        const int64_t p0 = c * kTR;
        {
            const uint4 z = make_uint4(0u, 0u, 0u, 0u);
            const __nv_bfloat16* src[4] = {q, k, v, g};
            const uint32_t dst[4] = {kSq, kSk, kSv, kSW};
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                for (int idx = tid; idx < kTR * 16; idx += kTailThreads) {
                    const int i = idx >> 4, part = idx & 15;
                    const int64_t p = p0 + i;
                    uint4 val = z;
                    if (p < N)
                        val = __ldg(reinterpret_cast<const uint4*>(src[a] + (p * H + h) * kTD) + part);
                    reinterpret_cast<uint4*>(sm + dst[a])[idx] = val;
                }
            }
            if (tid < kTR) {
                const int64_t p = p0 + tid;
                reinterpret_cast<float*>(sm + kSB)[tid] =
                    p < N ? __bfloat162float(beta[p * H + h]) : 0.f;
            }
        }
        __syncthreads();
        if (tid < kTD) {                          // G, one key channel per thread
            const __nv_bfloat16* gs = reinterpret_cast<const __nv_bfloat16*>(sm + kSW);
            float* G = reinterpret_cast<float*>(sm + kSG);
            float run = 0.f;
            for (int i = 0; i < kTR; ++i) {
                if ((m.valid >> i) & 1ull) run += __bfloat162float(gs[i * kTD + tid]);
                G[i * kTD + tid] = run;
            }
        }
        __syncthreads();

        if (tail) {
            float* S = fin + ((rb - 1) * int64_t(H) + h) * slot_elems;
            final_state(t, 0, (fc < kTR ? fc : kTR) - 1, S, S);
        }
        unsigned long long wk = work;
        while (wk != 0ull) {
            const int r = __ffsll((long long)wk) - 1;
            wk &= wk - 1ull;
            const int64_t rank = rb + __popcll(m.start & ((1ull << r) - 1ull));
            const unsigned long long after = (r >= 63) ? 0ull : (cut & (~0ull << (r + 1)));
            const int end = after ? __ffsll((long long)after) - 1 : kTR;
            const float* S0 = init ? init + (rank * H + h) * slot_elems : nullptr;
            if (S0) head_output<To>(t, r, end, S0, o, p0, H, h, scale);
            if (fin && (after != 0ull || next_cut))
                final_state(t, r, end - 1, S0, fin + (rank * H + h) * slot_elems);
        }
    }
}

template <typename To>
kda_status_t launch_tail_typed(const void* q, const void* k, const void* v, const void* g,
                               const void* beta, int64_t N, int32_t H, float scale, void* o,
                               void* ws, const float* init, float* fin, int64_t n_state,
                               cudaStream_t stream) {
    static const cudaError_t attr = cudaFuncSetAttribute(
        state_tail_kernel<To>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kTailSmem));
    if (attr != cudaSuccess) return KDA_ERR_CUDA;
    const int blocks = max(1, sm_count());
    state_tail_kernel<To><<<blocks, kTailThreads, kTailSmem, stream>>>(
        static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k),
        static_cast<const __nv_bfloat16*>(v), static_cast<const __nv_bfloat16*>(g),
        static_cast<const __nv_bfloat16*>(beta), N, H, scale, ws, init, fin, n_state,
        static_cast<To*>(o));
    return launch_status();
}

}  // namespace
}  // namespace tc

kda_status_t launch_state_tail(const void* q, const void* k, const void* v, const void* g,
                               const void* beta, int64_t N, int32_t H, float scale,
                               kda_dtype_t out_dtype, void* o, void* ws, const float* init,
                               float* fin, int64_t n_state, cudaStream_t stream) {
    if (out_dtype == KDA_F32)
        return tc::launch_tail_typed<float>(q, k, v, g, beta, N, H, scale, o, ws, init, fin,
                                            n_state, stream);
    return tc::launch_tail_typed<__nv_bfloat16>(q, k, v, g, beta, N, H, scale, o, ws, init, fin,
                                                n_state, stream);
}

}  // namespace kda
