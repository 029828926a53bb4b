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
// The planner lists the chunks holding a start or the end of a carried segment; each CTA
// takes the next (listed chunk, head) from a work counter, so that units of unequal cost
// spread evenly. fp32 arithmetic with exact exponentials (expf).
#include "kda_common.cuh"
#include "kda_plan.cuh"

namespace kda {
namespace tc {
namespace {

constexpr int kTD = 128;                  // head width of the bf16 path
constexpr int kTR = kChunk;               // rows per chunk
constexpr int kTailThreads = 512;
constexpr int kTailWarps = kTailThreads / 32;
// shared memory (bytes): q, k, v as stored (bf16 [64][128], row-major); the cumulative
// log-decay G [64][128]; work arrays W ([128][64] or [64][128]) and X ([128][64], or 64 rows
// of an initial state), fp32 (W holds g as bf16 while G is formed); a score tile A [64][64],
// beta [64] and G's per-quarter sums [4][128], fp32
constexpr uint32_t kSq = 0;
constexpr uint32_t kSk = kSq + kTR * kTD * 2;
constexpr uint32_t kSv = kSk + kTR * kTD * 2;
constexpr uint32_t kSG = kSv + kTR * kTD * 2;
constexpr uint32_t kSW = kSG + kTR * kTD * 4;
constexpr uint32_t kSX = kSW + kTR * kTD * 4;
constexpr uint32_t kSA = kSX + kTR * kTD * 4;
constexpr uint32_t kSB = kSA + kTR * kTR * 4;
constexpr uint32_t kSQ = kSB + kTR * 4;
// and the first 64 rows of an initial state, fetched ahead while its read-out's scores form
constexpr uint32_t kSS = kSQ + 4 * kTD * 4;
constexpr uint32_t kTailSmem = kSS + kTR * kTD * 4;  // 198,912 B: one CTA per SM

__device__ __forceinline__ float2 pfma(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 u, v, w, z;\n\tmov.b64 u, {%2, %3};\n\tmov.b64 v, {%4, %5};\n\t"
        "mov.b64 w, {%6, %7};\n\tfma.rn.f32x2 z, u, v, w;\n\tmov.b64 {%0, %1}, z;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

// 4 bf16 (one 8-byte word) -> 2 float pairs; exact (bf16 is the top half of an fp32 word)
__device__ __forceinline__ void unpack4(uint2 w, float2* x) {
    x[0] = make_float2(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u));
    x[1] = make_float2(__uint_as_float(w.y << 16), __uint_as_float(w.y & 0xffff0000u));
}

__device__ __forceinline__ uint32_t pack2(float a, float b) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
}

// dst[0..3] = scale * acc (4 channels of an output row), rounded once
__device__ __forceinline__ void store_out(__nv_bfloat16* dst, const float2* acc, float scale) {
    *reinterpret_cast<uint2*>(dst) =
        make_uint2(pack2(scale * acc[0].x, scale * acc[0].y), pack2(scale * acc[1].x, scale * acc[1].y));
}
__device__ __forceinline__ void store_out(float* dst, const float2* acc, float scale) {
    *reinterpret_cast<float4*>(dst) =
        make_float4(scale * acc[0].x, scale * acc[0].y, scale * acc[1].x, scale * acc[1].y);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" :: "r"(dst), "l"(src), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_all;" ::: "memory");
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
    const float* S;                        // rows 0..63 of an initial state
    uint32_t x_addr;                       // shared-state-space addresses of X and S
    uint32_t s_addr;
};

// Final state of rows a..e (one segment): out = exp(G_e - G_{a-1}) * base + sum_j Kf_j v_j^T,
// Kf_j = beta_j k_j * exp(G_e - G_j). base may be null (zero) or equal to out (in place:
// each thread reads its own 8 x 4 block before writing it).
__device__ void final_state(const Tile& t, int a, int e, const float* base, float* out) {
    const int tid = threadIdx.x;
    const float* Ge = t.G + e * kTD;
    const int rg = tid >> 5, cg = tid & 31;        // key rows 8 rg .., value columns 4 cg ..
    // the base state's block first: its loads are in flight while Kf is formed
    float4 bx[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        bx[i] = base ? *reinterpret_cast<const float4*>(base + (8 * rg + i) * kTD + 4 * cg)
                     : make_float4(0.f, 0.f, 0.f, 0.f);
    for (int idx = tid; idx < (e - a + 1) * kTD; idx += kTailThreads) {
        const int j = a + idx / kTD, c = idx % kTD;
        t.W[j * kTD + c] = t.beta[j] * __bfloat162float(t.k[j * kTD + c]) *
                           expf(Ge[c] - t.G[j * kTD + c]);
    }
    __syncthreads();
    float2 acc[8][2];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int c = 8 * rg + i;
        const float dec = expf(Ge[c] - (a > 0 ? t.G[(a - 1) * kTD + c] : 0.f));
        acc[i][0] = make_float2(dec * bx[i].x, dec * bx[i].y);
        acc[i][1] = make_float2(dec * bx[i].z, dec * bx[i].w);
    }
#pragma unroll 2
    for (int j = a; j <= e; ++j) {
        const float4* w4 = reinterpret_cast<const float4*>(t.W + j * kTD + 8 * rg);
        const float4 w0 = w4[0], w1 = w4[1];
        const float w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
        float2 vv[2];
        unpack4(*reinterpret_cast<const uint2*>(t.v + j * kTD + 4 * cg), vv);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float2 wi = make_float2(w[i], w[i]);
            acc[i][0] = pfma(wi, vv[0], acc[i][0]);
            acc[i][1] = pfma(wi, vv[1], acc[i][1]);
        }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i)
        *reinterpret_cast<float4*>(out + (8 * rg + i) * kTD + 4 * cg) =
            make_float4(acc[i][0].x, acc[i][0].y, acc[i][1].x, acc[i][1].y);
    __syncthreads();                              // W is free again
}

// Outputs of rows r..end-1, the rows of a segment (with initial state S0) in the chunk
// where it starts: o_t = scale (Qd_t^T S0 + sum_{j=r..t} (Qd_t . Kd_j) v_j). Qd and Kd are
// kept transposed (W, X: [key channel][row]) and so is the score tile (A: [j][t]), so that
// the loops below read 8- and 16-byte groups without bank conflicts; S0 then passes through
// X, 64 key rows at a time.
template <typename To>
__device__ void head_output(const Tile& t, int r, int end, const float* __restrict__ S0,
                            To* o, int64_t p0, int32_t H, int h, float scale) {
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    // S0's key rows 0..63 into S now; rows 64..127 go through X once the scores are formed
#pragma unroll
    for (int mm = 0; mm < kTR * kTD / 4 / kTailThreads; ++mm) {
        const int idx = tid + mm * kTailThreads;
        cp_async16(t.s_addr + idx * 16, S0 + idx * 4, 16);
    }
    {
        // transposing writes: a warp takes 32 rows x 32 key channels along a diagonal
        // (lane l: row 32 rt + l, channel 32 ct + (l + d) % 32), so that both the row-major
        // reads and the column-major writes fall in 32 different banks
        const int n_units = ((end - r + 31) / 32) * (kTD / 32) * 32;
        for (int wu = warp; wu < n_units; wu += kTailWarps) {
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
    // Kd's factor exp(G_{r-1} - G_j) leaves fp32's range once a key channel decays by more
    // than e^-80 over the segment's rows here; the scores are then formed from one
    // exponential per (t, j, channel) instead, which has no range limit.
    bool big = false;
    if (tid < kTD) {
        const float gr = r > 0 ? t.G[(r - 1) * kTD + tid] : 0.f;
        big = !(t.G[(end - 1) * kTD + tid] - gr >= -80.f);
    }
    const bool strong = __syncthreads_or(big) != 0;   // also orders W and X before their reads
    {                                             // A[j][t] = Qd_t . Kd_j for r <= j <= t < end
        const int ta = tid >> 4, jb = tid & 15;   // rows t 2 ta, 2 ta + 1; columns j 4 jb .. +3
        float acc[2][4] = {};
        if (2 * ta + 1 >= r && 2 * ta < end && 4 * jb < end && 4 * jb <= 2 * ta + 1) {
            if (!strong) {
#pragma unroll 4
                for (int c = 0; c < kTD; ++c) {
                    const float2 w = *reinterpret_cast<const float2*>(t.W + c * kTR + 2 * ta);
                    const float4 x = *reinterpret_cast<const float4*>(t.X + c * kTR + 4 * jb);
                    const float wv[2] = {w.x, w.y}, xv[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                    for (int i = 0; i < 2; ++i)
#pragma unroll
                        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(wv[i], xv[j], acc[i][j]);
                }
            } else {
                // q_tc k_jc exp(G_tc - G_jc), channels taken from a per-thread offset so that
                // the threads of a warp read different banks; the exponent is capped at 0
                // (pairs j > t are discarded below)
                for (int c0 = 0; c0 < kTD; ++c0) {
                    const int c = (c0 + jb) & (kTD - 1);
                    float gt[2], qt[2];
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        gt[i] = t.G[(2 * ta + i) * kTD + c];
                        qt[i] = __bfloat162float(t.q[(2 * ta + i) * kTD + c]);
                    }
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int jj = 4 * jb + j;
                        const float gj = t.G[jj * kTD + c];
                        const float kj = t.beta[jj] * __bfloat162float(t.k[jj * kTD + c]);
#pragma unroll
                        for (int i = 0; i < 2; ++i)
                            acc[i][j] = fmaf(qt[i] * kj, expf(fminf(gt[i] - gj, 0.f)), acc[i][j]);
                    }
                }
            }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int jj = 4 * jb + j;
            float out[2];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int ti = 2 * ta + i;
                out[i] = (jj >= r && jj <= ti && ti < end) ? acc[i][j] : 0.f;
            }
            *reinterpret_cast<float2*>(t.A + jj * kTR + 2 * ta) = make_float2(out[0], out[1]);
        }
    }
    __syncthreads();                              // X (Kd) is free: S0's rows 64.. go through it
    const int tr = tid >> 5, cg = tid & 31;        // rows 4 tr .. +3, value columns 4 cg ..
    const int i0 = 4 * tr;
    const bool mine = i0 + 3 >= r && i0 < end;
    float2 acc[4][2];
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i][0] = acc[i][1] = make_float2(0.f, 0.f);
#pragma unroll
    for (int mm = 0; mm < kTR * kTD / 4 / kTailThreads; ++mm) {
        const int idx = tid + mm * kTailThreads;              // 16-byte group of the 32 KB block
        cp_async16(t.x_addr + idx * 16, S0 + 64 * kTD + idx * 4, 16);
    }
    cp_async_wait_all();
    __syncthreads();
#pragma unroll 1
    for (int half = 0; half < 2; ++half) {        // Qd^T S0, key rows 64 half .. +63
        const float* blk = half == 0 ? t.S : t.X;
        if (mine) {
#pragma unroll 4
            for (int cc = 0; cc < 64; ++cc) {
                const float4 w = *reinterpret_cast<const float4*>(t.W + (64 * half + cc) * kTR + i0);
                const float4 sv4 = *reinterpret_cast<const float4*>(blk + cc * kTD + 4 * cg);
                const float2 sv[2] = {make_float2(sv4.x, sv4.y), make_float2(sv4.z, sv4.w)};
                const float wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 w2 = make_float2(wv[i], wv[i]);
                    acc[i][0] = pfma(w2, sv[0], acc[i][0]);
                    acc[i][1] = pfma(w2, sv[1], acc[i][1]);
                }
            }
        }
    }
    __syncthreads();                              // S and X are read before they are refilled
    if (mine) {
        const int j_hi = (i0 + 4 < end) ? i0 + 4 : end;
        for (int j = r; j < j_hi; ++j) {          // + A V (A is zero outside the segment)
            const float4 a = *reinterpret_cast<const float4*>(t.A + j * kTR + i0);
            const float av[4] = {a.x, a.y, a.z, a.w};
            float2 vv[2];
            unpack4(*reinterpret_cast<const uint2*>(t.v + j * kTD + 4 * cg), vv);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 a2 = make_float2(av[i], av[i]);
                acc[i][0] = pfma(a2, vv[0], acc[i][0]);
                acc[i][1] = pfma(a2, vv[1], acc[i][1]);
            }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int row = i0 + i;
            if (row < r || row >= end) continue;
            store_out(o + ((p0 + row) * H + h) * kTD + 4 * cg, acc[i], scale);
        }
    }
    __syncthreads();                              // W and A are free again
}

template <typename To>
__global__ void __launch_bounds__(kTailThreads, 1)
state_tail_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                  const __nv_bfloat16* __restrict__ v, const __nv_bfloat16* __restrict__ g,
                  const __nv_bfloat16* __restrict__ beta, int64_t N, int32_t H, float scale,
                  void* ws, const float* __restrict__ init, float* fin, int64_t n_state,
                  To* o) {
    extern __shared__ __align__(16) uint8_t sm[];
    const uint32_t sbase = static_cast<uint32_t>(__cvta_generic_to_shared(sm));
    Tile t;
    t.q = reinterpret_cast<const __nv_bfloat16*>(sm + kSq);
    t.k = reinterpret_cast<const __nv_bfloat16*>(sm + kSk);
    t.v = reinterpret_cast<const __nv_bfloat16*>(sm + kSv);
    t.G = reinterpret_cast<const float*>(sm + kSG);
    t.W = reinterpret_cast<float*>(sm + kSW);
    t.X = reinterpret_cast<float*>(sm + kSX);
    t.A = reinterpret_cast<float*>(sm + kSA);
    t.beta = reinterpret_cast<const float*>(sm + kSB);
    t.S = reinterpret_cast<const float*>(sm + kSS);
    t.x_addr = sbase + kSX;
    t.s_addr = sbase + kSS;
    const int64_t n_chunks = ceil_div(N, kTR);
    const Plan pl = plan_view(ws, n_chunks);
    const int tid = threadIdx.x;
    const int64_t slot_elems = int64_t(kTD) * kTD;

    const int64_t n_units = int64_t(pl.counters[3]) * H;
    __shared__ int s_unit;
    for (;;) {
        if (tid == 0) s_unit = atomicAdd(&pl.counters[4], 1);
        __syncthreads();
        const int64_t u = s_unit;
        __syncthreads();                          // all have read it before it is rewritten
        if (u >= n_units) break;
        const int64_t c = pl.active[u / H];
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
        // segments starting here with a slot: the outputs of their rows here, and their
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
            // all 64 rows of q, k, v and g in flight at once (16-byte asynchronous copies;
            // rows past the end are zero-filled), beta alongside
            const __nv_bfloat16* src[4] = {q, k, v, g};
            const uint32_t dst[4] = {kSq, kSk, kSv, kSW};
#pragma unroll
            for (int a = 0; a < 4; ++a) {
#pragma unroll
                for (int mm = 0; mm < kTR * 16 / kTailThreads; ++mm) {
                    const int idx = tid + mm * kTailThreads;
                    const int i = idx >> 4, part = idx & 15;
                    const int64_t p = p0 + i;
                    const bool in = p < N;
                    cp_async16(sbase + dst[a] + idx * 16,
                               src[a] + ((in ? p : 0) * H + h) * kTD + part * 8, in ? 16u : 0u);
                }
            }
            if (tid < kTR) {
                const int64_t p = p0 + tid;
                reinterpret_cast<float*>(sm + kSB)[tid] =
                    p < N ? __bfloat162float(beta[p * H + h]) : 0.f;
            }
            cp_async_wait_all();
        }
        __syncthreads();
        {                                         // G: four threads per key channel, 16 rows each
            const __nv_bfloat16* gs = reinterpret_cast<const __nv_bfloat16*>(sm + kSW);
            float* G = reinterpret_cast<float*>(sm + kSG);
            float* qsum = reinterpret_cast<float*>(sm + kSQ);
            const int ch = tid & (kTD - 1), qd = tid >> 7;
            float run = 0.f;
#pragma unroll 8
            for (int i = 16 * qd; i < 16 * qd + 16; ++i) {
                if ((m.valid >> i) & 1ull) run += __bfloat162float(gs[i * kTD + ch]);
                G[i * kTD + ch] = run;
            }
            qsum[qd * kTD + ch] = run;
            __syncthreads();
            float before = 0.f;
            for (int q2 = 0; q2 < qd; ++q2) before += qsum[q2 * kTD + ch];
            if (qd > 0) {
#pragma unroll 8
                for (int i = 16 * qd; i < 16 * qd + 16; ++i) G[i * kTD + ch] += before;
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
            if (fin && (after != 0ull || next_cut))
                final_state(t, r, end - 1, S0, fin + (rank * H + h) * slot_elems);
            if (S0) head_output<To>(t, r, end, S0, o, p0, H, h, scale);
        }
    }
}

template <typename To>
kda_status_t launch_tail_typed(const void* q, const void* k, const void* v, const void* g,
                               const void* beta, int64_t N, int32_t H, float scale, void* o,
                               void* ws, const float* init, float* fin, int64_t n_state,
                               cudaStream_t stream) {
    if (dynamic_smem_attr<state_tail_kernel<To>>(int(kTailSmem)) != cudaSuccess)
        return KDA_ERR_CUDA;
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
