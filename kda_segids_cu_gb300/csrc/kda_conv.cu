// kda_conv.cu -- segment-masked causal depthwise short convolution.
//
// [RFC-0025] "RFC-0025: 支持 Attention Varlen 功能并对齐 Loss", 方案 §3
// "ShortConvolution segment 边界 mask": y[b,t,f] = sum_j w[j,f] x[b,t-j,f] over
// taps j < K whose source token t-j exists and carries the destination's id.
//
// Design (HBM-bound: 2 x sizeof(dtype) bytes per element): a CTA of 128 threads
// owns 2 KB of features (1024 bf16 or 512 fp32) of one row and streams a span of
// its tokens, three CTAs per SM (two for K >= 7). Each thread owns one 16-byte feature
// vector and walks the span in tiles of kTok = 8 tokens through a ring of kRing = 4 tiles in
// shared memory, filled by 16-byte asynchronous copies (cp.async, kRing - 1 tiles requested
// ahead, no registers held). A thread reads back only what it copied, so the ring needs no
// barrier. It slides a window of K-1 unpacked inputs along the tokens (fully unrolled
// per tile, packed fp32x2 arithmetic); the window carries across tiles, so only a
// span's first K-1 tokens are read twice. Outputs are 16-byte stores, coalesced
// along F. Products accumulate in fp32 and round once to the output.
#include "kda_common.cuh"

namespace kda {
namespace {

// 8-token tiles, a ring of 4, three CTAs per SM: 47.3 us per conv of a [4, 8192, 2048] bf16
// input (width 4) against 47.8 us with 16-token tiles, a ring of 3 and two CTAs per SM
constexpr int kTok = 8;                // tokens per tile
constexpr int kRing = 4;               // tiles of the ring (kRing - 1 in flight while one is used)
// CTAs per SM: three (192 KB of rings), or two for the widest windows (K >= 7), whose
// registers would not fit three
constexpr int conv_ctas_per_sm(int k) { return k >= 7 ? 2 : 3; }
constexpr int kTileBytes = 2048;       // feature bytes per tile row
constexpr int kCols = kTileBytes / 16; // 16-byte feature vectors per tile row
constexpr int kConvThreads = kCols;       // one thread per 16-byte feature vector

template <typename T> struct Vec;
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 u, v, w;\n\tmov.b64 u, {%2, %3};\n\tmov.b64 v, {%4, %5};\n\t"
        "mul.rn.f32x2 w, u, v;\n\tmov.b64 {%0, %1}, w;\n\t}"
        : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 u, v, w, z;\n\tmov.b64 u, {%2, %3};\n\tmov.b64 v, {%4, %5};\n\t"
        "mov.b64 w, {%6, %7};\n\tfma.rn.f32x2 z, u, v, w;\n\tmov.b64 {%0, %1}, z;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

// 16-byte vectors as pairs of fp32 values (P pairs).
template <typename T> struct Pairs;
template <> struct Pairs<__nv_bfloat16> {
    static constexpr int P = 4;
    __device__ static void cvt(const uint4& u, float2 (&o)[P]) {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)     // bf16 -> fp32 is exact: the bits are the top half
            o[i] = make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
    }
    __device__ static uint4 pack(const float2 (&a)[P]) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __nv_bfloat162 h = __floats2bfloat162_rn(a[i].x, a[i].y);
            w[i] = *reinterpret_cast<const uint32_t*>(&h);
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
};
template <> struct Pairs<float> {
    static constexpr int P = 2;
    __device__ static void cvt(const uint4& u, float2 (&o)[P]) {
        o[0] = make_float2(__uint_as_float(u.x), __uint_as_float(u.y));
        o[1] = make_float2(__uint_as_float(u.z), __uint_as_float(u.w));
    }
    __device__ static uint4 pack(const float2 (&a)[P]) {
        return make_uint4(__float_as_uint(a[0].x), __float_as_uint(a[0].y), __float_as_uint(a[1].x),
                          __float_as_uint(a[1].y));
    }
};

template <> struct Vec<__nv_bfloat16> {
    static constexpr int N = 8;
    __device__ static void load(const void* p, float* out) {
        cvt(*reinterpret_cast<const uint4*>(p), out);
    }
    __device__ static void cvt(const uint4& u, float* out) {
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __bfloat1622float2(h[i]);
            out[2 * i] = f.x;
            out[2 * i + 1] = f.y;
        }
    }
    __device__ static void store(void* p, const float* in) {
        uint4 u;
        __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
        for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(in[2 * i], in[2 * i + 1]);
        *reinterpret_cast<uint4*>(p) = u;
    }
};
template <> struct Vec<float> {
    static constexpr int N = 4;
    __device__ static void load(const void* p, float* out) {
        cvt(*reinterpret_cast<const uint4*>(p), out);
    }
    __device__ static void cvt(const uint4& u, float* out) {
        out[0] = __uint_as_float(u.x); out[1] = __uint_as_float(u.y);
        out[2] = __uint_as_float(u.z); out[3] = __uint_as_float(u.w);
    }
    __device__ static void store(void* p, const float* in) {
        *reinterpret_cast<float4*>(p) = make_float4(in[0], in[1], in[2], in[3]);
    }
};

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(
                     __cvta_generic_to_shared(smem))), "l"(gmem) : "memory");
}

constexpr int conv_smem_bytes() { return kRing * kTok * kTileBytes; }

__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <typename T, int K>
__global__ void __launch_bounds__(kConvThreads, conv_ctas_per_sm(K))
short_conv_kernel(const T* __restrict__ x, const T* __restrict__ w,
                  const int32_t* __restrict__ seg, T* __restrict__ y, int64_t T_len,
                  int64_t F, int64_t span, int64_t spans_per_row) {
    constexpr int V = Vec<T>::N;
    constexpr int Hl = K - 1;                  // window: the K-1 tokens before the current one
    constexpr int P = Pairs<T>::P;
    extern __shared__ __align__(16) uint8_t ring[];
    const int64_t b = blockIdx.x / spans_per_row;      // (row, span) along x, feature block along y
    const int64_t s0 = (blockIdx.x % spans_per_row) * span;
    const int64_t s1 = (s0 + span < T_len) ? s0 + span : T_len;
    const int64_t fb = int64_t(blockIdx.y) * (kTileBytes / sizeof(T));   // first feature
    const int64_t f_left = F - fb;
    const int cols = f_left * int64_t(sizeof(T)) >= kTileBytes
                         ? kCols : int(f_left * int64_t(sizeof(T)) / 16);
    const int c = threadIdx.x;                  // this thread's feature vector
    if (c >= cols || s0 >= s1) return;          // no barrier below: leaving early is safe
    const T* xc = x + b * T_len * F + fb + c * V;   // token t of this vector at xc + t * F
    T* yc = y + b * T_len * F + fb + c * V;
    const int32_t* sr = seg ? seg + b * T_len : nullptr;
    uint8_t* mine = ring + c * 16;                  // this thread's column of every ring row
    const int n_tiles = int((s1 - s0 + kTok - 1) / kTok);

    auto issue = [&](int ti) {                  // tile ti of the span into ring slot ti % kRing
        if (ti < n_tiles) {
            const int64_t t0 = s0 + int64_t(ti) * kTok;
            uint8_t* slot = mine + (ti % kRing) * (kTok * kTileBytes);
#pragma unroll
            for (int r = 0; r < kTok; ++r)
                if (t0 + r < s1) cp_async16(slot + r * kTileBytes, xc + (t0 + r) * F);
        }
        cp_async_commit();                      // one group per tile, empty past the end
    };
#pragma unroll
    for (int ti = 0; ti < kRing - 1; ++ti) issue(ti);

    float2 wp[K][P];                            // the K taps of this vector, as pairs
#pragma unroll
    for (int j = 0; j < K; ++j)
        Pairs<T>::cvt(*reinterpret_cast<const uint4*>(w + int64_t(j) * F + fb + c * V), wp[j]);
    // the window before the span: win[j] is token s0-1-j, wid[j] its id
    float2 win[K > 1 ? K - 1 : 1][P];
    int32_t wid[K > 1 ? K - 1 : 1];
#pragma unroll
    for (int j = 0; j < Hl; ++j) {
        const int64_t t = s0 - 1 - j;
        if (t >= 0) {
            Pairs<T>::cvt(*reinterpret_cast<const uint4*>(xc + t * F), win[j]);
            wid[j] = sr ? sr[t] : 0;
        } else {
#pragma unroll
            for (int p = 0; p < P; ++p) win[j][p] = make_float2(0.f, 0.f);
            wid[j] = 0;
        }
    }

    for (int ti = 0; ti < n_tiles; ++ti) {
        issue(ti + kRing - 1);
        const int64_t t0 = s0 + int64_t(ti) * kTok;
        int32_t ids[kTok];
#pragma unroll
        for (int r = 0; r < kTok; ++r) ids[r] = (sr && t0 + r < s1) ? sr[t0 + r] : 0;
        cp_async_wait<kRing - 1>();             // this tile's copies have landed
        const uint8_t* slot = mine + (ti % kRing) * (kTok * kTileBytes);
#pragma unroll
        for (int r = 0; r < kTok; ++r) {
            const int64_t t = t0 + r;
            if (t >= s1) break;
            float2 cur[P];
            Pairs<T>::cvt(*reinterpret_cast<const uint4*>(slot + r * kTileBytes), cur);
            const int32_t id = ids[r];
            float2 acc[P];
#pragma unroll
            for (int p = 0; p < P; ++p) acc[p] = mul2(wp[0][p], cur[p]);
#pragma unroll
            for (int j = 0; j < Hl; ++j) {
                // source token t - 1 - j exists (t - 1 - j >= 0) and carries the same id
                if (t - 1 - j >= 0 && wid[j] == id) {
#pragma unroll
                    for (int p = 0; p < P; ++p) acc[p] = fma2(wp[j + 1][p], win[j][p], acc[p]);
                }
            }
            *reinterpret_cast<uint4*>(yc + t * F) = Pairs<T>::pack(acc);
#pragma unroll
            for (int j = Hl - 1; j > 0; --j) {
                wid[j] = wid[j - 1];
#pragma unroll
                for (int p = 0; p < P; ++p) win[j][p] = win[j - 1][p];
            }
            if (Hl > 0) {
                wid[0] = id;
#pragma unroll
                for (int p = 0; p < P; ++p) win[0][p] = cur[p];
            }
        }
    }
    cp_async_wait<0>();                         // nothing left in flight when the thread exits
}

template <typename T>
kda_status_t launch_typed(const void* x, const void* w, const int32_t* seg, void* y, int64_t B,
                          int64_t T_len, int64_t F, int32_t K, cudaStream_t stream) {
    const int64_t gy = ceil_div(F * int64_t(sizeof(T)), kTileBytes);
    // spans of whole tiles, about conv_ctas_per_sm(K) CTAs per SM over all (row, feature block)
    const int64_t target = int64_t(conv_ctas_per_sm(K)) * sm_count();
    const int64_t pairs = B * gy;
    int64_t spans = ceil_div(target, pairs > 0 ? pairs : 1);
    int64_t span = ceil_div(ceil_div(T_len, spans), int64_t(kTok)) * kTok;
    if (span < kTok) span = kTok;
    spans = ceil_div(T_len, span);
    const int64_t gx = B * spans;
    if (gx > 2147483647LL || gy > 65535) return KDA_ERR_UNSUPPORTED;
    const dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(gy), 1u);
    const T* xp = static_cast<const T*>(x);
    const T* wp = static_cast<const T*>(w);
    T* yp = static_cast<T*>(y);
    switch (K) {
#define KDA_CONV_CASE(KK)                                                                      \
    case KK: {                                                                                 \
        if (dynamic_smem_attr<short_conv_kernel<T, KK>>(conv_smem_bytes()) != cudaSuccess)     \
            return KDA_ERR_CUDA;                                                               \
        short_conv_kernel<T, KK><<<grid, kConvThreads, conv_smem_bytes(), stream>>>(           \
            xp, wp, seg, yp, T_len, F, span, spans);                                           \
        break;                                                                                 \
    }
        KDA_CONV_CASE(1) KDA_CONV_CASE(2) KDA_CONV_CASE(3) KDA_CONV_CASE(4)
        KDA_CONV_CASE(5) KDA_CONV_CASE(6) KDA_CONV_CASE(7) KDA_CONV_CASE(8)
#undef KDA_CONV_CASE
        default:
            return KDA_ERR_UNSUPPORTED;
    }
    return launch_status();
}

}  // namespace
}  // namespace kda

kda_status_t kda_launch_short_conv(const void* x, const void* w, const int32_t* seg, void* y,
                                   int64_t B, int64_t T, int64_t F, int32_t K, kda_dtype_t dtype,
                                   cudaStream_t stream) {
    if (dtype == KDA_BF16)
        return kda::launch_typed<__nv_bfloat16>(x, w, seg, y, B, T, F, K, stream);
    return kda::launch_typed<float>(x, w, seg, y, B, T, F, K, stream);
}
