// kda_conv.cu -- segment-masked causal depthwise short convolution.
//
// [RFC-0025] "RFC-0025: 支持 Attention Varlen 功能并对齐 Loss", 方案 §3
// "ShortConvolution segment 边界 mask": y[b,t,f] = sum_j w[j,f] x[b,t-j,f] over
// taps j < K whose source token t-j exists and carries the destination's id.
//
// Design (HBM-bound: 2 x sizeof(dtype) bytes per element): a CTA of 128 threads
// owns a tile of kTok consecutive tokens of one row and 2 KB of features (1024
// bf16 or 512 fp32). It stages the tile and its K-1 halo tokens in shared memory
// with 16-byte asynchronous copies (cp.async: the whole tile requested at once, no
// registers held), then each thread takes one 16-byte feature vector, slides a
// window of K-1 unpacked inputs along the tile's tokens (fully unrolled, packed
// fp32x2 arithmetic) and stores 16-byte outputs,
// coalesced along F. Small tiles let several CTAs per SM keep loads in flight while
// others compute. Halo tokens are re-read, mostly from L2. Products accumulate in
// fp32 and round once to the output.
#include "kda_common.cuh"

namespace kda {
namespace {

constexpr int kTok = 16;               // tokens per tile
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

template <int K>
constexpr int conv_smem_bytes() { return (kTok + K - 1) * kTileBytes; }

template <typename T, int K>
__global__ void __launch_bounds__(kConvThreads, (K <= 5 ? 5 : 2))
short_conv_kernel(const T* __restrict__ x, const T* __restrict__ w,
                  const int32_t* __restrict__ seg, T* __restrict__ y, int64_t T_len,
                  int64_t F, int64_t tiles_per_row) {
    constexpr int V = Vec<T>::N;
    constexpr int Hl = K - 1;                  // halo tokens before the tile
    constexpr int R = kTok + Hl;               // staged rows; row u holds token t0 - Hl + u
    extern __shared__ __align__(16) uint8_t tile[];
    __shared__ int32_t ids[R];
    const int64_t b = blockIdx.x / tiles_per_row;      // token tiles along x, feature tiles along y
    const int64_t t0 = (blockIdx.x % tiles_per_row) * kTok;
    const int64_t fb = int64_t(blockIdx.y) * (kTileBytes / sizeof(T));   // first feature
    const int64_t row = b * T_len;
    const int64_t f_left = F - fb;
    const int cols = f_left * int64_t(sizeof(T)) >= kTileBytes
                         ? kCols : int(f_left * int64_t(sizeof(T)) / 16);

    // stage rows of tokens that exist (rows outside the row are never read below)
    for (int i = threadIdx.x; i < R * kCols; i += kConvThreads) {
        const int u = i / kCols, c = i % kCols;
        const int64_t t = t0 - Hl + u;
        if (c < cols && t >= 0 && t < T_len)
            cp_async16(tile + u * kTileBytes + c * 16, x + (row + t) * F + fb + c * V);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    for (int u = threadIdx.x; u < R; u += kConvThreads) {
        const int64_t t = t0 - Hl + u;
        ids[u] = (seg && t >= 0 && t < T_len) ? seg[row + t] : 0;
    }
    const int c = threadIdx.x;                  // this thread's feature vector
    constexpr int P = Pairs<T>::P;
    float2 wp[K][P];                            // the K taps of this vector, as pairs
    if (c < cols) {
#pragma unroll
        for (int j = 0; j < K; ++j)
            Pairs<T>::cvt(*reinterpret_cast<const uint4*>(w + int64_t(j) * F + fb + c * V), wp[j]);
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncthreads();
    if (c >= cols) return;

    // The tile's tokens, fully unrolled: win[j] holds the unpacked input of token r-1-j,
    // so each input is converted once and the window shifts by renaming registers.
    // Rows past the end of the row were not staged: they are never stored and never
    // feed a stored output (sources precede their destinations).
    float2 win[K > 1 ? K - 1 : 1][P];
#pragma unroll
    for (int j = 0; j < Hl; ++j)
        Pairs<T>::cvt(*reinterpret_cast<const uint4*>(tile + (Hl - 1 - j) * kTileBytes + c * 16), win[j]);
#pragma unroll
    for (int r = 0; r < kTok; ++r) {
        const int u = Hl + r;
        const int64_t t = t0 + r;
        float2 cur[P];
        Pairs<T>::cvt(*reinterpret_cast<const uint4*>(tile + u * kTileBytes + c * 16), cur);
        const int32_t id = ids[u];
        float2 acc[P];
#pragma unroll
        for (int p = 0; p < P; ++p) acc[p] = mul2(wp[0][p], cur[p]);
#pragma unroll
        for (int j = 0; j < Hl; ++j) {
            // source token t - 1 - j exists (t - 1 - j >= 0) and carries the same id
            if (t - 1 - j >= 0 && ids[u - 1 - j] == id) {
#pragma unroll
                for (int p = 0; p < P; ++p) acc[p] = fma2(wp[j + 1][p], win[j][p], acc[p]);
            }
        }
        if (t < T_len) *reinterpret_cast<uint4*>(y + (row + t) * F + fb + c * V) = Pairs<T>::pack(acc);
#pragma unroll
        for (int j = Hl - 1; j > 0; --j) {
#pragma unroll
            for (int p = 0; p < P; ++p) win[j][p] = win[j - 1][p];
        }
        if (Hl > 0) {
#pragma unroll
            for (int p = 0; p < P; ++p) win[0][p] = cur[p];
        }
    }
}

template <typename T>
kda_status_t launch_typed(const void* x, const void* w, const int32_t* seg, void* y, int64_t B,
                          int64_t T_len, int64_t F, int32_t K, cudaStream_t stream) {
    const int64_t tiles = ceil_div(T_len, kTok);
    const int64_t gx = B * tiles;
    const int64_t gy = ceil_div(F * int64_t(sizeof(T)), kTileBytes);
    if (gx > 2147483647LL || gy > 65535) return KDA_ERR_UNSUPPORTED;
    const dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(gy), 1u);
    const T* xp = static_cast<const T*>(x);
    const T* wp = static_cast<const T*>(w);
    T* yp = static_cast<T*>(y);
    switch (K) {
#define KDA_CONV_CASE(KK)                                                                      \
    case KK: {                                                                                 \
        static cudaError_t attr = cudaFuncSetAttribute(                                        \
            short_conv_kernel<T, KK>, cudaFuncAttributeMaxDynamicSharedMemorySize,              \
            conv_smem_bytes<KK>());                                                            \
        if (attr != cudaSuccess) return KDA_ERR_CUDA;                                          \
        short_conv_kernel<T, KK><<<grid, kConvThreads, conv_smem_bytes<KK>(), stream>>>(       \
            xp, wp, seg, yp, T_len, F, tiles);                                                 \
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
