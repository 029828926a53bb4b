// kda_conv.cu -- segment-masked causal depthwise short convolution.
//
// [RFC-0025] "RFC-0025: 支持 Attention Varlen 功能并对齐 Loss", 方案 §3
// "ShortConvolution segment 边界 mask": y[b,t,f] = sum_j w[j,f] x[b,t-j,f] over
// taps j < K whose source token t-j exists and carries the destination's id.
//
// Design (HBM-bound: 2 x sizeof(dtype) bytes per element): a CTA of 256 threads
// owns a tile of kTok consecutive tokens of one row and 2 KB of features (1024
// bf16 or 512 fp32). It stages the tile and its K-1 halo tokens in shared memory
// with 16-byte asynchronous copies (cp.async: about 70 KB requested at once per
// CTA, no registers held), then each thread takes one 16-byte feature vector
// and half of the tile's tokens, slides a window of K-1 unpacked inputs along
// them and stores 16-byte outputs, coalesced along F. Halo tokens are re-read,
// mostly from L2. Products accumulate in fp32 and round once to the output.
#include "kda_common.cuh"

namespace kda {
namespace {

constexpr int kTok = 32;               // tokens per tile
constexpr int kTileBytes = 2048;       // feature bytes per tile row
constexpr int kCols = kTileBytes / 16; // 16-byte feature vectors per tile row
constexpr int kConvThreads = 2 * kCols;

template <typename T> struct Vec;
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
__global__ void __launch_bounds__(kConvThreads, (K <= 5 ? 3 : 2))
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
    const int c = threadIdx.x % kCols;          // this thread's feature vector
    const int half = threadIdx.x / kCols;       // tokens [16 half, 16 half + 16) of the tile
    float wr[K][V];
    if (c < cols) {
#pragma unroll
        for (int j = 0; j < K; ++j) Vec<T>::load(w + int64_t(j) * F + fb + c * V, wr[j]);
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncthreads();
    if (c >= cols) return;

    constexpr int kHalf = kTok / 2;
    const int r0 = half * kHalf;                // first output of this thread, tile-relative
    // window[j] holds the raw 16 bytes of token r - 1 - j (tile-relative r); they are
    // unpacked where used, which keeps the window at 4 registers per token
    uint4 win[K > 1 ? K - 1 : 1];
#pragma unroll
    for (int j = 0; j < Hl; ++j)
        win[j] = *reinterpret_cast<const uint4*>(tile + (Hl + r0 - 1 - j) * kTileBytes + c * 16);
#pragma unroll 1
    for (int r = r0; r < r0 + kHalf; ++r) {
        const int u = Hl + r;
        const int64_t t = t0 + r;
        if (t >= T_len) break;
        const uint4 cur_raw = *reinterpret_cast<const uint4*>(tile + u * kTileBytes + c * 16);
        const int32_t id = ids[u];
        float acc[V];
        {
            float cur[V];
            Vec<T>::cvt(cur_raw, cur);
#pragma unroll
            for (int e = 0; e < V; ++e) acc[e] = wr[0][e] * cur[e];
        }
#pragma unroll
        for (int j = 0; j < Hl; ++j) {
            // source token t - 1 - j exists (t - 1 - j >= 0) and carries the same id
            if (t - 1 - j >= 0 && ids[u - 1 - j] == id) {
                float src[V];
                Vec<T>::cvt(win[j], src);
#pragma unroll
                for (int e = 0; e < V; ++e) acc[e] = fmaf(wr[j + 1][e], src[e], acc[e]);
            }
        }
        Vec<T>::store(y + (row + t) * F + fb + c * V, acc);
#pragma unroll
        for (int j = Hl - 1; j > 0; --j) win[j] = win[j - 1];
        if (Hl > 0) win[0] = cur_raw;
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
