// kda_conv.cu -- segment-masked causal depthwise short convolution.
//
// [RFC-0025] "RFC-0025: 支持 Attention Varlen 功能并对齐 Loss", 方案 §3
// "ShortConvolution segment 边界 mask": y[b,t,f] = sum_j w[j,f] x[b,t-j,f] over
// taps j < K whose source token t-j exists and carries the destination's id.
//
// Design (HBM-bound: 2 x sizeof(dtype) bytes per element): each thread owns
// one 16-byte vector of features (8 bf16 or 4 fp32) and a run of kRun
// consecutive tokens of one row. It keeps the K-1 previous input vectors and
// their ids in registers, so every input vector is read from memory once per
// run (the K-1 halo tokens of a run are re-read, mostly from L2). Loads and
// stores are 16-byte and coalesced along F; the ids are warp-uniform
// broadcast loads. Products accumulate in fp32 and round once to the output.
#include "kda_common.cuh"

namespace kda {
namespace {

constexpr int kRun = 16;       // tokens per thread
constexpr int kThreadsX = 128; // feature vectors per block

template <typename T> struct Vec;
template <> struct Vec<__nv_bfloat16> {
    static constexpr int N = 8;
    __device__ static void load(const void* p, float* out) {
        const uint4 u = *reinterpret_cast<const uint4*>(p);
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
        const float4 f = *reinterpret_cast<const float4*>(p);
        out[0] = f.x; out[1] = f.y; out[2] = f.z; out[3] = f.w;
    }
    __device__ static void store(void* p, const float* in) {
        *reinterpret_cast<float4*>(p) = make_float4(in[0], in[1], in[2], in[3]);
    }
};

template <typename T, int K>
__global__ void __launch_bounds__(kThreadsX)
short_conv_kernel(const T* __restrict__ x, const T* __restrict__ w,
                  const int32_t* __restrict__ seg, T* __restrict__ y, int64_t T_len,
                  int64_t F, int64_t runs_per_row) {
    constexpr int V = Vec<T>::N;
    const int64_t fv = int64_t(blockIdx.x) * kThreadsX + threadIdx.x;   // feature vector
    if (fv * V >= F) return;
    const int64_t b = blockIdx.y / runs_per_row;
    const int64_t t0 = (blockIdx.y % runs_per_row) * kRun;
    const int64_t f0 = fv * V;
    const int64_t row = b * T_len;

    float wr[K][V];
#pragma unroll
    for (int j = 0; j < K; ++j) Vec<T>::load(w + int64_t(j) * F + f0, wr[j]);

    // window[j] holds x[t-1-j] and its id (or zeros / an impossible id before t = 0)
    float win[K > 1 ? K - 1 : 1][V];
    int32_t wid[K > 1 ? K - 1 : 1];
#pragma unroll
    for (int j = 0; j < K - 1; ++j) {
        const int64_t s = t0 - 1 - j;
        if (s >= 0) {
            Vec<T>::load(x + (row + s) * F + f0, win[j]);
            wid[j] = seg ? seg[row + s] : 0;
        } else {
#pragma unroll
            for (int e = 0; e < V; ++e) win[j][e] = 0.f;
            wid[j] = INT32_MIN;   // never equal to a real or padding id
        }
    }

    const int64_t t_end = (t0 + kRun < T_len) ? t0 + kRun : T_len;
    for (int64_t t = t0; t < t_end; ++t) {
        float cur[V];
        Vec<T>::load(x + (row + t) * F + f0, cur);
        const int32_t id = seg ? seg[row + t] : 0;
        float acc[V];
#pragma unroll
        for (int e = 0; e < V; ++e) acc[e] = wr[0][e] * cur[e];
#pragma unroll
        for (int j = 0; j < K - 1; ++j) {
            if (wid[j] == id) {
#pragma unroll
                for (int e = 0; e < V; ++e) acc[e] = fmaf(wr[j + 1][e], win[j][e], acc[e]);
            }
        }
        Vec<T>::store(y + (row + t) * F + f0, acc);
        // shift the window
#pragma unroll
        for (int j = K - 2; j > 0; --j) {
#pragma unroll
            for (int e = 0; e < V; ++e) win[j][e] = win[j - 1][e];
            wid[j] = wid[j - 1];
        }
        if (K > 1) {
#pragma unroll
            for (int e = 0; e < V; ++e) win[0][e] = cur[e];
            wid[0] = id;
        }
    }
}

template <typename T>
kda_status_t launch_typed(const void* x, const void* w, const int32_t* seg, void* y, int64_t B,
                          int64_t T_len, int64_t F, int32_t K, cudaStream_t stream) {
    constexpr int V = Vec<T>::N;
    const int64_t runs = ceil_div(T_len, kRun);
    const int64_t gy = B * runs;
    const int64_t gx = ceil_div(F / V, kThreadsX);
    if (gy > 2147483647LL || gx > 65535) return KDA_ERR_UNSUPPORTED;
    const dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(gy), 1u);
    const T* xp = static_cast<const T*>(x);
    const T* wp = static_cast<const T*>(w);
    T* yp = static_cast<T*>(y);
    switch (K) {
#define KDA_CONV_CASE(KK)                                                                   \
    case KK:                                                                                \
        short_conv_kernel<T, KK><<<grid, kThreadsX, 0, stream>>>(xp, wp, seg, yp, T_len, F, \
                                                                 runs);                     \
        break;
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
