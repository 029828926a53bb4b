// kda_api.cu -- libkda's C entry points: host-side validation, then launches
// on the caller's stream. Semantics and argument contracts are in kda.h.
#include "kda_common.cuh"

namespace kda {
size_t recurrent_workspace_bytes(int64_t N);
size_t tc_workspace_bytes(int64_t N, int32_t H, bool with_slots);
kda_status_t launch_recurrent(const void* q, const void* k, const void* v, const void* g,
                              const void* beta, const int32_t* seg, int64_t B, int64_t T,
                              int32_t H, int32_t D, float scale, kda_dtype_t dtype,
                              kda_dtype_t out_dtype, void* o, void* ws, cudaStream_t stream);
kda_status_t launch_recurrent_state(const void* q, const void* k, const void* v, const void* g,
                                    const void* beta, const int32_t* seg, int64_t B, int64_t T_len,
                                    int32_t H, int32_t D, float scale, kda_dtype_t dtype,
                                    kda_dtype_t out_dtype, void* o, void* ws, const float* init,
                                    float* fin, int64_t n_state, cudaStream_t stream);
kda_status_t launch_recurrent_delta(const void* q, const void* k, const void* v, const void* g,
                                    const void* beta, const int32_t* seg, int64_t B, int64_t T_len,
                                    int32_t H, int32_t D, float scale, kda_dtype_t dtype,
                                    kda_dtype_t out_dtype, void* o, void* ws, cudaStream_t stream);
kda_status_t launch_chunk_plan(const int32_t* seg, int64_t B, int64_t T, int32_t H, int32_t D,
                               bool with_state, void* ws, size_t ws_bytes, cudaStream_t stream);
kda_status_t launch_chunk_tc(const void* q, const void* k, const void* v, const void* g,
                             const void* beta, const int32_t* seg, int64_t B, int64_t T,
                             int32_t H, int32_t D, float scale, kda_dtype_t out_dtype, void* o,
                             void* ws, size_t ws_bytes, uint32_t* status_dev, const float* init,
                             float* fin, int64_t n_state, bool plan, cudaStream_t stream,
                             const ConvIn* conv = nullptr);
size_t bwd_workspace_bytes(int64_t N, int32_t H, int32_t D);
kda_status_t launch_bwd(const void* q, const void* k, const void* v, const void* g,
                        const void* beta, const void* d_o, const int32_t* seg, int64_t B,
                        int64_t T_len, int32_t H, int32_t D, float scale, kda_dtype_t dtype,
                        kda_dtype_t grad_dtype, void* dq, void* dk, void* dv, void* dg,
                        void* dbeta, void* ws, cudaStream_t stream);
size_t bwd_tc_workspace_bytes(int64_t N, int32_t H);
kda_status_t launch_bwd_tc(const void* q, const void* k, const void* v, const void* g,
                           const void* beta, const void* d_o, const int32_t* seg, int64_t B,
                           int64_t T_len, int32_t H, float scale, kda_dtype_t grad_dtype,
                           void* dq, void* dk, void* dv, void* dg, void* dbeta, void* ws,
                           uint32_t* status_dev, cudaStream_t stream);
}  // namespace kda

namespace {

constexpr int64_t kMaxTokens = 2147483647LL;   // B*T < 2^31 (int32 token indices)

bool valid_dtype(kda_dtype_t d) { return d == KDA_F32 || d == KDA_BF16; }
size_t dtype_bytes(kda_dtype_t d) { return d == KDA_BF16 ? 2 : 4; }

bool token_count_ok(int64_t B, int64_t T) {
    return B >= 1 && T >= 1 && B <= kMaxTokens / T;
}

}  // namespace

namespace kda {

// The checks of the inputs and outputs that every forward entry point shares (all of
// kda_chunk_fwd_varlen's checks but the workspace's), in the order kda.h documents.
kda_status_t check_fwd_inputs(const void* q, const void* k, const void* v, const void* g,
                              const void* beta, const int32_t* segment_ids, int64_t B, int64_t T,
                              int32_t H, int32_t d_qk, int32_t d_v, kda_dtype_t dtype,
                              kda_dtype_t out_dtype, const void* o, const uint32_t* status_dev) {
    if (!q || !k || !v || !g || !beta || !o) return KDA_ERR_INVALID_ARG;
    if (!valid_dtype(dtype) || !valid_dtype(out_dtype) || !token_count_ok(B, T) || H < 1 ||
        d_qk < 1 || d_v < 1)
        return KDA_ERR_INVALID_ARG;
    if (out_dtype != dtype && out_dtype != KDA_F32) return KDA_ERR_UNSUPPORTED;
    if (d_qk != d_v || (d_qk != 64 && d_qk != 128)) return KDA_ERR_UNSUPPORTED;
    if (int64_t(H) * d_qk > 65536) return KDA_ERR_UNSUPPORTED;
    const void* ptrs[] = {q, k, v, g, beta, o};
    for (const void* p : ptrs)
        if (!kda::aligned(p, 16)) return KDA_ERR_INVALID_ARG;
    if (segment_ids && !kda::aligned(segment_ids, 4)) return KDA_ERR_INVALID_ARG;
    if (status_dev && !kda::aligned(status_dev, 4)) return KDA_ERR_INVALID_ARG;
    return KDA_OK;
}

}  // namespace kda

extern "C" {

const char* kda_status_string(kda_status_t s) {
    switch (s) {
        case KDA_OK: return "KDA_OK";
        case KDA_ERR_INVALID_ARG: return "KDA_ERR_INVALID_ARG";
        case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED";
        case KDA_ERR_CUDA: return "KDA_ERR_CUDA";
        case KDA_ERR_WORKSPACE: return "KDA_ERR_WORKSPACE";
    }
    return "KDA_UNKNOWN_STATUS";
}

kda_status_t kda_segids_to_cu_seqlens(const int32_t* segment_ids, int64_t B, int64_t T,
                                      int32_t max_segs, int32_t* cu_seqlens,
                                      int32_t* n_segs_out, kda_stream_t stream) {
    if (!segment_ids || !cu_seqlens) return KDA_ERR_INVALID_ARG;
    if (!token_count_ok(B, T) || max_segs < 1) return KDA_ERR_INVALID_ARG;
    if (!kda::aligned(segment_ids, 4) || !kda::aligned(cu_seqlens, 4) ||
        (n_segs_out && !kda::aligned(n_segs_out, 4)))
        return KDA_ERR_INVALID_ARG;
    return kda_launch_segids_to_cu_seqlens(segment_ids, B, T, max_segs, cu_seqlens, n_segs_out,
                                           reinterpret_cast<cudaStream_t>(stream));
}

kda_status_t kda_short_conv_varlen(const void* x, const void* weight,
                                   const int32_t* segment_ids, void* y, int64_t B, int64_t T,
                                   int64_t F, int32_t k_conv, kda_dtype_t dtype,
                                   kda_stream_t stream) {
    if (!x || !weight || !y) return KDA_ERR_INVALID_ARG;
    if (!valid_dtype(dtype) || !token_count_ok(B, T) || F < 1) return KDA_ERR_INVALID_ARG;
    if (k_conv < 1 || k_conv > 8) return KDA_ERR_UNSUPPORTED;
    if ((F * int64_t(dtype_bytes(dtype))) % 16 != 0) return KDA_ERR_UNSUPPORTED;
    if (!kda::aligned(x, 16) || !kda::aligned(weight, 16) || !kda::aligned(y, 16) ||
        (segment_ids && !kda::aligned(segment_ids, 4)))
        return KDA_ERR_INVALID_ARG;
    return kda_launch_short_conv(x, weight, segment_ids, y, B, T, F, k_conv, dtype,
                                 reinterpret_cast<cudaStream_t>(stream));
}

namespace {
size_t fwd_workspace(int64_t B, int64_t T, int32_t H, int32_t d_qk, int32_t d_v,
                     kda_dtype_t dtype, bool with_slots) {
    if (!token_count_ok(B, T) || H < 1 || d_qk < 1 || d_v < 1 || !valid_dtype(dtype)) return 0;
    const int64_t N = B * T;
    const size_t rec = kda::recurrent_workspace_bytes(N);
    if (dtype != KDA_BF16) return rec;
    const size_t tc = kda::tc_workspace_bytes(N, H, with_slots && d_qk == 128 && d_v == 128);
    return tc > rec ? tc : rec;
}
}  // namespace

size_t kda_chunk_fwd_varlen_workspace_size(int64_t B, int64_t T, int32_t H, int32_t d_qk,
                                           int32_t d_v, kda_dtype_t dtype) {
    return fwd_workspace(B, T, H, d_qk, d_v, dtype, true);
}

size_t kda_chunk_fwd_varlen_workspace_min(int64_t B, int64_t T, int32_t H, int32_t d_qk,
                                          int32_t d_v, kda_dtype_t dtype) {
    return fwd_workspace(B, T, H, d_qk, d_v, dtype, false);
}


namespace {

// The checks kda_chunk_fwd_varlen and kda_chunk_fwd_varlen_planned share.
kda_status_t check_fwd_args(const void* q, const void* k, const void* v, const void* g,
                            const void* beta, const int32_t* segment_ids, int64_t B, int64_t T,
                            int32_t H, int32_t d_qk, int32_t d_v, kda_dtype_t dtype,
                            kda_dtype_t out_dtype, const void* o, const void* workspace,
                            size_t workspace_bytes, const uint32_t* status_dev) {
    const kda_status_t s = kda::check_fwd_inputs(q, k, v, g, beta, segment_ids, B, T, H, d_qk,
                                                 d_v, dtype, out_dtype, o, status_dev);
    if (s != KDA_OK) return s;
    const size_t need = kda_chunk_fwd_varlen_workspace_min(B, T, H, d_qk, d_v, dtype);
    if (!workspace || workspace_bytes < need || !kda::aligned(workspace, 256))
        return KDA_ERR_WORKSPACE;
    return KDA_OK;
}

kda_status_t chunk_fwd(const void* q, const void* k, const void* v, const void* g,
                       const void* beta, const int32_t* segment_ids, int64_t B, int64_t T,
                       int32_t H, int32_t d_qk, int32_t d_v, float scale, kda_dtype_t dtype,
                       kda_dtype_t out_dtype, void* o, void* workspace, size_t workspace_bytes,
                       uint32_t* status_dev, bool plan, kda_stream_t stream) {
    const kda_status_t chk = check_fwd_args(q, k, v, g, beta, segment_ids, B, T, H, d_qk, d_v,
                                            dtype, out_dtype, o, workspace, workspace_bytes,
                                            status_dev);
    if (chk != KDA_OK) return chk;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (dtype == KDA_BF16)
        return kda::launch_chunk_tc(q, k, v, g, beta, segment_ids, B, T, H, d_qk, scale,
                                    out_dtype, o, workspace, workspace_bytes, status_dev, nullptr,
                                    nullptr, 0, plan, st);
    return kda::launch_recurrent(q, k, v, g, beta, segment_ids, B, T, H, d_qk, scale, dtype,
                                 out_dtype, o, workspace, st);
}

}  // namespace

kda_status_t kda_chunk_fwd_varlen(const void* q, const void* k, const void* v, const void* g,
                                  const void* beta, const int32_t* segment_ids, int64_t B,
                                  int64_t T, int32_t H, int32_t d_qk, int32_t d_v, float scale,
                                  kda_dtype_t dtype, kda_dtype_t out_dtype, void* o,
                                  void* workspace, size_t workspace_bytes,
                                  uint32_t* status_dev, kda_stream_t stream) {
    return chunk_fwd(q, k, v, g, beta, segment_ids, B, T, H, d_qk, d_v, scale, dtype, out_dtype,
                     o, workspace, workspace_bytes, status_dev, true, stream);
}

kda_status_t kda_chunk_plan_varlen(const int32_t* segment_ids, int64_t B, int64_t T, int32_t H,
                                   int32_t d_qk, int32_t d_v, kda_dtype_t dtype, void* workspace,
                                   size_t workspace_bytes, kda_stream_t stream) {
    if (!valid_dtype(dtype) || !token_count_ok(B, T) || H < 1 || d_qk < 1 || d_v < 1)
        return KDA_ERR_INVALID_ARG;
    if (d_qk != d_v || (d_qk != 64 && d_qk != 128)) return KDA_ERR_UNSUPPORTED;
    if (int64_t(H) * d_qk > 65536) return KDA_ERR_UNSUPPORTED;
    if (segment_ids && !kda::aligned(segment_ids, 4)) return KDA_ERR_INVALID_ARG;
    const size_t need = kda_chunk_fwd_varlen_workspace_min(B, T, H, d_qk, d_v, dtype);
    if (!workspace || workspace_bytes < need || !kda::aligned(workspace, 256))
        return KDA_ERR_WORKSPACE;
    if (dtype != KDA_BF16) return KDA_OK;     // the fp32 path plans inside its call
    return kda::launch_chunk_plan(segment_ids, B, T, H, d_qk, false, workspace, workspace_bytes,
                                  reinterpret_cast<cudaStream_t>(stream));
}

kda_status_t kda_chunk_fwd_varlen_planned(const void* q, const void* k, const void* v,
                                          const void* g, const void* beta,
                                          const int32_t* segment_ids, int64_t B, int64_t T,
                                          int32_t H, int32_t d_qk, int32_t d_v, float scale,
                                          kda_dtype_t dtype, kda_dtype_t out_dtype, void* o,
                                          void* workspace, size_t workspace_bytes,
                                          uint32_t* status_dev, kda_stream_t stream) {
    return chunk_fwd(q, k, v, g, beta, segment_ids, B, T, H, d_qk, d_v, scale, dtype, out_dtype,
                     o, workspace, workspace_bytes, status_dev, false, stream);
}

kda_status_t kda_chunk_fwd_varlen_conv(const void* x_q, const void* x_k, const void* x_v,
                                       const void* w_q, const void* w_k, const void* w_v,
                                       int32_t k_conv, const void* g, const void* beta,
                                       const int32_t* segment_ids, int64_t B, int64_t T,
                                       int32_t H, int32_t d_qk, int32_t d_v, float scale,
                                       kda_dtype_t dtype, kda_dtype_t out_dtype, void* o,
                                       void* workspace, size_t workspace_bytes, int planned,
                                       uint32_t* status_dev, kda_stream_t stream) {
    if (!w_q || !w_k || !w_v) return KDA_ERR_INVALID_ARG;
    const kda_status_t chk = check_fwd_args(x_q, x_k, x_v, g, beta, segment_ids, B, T, H, d_qk,
                                            d_v, dtype, out_dtype, o, workspace, workspace_bytes,
                                            status_dev);
    if (chk != KDA_OK) return chk;
    if (!kda::aligned(w_q, 16) || !kda::aligned(w_k, 16) || !kda::aligned(w_v, 16))
        return KDA_ERR_INVALID_ARG;
    if (dtype != KDA_BF16 || d_qk != 128 || d_v != 128) return KDA_ERR_UNSUPPORTED;
    if (k_conv < 1 || k_conv > 4) return KDA_ERR_UNSUPPORTED;
    const kda::ConvIn conv = {{w_q, w_k, w_v}, k_conv};
    return kda::launch_chunk_tc(x_q, x_k, x_v, g, beta, segment_ids, B, T, H, d_qk, scale,
                                out_dtype, o, workspace, workspace_bytes, status_dev, nullptr,
                                nullptr, 0, planned == 0, reinterpret_cast<cudaStream_t>(stream),
                                &conv);
}

kda_status_t kda_delta_fwd_varlen(const void* q, const void* k, const void* v, const void* g,
                                  const void* beta, const int32_t* segment_ids, int64_t B,
                                  int64_t T, int32_t H, int32_t d_qk, int32_t d_v, float scale,
                                  kda_dtype_t dtype, kda_dtype_t out_dtype, void* o,
                                  void* workspace, size_t workspace_bytes, uint32_t* status_dev,
                                  kda_stream_t stream) {
    const kda_status_t chk = check_fwd_args(q, k, v, g, beta, segment_ids, B, T, H, d_qk, d_v,
                                            dtype, out_dtype, o, workspace, workspace_bytes,
                                            status_dev);
    if (chk != KDA_OK) return chk;
    return kda::launch_recurrent_delta(q, k, v, g, beta, segment_ids, B, T, H, d_qk, scale, dtype,
                                       out_dtype, o, workspace,
                                       reinterpret_cast<cudaStream_t>(stream));
}

kda_status_t kda_chunk_fwd_varlen_state(const void* q, const void* k, const void* v,
                                        const void* g, const void* beta,
                                        const int32_t* segment_ids, int64_t B, int64_t T,
                                        int32_t H, int32_t d_qk, int32_t d_v, float scale,
                                        kda_dtype_t dtype, kda_dtype_t out_dtype, void* o,
                                        const float* initial_state, float* final_state,
                                        int64_t n_state, void* workspace, size_t workspace_bytes,
                                        uint32_t* status_dev, kda_stream_t stream) {
    if (!q || !k || !v || !g || !beta || !o) return KDA_ERR_INVALID_ARG;
    if (!valid_dtype(dtype) || !valid_dtype(out_dtype) || !token_count_ok(B, T) || H < 1 ||
        d_qk < 1 || d_v < 1 || n_state < 0)
        return KDA_ERR_INVALID_ARG;
    if (out_dtype != dtype && out_dtype != KDA_F32) return KDA_ERR_UNSUPPORTED;
    if (d_qk != d_v || (d_qk != 64 && d_qk != 128)) return KDA_ERR_UNSUPPORTED;
    if (int64_t(H) * d_qk > 65536) return KDA_ERR_UNSUPPORTED;
    if (n_state > (int64_t(1) << 40) / (int64_t(H) * d_qk * d_v)) return KDA_ERR_UNSUPPORTED;
    const void* ptrs[] = {q, k, v, g, beta, o};
    for (const void* p : ptrs)
        if (!kda::aligned(p, 16)) return KDA_ERR_INVALID_ARG;
    if ((initial_state && !kda::aligned(initial_state, 16)) ||
        (final_state && !kda::aligned(final_state, 16)))
        return KDA_ERR_INVALID_ARG;
    if (segment_ids && !kda::aligned(segment_ids, 4)) return KDA_ERR_INVALID_ARG;
    if (status_dev && !kda::aligned(status_dev, 4)) return KDA_ERR_INVALID_ARG;
    const size_t need = kda_chunk_fwd_varlen_workspace_min(B, T, H, d_qk, d_v, dtype);
    if (!workspace || workspace_bytes < need || !kda::aligned(workspace, 256))
        return KDA_ERR_WORKSPACE;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (dtype == KDA_BF16 && d_qk == 128)   // tensor-core chunked form, then the state pass
        return kda::launch_chunk_tc(q, k, v, g, beta, segment_ids, B, T, H, d_qk, scale,
                                    out_dtype, o, workspace, workspace_bytes, status_dev,
                                    initial_state, final_state, n_state, true, st);
    return kda::launch_recurrent_state(q, k, v, g, beta, segment_ids, B, T, H, d_qk, scale, dtype,
                                       out_dtype, o, workspace, initial_state, final_state,
                                       n_state, st);
}

size_t kda_chunk_bwd_varlen_workspace_size(int64_t B, int64_t T, int32_t H, int32_t d_qk,
                                           int32_t d_v, kda_dtype_t dtype) {
    if (!token_count_ok(B, T) || H < 1 || d_qk < 1 || d_v < 1 || !valid_dtype(dtype)) return 0;
    if (d_qk != d_v || (d_qk != 64 && d_qk != 128)) return 0;
    const size_t walk = kda::bwd_workspace_bytes(B * T, H, d_qk);
    if (dtype != KDA_BF16 || d_qk != 128) return walk;
    const size_t tc = kda::bwd_tc_workspace_bytes(B * T, H);
    return walk > tc ? walk : tc;
}

kda_status_t kda_chunk_bwd_varlen_ex(const void* q, const void* k, const void* v, const void* g,
                                     const void* beta, const int32_t* segment_ids, int64_t B,
                                     int64_t T, int32_t H, int32_t d_qk, int32_t d_v, float scale,
                                     kda_dtype_t dtype, const void* d_o, kda_dtype_t grad_dtype,
                                     void* dq, void* dk, void* dv, void* dg, void* dbeta,
                                     void* workspace, size_t workspace_bytes, int32_t method,
                                     uint32_t* status_dev, kda_stream_t stream) {
    if (!q || !k || !v || !g || !beta || !d_o || !dq || !dk || !dv || !dg || !dbeta)
        return KDA_ERR_INVALID_ARG;
    if (!valid_dtype(dtype) || !valid_dtype(grad_dtype) || !token_count_ok(B, T) || H < 1 ||
        d_qk < 1 || d_v < 1)
        return KDA_ERR_INVALID_ARG;
    if (method != KDA_BWD_AUTO && method != KDA_BWD_WALK) return KDA_ERR_INVALID_ARG;
    if (grad_dtype != dtype && grad_dtype != KDA_F32) return KDA_ERR_UNSUPPORTED;
    if (d_qk != d_v || (d_qk != 64 && d_qk != 128)) return KDA_ERR_UNSUPPORTED;
    if (int64_t(H) * d_qk > 65536) return KDA_ERR_UNSUPPORTED;
    const void* ptrs[] = {q, k, v, g, beta, d_o, dq, dk, dv, dg, dbeta};
    for (const void* p : ptrs)
        if (!kda::aligned(p, 16)) return KDA_ERR_INVALID_ARG;
    if (segment_ids && !kda::aligned(segment_ids, 4)) return KDA_ERR_INVALID_ARG;
    if (status_dev && !kda::aligned(status_dev, 4)) return KDA_ERR_INVALID_ARG;
    const size_t need = kda_chunk_bwd_varlen_workspace_size(B, T, H, d_qk, d_v, dtype);
    if (!workspace || workspace_bytes < need || !kda::aligned(workspace, 256))
        return KDA_ERR_WORKSPACE;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (method == KDA_BWD_AUTO && dtype == KDA_BF16 && d_qk == 128)
        return kda::launch_bwd_tc(q, k, v, g, beta, d_o, segment_ids, B, T, H, scale, grad_dtype,
                                  dq, dk, dv, dg, dbeta, workspace, status_dev, st);
    return kda::launch_bwd(q, k, v, g, beta, d_o, segment_ids, B, T, H, d_qk, scale, dtype,
                           grad_dtype, dq, dk, dv, dg, dbeta, workspace, st);
}

kda_status_t kda_chunk_bwd_varlen(const void* q, const void* k, const void* v, const void* g,
                                  const void* beta, const int32_t* segment_ids, int64_t B,
                                  int64_t T, int32_t H, int32_t d_qk, int32_t d_v, float scale,
                                  kda_dtype_t dtype, const void* d_o, kda_dtype_t grad_dtype,
                                  void* dq, void* dk, void* dv, void* dg, void* dbeta,
                                  void* workspace, size_t workspace_bytes, kda_stream_t stream) {
    return kda_chunk_bwd_varlen_ex(q, k, v, g, beta, segment_ids, B, T, H, d_qk, d_v, scale,
                                   dtype, d_o, grad_dtype, dq, dk, dv, dg, dbeta, workspace,
                                   workspace_bytes, KDA_BWD_AUTO, nullptr, stream);
}

}  // extern "C"
