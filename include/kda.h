/*
 * kda.h -- C ABI of libkda: the packed (varlen) Kimi Delta Attention forward
 * on one NVIDIA GB300 GPU (sm_103a).
 *
 * Sources (web pages):
 *   [RFC-0025] "RFC-0025: 支持 Attention Varlen 功能并对齐 Loss"
 *   [RFC-0026] "RFC-0026: Ling3 KDA Varlen 支持（packing 文档间隔离）"
 *   [Drill]    "Drill: Sequence Packing from scratch"
 *
 * Conventions shared by every call
 *   - Tensor pointers are DEVICE pointers owned by the caller, dense
 *     (contiguous, row-major) and aligned to 16 bytes. The library never
 *     frees or retains them.
 *   - A call validates its arguments on the host, enqueues its kernels on
 *     `stream` (NULL: the legacy default stream) and returns without
 *     synchronising. The return value reports argument errors and launch
 *     errors only; conditions found on the device are written to device
 *     words the caller reads after its own synchronisation.
 *   - The library allocates no memory. Scratch space is passed in by the
 *     caller (see kda_chunk_fwd_varlen_workspace_size).
 *   - Segment ids are int32 [B, T]: documents carry non-zero ids, 0 marks
 *     padding. A segment starts where a non-zero id differs from the
 *     previous token's id, and at t = 0 of every row ([RFC-0026] §3.1.1
 *     "边界 reset 语义"). The batch is flattened to [1, B*T] ([RFC-0025]
 *     方案 §2), so tensors indexed by token use the flat index p = b*T + t.
 *   - Sizes: B*T < 2^31.
 *   - Every call can be captured in a CUDA graph: it makes no host round trip,
 *     allocates nothing and launches only on `stream`. Make one call of each
 *     entry point (per kernel variant) on a device before capturing there,
 *     since the first call on each device sets kernel attributes.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; NULL selects the legacy default stream. */
typedef struct CUstream_st *kda_stream_t;

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = -1, /* null/misaligned pointer, negative or inconsistent size */
    KDA_ERR_UNSUPPORTED = -2, /* valid request outside the shapes this build supports   */
    KDA_ERR_CUDA = -3,        /* a CUDA runtime call or a kernel launch failed          */
    KDA_ERR_WORKSPACE = -4    /* workspace missing or smaller than required             */
} kda_status_t;

typedef enum {
    KDA_F32 = 0, /* IEEE float32 */
    KDA_BF16 = 1 /* bfloat16     */
} kda_dtype_t;

/* Bits that kda_chunk_fwd_varlen ORs into *status_dev. */
#define KDA_DEV_DECAY_RANGE 0x1u /* a 16-token block's cumulative log-decay left the
                                    range the chunked factorisation handles (see below) */
#define KDA_DEV_TIMEOUT 0x2u     /* a bounded in-kernel wait (TMA or tensor-core
                                    completion) gave up; outputs are incomplete */

/*
 * kda_segids_to_cu_seqlens -- [RFC-0025] 方案 §1 "segment_ids → cu_seqlens 转换".
 *
 * Turns segment ids into cumulative sequence lengths in the FLA convention,
 * padded to a fixed length: cu_seqlens[0] = 0 and cu_seqlens[i] = end of the
 * i-th segment of the flattened [B*T] sequence, where a segment ends where
 * the next one starts ([Drill] 数学: cu[i] = l_1 + ... + l_i). The last real
 * segment ends one past the last non-padding token; entries past the real
 * segment count ("phantom" segments) repeat that end, i.e. have zero length.
 * If the real count exceeds max_segs, cu_seqlens[max_segs] = B*T and the
 * extra segments merge into the last slot, as on the page; *n_segs_out then
 * exceeds max_segs, which the caller should treat as an error.
 *
 *   segment_ids  device int32 [B, T], 4-byte aligned.
 *   B, T         B >= 1, T >= 1.
 *   max_segs     >= 1.
 *   cu_seqlens   device int32 [max_segs + 1], written entirely.
 *   n_segs_out   device int32 scalar or NULL: number of real segments.
 *
 * Returns KDA_OK, KDA_ERR_INVALID_ARG or KDA_ERR_CUDA. One kernel launch.
 */
kda_status_t kda_segids_to_cu_seqlens(const int32_t *segment_ids, int64_t B, int64_t T,
                                      int32_t max_segs, int32_t *cu_seqlens,
                                      int32_t *n_segs_out, kda_stream_t stream);

/*
 * kda_short_conv_varlen -- [RFC-0025] 方案 §3 "ShortConvolution segment 边界 mask".
 *
 * Causal depthwise convolution of width k_conv over time, per row:
 *     y[b,t,f] = sum_{j=0}^{k_conv-1} w[j,f] * x[b,t-j,f]
 * where a tap contributes only if t-j >= 0 and segment_ids[b,t-j] ==
 * segment_ids[b,t] (taps that cross a document boundary are zeroed; tap 0
 * weighs the current token). With segment_ids == NULL only t-j >= 0 is
 * required. Products are summed in fp32 and rounded once to `dtype`.
 *
 *   x, y         device [B, T, F] of `dtype`; y must not overlap x.
 *   weight       device [k_conv, F] of `dtype`.
 *   segment_ids  device int32 [B, T] or NULL.
 *   F            >= 1; F * sizeof(dtype) must be a multiple of 16.
 *   k_conv       1..8.
 *
 * Returns KDA_OK, KDA_ERR_INVALID_ARG, KDA_ERR_UNSUPPORTED or KDA_ERR_CUDA.
 */
kda_status_t kda_short_conv_varlen(const void *x, const void *weight,
                                   const int32_t *segment_ids, void *y, int64_t B, int64_t T,
                                   int64_t F, int32_t k_conv, kda_dtype_t dtype,
                                   kda_stream_t stream);

/*
 * kda_chunk_fwd_varlen_workspace_size -- bytes of device scratch that
 * kda_chunk_fwd_varlen uses for these sizes (0 on invalid sizes): the minimum
 * below, plus, for bf16 with 128-wide heads, room for the states that let it
 * split long segments (one 64 KB state per head per 64 chunks; see
 * kda_chunk_fwd_varlen).
 *
 * kda_chunk_fwd_varlen_workspace_min -- the least scratch the forward entry
 * points accept. With less than the full size they split fewer long segments,
 * or none; the results are the same to rounding.
 */
size_t kda_chunk_fwd_varlen_workspace_size(int64_t B, int64_t T, int32_t H, int32_t d_qk,
                                           int32_t d_v, kda_dtype_t dtype);
size_t kda_chunk_fwd_varlen_workspace_min(int64_t B, int64_t T, int32_t H, int32_t d_qk,
                                          int32_t d_v, kda_dtype_t dtype);

/*
 * kda_chunk_fwd_varlen -- the KDA recurrence over packed sequences,
 * [RFC-0026] 背景 "KDA 状态泄漏问题" and §3.1.1:
 *     S'_t = S_{t-1} * exp(g_t)          (g_t in R^{d_qk} scales the key rows)
 *     S_t  = S'_t + beta_t * k_t v_t^T   (S in R^{d_qk x d_v}, fp32)
 *     o_t  = scale * S_t^T q_t
 * with S = 0 at every segment start. Padding tokens contribute nothing and
 * their output is 0. segment_ids == NULL makes every row one segment.
 *
 * Layout: the flattened [1, B*T, H, D] view ([RFC-0025] 方案 §2):
 *   q, k, g      device [B*T, H, d_qk] of `dtype` (g is the log-decay, <= 0)
 *   v            device [B*T, H, d_v]  of `dtype`
 *   beta         device [B*T, H]       of `dtype`
 *   o            device [B*T, H, d_v]  of `out_dtype` (KDA_F32, or equal to
 *                `dtype`); values are rounded once, to nearest even, from fp32
 *   segment_ids  device int32 [B, T] or NULL
 *
 * dtype KDA_BF16 runs the chunked form (64-token chunks, tensor cores,
 * fp32 accumulation and fp32 state); KDA_F32 runs the token recurrence in
 * fp32 arithmetic. Supported: d_qk == d_v in {64, 128}; H >= 1.
 *
 * The chunked form factors the in-chunk decay into per-token scalings
 * exp(G_i - G_ref) and exp(G_ref - G_j), G the cumulative log-decay in the
 * chunk and G_ref its value at the chunk's end. Where some channel's log-decay
 * over a chunk falls below -80 (for instance g < -1.25 on every token) those
 * factors would leave fp32's range; such chunks are computed again with a
 * reference point at the end of each 16-token block instead, which holds
 * while every channel's log-decay over each 16-token block stays above -80
 * (a per-token average above -5). Past that the kernel sets
 * KDA_DEV_DECAY_RANGE in *status_dev and the affected outputs are
 * unreliable. (fp32 inputs and 64-wide heads run the token recurrence, which
 * has no such limit.)
 *
 * Long segments: the state is serial along a segment, so one long document
 * would keep a single multiprocessor busy while the others finish. When the
 * workspace has room, a segment longer than one multiprocessor's share of the
 * work (chunks x heads / multiprocessors) by more than 32 chunks is cut into
 * pieces. A state-only pass computes, in parallel, each leading piece's end
 * state from a zero start, and hands each piece's start state to the next one
 * along the segment; the forward then runs every piece from its start state.
 *
 *   workspace        device scratch of at least
 *                    kda_chunk_fwd_varlen_workspace_min(...) bytes, and best
 *                    kda_chunk_fwd_varlen_workspace_size(...), 256-byte
 *                    aligned; its contents on entry do not matter.
 *   workspace_bytes  its size, which bounds how many segments are split.
 *   status_dev       device uint32 or NULL; bits are ORed in, never cleared.
 *
 * Returns KDA_OK, KDA_ERR_INVALID_ARG, KDA_ERR_UNSUPPORTED, KDA_ERR_WORKSPACE
 * or KDA_ERR_CUDA. Calls that share a workspace must not overlap in time.
 */
kda_status_t kda_chunk_fwd_varlen(const void *q, const void *k, const void *v, const void *g,
                                  const void *beta, const int32_t *segment_ids, int64_t B,
                                  int64_t T, int32_t H, int32_t d_qk, int32_t d_v, float scale,
                                  kda_dtype_t dtype, kda_dtype_t out_dtype, void *o, void *workspace,
                                  size_t workspace_bytes, uint32_t *status_dev,
                                  kda_stream_t stream);

/*
 * kda_chunk_plan_varlen / kda_chunk_fwd_varlen_planned -- kda_chunk_fwd_varlen
 * in two calls. The plan (where segments start in each 64-token chunk, and the
 * chunk ranges that the kernel's CTAs take in turn) depends only on
 * segment_ids and the sizes. So a caller may compute it on another stream
 * while the kernels that produce q, k, v and g run, and join before the
 * forward. kda_chunk_plan_varlen(segment_ids, B, T, H, d_qk, d_v, dtype, ws)
 * followed by kda_chunk_fwd_varlen_planned(..., ws, ...) with the same
 * segment_ids contents and sizes gives kda_chunk_fwd_varlen's result bit for
 * bit.
 *
 *   kda_chunk_plan_varlen    writes the plan into `workspace` (the forward's
 *                            workspace: same size rule, alignment and
 *                            argument checks). It reads segment_ids only.
 *   kda_chunk_fwd_varlen_planned
 *                            takes kda_chunk_fwd_varlen's arguments. Its
 *                            workspace must hold a plan of the same
 *                            segment_ids contents, B, T, H, d_qk, d_v and
 *                            dtype, and the same workspace_bytes (which
 *                            fix how long segments are split), complete or
 *                            ordered before the call (same stream, or an
 *                            event). A plan serves any number of planned
 *                            calls, one at a time, until another call
 *                            writes the workspace.
 *
 * Paths that plan inside the forward (dtype KDA_F32, or 64-wide heads) have
 * nothing to plan ahead: kda_chunk_plan_varlen only checks its arguments and
 * the planned call plans for itself. A planned call on a workspace without a
 * matching plan is undefined (wrong or missing outputs). Returns as
 * kda_chunk_fwd_varlen.
 */
kda_status_t kda_chunk_plan_varlen(const int32_t *segment_ids, int64_t B, int64_t T, int32_t H,
                                   int32_t d_qk, int32_t d_v, kda_dtype_t dtype, void *workspace,
                                   size_t workspace_bytes, kda_stream_t stream);

kda_status_t kda_chunk_fwd_varlen_planned(const void *q, const void *k, const void *v,
                                          const void *g, const void *beta,
                                          const int32_t *segment_ids, int64_t B, int64_t T,
                                          int32_t H, int32_t d_qk, int32_t d_v, float scale,
                                          kda_dtype_t dtype, kda_dtype_t out_dtype, void *o,
                                          void *workspace, size_t workspace_bytes,
                                          uint32_t *status_dev, kda_stream_t stream);

/*
 * kda_chunk_fwd_varlen_conv -- kda_chunk_fwd_varlen with the three
 * segment-masked short convolutions that produce q, k and v ([RFC-0025] 方案 §3
 * "ShortConvolution segment 边界 mask") done inside the chunk kernel: the
 * prologue fusion that [RFC-0026] §3.3's kernel wrapper implies. The result is
 *     q = conv(x_q, w_q), k = conv(x_k, w_k), v = conv(x_v, w_v)   (each as
 *     kda_short_conv_varlen with these segment_ids, rounded to dtype)
 *     o = kda_chunk_fwd_varlen(q, k, v, g, beta, ...)
 * equal to those four calls bit for bit, but q, k and v are never written to
 * device memory: the kernel reads x_q, x_k and x_v (plus the k_conv - 1 tokens
 * before each 64-token chunk) and convolves them in shared memory. No L2
 * normalisation of q and k is applied (the pages give no epsilon for it).
 *
 *   x_q, x_k, x_v  device [B*T, H*d_qk] of `dtype` (the convs' inputs, laid out
 *                  like q, k, v); none may overlap o.
 *   w_q, w_k, w_v  device [k_conv, H*d_qk] of `dtype`, 16-byte aligned: tap j
 *                  weighs the token j steps back, as in kda_short_conv_varlen.
 *   k_conv         1..4.
 *   planned        0: plan inside the call, as kda_chunk_fwd_varlen; 1: the
 *                  workspace holds the plan of kda_chunk_plan_varlen, under the
 *                  rules of kda_chunk_fwd_varlen_planned.
 *
 * The other arguments are kda_chunk_fwd_varlen's, with the same workspace
 * sizes (long segments are split the same way). Supported: dtype KDA_BF16 with
 * d_qk == d_v == 128; other dtypes, widths or k_conv return
 * KDA_ERR_UNSUPPORTED (run the convs, then kda_chunk_fwd_varlen). Returns as
 * kda_chunk_fwd_varlen. Calls that share a workspace must not overlap in time.
 */
kda_status_t kda_chunk_fwd_varlen_conv(const void *x_q, const void *x_k, const void *x_v,
                                       const void *w_q, const void *w_k, const void *w_v,
                                       int32_t k_conv, const void *g, const void *beta,
                                       const int32_t *segment_ids, int64_t B, int64_t T,
                                       int32_t H, int32_t d_qk, int32_t d_v, float scale,
                                       kda_dtype_t dtype, kda_dtype_t out_dtype, void *o,
                                       void *workspace, size_t workspace_bytes, int planned,
                                       uint32_t *status_dev, kda_stream_t stream);

/*
 * kda_delta_fwd_varlen -- the delta-rule form of the recurrence. [RFC-0026]
 * names the method Kimi Delta Attention but its pages state only the additive
 * update of kda_chunk_fwd_varlen; this is the reading of that name, the gated
 * delta rule with a decay per key channel:
 *     S'_t = S_{t-1} * exp(g_t)                      (key rows)
 *     S_t  = S'_t + beta_t * k_t (v_t - S'_t^T k_t)^T  = (I - beta_t k_t k_t^T) S'_t
 *                                                      + beta_t k_t v_t^T
 *     o_t  = scale * S_t^T q_t
 * with S = 0 at every segment start and padding outputs 0, as in
 * kda_chunk_fwd_varlen. It runs the token recurrence in fp32 arithmetic (one
 * walk per segment and head; each token's S'^T k is a reduction over the
 * walk's threads), for either dtype; there is no chunked (tensor-core) form of
 * it here. The arguments, layouts, workspace sizes and return codes are
 * kda_chunk_fwd_varlen's; d_qk == d_v in {64, 128}.
 */
kda_status_t kda_delta_fwd_varlen(const void *q, const void *k, const void *v, const void *g,
                                  const void *beta, const int32_t *segment_ids, int64_t B,
                                  int64_t T, int32_t H, int32_t d_qk, int32_t d_v, float scale,
                                  kda_dtype_t dtype, kda_dtype_t out_dtype, void *o,
                                  void *workspace, size_t workspace_bytes, uint32_t *status_dev,
                                  kda_stream_t stream);

/*
 * kda_chunk_fwd_varlen_state -- kda_chunk_fwd_varlen with per-segment recurrent
 * state in and out: the initial_state and output_final_state kwargs that
 * [RFC-0026] passes to the chunked KDA call, one state per packed sequence.
 *
 * Segment r is the r-th segment of the flattened [B*T] sequence in token order
 * (the r-th entry of cu_seqlens; rows first, padding is no segment, and with
 * segment_ids == NULL segment r is row r). For r < n_state:
 *   initial_state  device fp32 [n_state, H, d_qk, d_v] or NULL: segment r starts
 *                  from initial_state[r] instead of 0 (rows are key channels:
 *                  S[i][j], i < d_qk, j < d_v);
 *   final_state    device fp32 [n_state, H, d_qk, d_v] or NULL: receives segment
 *                  r's state after its last token. Slots r >= the segment count
 *                  are left untouched.
 * Segments r >= n_state start from 0 and are not written out. Both arrays are
 * owned by the caller, 16-byte aligned, and must not overlap.
 *
 * The other arguments are those of kda_chunk_fwd_varlen, with the same
 * workspace size. dtype KDA_BF16 with d_qk == 128 runs the tensor-core
 * chunked form. It seeds each segment's state at the chunk where the segment
 * starts and keeps the state carried into the chunk where it ends (in
 * final_state). A second pass then works chunk by chunk in fp32. It writes
 * the outputs of each segment's rows in its first chunk, whose read-out of
 * the initial state the chunked form leaves out, and it forms the final
 * states. Outputs meet the bf16 bound of kda_chunk_fwd_varlen for either
 * out_dtype. Other dtypes and widths run the token recurrence in fp32
 * arithmetic, one walk per segment and head.
 *
 * Returns KDA_OK, KDA_ERR_INVALID_ARG, KDA_ERR_UNSUPPORTED, KDA_ERR_WORKSPACE or
 * KDA_ERR_CUDA. Calls that share a workspace must not overlap in time.
 */
kda_status_t kda_chunk_fwd_varlen_state(const void *q, const void *k, const void *v,
                                        const void *g, const void *beta,
                                        const int32_t *segment_ids, int64_t B, int64_t T,
                                        int32_t H, int32_t d_qk, int32_t d_v, float scale,
                                        kda_dtype_t dtype, kda_dtype_t out_dtype, void *o,
                                        const float *initial_state, float *final_state,
                                        int64_t n_state, void *workspace, size_t workspace_bytes,
                                        uint32_t *status_dev, kda_stream_t stream);

/*
 * kda_chunk_bwd_varlen_workspace_size -- bytes of device scratch that
 * kda_chunk_bwd_varlen and kda_chunk_bwd_varlen_ex need, with either method (0 on
 * invalid or unsupported sizes). The fp32 walks keep the segment list, dq in
 * fp32 and one fp32 state per 64-token chunk and head, about
 * (B*T) * H * (4 d_qk + 4 d_qk d_v / 64) bytes; the tensor-core path keeps two
 * fp32 states per chunk and head (the state entering the chunk and the adjoint
 * at its end), about (B*T) * H * 8 d_qk d_v / 64 bytes. The size is the larger.
 */
size_t kda_chunk_bwd_varlen_workspace_size(int64_t B, int64_t T, int32_t H, int32_t d_qk,
                                           int32_t d_v, kda_dtype_t dtype);

/*
 * kda_chunk_bwd_varlen -- gradients of kda_chunk_fwd_varlen (no per-segment
 * state) with respect to q, k, v, g and beta, for an upstream gradient d_o of o.
 * The pages state the forward only; these are its derivatives:
 *     A_t     = dL/dS_t = scale q_t d_o_t^T + exp(g_{t+1}) * A_{t+1}
 *               (rows scaled; zero past a segment's last token)
 *     dq_t    = scale S_t d_o_t
 *     dk_t    = beta_t A_t v_t      dv_t = beta_t A_t^T k_t
 *     dbeta_t = k_t^T A_t v_t
 *     dg_t    = sum over the segment's tokens u >= t of (q_u * dq_u - k_u * dk_u)
 * Padding tokens get zero gradients. The running sum for dg restarts at every
 * 64-token chunk start from its direct form exp(g_t) * sum_j A_t[i][j] S_{t-1}[i][j]
 * (the sum cancels, so its rounding error would otherwise grow with the segment).
 *
 * Layout and arguments are those of kda_chunk_fwd_varlen, with the workspace size
 * from kda_chunk_bwd_varlen_workspace_size, plus:
 *   d_o          device [B*T, H, d_v] of `dtype`
 *   dq, dk, dg   device [B*T, H, d_qk] of `grad_dtype`
 *   dv           device [B*T, H, d_v] of `grad_dtype`
 *   dbeta        device [B*T, H] of `grad_dtype`
 *   grad_dtype   KDA_F32, or equal to `dtype`; values rounded once to nearest even
 * It is kda_chunk_bwd_varlen_ex with method KDA_BWD_AUTO and no status word.
 *
 * Returns KDA_OK, KDA_ERR_INVALID_ARG, KDA_ERR_UNSUPPORTED, KDA_ERR_WORKSPACE or
 * KDA_ERR_CUDA. Calls that share a workspace must not overlap in time.
 */
kda_status_t kda_chunk_bwd_varlen(const void *q, const void *k, const void *v, const void *g,
                                  const void *beta, const int32_t *segment_ids, int64_t B,
                                  int64_t T, int32_t H, int32_t d_qk, int32_t d_v, float scale,
                                  kda_dtype_t dtype, const void *d_o, kda_dtype_t grad_dtype,
                                  void *dq, void *dk, void *dv, void *dg, void *dbeta,
                                  void *workspace, size_t workspace_bytes, kda_stream_t stream);

/* Methods of kda_chunk_bwd_varlen_ex. */
#define KDA_BWD_AUTO 0 /* tensor cores for bf16 inputs with d_qk = d_v = 128, else the walks */
#define KDA_BWD_WALK 1 /* the fp32 walks, for every supported shape and dtype */

/*
 * kda_chunk_bwd_varlen_ex -- kda_chunk_bwd_varlen with a choice of method and a
 * device status word. Arguments and results are kda_chunk_bwd_varlen's, plus:
 *   method       KDA_BWD_AUTO or KDA_BWD_WALK (anything else: KDA_ERR_INVALID_ARG)
 *   status_dev   device uint32, nullable: KDA_DEV_* bits are ORed into it, as in
 *                kda_chunk_fwd_varlen
 *
 * KDA_BWD_WALK runs in fp32 arithmetic as two walks per (segment, head): forward
 * for dq and the chunk-start states, then backward for the rest, which reads
 * them back. Its gradients hold the fp32 bound (1e-4 RMS per head).
 *
 * KDA_BWD_AUTO, for bf16 inputs with d_qk = d_v = 128, runs the chunked form on
 * tcgen05 tensor cores in three launches: a forward scan over the chunks that
 * one segment links stores the state entering every chunk; a backward scan
 * stores the adjoint at every chunk's end; then, per (chunk, head) and with no
 * dependence between them, eight tensor-core products give dq, dk, dv, and the
 * epilogue dg and dbeta (dg from its sum within the chunk plus the direct form
 * past it). Operands are bf16 (decayed ones as hi + lo pairs), accumulation
 * fp32, as in the forward kernel, so the gradients hold the bf16 bound of the
 * forward's output (2e-2 RMS per head). A (chunk, head) whose log-decay on some
 * key channel falls below -80 is outside the factorised products' range: a last
 * launch recomputes its gradients by an fp32 token walk over the chunk, from the
 * stored state and adjoint. Other inputs take the walks.
 */
kda_status_t kda_chunk_bwd_varlen_ex(const void *q, const void *k, const void *v, const void *g,
                                     const void *beta, const int32_t *segment_ids, int64_t B,
                                     int64_t T, int32_t H, int32_t d_qk, int32_t d_v, float scale,
                                     kda_dtype_t dtype, const void *d_o, kda_dtype_t grad_dtype,
                                     void *dq, void *dk, void *dv, void *dg, void *dbeta,
                                     void *workspace, size_t workspace_bytes, int32_t method,
                                     uint32_t *status_dev, kda_stream_t stream);

/*
 * kda_chunk_fwd_varlen_noalloc -- kda_chunk_fwd_varlen for callers that cannot
 * allocate device memory. The pages have no counterpart: this is a calling
 * convention of this library, not part of the method.
 *
 * Some callers hold no device allocator: a plain C host program that only
 * receives device buffers from another runtime, or a serving loop whose memory
 * pool owns all free device memory and forbids further cudaMalloc/cudaFree on
 * its hot path (those calls can also synchronise the device). They cannot hand
 * kda_chunk_fwd_varlen a workspace, so this entry point takes its scratch from
 * an array compiled into the library instead: KDA_NOALLOC_SCRATCH_BYTES bytes of
 * device memory that every GPU loading the library holds until the process
 * exits. It allocates nothing and calls no allocating routine.
 *
 * Arguments, layouts and results are those of kda_chunk_fwd_varlen without the
 * workspace pair, and the arguments are checked in the same order, so a null
 * or misaligned tensor returns KDA_ERR_INVALID_ARG whatever the size. Then
 * problems whose kda_chunk_fwd_varlen_workspace_size exceeds
 * KDA_NOALLOC_SCRATCH_BYTES are refused with KDA_ERR_WORKSPACE before anything
 * is launched (the 4 MiB array covers up to 524,256 tokens, B*T, for either
 * dtype).
 *
 * The first call on a device looks up the array's device address on that
 * device (with it current) and caches it; make that first call before any
 * stream capture. A lookup that fails returns KDA_ERR_CUDA and is not cached:
 * the next call on that device tries again. Every call shares the one array
 * and leaves its contents behind; the kernels write every scratch word before
 * they read it, so stale contents do not matter, but calls whose kernels
 * overlap on the GPU race on the array: issue them on one stream, or order
 * them.
 */
#define KDA_NOALLOC_SCRATCH_BYTES (4u << 20)

kda_status_t kda_chunk_fwd_varlen_noalloc(const void *q, const void *k, const void *v,
                                          const void *g, const void *beta,
                                          const int32_t *segment_ids, int64_t B, int64_t T,
                                          int32_t H, int32_t d_qk, int32_t d_v, float scale,
                                          kda_dtype_t dtype, kda_dtype_t out_dtype, void *o,
                                          uint32_t *status_dev, kda_stream_t stream);

/*
 * kda_selftest_wait_timeout -- a check of the failure detection behind
 * KDA_DEV_TIMEOUT; not part of the method. The chunk kernels bound every
 * in-kernel wait by wall time, after which they set KDA_DEV_TIMEOUT and return
 * with the context intact. This call launches one small kernel that waits,
 * through the same bounded wait, on a barrier that nothing arrives on, for about
 * timeout_ns nanoseconds of GPU time, then ORs KDA_DEV_TIMEOUT into *status_dev
 * and returns. Synchronise, then read the word.
 *
 *   timeout_ns   1e6 .. 1e10 (1 ms .. 10 s).
 *   status_dev   device uint32, 4-byte aligned.
 *
 * Returns KDA_OK, KDA_ERR_INVALID_ARG or KDA_ERR_CUDA.
 */
kda_status_t kda_selftest_wait_timeout(uint64_t timeout_ns, uint32_t *status_dev,
                                       kda_stream_t stream);

/* Static, human-readable name of a status code. */
const char *kda_status_string(kda_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
