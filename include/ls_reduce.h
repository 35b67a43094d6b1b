/*
 * ls_reduce.h -- C ABI of libls_reduce.so: fused softmax and LayerNorm reduce
 * kernels of a Transformer layer (forward and backward) for NVIDIA GB300
 * (sm_103a).
 *
 * The operations are the LightSeq-style reduce kernels described on the pages
 *   "CMU 11-868 L10: Accelerating Transformers on GPUs, and Where LightSeq
 *    Finds the Time", section "Technique 2: rewrite the formula, drop a
 *    synchronization" (slides 21-26), and
 *   "CMU 11-868 HW4：把 Softmax 與 LayerNorm 寫成 CUDA 融合 kernel",
 *    section 題目結構與配分 (Problems 1.1, 1.2, 2.1, 2.2).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Pointers named as device buffers must be CUDA device (or managed) memory
 *    owned by the caller.  The library never allocates, frees or
 *    synchronises; it only enqueues kernels on `stream`.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream).  All work is asynchronous with respect to the host.
 *  - Tensors are dense, row-major, with the last dimension contiguous.
 *  - Storage dtype `dt` applies to every `void*` tensor of a call (scores,
 *    mask, gamma, beta, activations and their gradients).  Arithmetic is FP32
 *    for every storage dtype; 16-bit outputs are rounded to nearest-even.
 *    LayerNorm statistics (mean, rstd) and the gamma/beta gradients are
 *    always FP32.
 *  - Pointers must be aligned to their element size.  Buffers that are also
 *    16-byte aligned, with a row length in bytes that is a multiple of 16,
 *    take the 128-bit vector path; all others take a scalar path of the same
 *    kernel family (same results, lower bandwidth).  There is no CPU path.
 *  - A zero-sized problem (no rows, or an empty row for softmax) is a valid
 *    no-op, except where stated.  Negative sizes, NULL required pointers,
 *    unsupported dtypes and inconsistent shapes are rejected on the host
 *    before anything is launched; nothing is written in that case.
 *  - Return value: LS_OK once the kernels are enqueued.  A launch failure
 *    reported by the CUDA runtime is LS_ERR_CUDA.  Faults that happen while
 *    the kernels run surface at the caller's next synchronisation, as for any
 *    CUDA work.
 */
#ifndef LS_REDUCE_H
#define LS_REDUCE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum ls_dtype {
    LS_F32 = 0,  /* IEEE binary32 */
    LS_F16 = 1,  /* IEEE binary16 */
    LS_BF16 = 2  /* bfloat16 */
} ls_dtype;

typedef enum ls_status {
    LS_OK = 0,
    LS_ERR_INVALID_ARG = 1,  /* NULL pointer, negative size, inconsistent shape */
    LS_ERR_UNSUPPORTED = 2,  /* unknown dtype, or a size beyond the limits below */
    LS_ERR_MISALIGNED = 3,   /* pointer not aligned to its element size */
    LS_ERR_WORKSPACE = 4,    /* workspace missing or smaller than required */
    LS_ERR_CUDA = 5          /* the CUDA runtime rejected a launch */
} ls_status;

/* Largest row length (Tk for softmax, hidden for LayerNorm) accepted. */
#define LS_MAX_ROW_LENGTH ((int64_t)1 << 30)

/*
 * Attention softmax forward ("Problem 1.1" of the HW4 page; slides 23-26 of
 * the L10 page).  For every row (b, h, i) of the score tensor:
 *     z_j = -inf                       if causal and j > i + (Tk - Tq)  (future key)
 *     z_j = inp[b,h,i,j] + mask[b,j]   otherwise
 *     out[b,h,i,j] = exp(z_j - max_k z_k) / sum_k exp(z_k - max_k z_k)
 * A row whose every key is -inf is written as zeros.
 *
 *   out   [B,H,Tq,Tk] dt, device, written.  May equal `inp` (in place).
 *   inp   [B,H,Tq,Tk] dt, device, read.  Scores are expected to be finite.
 *   mask  [B,Tk] dt additive mask (0 = keep, -inf = padded key), device,
 *         read; NULL means no mask.  Shared by all heads and queries of a
 *         batch entry.  Keys whose mask is -inf are not read from `inp`.
 *   causal  nonzero: mask future keys.  Requires Tq <= Tk; the Tq queries are
 *           the last Tq positions of the key sequence (bottom-right
 *           alignment), so query i sees keys j <= i + (Tk - Tq); with
 *           Tq == Tk that is j <= i.
 * Errors: LS_ERR_INVALID_ARG for NULL out/inp with a non-empty problem,
 * negative sizes, or causal with Tq > Tk; LS_ERR_UNSUPPORTED for Tk beyond
 * LS_MAX_ROW_LENGTH or an unknown dtype.
 */
ls_status ls_softmax_fw(void *out, const void *inp, const void *mask,
                        int64_t B, int64_t H, int64_t Tq, int64_t Tk,
                        int causal, ls_dtype dt, void *stream);

/*
 * Attention softmax backward ("Problem 1.2" of the HW4 page).  For every
 * row:  dinp_j = out_j * (dout_j - sum_k out_k * dout_k),
 * the vector-Jacobian product of the forward softmax at its output `out_fw`.
 * Masked and future keys need no mask argument: their forward output is 0.
 *
 *   dinp    [B,H,Tq,Tk] dt, device, written.  May equal `dout`.
 *   dout    [B,H,Tq,Tk] dt, device, read (gradient of the softmax output).
 *   out_fw  [B,H,Tq,Tk] dt, device, read (the forward output).
 * Errors as for ls_softmax_fw (no causal/mask arguments here).
 */
ls_status ls_softmax_bw(void *dinp, const void *dout, const void *out_fw,
                        int64_t B, int64_t H, int64_t Tq, int64_t Tk,
                        ls_dtype dt, void *stream);

/*
 * Attention softmax backward that skips invisible keys: the same result as
 * ls_softmax_bw when `out_fw` is the forward output (0 on masked and future
 * keys), but keys that are masked (mask == -inf) or in the causal future are
 * neither read from `dout` / `out_fw` nor summed; their gradient is written
 * as 0.  Per row:
 *     s      = sum over visible k of out_k * dout_k
 *     dinp_j = out_j * (dout_j - s)   on visible keys, 0 elsewhere
 * It is the backward counterpart of ls_softmax_fw's read skipping (the L10
 * page's slide 30 names the score gradient as the O(T^2) tensor of the
 * attention backward).
 *
 *   dinp    [B,H,Tq,Tk] dt, device, written.  May equal `dout`.
 *   dout, out_fw  [B,H,Tq,Tk] dt, device, read on visible keys only.
 *   mask    [B,Tk] dt additive mask or NULL, as for ls_softmax_fw.
 *   causal  as for ls_softmax_fw (Tq <= Tk, bottom-right alignment).
 * Errors as for ls_softmax_fw.
 */
ls_status ls_softmax_bw_masked(void *dinp, const void *dout, const void *out_fw,
                               const void *mask, int64_t B, int64_t H, int64_t Tq,
                               int64_t Tk, int causal, ls_dtype dt, void *stream);

/*
 * Scaled softmax, forward: the fused "scale + mask + softmax" of an attention
 * layer (the L10 page, section "Technique 1", fuses the operations between
 * the GEMMs into custom kernels; the score scale is one of them).  As
 * ls_softmax_fw, with the scores multiplied by `scale` (e.g. 1/sqrt(head
 * dimension)) before the additive mask:
 *     z_j = scale * x_j + mask[b, j]   (-inf for causal future keys)
 *     y   = softmax(z)
 * The scale is folded into the exponent (no extra pass, no extra arithmetic
 * on unmasked chunks).  scale must be finite and > 0, else
 * LS_ERR_INVALID_ARG.  Other arguments and errors as for ls_softmax_fw;
 * ls_softmax_fw is this function with scale = 1 (bitwise).
 */
ls_status ls_softmax_fw_scaled(void *out, const void *inp, const void *mask, int64_t B,
                               int64_t H, int64_t Tq, int64_t Tk, int causal, float scale,
                               ls_dtype dt, void *stream);

/*
 * Scaled softmax, backward over the visible keys: the gradient of the scores
 * of ls_softmax_fw_scaled,
 *     dinp_j = scale * y_j * (dout_j - sum over visible k of y_k dout_k)
 * on visible keys and 0 on the others (as ls_softmax_bw_masked, which is this
 * function with scale = 1, bitwise).  scale must be finite and > 0.
 */
ls_status ls_softmax_bw_masked_scaled(void *dinp, const void *dout, const void *out_fw,
                                      const void *mask, int64_t B, int64_t H, int64_t Tq,
                                      int64_t Tk, int causal, float scale, ls_dtype dt,
                                      void *stream);

/*
 * LayerNorm forward ("Problem 2.1" of the HW4 page; slide 21 of the L10
 * page).  For every row of x [rows, hidden], the mean and variance come from
 * ONE fused reduction of the two sums sum(x') and sum(x'^2), x' = x - x_0
 * (x_0 the row's first element; the variance is shift-invariant and the
 * shift keeps the one-pass form exact for constant rows):
 *     mu   = x_0 + mean(x'),   var = max(mean(x'^2) - mean(x')^2, 0)
 *     rstd = 1 / sqrt(var + eps)
 *     y_j  = (x_j - mu) * rstd * gamma_j + beta_j
 *
 *   y      [rows, hidden] dt, device, written.
 *   mean   [rows] float32, device, written (the saved mu).
 *   rstd   [rows] float32, device, written (the saved 1/sqrt(var + eps)).
 *   x      [rows, hidden] dt, device, read.
 *   gamma, beta  [hidden] dt, device, read.
 *   eps    added to the variance inside the square root (the pages use 1e-8).
 * Errors: LS_ERR_INVALID_ARG for NULL pointers with rows > 0, negative rows,
 * hidden < 1, or eps < 0 / not finite; LS_ERR_UNSUPPORTED for hidden beyond
 * LS_MAX_ROW_LENGTH or an unknown dtype.
 */
ls_status ls_layernorm_fw(void *y, float *mean, float *rstd, const void *x,
                          const void *gamma, const void *beta, int64_t rows,
                          int64_t hidden, float eps, ls_dtype dt, void *stream);

/*
 * LayerNorm backward, input gradient ("Problem 2.2" of the HW4 page; slide
 * 22 of the L10 page: two sums computed in parallel, then elementwise work).
 * With xhat = (x - mean) * rstd and g = gamma * dy, per row:
 *     S1 = sum_j g_j,   S2 = sum_j g_j * xhat_j      (one fused reduction)
 *     dx_j = rstd * (g_j - S1 / hidden - xhat_j * S2 / hidden)
 *
 *   dx     [rows, hidden] dt, device, written.  May equal `dy`.
 *   dy     [rows, hidden] dt, device, read (gradient of y).
 *   x      [rows, hidden] dt, device, read (the forward input).
 *   gamma  [hidden] dt, device, read.
 *   mean, rstd  [rows] float32, device, read (as saved by ls_layernorm_fw).
 * Errors as for ls_layernorm_fw.
 */
ls_status ls_layernorm_bw_dinp(void *dx, const void *dy, const void *x,
                               const void *gamma, const float *mean,
                               const float *rstd, int64_t rows, int64_t hidden,
                               ls_dtype dt, void *stream);

/*
 * Bytes of device workspace ls_layernorm_bw_dgamma_dbeta needs for a
 * [rows, hidden] problem (the same for every dtype).  Returns 0 for
 * rows <= 0 or hidden <= 0.  Host-only; launches nothing.
 */
size_t ls_layernorm_bw_dgamma_dbeta_workspace_size(int64_t rows, int64_t hidden);

/*
 * LayerNorm backward, gamma and beta gradients ("Problem 2.2" of the HW4
 * page: the cross-row kernel).  Column sums over all rows:
 *     dgamma_j = sum_r dy_rj * (x_rj - mean_r) * rstd_r
 *     dbeta_j  = sum_r dy_rj
 * computed in a fixed order that depends only on (rows, hidden): the result
 * is bitwise reproducible from run to run and GPU to GPU.  With rows == 0 the
 * outputs are set to zero.
 *
 *   dgamma, dbeta  [hidden] float32, device, written (overwritten, not
 *                  accumulated into).
 *   dy, x          [rows, hidden] dt, device, read.
 *   mean, rstd     [rows] float32, device, read.
 *   workspace      device scratch of at least
 *                  ls_layernorm_bw_dgamma_dbeta_workspace_size(rows, hidden)
 *                  bytes, 16-byte aligned; its contents on entry do not
 *                  matter and are left undefined.  May be NULL when that size
 *                  is 0.  Calls that overlap on the GPU must not share it.
 * Errors as for ls_layernorm_fw, plus LS_ERR_WORKSPACE when the workspace is
 * NULL, too small or not 16-byte aligned.
 */
ls_status ls_layernorm_bw_dgamma_dbeta(float *dgamma, float *dbeta,
                                       const void *dy, const void *x,
                                       const float *mean, const float *rstd,
                                       int64_t rows, int64_t hidden,
                                       void *workspace, size_t workspace_bytes,
                                       ls_dtype dt, void *stream);

/*
 * Bytes of device workspace ls_layernorm_bw needs for a [rows, hidden]
 * problem (the same for every dtype): 8 * hidden bytes for each of at most
 * 456 partial sums, or what ls_layernorm_bw_dgamma_dbeta needs when that is
 * more (the scalar path below).  Returns 0 for rows <= 0 or hidden <= 0.
 * Host-only; launches nothing.
 */
size_t ls_layernorm_bw_workspace_size(int64_t rows, int64_t hidden);

/*
 * Fused LayerNorm backward: the input gradient of ls_layernorm_bw_dinp and the
 * gamma / beta gradients of ls_layernorm_bw_dgamma_dbeta from one read of dy
 * and x ("Problem 2.2" of the HW4 page asks for both halves of the backward;
 * slide 22 of the L10 page lists the per-row sums).  The rows are cut into
 * contiguous chunks (at most 456 for rows of one 16-byte vector, 304 for up
 * to 512 vectors, 152 for wider rows) by a rule that depends only on (rows,
 * hidden, dt); one thread block per chunk writes dx for its rows and its
 * chunk's column sums of dy * xhat and dy, and a second kernel adds the
 * chunks in index order.  dgamma and dbeta are therefore bitwise
 * reproducible from run to run and GPU to GPU; their rounding, and dx's (the
 * row sums are split across threads differently), may differ from the
 * separate kernels' in the last bits.
 *
 *   dx             [rows, hidden] dt, device, written.  May equal dy (each
 *                  row's dy is staged on chip before its dx is written).
 *   dgamma, dbeta  [hidden] float32, device, written (overwritten).
 *   dy, x          [rows, hidden] dt, device, read.
 *   gamma          [hidden] dt, device, read.
 *   mean, rstd     [rows] float32, device, read (as saved by ls_layernorm_fw).
 *   workspace      device scratch of at least
 *                  ls_layernorm_bw_workspace_size(rows, hidden) bytes,
 *                  16-byte aligned, contents ignored; may be NULL when that
 *                  size is 0.  Calls that overlap on the GPU must not share it.
 * Errors as for ls_layernorm_bw_dgamma_dbeta.  Rows wider than 2048 16-byte
 * vectors (hidden > 16384 for 16-bit storage, > 8192 for fp32), or pointers
 * or widths that are not 16-byte multiples, run the two separate kernels
 * instead, with the same results as calling them.
 */
ls_status ls_layernorm_bw(void *dx, float *dgamma, float *dbeta, const void *dy,
                          const void *x, const void *gamma, const float *mean,
                          const float *rstd, int64_t rows, int64_t hidden,
                          void *workspace, size_t workspace_bytes, ls_dtype dt,
                          void *stream);

/*
 * Size of the device array that ls_layernorm_bw_dgamma_dbeta_noalloc uses as
 * scratch (4 MiB).  It covers every problem with hidden <= 524288 (2^19),
 * whatever the row count: the partial sums take at most 456 * 2048 bytes
 * for hidden below 116736 (456 tiles of 256), and 8 * hidden bytes (one
 * row chunk) above it.
 */
#define LS_DGDB_NOALLOC_SCRATCH_BYTES ((size_t)4 << 20)

/*
 * LayerNorm gamma/beta gradients without any allocation.  The pages have no
 * counterpart to this entry point; it exists for callers that cannot hand the
 * library a workspace -- code that receives only tensor pointers and a stream
 * from a host program (a plugin, or C code with no access to the host's
 * allocator), or code that may not call cudaMalloc at that moment because
 * cudaMalloc can synchronise the device or break the host's memory budget.
 *
 * Computes exactly what ls_layernorm_bw_dgamma_dbeta computes (same kernels,
 * same fixed summation order, bitwise the same result), but keeps the partial
 * sums in a fixed device array of LS_DGDB_NOALLOC_SCRATCH_BYTES compiled into
 * the library, which every GPU that loads the library holds until the process
 * exits.  It calls no cudaMalloc, cudaFree or other allocating routine.
 *
 *   Arguments as for ls_layernorm_bw_dgamma_dbeta, without the workspace.
 *   Problems whose partial sums need more than LS_DGDB_NOALLOC_SCRATCH_BYTES
 *   (ls_layernorm_bw_dgamma_dbeta_workspace_size(rows, hidden) larger than
 *   that) are refused with LS_ERR_UNSUPPORTED before anything is launched.
 *
 * Every call looks up the array's device address (cudaGetSymbolAddress) with
 * the caller's device current; once the library's module is loaded on that
 * device the lookup is a host-side query that allocates nothing, and a fresh
 * lookup stays valid after cudaDeviceReset.  The first call on a device may
 * be the one that loads the module, which places the array in device memory
 * and can synchronise: make one call during set-up, before any stream
 * capture, if that must not happen later.  All calls on a device share the one
 * array: calls that may overlap on the GPU (different streams without
 * ordering between them) race on it and must not be issued that way.  The
 * array keeps the last call's partial sums; each call overwrites every
 * partial it reads, so nothing needs to be cleared between calls.
 */
ls_status ls_layernorm_bw_dgamma_dbeta_noalloc(float *dgamma, float *dbeta,
                                               const void *dy, const void *x,
                                               const float *mean, const float *rstd,
                                               int64_t rows, int64_t hidden,
                                               ls_dtype dt, void *stream);

/*
 * RMSNorm forward: the one-reduction LayerNorm variant of the page
 * "FastTransformer: Breaking the Compiler Ceiling via Architectural
 * Co-Design", section 5.4 "Vectorized Pre-RMSNorm" (no mean centring, no
 * bias).  Per row of x [rows, hidden]:
 *     rstd = 1 / sqrt(mean(x^2) + eps),   y_j = x_j * rstd * gamma_j
 *
 *   y      [rows, hidden] dt, device, written.
 *   rstd   [rows] float32, device, written (saved for the backward).
 *   x      [rows, hidden] dt, device, read.
 *   gamma  [hidden] dt, device, read.
 *   eps    added inside the square root (the page uses 1e-6).
 * Errors as for ls_layernorm_fw.
 */
ls_status ls_rmsnorm_fw(void *y, float *rstd, const void *x, const void *gamma, int64_t rows,
                        int64_t hidden, float eps, ls_dtype dt, void *stream);

/*
 * RMSNorm backward, input gradient.  With xhat = x * rstd and g = gamma * dy,
 * per row:  S = sum_j g_j * xhat_j,  dx_j = rstd * (g_j - xhat_j * S / hidden).
 *
 *   dx     [rows, hidden] dt, device, written.  May equal `dy`.
 *   dy, x  [rows, hidden] dt, device, read.
 *   gamma  [hidden] dt, device, read.
 *   rstd   [rows] float32, device, read (as saved by ls_rmsnorm_fw).
 * Errors as for ls_layernorm_bw_dinp.
 */
ls_status ls_rmsnorm_bw_dinp(void *dx, const void *dy, const void *x, const void *gamma,
                             const float *rstd, int64_t rows, int64_t hidden, ls_dtype dt,
                             void *stream);

/*
 * RMSNorm backward, gamma gradient: dgamma_j = sum_r dy_rj * x_rj * rstd_r,
 * in the same fixed order as ls_layernorm_bw_dgamma_dbeta (bitwise
 * reproducible).  `workspace` as for that function, sized by
 * ls_layernorm_bw_dgamma_dbeta_workspace_size(rows, hidden).
 *
 *   dgamma  [hidden] float32, device, written (overwritten).
 *   dy, x   [rows, hidden] dt, device, read.
 *   rstd    [rows] float32, device, read.
 * Errors as for ls_layernorm_bw_dgamma_dbeta.
 */
ls_status ls_rmsnorm_bw_dgamma(float *dgamma, const void *dy, const void *x, const float *rstd,
                               int64_t rows, int64_t hidden, void *workspace,
                               size_t workspace_bytes, ls_dtype dt, void *stream);

/*
 * Softmax cross entropy over a vocabulary, forward.  The L10 page, section
 * "Technique 1: kernel fusion, leaving only GEMMs to cuBLAS" (slide 12),
 * makes cross entropy the third custom reduce kernel beside LayerNorm and
 * softmax; the page gives no formula, so this is the textbook one, in FP32.
 * For each row r of logits z [rows, vocab] with target class t = target[r]:
 *     lse_r  = log sum_j exp(z_rj)        (computed as max + log sum exp(z - max))
 *     loss_r = lse_r - z_rt               (= -log softmax(z_r)_t)
 * A negative target marks an ignored row (padding): loss_r = lse_r = 0 and
 * the row is not read.  A target >= vocab gives loss_r = lse_r = NaN (there
 * is no device-side trap).  No label smoothing; one loss per row (the caller
 * reduces, e.g. sums over its non-ignored rows).
 *
 *   loss, lse  [rows] float32, device, written.
 *   logits     [rows, vocab] dt, device, read; any vocab >= 1 (rows need
 *              not start on 16-byte boundaries).
 *   target     [rows] int32, device, read.
 * Errors: LS_ERR_INVALID_ARG for rows < 0, vocab < 1 or a NULL pointer when
 * rows > 0; LS_ERR_UNSUPPORTED for an unknown dtype or vocab above
 * LS_MAX_ROW_LENGTH; LS_ERR_MISALIGNED for a pointer not aligned to its
 * element; LS_ERR_CUDA for a failed launch.  rows == 0 launches nothing.
 */
ls_status ls_cross_entropy_fw(float *loss, float *lse, const void *logits,
                              const int32_t *target, int64_t rows, int64_t vocab,
                              ls_dtype dt, void *stream);

/*
 * Softmax cross entropy, backward: the gradient of loss_r * dloss_r with
 * respect to the logits, from the lse saved by the forward:
 *     dlogits_rj = dloss_r * ( exp(z_rj - lse_r) - [j == t_r] )
 * Ignored rows (t_r < 0) are written as zeros and rows with t_r >= vocab as
 * NaN; neither is read.
 *
 *   dlogits  [rows, vocab] dt, device, written.  May equal logits.
 *   logits   [rows, vocab] dt, device, read.
 *   target   [rows] int32, device, read.
 *   lse      [rows] float32, device, read (as written by ls_cross_entropy_fw).
 *   dloss    [rows] float32, device, read (upstream gradient of each row's
 *            loss; 1 / (number of non-ignored rows) for a mean loss).
 * Errors as for ls_cross_entropy_fw.  When logits and dlogits do not sit at
 * the same offset modulo 16 bytes, every element is moved singly (slower,
 * same result).
 */
ls_status ls_cross_entropy_bw(void *dlogits, const void *logits, const int32_t *target,
                              const float *lse, const float *dloss, int64_t rows,
                              int64_t vocab, ls_dtype dt, void *stream);

/* Static, human-readable name of a status code (never NULL). */
const char *ls_status_string(ls_status s);

#ifdef __cplusplus
}
#endif

#endif /* LS_REDUCE_H */
