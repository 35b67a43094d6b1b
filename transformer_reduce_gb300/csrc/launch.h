// launch.h -- internal C++ launchers behind the C ABI (one instantiation per
// storage dtype, compiled in its own translation unit).  Arguments have been
// validated by the ABI layer; `vec` says whether every tensor of the call is
// 16-byte aligned with a row length in bytes that is a multiple of 16.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace lsr {

// Rows per partial-sum chunk of the gamma/beta reduction, and the chunk count.
// Chosen so that column tiles x chunks gives roughly 1024 blocks; depends only
// on (rows, hidden), never on the GPU, so the summation order is fixed.
int64_t dgdb_rows_per_chunk(int64_t rows, int64_t hidden);
int64_t dgdb_num_chunks(int64_t rows, int64_t hidden);

// Number of SMs of the current device (cached per device).
int device_sm_count();

// qoff = Tk - Tq: a causal row sees keys j <= (query index) + qoff.  scale
// (> 0) multiplies the scores before the mask is added (1 for plain softmax).
template <typename T>
cudaError_t launch_softmax_fw(T *out, const T *inp, const T *mask, int64_t rows,
                              int64_t rows_per_batch, int64_t Tq, int64_t Tk,
                              int causal, int64_t qoff, float scale, bool vec, cudaStream_t st);
template <typename T>
cudaError_t launch_softmax_bw_masked(T *dinp, const T *dout, const T *y, const T *mask,
                                     int64_t rows, int64_t rows_per_batch, int64_t Tq,
                                     int64_t Tk, int causal, int64_t qoff, float scale, bool vec,
                                     cudaStream_t st);
template <typename T>
cudaError_t launch_softmax_bw(T *dinp, const T *dout, const T *y, int64_t rows,
                              int64_t Tk, bool vec, cudaStream_t st);
template <typename T>
cudaError_t launch_ln_fw(T *y, float *mean, float *rstd, const T *x, const T *gamma,
                         const T *beta, int64_t rows, int64_t N, float eps, bool vec,
                         cudaStream_t st);
template <typename T>
cudaError_t launch_ln_dinp(T *dx, const T *dy, const T *x, const T *gamma,
                           const float *mean, const float *rstd, int64_t rows,
                           int64_t N, bool vec, cudaStream_t st);
template <typename T>
cudaError_t launch_ln_dgdb(float *dgamma, float *dbeta, const T *dy, const T *x,
                           const float *mean, const float *rstd, int64_t rows,
                           int64_t N, float *part, bool vec, cudaStream_t st);

// Partial-sum slots the fused LayerNorm backward may use for `rows` rows:
// one per row chunk, at most 456.
int64_t ln_bw_fused_max_parts(int64_t rows);

// Fused LayerNorm backward: dx, dgamma, dbeta from one read of dy and x.
template <typename T>
cudaError_t launch_ln_bw_fused(T *dx, float *dgamma, float *dbeta, const T *dy, const T *x,
                               const T *gamma, const float *mean, const float *rstd,
                               int64_t rows, int64_t N, float *part, bool vec, cudaStream_t st);

// RMSNorm (no mean, no beta): forward, input gradient, gamma gradient.
template <typename T>
cudaError_t launch_rms_fw(T *y, float *rstd, const T *x, const T *gamma, int64_t rows, int64_t N,
                          float eps, bool vec, cudaStream_t st);
template <typename T>
cudaError_t launch_rms_dinp(T *dx, const T *dy, const T *x, const T *gamma, const float *rstd,
                            int64_t rows, int64_t N, bool vec, cudaStream_t st);
template <typename T>
cudaError_t launch_rms_dgamma(float *dgamma, const T *dy, const T *x, const float *rstd,
                              int64_t rows, int64_t N, float *part, bool vec, cudaStream_t st);

// Softmax cross entropy over a vocabulary (forward: loss and log-sum-exp per
// row; backward: dz from the saved log-sum-exp).  vec: take 16-byte vectors
// for the aligned middle of each row (the backward needs z and dz at the same
// offset modulo 16 bytes).
template <typename T>
cudaError_t launch_ce_fw(float *loss, float *lse, const T *z, const int32_t *target, int64_t rows,
                         int64_t V, bool vec, cudaStream_t st);
template <typename T>
cudaError_t launch_ce_bw(T *dz, const T *z, const int32_t *target, const float *lse,
                         const float *dloss, int64_t rows, int64_t V, bool vec, cudaStream_t st);

}  // namespace lsr
