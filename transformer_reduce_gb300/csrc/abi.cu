// abi.cu -- the extern "C" entry points of libls_reduce.so (declared and
// documented in include/ls_reduce.h).  This layer validates every argument on
// the host, picks the storage dtype and the vector/scalar path, and enqueues
// the kernels on the caller's stream.  It never allocates, frees or
// synchronises.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>

#include "launch.h"
#include "ls_reduce.h"

namespace lsr {

int64_t dgdb_rows_per_chunk(int64_t rows, int64_t hidden) {
    // At most about 456 blocks (256-column tiles x row chunks): three
    // resident blocks on each of a GB300's 152 SMs, one wave with no partial
    // second wave.  A constant, not the device's SM count, so the summation
    // order depends only on (rows, hidden).
    if (rows <= 0 || hidden <= 0) return 1;
    const int64_t tiles = (hidden + 255) / 256;
    const int64_t target_chunks = tiles < 456 ? 456 / tiles : 1;
    int64_t rpc = (rows + target_chunks - 1) / target_chunks;
    if (rpc < 16) rpc = 16;
    while ((rows + rpc - 1) / rpc > 65535) rpc *= 2;
    return rpc;
}

int64_t dgdb_num_chunks(int64_t rows, int64_t hidden) {
    if (rows <= 0 || hidden <= 0) return 0;
    const int64_t rpc = dgdb_rows_per_chunk(rows, hidden);
    return (rows + rpc - 1) / rpc;
}

int64_t ln_bw_fused_max_parts(int64_t rows) {
    // 456 chunks is the most any bucket uses (fewer chunks of more rows never
    // need more slots); one slot per chunk
    if (rows <= 0) return 0;
    const int64_t rpc = (rows + 455) / 456;
    return (rows + rpc - 1) / rpc;
}

int device_sm_count() {
    constexpr int kMaxDev = 64;
    static std::atomic<int> cache[kMaxDev];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 1;
    if (dev < kMaxDev) {
        int v = cache[dev].load(std::memory_order_relaxed);
        if (v > 0) return v;
    }
    int n = 1;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
        n = 1;
    if (dev < kMaxDev) cache[dev].store(n, std::memory_order_relaxed);
    return n;
}

}  // namespace lsr

namespace {

size_t elem_size(ls_dtype dt) {
    switch (dt) {
        case LS_F32: return 4;
        case LS_F16: return 2;
        case LS_BF16: return 2;
    }
    return 0;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// 16-byte vector path: every tensor 16-byte aligned and rows a whole number of
// 16-byte chunks (so every row starts on a 16-byte boundary too).
bool vec_ok(int64_t row_len, size_t es, std::initializer_list<const void *> ptrs) {
    if ((row_len * (int64_t)es) % 16 != 0) return false;
    for (const void *p : ptrs)
        if (p && !aligned(p, 16)) return false;
    return true;
}

ls_status from_cuda(cudaError_t e) { return e == cudaSuccess ? LS_OK : LS_ERR_CUDA; }

}  // namespace

extern "C" {

const char *ls_status_string(ls_status s) {
    switch (s) {
        case LS_OK: return "LS_OK";
        case LS_ERR_INVALID_ARG: return "LS_ERR_INVALID_ARG: null pointer, negative size or inconsistent shape";
        case LS_ERR_UNSUPPORTED: return "LS_ERR_UNSUPPORTED: unknown dtype or size beyond the library limits";
        case LS_ERR_MISALIGNED: return "LS_ERR_MISALIGNED: pointer not aligned to its element size";
        case LS_ERR_WORKSPACE: return "LS_ERR_WORKSPACE: workspace missing, too small or not 16-byte aligned";
        case LS_ERR_CUDA: return "LS_ERR_CUDA: the CUDA runtime rejected a launch";
    }
    return "unknown ls_status";
}

static ls_status softmax_fw_impl(void *out, const void *inp, const void *mask, int64_t B,
                                 int64_t H, int64_t Tq, int64_t Tk, int causal, float scale,
                                 ls_dtype dt, void *stream) {
    const size_t es = elem_size(dt);
    if (es == 0) return LS_ERR_UNSUPPORTED;
    if (B < 0 || H < 0 || Tq < 0 || Tk < 0) return LS_ERR_INVALID_ARG;
    if (causal && Tq > Tk) return LS_ERR_INVALID_ARG;
    if (Tk > LS_MAX_ROW_LENGTH) return LS_ERR_UNSUPPORTED;
    if (B == 0 || H == 0 || Tq == 0 || Tk == 0) return LS_OK;
    if (!out || !inp) return LS_ERR_INVALID_ARG;
    if (H > INT64_MAX / B || Tq > INT64_MAX / (B * H) || Tk > INT64_MAX / (B * H * Tq))
        return LS_ERR_UNSUPPORTED;
    if (!aligned(out, es) || !aligned(inp, es) || (mask && !aligned(mask, es)))
        return LS_ERR_MISALIGNED;
    const int64_t rows = B * H * Tq;
    const bool vec = vec_ok(Tk, es, {out, inp, mask});
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    switch (dt) {
        case LS_F32:
            return from_cuda(lsr::launch_softmax_fw<float>(
                (float *)out, (const float *)inp, (const float *)mask, rows, H * Tq, Tq, Tk,
                causal ? 1 : 0, Tk - Tq, scale, vec, st));
        case LS_F16:
            return from_cuda(lsr::launch_softmax_fw<__half>(
                (__half *)out, (const __half *)inp, (const __half *)mask, rows, H * Tq, Tq, Tk,
                causal ? 1 : 0, Tk - Tq, scale, vec, st));
        case LS_BF16:
            return from_cuda(lsr::launch_softmax_fw<__nv_bfloat16>(
                (__nv_bfloat16 *)out, (const __nv_bfloat16 *)inp, (const __nv_bfloat16 *)mask,
                rows, H * Tq, Tq, Tk, causal ? 1 : 0, Tk - Tq, scale, vec, st));
    }
    return LS_ERR_UNSUPPORTED;
}

static bool scale_ok(float scale) { return std::isfinite(scale) && scale > 0.f; }

ls_status ls_softmax_fw(void *out, const void *inp, const void *mask, int64_t B, int64_t H,
                        int64_t Tq, int64_t Tk, int causal, ls_dtype dt, void *stream) {
    return softmax_fw_impl(out, inp, mask, B, H, Tq, Tk, causal, 1.0f, dt, stream);
}

ls_status ls_softmax_fw_scaled(void *out, const void *inp, const void *mask, int64_t B,
                               int64_t H, int64_t Tq, int64_t Tk, int causal, float scale,
                               ls_dtype dt, void *stream) {
    if (elem_size(dt) == 0) return LS_ERR_UNSUPPORTED;
    if (!scale_ok(scale)) return LS_ERR_INVALID_ARG;
    return softmax_fw_impl(out, inp, mask, B, H, Tq, Tk, causal, scale, dt, stream);
}

ls_status ls_softmax_bw(void *dinp, const void *dout, const void *out_fw, int64_t B, int64_t H,
                        int64_t Tq, int64_t Tk, ls_dtype dt, void *stream) {
    const size_t es = elem_size(dt);
    if (es == 0) return LS_ERR_UNSUPPORTED;
    if (B < 0 || H < 0 || Tq < 0 || Tk < 0) return LS_ERR_INVALID_ARG;
    if (Tk > LS_MAX_ROW_LENGTH) return LS_ERR_UNSUPPORTED;
    if (B == 0 || H == 0 || Tq == 0 || Tk == 0) return LS_OK;
    if (!dinp || !dout || !out_fw) return LS_ERR_INVALID_ARG;
    if (H > INT64_MAX / B || Tq > INT64_MAX / (B * H) || Tk > INT64_MAX / (B * H * Tq))
        return LS_ERR_UNSUPPORTED;
    if (!aligned(dinp, es) || !aligned(dout, es) || !aligned(out_fw, es))
        return LS_ERR_MISALIGNED;
    const int64_t rows = B * H * Tq;
    const bool vec = vec_ok(Tk, es, {dinp, dout, out_fw});
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    switch (dt) {
        case LS_F32:
            return from_cuda(lsr::launch_softmax_bw<float>(
                (float *)dinp, (const float *)dout, (const float *)out_fw, rows, Tk, vec, st));
        case LS_F16:
            return from_cuda(lsr::launch_softmax_bw<__half>(
                (__half *)dinp, (const __half *)dout, (const __half *)out_fw, rows, Tk, vec, st));
        case LS_BF16:
            return from_cuda(lsr::launch_softmax_bw<__nv_bfloat16>(
                (__nv_bfloat16 *)dinp, (const __nv_bfloat16 *)dout,
                (const __nv_bfloat16 *)out_fw, rows, Tk, vec, st));
    }
    return LS_ERR_UNSUPPORTED;
}

static ls_status softmax_bw_masked_impl(void *dinp, const void *dout, const void *out_fw,
                                        const void *mask, int64_t B, int64_t H, int64_t Tq,
                                        int64_t Tk, int causal, float scale, ls_dtype dt,
                                        void *stream) {
    const size_t es = elem_size(dt);
    if (es == 0) return LS_ERR_UNSUPPORTED;
    if (B < 0 || H < 0 || Tq < 0 || Tk < 0) return LS_ERR_INVALID_ARG;
    if (causal && Tq > Tk) return LS_ERR_INVALID_ARG;
    if (Tk > LS_MAX_ROW_LENGTH) return LS_ERR_UNSUPPORTED;
    if (B == 0 || H == 0 || Tq == 0 || Tk == 0) return LS_OK;
    if (!dinp || !dout || !out_fw) return LS_ERR_INVALID_ARG;
    if (H > INT64_MAX / B || Tq > INT64_MAX / (B * H) || Tk > INT64_MAX / (B * H * Tq))
        return LS_ERR_UNSUPPORTED;
    if (!aligned(dinp, es) || !aligned(dout, es) || !aligned(out_fw, es) ||
        (mask && !aligned(mask, es)))
        return LS_ERR_MISALIGNED;
    const int64_t rows = B * H * Tq;
    const bool vec = vec_ok(Tk, es, {dinp, dout, out_fw, mask});
    const int c = causal ? 1 : 0;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    switch (dt) {
        case LS_F32:
            return from_cuda(lsr::launch_softmax_bw_masked<float>(
                (float *)dinp, (const float *)dout, (const float *)out_fw, (const float *)mask,
                rows, H * Tq, Tq, Tk, c, Tk - Tq, scale, vec, st));
        case LS_F16:
            return from_cuda(lsr::launch_softmax_bw_masked<__half>(
                (__half *)dinp, (const __half *)dout, (const __half *)out_fw,
                (const __half *)mask, rows, H * Tq, Tq, Tk, c, Tk - Tq, scale, vec, st));
        case LS_BF16:
            return from_cuda(lsr::launch_softmax_bw_masked<__nv_bfloat16>(
                (__nv_bfloat16 *)dinp, (const __nv_bfloat16 *)dout,
                (const __nv_bfloat16 *)out_fw, (const __nv_bfloat16 *)mask, rows, H * Tq, Tq,
                Tk, c, Tk - Tq, scale, vec, st));
    }
    return LS_ERR_UNSUPPORTED;
}

ls_status ls_softmax_bw_masked(void *dinp, const void *dout, const void *out_fw,
                               const void *mask, int64_t B, int64_t H, int64_t Tq, int64_t Tk,
                               int causal, ls_dtype dt, void *stream) {
    return softmax_bw_masked_impl(dinp, dout, out_fw, mask, B, H, Tq, Tk, causal, 1.0f, dt,
                                  stream);
}

ls_status ls_softmax_bw_masked_scaled(void *dinp, const void *dout, const void *out_fw,
                                      const void *mask, int64_t B, int64_t H, int64_t Tq,
                                      int64_t Tk, int causal, float scale, ls_dtype dt,
                                      void *stream) {
    if (elem_size(dt) == 0) return LS_ERR_UNSUPPORTED;
    if (!scale_ok(scale)) return LS_ERR_INVALID_ARG;
    return softmax_bw_masked_impl(dinp, dout, out_fw, mask, B, H, Tq, Tk, causal, scale, dt,
                                  stream);
}

// Shared checks of the LayerNorm entry points.
static ls_status ln_check(int64_t rows, int64_t hidden, size_t es) {
    if (es == 0) return LS_ERR_UNSUPPORTED;
    if (rows < 0 || hidden < 1) return LS_ERR_INVALID_ARG;
    if (hidden > LS_MAX_ROW_LENGTH) return LS_ERR_UNSUPPORTED;
    if (rows > 0 && hidden > INT64_MAX / rows) return LS_ERR_UNSUPPORTED;
    return LS_OK;
}

ls_status ls_layernorm_fw(void *y, float *mean, float *rstd, const void *x, const void *gamma,
                          const void *beta, int64_t rows, int64_t hidden, float eps,
                          ls_dtype dt, void *stream) {
    const size_t es = elem_size(dt);
    ls_status s = ln_check(rows, hidden, es);
    if (s != LS_OK) return s;
    if (!(eps >= 0.f) || !std::isfinite(eps)) return LS_ERR_INVALID_ARG;
    if (rows == 0) return LS_OK;
    if (!y || !mean || !rstd || !x || !gamma || !beta) return LS_ERR_INVALID_ARG;
    if (!aligned(y, es) || !aligned(x, es) || !aligned(gamma, es) || !aligned(beta, es) ||
        !aligned(mean, 4) || !aligned(rstd, 4))
        return LS_ERR_MISALIGNED;
    const bool vec = vec_ok(hidden, es, {y, x, gamma, beta});
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    switch (dt) {
        case LS_F32:
            return from_cuda(lsr::launch_ln_fw<float>((float *)y, mean, rstd, (const float *)x,
                                                      (const float *)gamma, (const float *)beta,
                                                      rows, hidden, eps, vec, st));
        case LS_F16:
            return from_cuda(lsr::launch_ln_fw<__half>(
                (__half *)y, mean, rstd, (const __half *)x, (const __half *)gamma,
                (const __half *)beta, rows, hidden, eps, vec, st));
        case LS_BF16:
            return from_cuda(lsr::launch_ln_fw<__nv_bfloat16>(
                (__nv_bfloat16 *)y, mean, rstd, (const __nv_bfloat16 *)x,
                (const __nv_bfloat16 *)gamma, (const __nv_bfloat16 *)beta, rows, hidden, eps,
                vec, st));
    }
    return LS_ERR_UNSUPPORTED;
}

ls_status ls_layernorm_bw_dinp(void *dx, const void *dy, const void *x, const void *gamma,
                               const float *mean, const float *rstd, int64_t rows,
                               int64_t hidden, ls_dtype dt, void *stream) {
    const size_t es = elem_size(dt);
    ls_status s = ln_check(rows, hidden, es);
    if (s != LS_OK) return s;
    if (rows == 0) return LS_OK;
    if (!dx || !dy || !x || !gamma || !mean || !rstd) return LS_ERR_INVALID_ARG;
    if (!aligned(dx, es) || !aligned(dy, es) || !aligned(x, es) || !aligned(gamma, es) ||
        !aligned(mean, 4) || !aligned(rstd, 4))
        return LS_ERR_MISALIGNED;
    const bool vec = vec_ok(hidden, es, {dx, dy, x, gamma});
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    switch (dt) {
        case LS_F32:
            return from_cuda(lsr::launch_ln_dinp<float>((float *)dx, (const float *)dy,
                                                        (const float *)x, (const float *)gamma,
                                                        mean, rstd, rows, hidden, vec, st));
        case LS_F16:
            return from_cuda(lsr::launch_ln_dinp<__half>((__half *)dx, (const __half *)dy,
                                                         (const __half *)x,
                                                         (const __half *)gamma, mean, rstd,
                                                         rows, hidden, vec, st));
        case LS_BF16:
            return from_cuda(lsr::launch_ln_dinp<__nv_bfloat16>(
                (__nv_bfloat16 *)dx, (const __nv_bfloat16 *)dy, (const __nv_bfloat16 *)x,
                (const __nv_bfloat16 *)gamma, mean, rstd, rows, hidden, vec, st));
    }
    return LS_ERR_UNSUPPORTED;
}

ls_status ls_rmsnorm_fw(void *y, float *rstd, const void *x, const void *gamma, int64_t rows,
                        int64_t hidden, float eps, ls_dtype dt, void *stream) {
    const size_t es = elem_size(dt);
    ls_status s = ln_check(rows, hidden, es);
    if (s != LS_OK) return s;
    if (!(eps >= 0.f) || !std::isfinite(eps)) return LS_ERR_INVALID_ARG;
    if (rows == 0) return LS_OK;
    if (!y || !rstd || !x || !gamma) return LS_ERR_INVALID_ARG;
    if (!aligned(y, es) || !aligned(x, es) || !aligned(gamma, es) || !aligned(rstd, 4))
        return LS_ERR_MISALIGNED;
    const bool vec = vec_ok(hidden, es, {y, x, gamma});
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    switch (dt) {
        case LS_F32:
            return from_cuda(lsr::launch_rms_fw<float>((float *)y, rstd, (const float *)x,
                                                       (const float *)gamma, rows, hidden, eps,
                                                       vec, st));
        case LS_F16:
            return from_cuda(lsr::launch_rms_fw<__half>((__half *)y, rstd, (const __half *)x,
                                                        (const __half *)gamma, rows, hidden, eps,
                                                        vec, st));
        case LS_BF16:
            return from_cuda(lsr::launch_rms_fw<__nv_bfloat16>(
                (__nv_bfloat16 *)y, rstd, (const __nv_bfloat16 *)x, (const __nv_bfloat16 *)gamma,
                rows, hidden, eps, vec, st));
    }
    return LS_ERR_UNSUPPORTED;
}

ls_status ls_rmsnorm_bw_dinp(void *dx, const void *dy, const void *x, const void *gamma,
                             const float *rstd, int64_t rows, int64_t hidden, ls_dtype dt,
                             void *stream) {
    const size_t es = elem_size(dt);
    ls_status s = ln_check(rows, hidden, es);
    if (s != LS_OK) return s;
    if (rows == 0) return LS_OK;
    if (!dx || !dy || !x || !gamma || !rstd) return LS_ERR_INVALID_ARG;
    if (!aligned(dx, es) || !aligned(dy, es) || !aligned(x, es) || !aligned(gamma, es) ||
        !aligned(rstd, 4))
        return LS_ERR_MISALIGNED;
    const bool vec = vec_ok(hidden, es, {dx, dy, x, gamma});
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    switch (dt) {
        case LS_F32:
            return from_cuda(lsr::launch_rms_dinp<float>((float *)dx, (const float *)dy,
                                                         (const float *)x, (const float *)gamma,
                                                         rstd, rows, hidden, vec, st));
        case LS_F16:
            return from_cuda(lsr::launch_rms_dinp<__half>((__half *)dx, (const __half *)dy,
                                                          (const __half *)x,
                                                          (const __half *)gamma, rstd, rows,
                                                          hidden, vec, st));
        case LS_BF16:
            return from_cuda(lsr::launch_rms_dinp<__nv_bfloat16>(
                (__nv_bfloat16 *)dx, (const __nv_bfloat16 *)dy, (const __nv_bfloat16 *)x,
                (const __nv_bfloat16 *)gamma, rstd, rows, hidden, vec, st));
    }
    return LS_ERR_UNSUPPORTED;
}

ls_status ls_rmsnorm_bw_dgamma(float *dgamma, const void *dy, const void *x, const float *rstd,
                               int64_t rows, int64_t hidden, void *workspace,
                               size_t workspace_bytes, ls_dtype dt, void *stream) {
    const size_t es = elem_size(dt);
    ls_status s = ln_check(rows, hidden, es);
    if (s != LS_OK) return s;
    if (!dgamma) return LS_ERR_INVALID_ARG;
    if (rows > 0 && (!dy || !x || !rstd)) return LS_ERR_INVALID_ARG;
    if (!aligned(dgamma, 4) || (dy && !aligned(dy, es)) || (x && !aligned(x, es)) ||
        (rstd && !aligned(rstd, 4)))
        return LS_ERR_MISALIGNED;
    const size_t need = ls_layernorm_bw_dgamma_dbeta_workspace_size(rows, hidden);
    if (need > 0 && (!workspace || workspace_bytes < need || !aligned(workspace, 16)))
        return LS_ERR_WORKSPACE;
    const bool vec = vec_ok(hidden, es, {dy, x});
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    float *part = static_cast<float *>(workspace);
    switch (dt) {
        case LS_F32:
            return from_cuda(lsr::launch_rms_dgamma<float>(dgamma, (const float *)dy,
                                                           (const float *)x, rstd, rows, hidden,
                                                           part, vec, st));
        case LS_F16:
            return from_cuda(lsr::launch_rms_dgamma<__half>(dgamma, (const __half *)dy,
                                                            (const __half *)x, rstd, rows, hidden,
                                                            part, vec, st));
        case LS_BF16:
            return from_cuda(lsr::launch_rms_dgamma<__nv_bfloat16>(
                dgamma, (const __nv_bfloat16 *)dy, (const __nv_bfloat16 *)x, rstd, rows, hidden,
                part, vec, st));
    }
    return LS_ERR_UNSUPPORTED;
}

size_t ls_layernorm_bw_workspace_size(int64_t rows, int64_t hidden) {
    if (rows <= 0 || hidden <= 0) return 0;
    const size_t fused = (size_t)lsr::ln_bw_fused_max_parts(rows) * 2u * (size_t)hidden * 4u;
    const size_t split = ls_layernorm_bw_dgamma_dbeta_workspace_size(rows, hidden);
    return fused > split ? fused : split;
}

ls_status ls_layernorm_bw(void *dx, float *dgamma, float *dbeta, const void *dy, const void *x,
                          const void *gamma, const float *mean, const float *rstd, int64_t rows,
                          int64_t hidden, void *workspace, size_t workspace_bytes, ls_dtype dt,
                          void *stream) {
    const size_t es = elem_size(dt);
    ls_status s = ln_check(rows, hidden, es);
    if (s != LS_OK) return s;
    if (!dgamma || !dbeta) return LS_ERR_INVALID_ARG;
    if (rows > 0 && (!dx || !dy || !x || !gamma || !mean || !rstd)) return LS_ERR_INVALID_ARG;
    if (!aligned(dgamma, 4) || !aligned(dbeta, 4) || (dx && !aligned(dx, es)) ||
        (dy && !aligned(dy, es)) || (x && !aligned(x, es)) || (gamma && !aligned(gamma, es)) ||
        (mean && !aligned(mean, 4)) || (rstd && !aligned(rstd, 4)))
        return LS_ERR_MISALIGNED;
    const size_t need = ls_layernorm_bw_workspace_size(rows, hidden);
    if (need > 0 && (!workspace || workspace_bytes < need || !aligned(workspace, 16)))
        return LS_ERR_WORKSPACE;
    const bool vec = vec_ok(hidden, es, {dx, dy, x, gamma});
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    float *part = static_cast<float *>(workspace);
    switch (dt) {
        case LS_F32:
            return from_cuda(lsr::launch_ln_bw_fused<float>(
                (float *)dx, dgamma, dbeta, (const float *)dy, (const float *)x,
                (const float *)gamma, mean, rstd, rows, hidden, part, vec, st));
        case LS_F16:
            return from_cuda(lsr::launch_ln_bw_fused<__half>(
                (__half *)dx, dgamma, dbeta, (const __half *)dy, (const __half *)x,
                (const __half *)gamma, mean, rstd, rows, hidden, part, vec, st));
        case LS_BF16:
            return from_cuda(lsr::launch_ln_bw_fused<__nv_bfloat16>(
                (__nv_bfloat16 *)dx, dgamma, dbeta, (const __nv_bfloat16 *)dy,
                (const __nv_bfloat16 *)x, (const __nv_bfloat16 *)gamma, mean, rstd, rows, hidden,
                part, vec, st));
    }
    return LS_ERR_UNSUPPORTED;
}

size_t ls_layernorm_bw_dgamma_dbeta_workspace_size(int64_t rows, int64_t hidden) {
    if (rows <= 0 || hidden <= 0) return 0;
    const int64_t nchunks = lsr::dgdb_num_chunks(rows, hidden);
    return (size_t)nchunks * 2u * (size_t)hidden * sizeof(float);
}

ls_status ls_layernorm_bw_dgamma_dbeta(float *dgamma, float *dbeta, const void *dy, const void *x,
                                       const float *mean, const float *rstd, int64_t rows,
                                       int64_t hidden, void *workspace, size_t workspace_bytes,
                                       ls_dtype dt, void *stream) {
    const size_t es = elem_size(dt);
    ls_status s = ln_check(rows, hidden, es);
    if (s != LS_OK) return s;
    if (!dgamma || !dbeta) return LS_ERR_INVALID_ARG;
    if (rows > 0 && (!dy || !x || !mean || !rstd)) return LS_ERR_INVALID_ARG;
    if (!aligned(dgamma, 4) || !aligned(dbeta, 4) || (dy && !aligned(dy, es)) ||
        (x && !aligned(x, es)) || (mean && !aligned(mean, 4)) || (rstd && !aligned(rstd, 4)))
        return LS_ERR_MISALIGNED;
    const size_t need = ls_layernorm_bw_dgamma_dbeta_workspace_size(rows, hidden);
    if (need > 0 && (!workspace || workspace_bytes < need || !aligned(workspace, 16)))
        return LS_ERR_WORKSPACE;
    const bool vec = vec_ok(hidden, es, {dy, x});
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    float *part = static_cast<float *>(workspace);
    switch (dt) {
        case LS_F32:
            return from_cuda(lsr::launch_ln_dgdb<float>(dgamma, dbeta, (const float *)dy,
                                                        (const float *)x, mean, rstd, rows,
                                                        hidden, part, vec, st));
        case LS_F16:
            return from_cuda(lsr::launch_ln_dgdb<__half>(dgamma, dbeta, (const __half *)dy,
                                                         (const __half *)x, mean, rstd, rows,
                                                         hidden, part, vec, st));
        case LS_BF16:
            return from_cuda(lsr::launch_ln_dgdb<__nv_bfloat16>(
                dgamma, dbeta, (const __nv_bfloat16 *)dy, (const __nv_bfloat16 *)x, mean, rstd,
                rows, hidden, part, vec, st));
    }
    return LS_ERR_UNSUPPORTED;
}

// ----------------------------------------------------------------------------
// cross entropy over a vocabulary
// ----------------------------------------------------------------------------
ls_status ls_cross_entropy_fw(float *loss, float *lse, const void *logits, const int32_t *target,
                              int64_t rows, int64_t vocab, ls_dtype dt, void *stream) {
    const size_t es = elem_size(dt);
    ls_status s = ln_check(rows, vocab, es);
    if (s != LS_OK) return s;
    if (rows > 0 && (!loss || !lse || !logits || !target)) return LS_ERR_INVALID_ARG;
    if ((loss && !aligned(loss, 4)) || (lse && !aligned(lse, 4)) ||
        (logits && !aligned(logits, es)) || (target && !aligned(target, 4)))
        return LS_ERR_MISALIGNED;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // the aligned middle of every row is read in 16-byte vectors whatever the
    // row's start offset
    switch (dt) {
        case LS_F32:
            return from_cuda(lsr::launch_ce_fw<float>(loss, lse, (const float *)logits, target,
                                                      rows, vocab, true, st));
        case LS_F16:
            return from_cuda(lsr::launch_ce_fw<__half>(loss, lse, (const __half *)logits, target,
                                                       rows, vocab, true, st));
        case LS_BF16:
            return from_cuda(lsr::launch_ce_fw<__nv_bfloat16>(
                loss, lse, (const __nv_bfloat16 *)logits, target, rows, vocab, true, st));
    }
    return LS_ERR_UNSUPPORTED;
}

ls_status ls_cross_entropy_bw(void *dlogits, const void *logits, const int32_t *target,
                              const float *lse, const float *dloss, int64_t rows, int64_t vocab,
                              ls_dtype dt, void *stream) {
    const size_t es = elem_size(dt);
    ls_status s = ln_check(rows, vocab, es);
    if (s != LS_OK) return s;
    if (rows > 0 && (!dlogits || !logits || !target || !lse || !dloss)) return LS_ERR_INVALID_ARG;
    if ((dlogits && !aligned(dlogits, es)) || (logits && !aligned(logits, es)) ||
        (target && !aligned(target, 4)) || (lse && !aligned(lse, 4)) ||
        (dloss && !aligned(dloss, 4)))
        return LS_ERR_MISALIGNED;
    // vectors need logits and dlogits at the same offset within 16 bytes
    const bool vec =
        ((reinterpret_cast<uintptr_t>(dlogits) ^ reinterpret_cast<uintptr_t>(logits)) & 15u) == 0;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    switch (dt) {
        case LS_F32:
            return from_cuda(lsr::launch_ce_bw<float>((float *)dlogits, (const float *)logits,
                                                      target, lse, dloss, rows, vocab, vec, st));
        case LS_F16:
            return from_cuda(lsr::launch_ce_bw<__half>((__half *)dlogits, (const __half *)logits,
                                                       target, lse, dloss, rows, vocab, vec, st));
        case LS_BF16:
            return from_cuda(lsr::launch_ce_bw<__nv_bfloat16>(
                (__nv_bfloat16 *)dlogits, (const __nv_bfloat16 *)logits, target, lse, dloss, rows,
                vocab, vec, st));
    }
    return LS_ERR_UNSUPPORTED;
}

}  // extern "C"
