// dispatch.cuh -- launch-time choice of the compile-time row shape.
//
// As the L10 page ("Technique 2", slides 24-26) describes for LightSeq, the
// number of threads per row (TPR) and of 16-byte chunks per thread (CPT) are
// template parameters; the launcher picks the smallest instantiation whose
// capacity covers the row.  The HW4 page's ITERATIONS buckets for the softmax
// backward (row lengths 32 ... 2048) all land on register-resident buckets
// here: 16-bit storage holds up to 1024 elements in one warp (32 threads x 4
// chunks x 8 elements), and longer rows use several warps per row, up to
// 16384 elements, with the looped path beyond.
#pragma once

#include "launch.h"
#include "layernorm.cuh"
#include "softmax.cuh"

#include <atomic>

namespace lsr {

// Buckets: threads per row up to a cap chosen so that the launch bounds
// (TPR threads per block) leave enough registers for CPT chunks per thread
// without spilling.  Longer rows take the looped path.
constexpr int kSoftmaxFwMaxCpt = 4;  // chunks per thread, softmax forward buckets
constexpr int kSoftmaxFwMaxTpr = 512;  // 16-bit: 16384 keys per row in registers
// The backward holds both y and dout: at most four chunks per thread (80
// registers), two or more warps per row beyond 128 chunks (2048 keys of
// 16-bit storage: 32 x 8 took 154 registers, one block per SM, 0.88 of peak;
// 64 x 4 reaches the copy peak)
constexpr int kSoftmaxBwMaxCpt = 4;  // chunks per thread, softmax backward buckets
constexpr int kSoftmaxBwMaxTpr = 512;  // 16-bit: 16384 keys per row in registers
constexpr int kLnMaxCpt = 4;         // chunks per thread, LayerNorm buckets
constexpr int kLnMaxTpr = 512;       // 16-bit: 16384 features per row in registers
constexpr int kLoopWarpRowMax = 2048;  // looped path: one warp per row up to here

template <int TPR>
constexpr int block_threads() { return TPR <= 32 ? 256 : TPR; }
template <int TPR>
constexpr int rows_per_block() { return TPR <= 32 ? 256 / TPR : 1; }

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

inline int next_pow2(int64_t v) {
    int p = 1;
    while (p < v) p <<= 1;
    return p;
}

// Bucket for a row of nchunk 16-byte chunks; false if it needs the looped path.
inline bool pick_bucket(int64_t nchunk, int maxcpt, int maxtpr, int *tpr, int *cpt) {
    if (nchunk <= 32) {
        *tpr = next_pow2(nchunk < 1 ? 1 : nchunk);
        *cpt = 1;
    } else if (nchunk <= 32 * maxcpt) {
        *tpr = 32;
        *cpt = (int)ceil_div(nchunk, 32);
    } else {
        int64_t t = next_pow2(ceil_div(nchunk, maxcpt));
        if (t > maxtpr) return false;
        *tpr = (int)t;
        *cpt = maxcpt;
    }
    return true;
}

constexpr int kMaxDevices = 64;

// Bucket of the pipelined row kernels: as many chunks per thread as allowed
// (maxcpt) and as few threads per row as that permits, so that per-row costs
// (the shuffle reductions, the pipeline bookkeeping) are shared by as many
// elements as possible and short rows pack several rows into one warp.
inline bool pick_bucket_dense(int64_t nchunk, int maxcpt, int maxtpr, int *tpr, int *cpt) {
    if (nchunk <= maxcpt) {
        *tpr = 1;
        *cpt = (int)(nchunk < 1 ? 1 : nchunk);
        return true;
    }
    const int64_t t = next_pow2(ceil_div(nchunk, maxcpt));
    if (t > maxtpr) return false;
    *tpr = (int)t;
    *cpt = (int)ceil_div(nchunk, t);
    return true;
}

// Launch with programmatic stream serialisation (see pdl_begin): the kernel
// may be scheduled while the previous kernel in the stream finishes.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, static_cast<KArgs>(args)...);
}

// Resident blocks per SM of one kernel instantiation with `smem` bytes of
// dynamic shared memory (queried once).  The opt-in to more than 48 KB per
// block is set once per device before the first launch there, for any
// dynamic size: the 48 KB default counts the kernel's static shared memory
// too, so a dynamic size just under it can already need the opt-in.
template <auto K>
void ensure_dynamic_smem(size_t smem) {
    static std::atomic<int> configured[kMaxDevices];
    int dev = 0;
    if (smem > 0 && cudaGetDevice(&dev) == cudaSuccess && dev >= 0 &&
        dev < kMaxDevices && !configured[dev].load(std::memory_order_acquire)) {
        cudaFuncSetAttribute(K, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        configured[dev].store(1, std::memory_order_release);
    }
}

template <auto K>
int occupancy_per_sm(int block, size_t smem) {
    ensure_dynamic_smem<K>(smem);
    static const int occ = [block, smem] {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, K, block, smem) != cudaSuccess ||
            n < 1)
            n = 1;
        return n;
    }();
    return occ;
}

// Persistent launch: as many blocks as fit on the GPU at once (never more than
// there is work for); the kernels loop over their rows.
template <auto K, typename... Args>
cudaError_t launch_persistent(int block, size_t smem, int64_t work_blocks, cudaStream_t st,
                              Args... args) {
    const int64_t cap = (int64_t)device_sm_count() * occupancy_per_sm<K>(block, smem);
    const int64_t grid = work_blocks < cap ? (work_blocks < 1 ? 1 : work_blocks) : cap;
    return launch_pdl(K, dim3((unsigned)grid), dim3(block), smem, st, args...);
}

// Stages of the cp.async row pipelines (rows in flight per row group = S - 1).
// LayerNorm: rows of up to 4 KB keep three (forward) or two (input gradient)
// rows in flight -- inside a layer's pass, where they often find their input
// warm in L2, that measured about 1 us per encoder pass faster -- and wider,
// HBM-bound rows keep one, which measured 3-5 % faster there (GB300, bf16,
// 16384 rows: forward 90.7 -> 87.5 us at 8192 features, input gradient
// 126.2 -> 119.7 us).  The fused backward keeps one at every width (75.2 ->
// 71.9 us at 4096 features).
constexpr int kSoftmaxFwStages = 4;
template <int TPR, int CPT>
constexpr int ln_fw_stages() { return TPR * CPT * 16 <= 4096 ? 4 : 2; }
template <int TPR, int CPT>
constexpr int ln_dinp_stages() { return TPR * CPT * 16 <= 4096 ? 3 : 2; }
constexpr int kLnBwFusedStages = 2;

// ----------------------------------------------------------------------------
// softmax
// ----------------------------------------------------------------------------
// (threads per row, chunks per thread) pairs pick_bucket_dense can return
// with at most 4 chunks per thread.
#define LSR_DENSE4_BUCKETS(X)                                                   \
    X(1, 1) X(1, 2) X(1, 3) X(1, 4) X(2, 3) X(2, 4) X(4, 3) X(4, 4) X(8, 3)      \
    X(8, 4) X(16, 3) X(16, 4) X(32, 3) X(32, 4) X(64, 3) X(64, 4) X(128, 3)      \
    X(128, 4) X(256, 3) X(256, 4) X(512, 3) X(512, 4)
#define LSR_SOFTMAX_FW_BUCKETS(X) LSR_DENSE4_BUCKETS(X)
#define LSR_SOFTMAX_BW_BUCKETS(X)                                               \
    X(1, 1) X(2, 1) X(4, 1) X(8, 1) X(16, 1) X(32, 1) X(32, 2) X(32, 3) X(32, 4) \
    X(64, 4) X(128, 4) X(256, 4) X(512, 4)
#define LSR_LN_BUCKETS(X) LSR_DENSE4_BUCKETS(X)

template <typename T>
cudaError_t launch_softmax_fw(T *out, const T *inp, const T *mask, int64_t rows,
                              int64_t rows_per_batch, int64_t Tq, int64_t Tk,
                              int causal, int64_t qoff, float scale, bool vec, cudaStream_t st) {
    constexpr int V = Traits<T>::kVec;
    int tpr = 0, cpt = 0;
    if (vec && rows <= INT32_MAX &&
        pick_bucket_dense(Tk / V, kSoftmaxFwMaxCpt, kSoftmaxFwMaxTpr, &tpr, &cpt)) {
#define X(TPR_, CPT_)                                                                   \
    if (tpr == TPR_ && cpt == CPT_) {                                                   \
        if (scale == 1.0f)                                                              \
            return launch_persistent<softmax_fw_vec<T, TPR_, CPT_, kSoftmaxFwStages, false>>( \
                block_threads<TPR_>(), softmax_fw_smem<TPR_, CPT_, kSoftmaxFwStages>(),    \
                ceil_div(rows, rows_per_block<TPR_>()), st, out, inp, mask, rows,           \
                rows_per_batch, Tq, (int)Tk, causal, qoff, scale);                          \
        return launch_persistent<softmax_fw_vec<T, TPR_, CPT_, kSoftmaxFwStages, true>>(  \
            block_threads<TPR_>(), softmax_fw_smem<TPR_, CPT_, kSoftmaxFwStages>(),        \
            ceil_div(rows, rows_per_block<TPR_>()), st, out, inp, mask, rows,               \
            rows_per_batch, Tq, (int)Tk, causal, qoff, scale);                              \
    }
        LSR_SOFTMAX_FW_BUCKETS(X)
#undef X
    }
    if (Tk <= kLoopWarpRowMax)
        return launch_persistent<softmax_fw_loop<T, 32>>(256, 0, ceil_div(rows, 8), st, out, inp,
                                                         mask, rows, rows_per_batch, Tq, Tk,
                                                         causal, qoff, scale);
    return launch_persistent<softmax_fw_loop<T, 256>>(256, 0, rows, st, out, inp, mask, rows,
                                                      rows_per_batch, Tq, Tk, causal, qoff,
                                                      scale);
}

template <typename T>
cudaError_t launch_softmax_bw(T *dinp, const T *dout, const T *y, int64_t rows,
                              int64_t Tk, bool vec, cudaStream_t st) {
    constexpr int V = Traits<T>::kVec;
    int tpr = 0, cpt = 0;
    if (vec && pick_bucket(Tk / V, kSoftmaxBwMaxCpt, kSoftmaxBwMaxTpr, &tpr, &cpt)) {
#define X(TPR_, CPT_)                                                                   \
    if (tpr == TPR_ && cpt == CPT_)                                                     \
        return launch_persistent<softmax_bw_vec<T, TPR_, CPT_>>(                        \
            block_threads<TPR_>(), 0, ceil_div(rows, rows_per_block<TPR_>()), st, dinp,     \
            dout, y, rows, (int)Tk);
        LSR_SOFTMAX_BW_BUCKETS(X)
#undef X
    }
    if (Tk <= kLoopWarpRowMax)
        return launch_persistent<softmax_bw_loop<T, 32>>(256, 0, ceil_div(rows, 8), st, dinp, dout,
                                                         y, rows, Tk);
    return launch_persistent<softmax_bw_loop<T, 256>>(256, 0, rows, st, dinp, dout, y, rows, Tk);
}

template <typename T>
cudaError_t launch_softmax_bw_masked(T *dinp, const T *dout, const T *y, const T *mask,
                                     int64_t rows, int64_t rows_per_batch, int64_t Tq,
                                     int64_t Tk, int causal, int64_t qoff, float scale, bool vec,
                                     cudaStream_t st) {
    constexpr int V = Traits<T>::kVec;
    int tpr = 0, cpt = 0;
    if (vec && rows <= INT32_MAX &&
        pick_bucket(Tk / V, kSoftmaxBwMaxCpt, kSoftmaxBwMaxTpr, &tpr, &cpt)) {
#define X(TPR_, CPT_)                                                                   \
    if (tpr == TPR_ && cpt == CPT_)                                                     \
        return launch_persistent<softmax_bw_masked_vec<T, TPR_, CPT_>>(                 \
            block_threads<TPR_>(), 0, ceil_div(rows, rows_per_block<TPR_>()), st, dinp,     \
            dout, y, mask, rows, rows_per_batch, Tq, (int)Tk, causal, qoff, scale);
        LSR_SOFTMAX_BW_BUCKETS(X)
#undef X
    }
    if (Tk <= kLoopWarpRowMax)
        return launch_persistent<softmax_bw_masked_loop<T, 32>>(
            256, 0, ceil_div(rows, 8), st, dinp, dout, y, mask, rows, rows_per_batch, Tq, Tk,
            causal, qoff, scale);
    return launch_persistent<softmax_bw_masked_loop<T, 256>>(
        256, 0, rows, st, dinp, dout, y, mask, rows, rows_per_batch, Tq, Tk, causal, qoff, scale);
}

// ----------------------------------------------------------------------------
// LayerNorm
// ----------------------------------------------------------------------------
template <typename T, bool RMS>
cudaError_t launch_norm_fw(T *y, float *mean, float *rstd, const T *x, const T *gamma,
                           const T *beta, int64_t rows, int64_t N, float eps, bool vec,
                           cudaStream_t st) {
    constexpr int V = Traits<T>::kVec;
    int tpr = 0, cpt = 0;
    if (vec && pick_bucket_dense(N / V, kLnMaxCpt, kLnMaxTpr, &tpr, &cpt)) {
#define X(TPR_, CPT_)                                                                     \
    if (tpr == TPR_ && cpt == CPT_)                                                       \
        return launch_persistent<ln_fw_vec<T, TPR_, CPT_, ln_fw_stages<TPR_, CPT_>(), RMS>>(  \
            block_threads<TPR_>(), ln_smem<TPR_, CPT_, ln_fw_stages<TPR_, CPT_>(), 1, 1>(),   \
            ceil_div(rows, rows_per_block<TPR_>()), st, y, mean, rstd, x, gamma, beta, rows,  \
            (int)N, eps);
        LSR_LN_BUCKETS(X)
#undef X
    }
    if (N <= kLoopWarpRowMax)
        return launch_persistent<ln_fw_loop<T, 32, RMS>>(256, 0, ceil_div(rows, 8), st, y, mean, rstd, x,
                                                    gamma, beta, rows, N, eps);
    return launch_persistent<ln_fw_loop<T, 256, RMS>>(256, 0, rows, st, y, mean, rstd, x, gamma, beta,
                                                 rows, N, eps);
}

template <typename T>
cudaError_t launch_ln_fw(T *y, float *mean, float *rstd, const T *x, const T *gamma,
                         const T *beta, int64_t rows, int64_t N, float eps, bool vec,
                         cudaStream_t st) {
    return launch_norm_fw<T, false>(y, mean, rstd, x, gamma, beta, rows, N, eps, vec, st);
}

template <typename T>
cudaError_t launch_rms_fw(T *y, float *rstd, const T *x, const T *gamma, int64_t rows, int64_t N,
                          float eps, bool vec, cudaStream_t st) {
    return launch_norm_fw<T, true>(y, nullptr, rstd, x, gamma, nullptr, rows, N, eps, vec, st);
}

template <typename T, bool RMS>
cudaError_t launch_norm_dinp(T *dx, const T *dy, const T *x, const T *gamma,
                             const float *mean, const float *rstd, int64_t rows,
                             int64_t N, bool vec, cudaStream_t st) {
    constexpr int V = Traits<T>::kVec;
    int tpr = 0, cpt = 0;
    if (vec && pick_bucket_dense(N / V, kLnMaxCpt, kLnMaxTpr, &tpr, &cpt)) {
#define X(TPR_, CPT_)                                                                       \
    if (tpr == TPR_ && cpt == CPT_)                                                         \
        return launch_persistent<ln_dinp_vec<T, TPR_, CPT_, ln_dinp_stages<TPR_, CPT_>(), RMS>>( \
            block_threads<TPR_>(), ln_smem<TPR_, CPT_, ln_dinp_stages<TPR_, CPT_>(), 2, 2>(),  \
            ceil_div(rows, rows_per_block<TPR_>()), st, dx, dy, x, gamma, mean, rstd, rows,     \
            (int)N);
        LSR_LN_BUCKETS(X)
#undef X
    }
    if (N <= kLoopWarpRowMax)
        return launch_persistent<ln_dinp_loop<T, 32, RMS>>(256, 0, ceil_div(rows, 8), st, dx, dy, x,
                                                      gamma, mean, rstd, rows, N);
    return launch_persistent<ln_dinp_loop<T, 256, RMS>>(256, 0, rows, st, dx, dy, x, gamma, mean, rstd,
                                                   rows, N);
}

template <typename T>
cudaError_t launch_ln_dinp(T *dx, const T *dy, const T *x, const T *gamma,
                           const float *mean, const float *rstd, int64_t rows,
                           int64_t N, bool vec, cudaStream_t st) {
    return launch_norm_dinp<T, false>(dx, dy, x, gamma, mean, rstd, rows, N, vec, st);
}

template <typename T>
cudaError_t launch_rms_dinp(T *dx, const T *dy, const T *x, const T *gamma, const float *rstd,
                            int64_t rows, int64_t N, bool vec, cudaStream_t st) {
    return launch_norm_dinp<T, true>(dx, dy, x, gamma, nullptr, rstd, rows, N, vec, st);
}

template <typename T>
cudaError_t launch_ln_dgdb(float *dgamma, float *dbeta, const T *dy, const T *x,
                           const float *mean, const float *rstd, int64_t rows,
                           int64_t N, float *part, bool vec, cudaStream_t st) {
    const int64_t rpc = dgdb_rows_per_chunk(rows, N);
    const int64_t nchunks = dgdb_num_chunks(rows, N);
    if (nchunks > 0) {
        if (nchunks > 65535) return cudaErrorInvalidConfiguration;  // not reachable (rpc grows)
        if (vec) {
            constexpr int V = Traits<T>::kVec;
            dim3 grid((unsigned)ceil_div(N, 32 * V), (unsigned)nchunks);
            // Ring depth: four stages (six rows in flight per warp) for rows of
            // up to 4 KB, which inside a layer's backward usually follow the
            // input gradient's read of the same dy and x (warm in L2; the
            // encoder pass measured 1.7 us faster than with two); two stages
            // for wider rows (cold, HBM-bound: 2-4 % faster than four).
            cudaError_t e;
            if (N * (int64_t)sizeof(T) <= 4096) {
                constexpr size_t smem = ln_dgdb_staged_smem<4>();
                ensure_dynamic_smem<ln_dgdb_staged<T, 4>>(smem);
                e = launch_pdl(ln_dgdb_staged<T, 4>, grid, dim3(kDgdbWarps * 32), smem, st, part,
                               dy, x, mean, rstd, rows, N, rpc);
            } else {
                constexpr size_t smem = ln_dgdb_staged_smem<2>();
                ensure_dynamic_smem<ln_dgdb_staged<T, 2>>(smem);
                e = launch_pdl(ln_dgdb_staged<T, 2>, grid, dim3(kDgdbWarps * 32), smem, st, part,
                               dy, x, mean, rstd, rows, N, rpc);
            }
            if (e != cudaSuccess) return e;
        } else {
            dim3 grid((unsigned)ceil_div(N, 32), (unsigned)nchunks);
            cudaError_t e = launch_pdl(ln_dgdb_partial<T>, grid, dim3(kDgdbWarps * 32), 0, st,
                                       part, dy, x, mean, rstd, rows, N, rpc);
            if (e != cudaSuccess) return e;
        }
    }
    return launch_pdl(ln_dgdb_final, dim3((unsigned)ceil_div(N, kFinalCols)),
                      dim3(kFinalCols * kFinalLanes), 0, st, dgamma, dbeta,
                      (const float *)part, nchunks, N);
}

// Fused LayerNorm backward: a fixed cut of the rows into ln_bw_fused_chunks
// chunks (at most 456), one block per chunk.  At most two 16-byte chunks per
// thread: the per-column accumulators then fit in registers next to the row
// (one chunk per thread measured slower: more threads and barriers per row).
#define LSR_FUSED_BW_BUCKETS(X)                                                 \
    X(1, 1) X(1, 2) X(2, 2) X(4, 2) X(8, 2) X(16, 2) X(32, 2) X(32, 3) X(64, 2)  \
    X(64, 3) X(128, 2) X(128, 3) X(128, 4) X(256, 2) X(256, 3) X(256, 4) X(512, 3) \
    X(512, 4)
constexpr int kFusedMaxCpt = 2;


template <typename T>
cudaError_t launch_ln_bw_fused(T *dx, float *dgamma, float *dbeta, const T *dy, const T *x,
                               const T *gamma, const float *mean, const float *rstd,
                               int64_t rows, int64_t N, float *part, bool vec, cudaStream_t st) {
    constexpr int V = Traits<T>::kVec;
    int tpr = 0, cpt = 0;
    // Chunks per thread: two (the row's g and xhat held for the epilogue) up
    // to 256 vectors; four above (g and xhat unpacked again from the staged
    // row), where 256 threads with four chunks beat 512 with two (8192
    // features on GB300: 179 -> 143 us).  From 64 vectors up, the bucket of
    // up to four chunks is also taken when it covers the row with fewer idle
    // slots (768 features: 32 x 3 instead of 64 x 2, 20.8 -> 17.2 us).
    const int64_t nvec = N / V;
    int tpr2 = 0, cpt2 = 0, tpr4 = 0, cpt4 = 0;
    const bool ok2 = pick_bucket_dense(nvec, kFusedMaxCpt, kLnMaxTpr, &tpr2, &cpt2);
    const bool ok4 = pick_bucket_dense(nvec, kLnMaxCpt, kLnMaxTpr, &tpr4, &cpt4);
    const bool four = nvec > 256 ||
                      (nvec >= 64 && ok4 && (!ok2 || tpr4 * cpt4 < tpr2 * cpt2));
    const bool picked = four ? ok4 : ok2;
    tpr = four ? tpr4 : tpr2;
    cpt = four ? cpt4 : cpt2;
    if (rows > 0 && vec && picked) {
        int64_t nparts = 0;
        cudaError_t e = cudaErrorInvalidValue;
#define X(TPR_, CPT_)                                                                       \
    if (tpr == TPR_ && cpt == CPT_) {                                                       \
        const int64_t rpc = ceil_div(rows, (int64_t)ln_bw_fused_chunks<TPR_, CPT_>());      \
        nparts = ceil_div(rows, rpc);                                                       \
        constexpr size_t smem = ln_bw_fused_smem<TPR_, CPT_, kLnBwFusedStages, V>();            \
        ensure_dynamic_smem<ln_bw_fused_vec<T, TPR_, CPT_, kLnBwFusedStages>>(smem);            \
        e = launch_pdl(ln_bw_fused_vec<T, TPR_, CPT_, kLnBwFusedStages>,                        \
                       dim3((unsigned)nparts),                                               \
                       dim3(ln_bw_fused_block<TPR_>()), smem, st, dx, part, dy, x, gamma,    \
                       mean, rstd, rows, (int)N, rpc);                                       \
    }
        LSR_FUSED_BW_BUCKETS(X)
#undef X
        if (e != cudaSuccess) return e;
        return launch_pdl(ln_dgdb_final, dim3((unsigned)ceil_div(N, kFinalCols)),
                          dim3(kFinalCols * kFinalLanes), 0, st, dgamma, dbeta,
                          (const float *)part, nparts, N);
    }
    // rows that take the scalar path, or wider than 4 * 512 vectors: the two
    // kernels one after the other
    cudaError_t e = launch_ln_dinp<T>(dx, dy, x, gamma, mean, rstd, rows, N, vec, st);
    if (e != cudaSuccess) return e;
    return launch_ln_dgdb<T>(dgamma, dbeta, dy, x, mean, rstd, rows, N, part, vec, st);
}

// RMSNorm gamma gradient: the LayerNorm column sums with mean 0 and no dbeta.
template <typename T>
cudaError_t launch_rms_dgamma(float *dgamma, const T *dy, const T *x, const float *rstd,
                              int64_t rows, int64_t N, float *part, bool vec, cudaStream_t st) {
    return launch_ln_dgdb<T>(dgamma, nullptr, dy, x, nullptr, rstd, rows, N, part, vec, st);
}

#define LSR_INSTANTIATE(T)                                                                      \
    template cudaError_t launch_softmax_fw<T>(T *, const T *, const T *, int64_t, int64_t,     \
                                              int64_t, int64_t, int, int64_t, float, bool,     \
                                              cudaStream_t);                                   \
    template cudaError_t launch_softmax_bw_masked<T>(T *, const T *, const T *, const T *,     \
                                                     int64_t, int64_t, int64_t, int64_t, int,  \
                                                     int64_t, float, bool, cudaStream_t);      \
    template cudaError_t launch_softmax_bw<T>(T *, const T *, const T *, int64_t, int64_t,     \
                                              bool, cudaStream_t);                             \
    template cudaError_t launch_ln_fw<T>(T *, float *, float *, const T *, const T *,          \
                                         const T *, int64_t, int64_t, float, bool,             \
                                         cudaStream_t);                                        \
    template cudaError_t launch_ln_dinp<T>(T *, const T *, const T *, const T *,               \
                                           const float *, const float *, int64_t, int64_t,     \
                                           bool, cudaStream_t);                                \
    template cudaError_t launch_ln_dgdb<T>(float *, float *, const T *, const T *,             \
                                           const float *, const float *, int64_t, int64_t,     \
                                           float *, bool, cudaStream_t);                       \
    template cudaError_t launch_ln_bw_fused<T>(T *, float *, float *, const T *, const T *,     \
                                               const T *, const float *, const float *,         \
                                               int64_t, int64_t, float *, bool, cudaStream_t);  \
    template cudaError_t launch_rms_fw<T>(T *, float *, const T *, const T *, int64_t, int64_t, \
                                          float, bool, cudaStream_t);                          \
    template cudaError_t launch_rms_dinp<T>(T *, const T *, const T *, const T *,              \
                                            const float *, int64_t, int64_t, bool,             \
                                            cudaStream_t);                                     \
    template cudaError_t launch_rms_dgamma<T>(float *, const T *, const T *, const float *,    \
                                              int64_t, int64_t, float *, bool, cudaStream_t);

}  // namespace lsr
