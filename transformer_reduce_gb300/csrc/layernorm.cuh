// layernorm.cuh -- LayerNorm forward, input-gradient and gamma/beta-gradient
// kernels (sm_103a).
//
// The operations are those of the page "CMU 11-868 HW4：把 Softmax 與
// LayerNorm 寫成 CUDA 融合 kernel" (section 題目結構與配分, Problems 2.1 and
// 2.2: eps = 1e-8 inside the root, 128-bit vector access, the backward split
// into an input-gradient kernel and a cross-row gamma/beta kernel) and of
// "CMU 11-868 L10: Accelerating Transformers on GPUs, and Where LightSeq
// Finds the Time" (section "Technique 2", slide 21: mean and mean of squares
// reduced together, one synchronisation instead of two; slide 22: the
// backward's two sums reduced together).
//
// GB300 design: the same row-group mapping as the softmax kernels (TPR
// threads per row, CPT 16-byte chunks per thread held in registers, one HBM
// read and one write per element, persistent grid).  gamma and beta are
// re-read per row through the read-only cache (they stay resident in L1/L2).
// The gamma/beta gradient is a column reduction over rows: column tiles x
// fixed row chunks, FP32 partial sums per chunk in a caller-provided
// workspace, then a fixed-order sum over the chunks.  The chunking depends
// only on (rows, hidden), so the result is bitwise reproducible.
#pragma once

#include "ls_device.cuh"

namespace lsr {

// ----------------------------------------------------------------------------
// Forward, register resident.  The two statistics come from ONE fused
// reduction of sum(x') and sum(x'^2) with x' = x - x0 (x0 = the row's first
// element): var = mean(x'^2) - mean(x')^2 is the one-pass form, and the shift
// removes its cancellation when |mean| >> std (it is exact for constant rows).
// ----------------------------------------------------------------------------
template <typename T, int TPR, int CPT>
__global__ void __launch_bounds__(TPR <= 32 ? 256 : TPR)
ln_fw_vec(T *y, float *mean, float *rstd, const T *x, const T *gamma,
          const T *beta, int64_t rows, int N, float eps) {
    using Tr = Traits<T>;
    constexpr int V = Tr::kVec;
    constexpr int BLOCK = TPR <= 32 ? 256 : TPR;
    constexpr int G = BLOCK / TPR;
    __shared__ float red[TPR > 32 ? 64 : 1];

    const int lane = threadIdx.x % TPR;
    const int grp = threadIdx.x / TPR;
    const int nchunk = N / V;
    const float invN = 1.f / (float)N;

    for (int64_t base = (int64_t)blockIdx.x * G; base < rows;
         base += (int64_t)gridDim.x * G) {
        const int64_t row = base + grp;
        const bool valid = row < rows;
        const T *xrow = x + row * (int64_t)N;
        const float x0 = valid ? Tr::load1_cached(xrow) : 0.f;

        float d[CPT][V];
        float s1 = 0.f, s2 = 0.f;
#pragma unroll
        for (int k = 0; k < CPT; ++k) {
            const int c = k * TPR + lane;
            if (valid && c < nchunk) {
                Tr::unpack(ld_stream16(xrow + c * V), d[k]);
#pragma unroll
                for (int e = 0; e < V; ++e) {
                    d[k][e] -= x0;
                    s1 += d[k][e];
                    s2 = fmaf(d[k][e], d[k][e], s2);
                }
            }
        }
        group_sum2<TPR>(s1, s2, red);
        const float m1 = s1 * invN;
        const float var = fmaxf(s2 * invN - m1 * m1, 0.f);
        const float rs = rsqrtf(var + eps);

        T *yrow = y + row * (int64_t)N;
#pragma unroll
        for (int k = 0; k < CPT; ++k) {
            const int c = k * TPR + lane;
            if (valid && c < nchunk) {
                float gv[V], bv[V], yv[V];
                Tr::unpack(ld_cached16(gamma + c * V), gv);
                Tr::unpack(ld_cached16(beta + c * V), bv);
#pragma unroll
                for (int e = 0; e < V; ++e)
                    yv[e] = fmaf((d[k][e] - m1) * rs, gv[e], bv[e]);
                st_stream16(yrow + c * V, Tr::pack(yv));
            }
        }
        if (valid && lane == 0) {
            mean[row] = x0 + m1;
            rstd[row] = rs;
        }
    }
}

// ----------------------------------------------------------------------------
// Input gradient, register resident.  g = gamma * dy, xhat = (x - mean)*rstd;
// S1 = sum g and S2 = sum g*xhat in one fused reduction; then
// dx = rstd * (g - S1/N - xhat * S2/N).
// ----------------------------------------------------------------------------
template <typename T, int TPR, int CPT>
__global__ void __launch_bounds__(TPR <= 32 ? 256 : TPR)
ln_dinp_vec(T *dx, const T *dy, const T *x, const T *gamma, const float *mean,
            const float *rstd, int64_t rows, int N) {
    using Tr = Traits<T>;
    constexpr int V = Tr::kVec;
    constexpr int BLOCK = TPR <= 32 ? 256 : TPR;
    constexpr int G = BLOCK / TPR;
    __shared__ float red[TPR > 32 ? 64 : 1];

    const int lane = threadIdx.x % TPR;
    const int grp = threadIdx.x / TPR;
    const int nchunk = N / V;
    const float invN = 1.f / (float)N;

    for (int64_t base = (int64_t)blockIdx.x * G; base < rows;
         base += (int64_t)gridDim.x * G) {
        const int64_t row = base + grp;
        const bool valid = row < rows;
        const int64_t off = row * (int64_t)N;
        const float mu = valid ? __ldg(mean + row) : 0.f;
        const float rs = valid ? __ldg(rstd + row) : 0.f;

        float g[CPT][V], xh[CPT][V];
        float s1 = 0.f, s2 = 0.f;
#pragma unroll
        for (int k = 0; k < CPT; ++k) {
            const int c = k * TPR + lane;
            if (valid && c < nchunk) {
                float gv[V];
                Tr::unpack(ld_stream16(dy + off + c * V), g[k]);
                Tr::unpack(ld_stream16(x + off + c * V), xh[k]);
                Tr::unpack(ld_cached16(gamma + c * V), gv);
#pragma unroll
                for (int e = 0; e < V; ++e) {
                    // rounded product (never fused into a later add), so that
                    // S1 sums exactly the g the epilogue uses
                    g[k][e] = __fmul_rn(g[k][e], gv[e]);
                    xh[k][e] = (xh[k][e] - mu) * rs;
                    s1 += g[k][e];
                    s2 = fmaf(g[k][e], xh[k][e], s2);
                }
            }
        }
        group_sum2<TPR>(s1, s2, red);
        const float a = s1 * invN, b = s2 * invN;
#pragma unroll
        for (int k = 0; k < CPT; ++k) {
            const int c = k * TPR + lane;
            if (valid && c < nchunk) {
                float dv[V];
#pragma unroll
                for (int e = 0; e < V; ++e) dv[e] = rs * (g[k][e] - a - xh[k][e] * b);
                st_stream16(dx + off + c * V, Tr::pack(dv));
            }
        }
    }
}

// ----------------------------------------------------------------------------
// Looped variants (scalar accesses, any alignment, any row length).
// ----------------------------------------------------------------------------
template <typename T, int TPR>
__global__ void __launch_bounds__(TPR <= 32 ? 256 : TPR)
ln_fw_loop(T *y, float *mean, float *rstd, const T *x, const T *gamma,
           const T *beta, int64_t rows, int64_t N, float eps) {
    using Tr = Traits<T>;
    constexpr int BLOCK = TPR <= 32 ? 256 : TPR;
    constexpr int G = BLOCK / TPR;
    __shared__ float red[TPR > 32 ? 64 : 1];
    const int lane = threadIdx.x % TPR;
    const int grp = threadIdx.x / TPR;
    const float invN = 1.f / (float)N;

    for (int64_t base = (int64_t)blockIdx.x * G; base < rows;
         base += (int64_t)gridDim.x * G) {
        const int64_t row = base + grp;
        const bool valid = row < rows;
        const T *xrow = x + row * N;
        const float x0 = valid ? Tr::load1_cached(xrow) : 0.f;
        float s1 = 0.f, s2 = 0.f;
        if (valid)
            for (int64_t j = lane; j < N; j += TPR) {
                const float d = Tr::load1(xrow + j) - x0;
                s1 += d;
                s2 = fmaf(d, d, s2);
            }
        group_sum2<TPR>(s1, s2, red);
        const float m1 = s1 * invN;
        const float var = fmaxf(s2 * invN - m1 * m1, 0.f);
        const float rs = rsqrtf(var + eps);
        if (valid) {
            T *yrow = y + row * N;
            for (int64_t j = lane; j < N; j += TPR) {
                const float d = Tr::load1(xrow + j) - x0;
                Tr::store1(yrow + j, fmaf((d - m1) * rs, Tr::load1_cached(gamma + j),
                                          Tr::load1_cached(beta + j)));
            }
            if (lane == 0) {
                mean[row] = x0 + m1;
                rstd[row] = rs;
            }
        }
    }
}

template <typename T, int TPR>
__global__ void __launch_bounds__(TPR <= 32 ? 256 : TPR)
ln_dinp_loop(T *dx, const T *dy, const T *x, const T *gamma, const float *mean,
             const float *rstd, int64_t rows, int64_t N) {
    using Tr = Traits<T>;
    constexpr int BLOCK = TPR <= 32 ? 256 : TPR;
    constexpr int G = BLOCK / TPR;
    __shared__ float red[TPR > 32 ? 64 : 1];
    const int lane = threadIdx.x % TPR;
    const int grp = threadIdx.x / TPR;
    const float invN = 1.f / (float)N;

    for (int64_t base = (int64_t)blockIdx.x * G; base < rows;
         base += (int64_t)gridDim.x * G) {
        const int64_t row = base + grp;
        const bool valid = row < rows;
        const int64_t off = row * N;
        const float mu = valid ? __ldg(mean + row) : 0.f;
        const float rs = valid ? __ldg(rstd + row) : 0.f;
        float s1 = 0.f, s2 = 0.f;
        if (valid)
            for (int64_t j = lane; j < N; j += TPR) {
                // rounded product (never fused), identical in both passes
                const float g = __fmul_rn(Tr::load1_cached(gamma + j), Tr::load1(dy + off + j));
                const float xh = (Tr::load1(x + off + j) - mu) * rs;
                s1 += g;
                s2 = fmaf(g, xh, s2);
            }
        group_sum2<TPR>(s1, s2, red);
        const float a = s1 * invN, b = s2 * invN;
        if (valid)
            for (int64_t j = lane; j < N; j += TPR) {
                const float g = __fmul_rn(Tr::load1_cached(gamma + j), Tr::load1(dy + off + j));
                const float xh = (Tr::load1(x + off + j) - mu) * rs;
                Tr::store1(dx + off + j, rs * (g - a - xh * b));
            }
    }
}

// ----------------------------------------------------------------------------
// gamma / beta gradient, stage 1: partial column sums of one row chunk.
// Block = 8 warps.  A warp spans one column tile (32 lanes x V columns: 16
// bytes per lane, 512 contiguous bytes per row for 16-bit storage); warp w
// takes rows w, w+8, ... of the chunk.  The 8 per-warp sums are then added in
// warp order through shared memory and written to
//   part[(chunk * 2 + 0) * N + col] (dgamma),  part[(chunk * 2 + 1) * N + col] (dbeta).
// V = 1 is the scalar path (any alignment).
// ----------------------------------------------------------------------------
constexpr int kDgdbWarps = 8;

template <typename T, int V>
__global__ void __launch_bounds__(kDgdbWarps * 32)
ln_dgdb_partial(float *part, const T *dy, const T *x, const float *mean,
                const float *rstd, int64_t rows, int64_t N, int64_t rows_per_chunk) {
    using Tr = Traits<T>;
    constexpr int CT = 32 * V;  // columns per tile
    __shared__ float sg[kDgdbWarps][CT];
    __shared__ float sb[kDgdbWarps][CT];

    const int lane = threadIdx.x & 31;
    const int w = threadIdx.x >> 5;
    const int64_t col0 = (int64_t)blockIdx.x * CT + lane * V;
    const int64_t chunk = blockIdx.y;
    const int64_t r0 = chunk * rows_per_chunk;
    const int64_t r1 = min(rows, r0 + rows_per_chunk);

    float ag[V], ab[V];
#pragma unroll
    for (int e = 0; e < V; ++e) ag[e] = ab[e] = 0.f;

    if (col0 < N) {
        int64_t r = r0 + w;
        // Four rows in flight per warp per iteration.
        for (; r + 3 * kDgdbWarps < r1; r += 4 * kDgdbWarps) {
            float dv[4][V], xv[4][V], mu[4], rs[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int64_t rr = r + u * kDgdbWarps;
                mu[u] = __ldg(mean + rr);
                rs[u] = __ldg(rstd + rr);
                if constexpr (V == 1) {
                    dv[u][0] = Tr::load1(dy + rr * N + col0);
                    xv[u][0] = Tr::load1(x + rr * N + col0);
                } else {
                    Tr::unpack(ld_stream16(dy + rr * N + col0), dv[u]);
                    Tr::unpack(ld_stream16(x + rr * N + col0), xv[u]);
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int e = 0; e < V; ++e) {
                    ag[e] = fmaf(dv[u][e], (xv[u][e] - mu[u]) * rs[u], ag[e]);
                    ab[e] += dv[u][e];
                }
        }
        for (; r < r1; r += kDgdbWarps) {
            float dv[V], xv[V];
            const float mu = __ldg(mean + r), rs = __ldg(rstd + r);
            if constexpr (V == 1) {
                dv[0] = Tr::load1(dy + r * N + col0);
                xv[0] = Tr::load1(x + r * N + col0);
            } else {
                Tr::unpack(ld_stream16(dy + r * N + col0), dv);
                Tr::unpack(ld_stream16(x + r * N + col0), xv);
            }
#pragma unroll
            for (int e = 0; e < V; ++e) {
                ag[e] = fmaf(dv[e], (xv[e] - mu) * rs, ag[e]);
                ab[e] += dv[e];
            }
        }
    }
#pragma unroll
    for (int e = 0; e < V; ++e) {
        sg[w][lane * V + e] = ag[e];
        sb[w][lane * V + e] = ab[e];
    }
    __syncthreads();
    for (int cc = threadIdx.x; cc < CT; cc += kDgdbWarps * 32) {
        const int64_t col = (int64_t)blockIdx.x * CT + cc;
        if (col < N) {
            float a = sg[0][cc], b = sb[0][cc];
#pragma unroll
            for (int ww = 1; ww < kDgdbWarps; ++ww) {
                a += sg[ww][cc];
                b += sb[ww][cc];
            }
            part[(chunk * 2 + 0) * N + col] = a;
            part[(chunk * 2 + 1) * N + col] = b;
        }
    }
}

// ----------------------------------------------------------------------------
// gamma / beta gradient, stage 2: sum the chunk partials in a fixed order.
// Block = 32 columns x 8 chunk lanes; chunk lane t sums chunks t, t+8, ...;
// the 8 lane sums are then added in lane order.  nchunks == 0 writes zeros.
// ----------------------------------------------------------------------------
constexpr int kFinalCols = 32;
constexpr int kFinalLanes = 8;

static __global__ void __launch_bounds__(kFinalCols * kFinalLanes)
ln_dgdb_final(float *dgamma, float *dbeta, const float *part, int64_t nchunks, int64_t N) {
    __shared__ float sg[kFinalLanes][kFinalCols];
    __shared__ float sb[kFinalLanes][kFinalCols];
    const int tx = threadIdx.x % kFinalCols;
    const int ty = threadIdx.x / kFinalCols;
    const int64_t col = (int64_t)blockIdx.x * kFinalCols + tx;
    float a = 0.f, b = 0.f;
    if (col < N)
        for (int64_t c = ty; c < nchunks; c += kFinalLanes) {
            a += __ldcs(part + (c * 2 + 0) * N + col);
            b += __ldcs(part + (c * 2 + 1) * N + col);
        }
    sg[ty][tx] = a;
    sb[ty][tx] = b;
    __syncthreads();
    if (ty == 0 && col < N) {
        float ga = sg[0][tx], gb = sb[0][tx];
#pragma unroll
        for (int t = 1; t < kFinalLanes; ++t) {
            ga += sg[t][tx];
            gb += sb[t][tx];
        }
        dgamma[col] = ga;
        dbeta[col] = gb;
    }
}

}  // namespace lsr
