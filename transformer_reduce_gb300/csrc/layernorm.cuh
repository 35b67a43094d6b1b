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

// First element of a row from the 4 bytes copied at its start.
template <typename T>
__device__ __forceinline__ float first_elem(uint32_t w);
template <>
__device__ __forceinline__ float first_elem<float>(uint32_t w) { return __uint_as_float(w); }
template <>
__device__ __forceinline__ float first_elem<__half>(uint32_t w) {
    return __half2float(__ushort_as_half((unsigned short)(w & 0xffffu)));
}
template <>
__device__ __forceinline__ float first_elem<__nv_bfloat16>(uint32_t w) {
    return __uint_as_float(w << 16);
}

// Shared memory of the staged LayerNorm kernels: S stages of A tensors x CPT
// 16-byte chunks per thread, plus W words of per-row scalars per stage.
template <int TPR, int CPT, int S, int A, int W>
constexpr size_t ln_smem() {
    return (size_t)S * (TPR <= 32 ? 256 : TPR) * (A * CPT * 16 + W * 4);
}

// ----------------------------------------------------------------------------
// Forward.  The two statistics come from ONE fused reduction of sum(x') and
// sum(x'^2) with x' = x - x0 (x0 = the row's first element): var =
// mean(x'^2) - mean(x')^2 is the one-pass form, and the shift removes its
// cancellation when |mean| >> std (it is exact for constant rows).
//
// Each row group owns a contiguous range of rows.  Rows are staged into
// shared memory S-1 rows ahead with per-thread cp.async copies (each thread
// reads back only its own chunks), so the loads of the next rows are in
// flight while one is reduced (the launcher picks S by the row's width).  A
// thread's columns are the same for every row: its gamma/beta chunks are
// loaded once.  x0 reaches a row's threads by a shuffle from the first
// lane's staged chunk when the row fits one warp (a per-thread 4-byte copy of
// it cost the encoder-width forward 5 %); in a multi-warp row each warp's
// first lane stages it with a 4-byte copy and shuffles it to its warp.
// ----------------------------------------------------------------------------
// RMS = true is RMSNorm (the FastTransformer page, section 5.4): no shift and
// no mean, one sum of squares, y = x * rstd * gamma; `mean` and `beta` are
// unused.
template <typename T, int TPR, int CPT, int S, bool RMS>
__global__ void __launch_bounds__(TPR <= 32 ? 256 : TPR, (row_kernel_min_blocks<TPR, CPT>()))
ln_fw_vec(T *y, float *mean, float *rstd, const T *x, const T *gamma,
          const T *beta, int64_t rows, int N, float eps) {
    pdl_begin();
    using Tr = Traits<T>;
    constexpr int V = Tr::kVec;
    constexpr int H2 = V / 2;
    constexpr int BLOCK = TPR <= 32 ? 256 : TPR;
    constexpr int G = BLOCK / TPR;
    extern __shared__ uint4 dsmem[];
    uint4 *stage = dsmem;                                                  // [S][CPT][BLOCK]
    uint32_t *x0b = reinterpret_cast<uint32_t *>(dsmem + S * CPT * BLOCK);  // [S][BLOCK]
    __shared__ float red[TPR > 32 ? 64 : 1];

    const int tid = threadIdx.x;
    const int lane = tid % TPR;
    const int grp = tid / TPR;
    const int nchunk = N / V;
    const float invN = 1.f / (float)N;
    const int64_t ngroups = (int64_t)gridDim.x * G;
    const int64_t per = (rows + ngroups - 1) / ngroups;
    const int64_t rbeg = ((int64_t)blockIdx.x * G + grp) * per;
    const int64_t rend = rbeg + per < rows ? rbeg + per : rows;

    uint4 gr[CPT], br[CPT];
#pragma unroll
    for (int k = 0; k < CPT; ++k) {
        const int c = k * TPR + lane;
        if (c < nchunk) {
            gr[k] = ld_cached16(gamma + c * V);
            if constexpr (!RMS) br[k] = ld_cached16(beta + c * V);
        }
    }
    int64_t inext = rbeg;
    auto issue = [&](int s) {
        if (inext < rend) {
            const T *xrow = x + inext * (int64_t)N;
#pragma unroll
            for (int k = 0; k < CPT; ++k) {
                const int c = k * TPR + lane;
                if (c < nchunk) cp_async16(&stage[(s * CPT + k) * BLOCK + tid], xrow + c * V);
            }
            // the shift: a row inside one warp takes it from its first
            // lane's staged chunk by a shuffle; for a multi-warp row each
            // warp's first lane stages it and shuffles it to the warp
            if constexpr (!RMS && TPR > 32) {
                if ((tid & 31) == 0) cp_async4(&x0b[s * BLOCK + tid], xrow);
            }
        }
        ++inext;
        cp_async_commit();
    };
#pragma unroll
    for (int s = 0; s < S - 1; ++s) issue(s);

    int s_cur = 0, s_iss = S - 1;
    for (int64_t k = 0; k < per; ++k) {
        issue(s_iss);
        s_iss = s_iss + 1 == S ? 0 : s_iss + 1;
        cp_async_wait<S - 1>();

        const int64_t row = rbeg + k;
        const bool valid = row < rend;
        float x0 = 0.f;
        if constexpr (!RMS) {
            if constexpr (TPR > 32) {
                const float f =
                    (valid && (tid & 31) == 0) ? first_elem<T>(x0b[s_cur * BLOCK + tid]) : 0.f;
                x0 = __shfl_sync(0xffffffffu, f, 0);
            } else {
                const float f =
                    (valid && lane == 0) ? first_elem<T>(stage[s_cur * CPT * BLOCK + tid].x) : 0.f;
                x0 = __shfl_sync(0xffffffffu, f, 0, TPR);
            }
        }
        float2 d[CPT][H2];
        float2 s1 = f2(0.f), s2 = f2(0.f);
#pragma unroll
        for (int kk = 0; kk < CPT; ++kk) {
            const int c = kk * TPR + lane;
            if (valid && c < nchunk) {
                unpack2<T>(stage[(s_cur * CPT + kk) * BLOCK + tid], d[kk]);
#pragma unroll
                for (int h = 0; h < H2; ++h) {
                    if constexpr (!RMS) {
                        d[kk][h] = add2(d[kk][h], f2(-x0));
                        s1 = add2(s1, d[kk][h]);
                    }
                    s2 = fma2(d[kk][h], d[kk][h], s2);
                }
            }
        }
        float m1 = 0.f, rs;
        if constexpr (RMS) {
            const float a2 = group_reduce<TPR, OpSum>(s2.x + s2.y, red);
            rs = rsqrtf(a2 * invN + eps);
        } else {
            float a1 = s1.x + s1.y, a2 = s2.x + s2.y;
            group_sum2<TPR>(a1, a2, red);
            m1 = a1 * invN;
            const float var = fmaxf(a2 * invN - m1 * m1, 0.f);
            rs = rsqrtf(var + eps);
        }

        T *yrow = y + row * (int64_t)N;
#pragma unroll
        for (int kk = 0; kk < CPT; ++kk) {
            const int c = kk * TPR + lane;
            if (valid && c < nchunk) {
                float2 gv[H2], yv[H2];
                unpack2<T>(gr[kk], gv);
                if constexpr (RMS) {
#pragma unroll
                    for (int h = 0; h < H2; ++h)
                        yv[h] = mul2(mul2(d[kk][h], f2(rs)), gv[h]);
                } else {
                    float2 bv[H2];
                    unpack2<T>(br[kk], bv);
#pragma unroll
                    for (int h = 0; h < H2; ++h) {
                        const float2 t = mul2(add2(d[kk][h], f2(-m1)), f2(rs));
                        yv[h] = fma2(t, gv[h], bv[h]);
                    }
                }
                st_stream16(yrow + c * V, pack2<T>(yv));
            }
        }
        if (valid && lane == 0) {
            if constexpr (!RMS) mean[row] = x0 + m1;
            rstd[row] = rs;
        }
        s_cur = s_cur + 1 == S ? 0 : s_cur + 1;
    }
}

// ----------------------------------------------------------------------------
// Input gradient.  g = gamma * dy, xhat = (x - mean)*rstd; S1 = sum g and
// S2 = sum g*xhat in one fused reduction; then dx = rstd*(g - S1/N - xhat*S2/N).
// Same staging as the forward: dy and x per stage, and the row's mean / rstd
// staged by the group's (or, for a multi-warp row, each warp's) first lane
// and shuffled to its threads (a 4-byte copy by every thread cost 8-16 % at
// 768-1024 features).
// ----------------------------------------------------------------------------
// RMS = true is the RMSNorm input gradient: xhat = x * rstd, one sum
// S2 = sum g*xhat, dx = rstd * (g - xhat * S2/N); `mean` is unused.
template <typename T, int TPR, int CPT, int S, bool RMS>
__global__ void __launch_bounds__(TPR <= 32 ? 256 : TPR, (row_kernel_min_blocks<TPR, CPT>()))
ln_dinp_vec(T *dx, const T *dy, const T *x, const T *gamma, const float *mean,
            const float *rstd, int64_t rows, int N) {
    pdl_begin();
    using Tr = Traits<T>;
    constexpr int V = Tr::kVec;
    constexpr int H2 = V / 2;
    constexpr int BLOCK = TPR <= 32 ? 256 : TPR;
    constexpr int G = BLOCK / TPR;
    constexpr int SW = TPR < 32 ? TPR : 32;  // threads sharing one staged copy of the scalars
    extern __shared__ uint4 dsmem[];
    uint4 *stage = dsmem;                                                    // [S][2][CPT][BLOCK]
    float *stat = reinterpret_cast<float *>(dsmem + S * 2 * CPT * BLOCK);    // [S][2][BLOCK]
    __shared__ float red[TPR > 32 ? 64 : 1];

    const int tid = threadIdx.x;
    const int lane = tid % TPR;
    const int grp = tid / TPR;
    const int nchunk = N / V;
    const float invN = 1.f / (float)N;
    const int64_t ngroups = (int64_t)gridDim.x * G;
    const int64_t per = (rows + ngroups - 1) / ngroups;
    const int64_t rbeg = ((int64_t)blockIdx.x * G + grp) * per;
    const int64_t rend = rbeg + per < rows ? rbeg + per : rows;

    uint4 gr[CPT];
#pragma unroll
    for (int k = 0; k < CPT; ++k) {
        const int c = k * TPR + lane;
        if (c < nchunk) gr[k] = ld_cached16(gamma + c * V);
    }
    int64_t inext = rbeg;
    auto issue = [&](int s) {
        if (inext < rend) {
            const int64_t off = inext * (int64_t)N;
#pragma unroll
            for (int k = 0; k < CPT; ++k) {
                const int c = k * TPR + lane;
                if (c < nchunk) {
                    cp_async16(&stage[((s * 2 + 0) * CPT + k) * BLOCK + tid], dy + off + c * V);
                    cp_async16(&stage[((s * 2 + 1) * CPT + k) * BLOCK + tid], x + off + c * V);
                }
            }
            // the row's statistics: staged by the first lane of each slice of
            // SW threads (the row group, or one warp of a multi-warp row),
            // then shuffled to the slice
            if (tid % SW == 0) {
                if constexpr (!RMS) cp_async4(&stat[(s * 2 + 0) * BLOCK + tid], mean + inext);
                cp_async4(&stat[(s * 2 + 1) * BLOCK + tid], rstd + inext);
            }
        }
        ++inext;
        cp_async_commit();
    };
#pragma unroll
    for (int s = 0; s < S - 1; ++s) issue(s);

    int s_cur = 0, s_iss = S - 1;
    for (int64_t k = 0; k < per; ++k) {
        issue(s_iss);
        s_iss = s_iss + 1 == S ? 0 : s_iss + 1;
        cp_async_wait<S - 1>();

        const int64_t row = rbeg + k;
        const bool valid = row < rend;
        const bool mine = valid && tid % SW == 0;
        const float m0 = (mine && !RMS) ? stat[(s_cur * 2 + 0) * BLOCK + tid] : 0.f;
        const float r0 = mine ? stat[(s_cur * 2 + 1) * BLOCK + tid] : 0.f;
        const float mu = __shfl_sync(0xffffffffu, m0, 0, SW);
        const float rs = __shfl_sync(0xffffffffu, r0, 0, SW);
        float2 g[CPT][H2], xh[CPT][H2];
        float2 s1 = f2(0.f), s2 = f2(0.f);
#pragma unroll
        for (int kk = 0; kk < CPT; ++kk) {
            const int c = kk * TPR + lane;
            if (valid && c < nchunk) {
                float2 gv[H2];
                unpack2<T>(stage[((s_cur * 2 + 0) * CPT + kk) * BLOCK + tid], g[kk]);
                unpack2<T>(stage[((s_cur * 2 + 1) * CPT + kk) * BLOCK + tid], xh[kk]);
                unpack2<T>(gr[kk], gv);
#pragma unroll
                for (int h = 0; h < H2; ++h) {
                    // rounded product (never fused into a later add), so that
                    // S1 sums exactly the g the epilogue uses
                    g[kk][h] = mul2(g[kk][h], gv[h]);
                    if constexpr (RMS) {
                        xh[kk][h] = mul2(xh[kk][h], f2(rs));
                    } else {
                        xh[kk][h] = mul2(add2(xh[kk][h], f2(-mu)), f2(rs));
                        s1 = add2(s1, g[kk][h]);
                    }
                    s2 = fma2(g[kk][h], xh[kk][h], s2);
                }
            }
        }
        float a1 = 0.f, a2;
        if constexpr (RMS) {
            a2 = group_reduce<TPR, OpSum>(s2.x + s2.y, red);
        } else {
            a1 = s1.x + s1.y;
            a2 = s2.x + s2.y;
            group_sum2<TPR>(a1, a2, red);
        }
        const float2 na = f2(-a1 * invN), nb = f2(-a2 * invN);
        const int64_t off = row * (int64_t)N;
#pragma unroll
        for (int kk = 0; kk < CPT; ++kk) {
            const int c = kk * TPR + lane;
            if (valid && c < nchunk) {
                float2 ov[H2];
#pragma unroll
                for (int h = 0; h < H2; ++h)
                    ov[h] = mul2(f2(rs), fma2(xh[kk][h], nb, add2(g[kk][h], na)));
                st_stream16(dx + off + c * V, pack2<T>(ov));
            }
        }
        s_cur = s_cur + 1 == S ? 0 : s_cur + 1;
    }
}

// ----------------------------------------------------------------------------
// Fused backward: dx, and the dgamma / dbeta partial sums of one row chunk,
// from one read of dy and x.  Block b owns rows [b*rpc, (b+1)*rpc) (a fixed
// cut of the rows, independent of the GPU); its G row groups split them into
// contiguous runs and stage dy and x as ln_dinp_vec does, while each thread
// reads the row's mean and rstd into registers one row ahead (staged with a
// 4-byte cp.async by every thread, they made this kernel 11-30 % slower at
// 768-2048 features).
// Each thread also accumulates dgamma += dy * xhat and dbeta += dy for its
// columns; the G groups' sums are added in group order through shared memory
// and written as the chunk's partial part[(b*2 + {0,1}) * N + col], which
// ln_dgdb_final then sums over chunks in a fixed order.  The epilogue re-reads
// the staged row instead of keeping g and xhat in registers (the stage is not
// refilled before the next iteration).
// ----------------------------------------------------------------------------
// Threads of a fused-backward block: at least 256 (several row groups when a
// group is smaller), so that the fixed grid of row chunks still fills an SM.
template <int TPR>
constexpr int ln_bw_fused_block() { return TPR < 256 ? 256 : TPR; }

// Resident blocks per SM the fused backward is compiled for (its register
// budget): one 512-thread block, else three 256-thread blocks when a thread
// holds one 16-byte chunk of the row, two when it holds two.
template <int TPR, int CPT>
constexpr int ln_bw_fused_resident() {
    return ln_bw_fused_block<TPR>() > 256 ? 1 : (CPT == 1 ? 3 : 2);
}

// Row chunks (= blocks) of the fused backward: the resident blocks of a
// 152-SM GB300.  A constant of the bucket, not the device's SM count, so that
// the summation order depends only on the problem.
constexpr int kFusedMaxChunks = 3 * 152;
template <int TPR, int CPT>
constexpr int ln_bw_fused_chunks() { return 152 * ln_bw_fused_resident<TPR, CPT>(); }

template <int TPR, int CPT, int S, int V>
constexpr size_t ln_bw_fused_smem() {
    // the stage ring, reused at the end for the [G][2][TPR*CPT*V] group sums
    constexpr int BLOCK = ln_bw_fused_block<TPR>();
    constexpr size_t ring = (size_t)S * BLOCK * 2 * CPT * 16;
    constexpr size_t sums = (size_t)BLOCK * 2 * CPT * V * 4;
    return ring > sums ? ring : sums;
}

// Block b owns rows [b*rpc, min(rows, (b+1)*rpc)) (blocks past the last row
// own none and contribute zeros); its G row groups split them into
// contiguous runs.  Per row: the input gradient as ln_dinp_vec computes it
// (same staging, same fused two-sum reduction), and each thread adds dy*xhat
// and dy into per-column accumulators.  At the end the groups' accumulators
// are added in group order in shared memory and the block writes its chunk's
// part[(b*2 + {0,1}) * N + col].  (Pairing blocks in a thread-block cluster
// to add two chunks through distributed shared memory first measured no
// faster: the cluster barrier waits for the block's last dx stores.)
template <typename T, int TPR, int CPT, int S>
__global__ void __launch_bounds__(ln_bw_fused_block<TPR>(), (ln_bw_fused_resident<TPR, CPT>()))
ln_bw_fused_vec(T *dx, float *part, const T *dy, const T *x, const T *gamma, const float *mean,
                const float *rstd, int64_t rows, int N, int64_t rows_per_chunk) {
    pdl_begin();
    using Tr = Traits<T>;
    constexpr int V = Tr::kVec;
    constexpr int H2 = V / 2;
    constexpr int BLOCK = ln_bw_fused_block<TPR>();
    constexpr int G = BLOCK / TPR;
    constexpr int W = TPR * CPT * V;  // columns a row group covers (>= N)
    extern __shared__ uint4 dsmem[];
    uint4 *stage = dsmem;  // [S][2][CPT][BLOCK]
    __shared__ float red[TPR > 32 ? 64 : 1];  // >= 2 * BLOCK / 32 and group_sum2's 48

    const int tid = threadIdx.x;
    const int lane = tid % TPR;
    const int grp = tid / TPR;
    const int nchunk = N / V;
    const float invN = 1.f / (float)N;
    const int64_t c0 = (int64_t)blockIdx.x * rows_per_chunk;
    const int64_t c1 = c0 + rows_per_chunk < rows ? c0 + rows_per_chunk : rows;
    const int64_t per = (rows_per_chunk + G - 1) / G;  // rows per group (uniform)
    const int64_t rbeg = c0 + grp * per;
    const int64_t rend = rbeg + per < c1 ? rbeg + per : c1;

    uint4 gr[CPT];
    float2 ag[CPT][H2], ab[CPT][H2];
#pragma unroll
    for (int k = 0; k < CPT; ++k) {
        const int c = k * TPR + lane;
        if (c < nchunk) gr[k] = ld_cached16(gamma + c * V);
#pragma unroll
        for (int h = 0; h < H2; ++h) ag[k][h] = ab[k][h] = f2(0.f);
    }
    int64_t inext = rbeg;
    auto issue = [&](int s) {
        if (inext < rend) {
            const int64_t off = inext * (int64_t)N;
#pragma unroll
            for (int k = 0; k < CPT; ++k) {
                const int c = k * TPR + lane;
                if (c < nchunk) {
                    cp_async16(&stage[((s * 2 + 0) * CPT + k) * BLOCK + tid], dy + off + c * V);
                    cp_async16(&stage[((s * 2 + 1) * CPT + k) * BLOCK + tid], x + off + c * V);
                }
            }
        }
        ++inext;
        cp_async_commit();
    };
#pragma unroll
    for (int s = 0; s < S - 1; ++s) issue(s);

    // the current row's statistics; the next row's are loaded while this
    // row's data lands and is reduced
    float mu_c = 0.f, rs_c = 0.f;
    if (rbeg < rend) {
        mu_c = __ldg(mean + rbeg);
        rs_c = __ldg(rstd + rbeg);
    }
    int s_cur = 0, s_iss = S - 1;
    for (int64_t k = 0; k < per; ++k) {
        issue(s_iss);
        s_iss = s_iss + 1 == S ? 0 : s_iss + 1;
        const int64_t row = rbeg + k;
        float mu_n = 0.f, rs_n = 0.f;
        if (row + 1 < rend) {
            mu_n = __ldg(mean + row + 1);
            rs_n = __ldg(rstd + row + 1);
        }
        cp_async_wait<S - 1>();

        const bool valid = row < rend;
        const float mu = valid ? mu_c : 0.f;
        const float rs = valid ? rs_c : 0.f;
        mu_c = mu_n;
        rs_c = rs_n;
        // Up to two chunks per thread the row's g and xhat stay in registers
        // for the epilogue; wider buckets (whose column accumulators already
        // take 64 registers) unpack them again from the stage instead.
        constexpr bool kKeep = CPT <= 2;
        float2 g[kKeep ? CPT : 1][H2], xh[kKeep ? CPT : 1][H2];
        float2 s1 = f2(0.f), s2 = f2(0.f);
        auto load_row = [&](int kk, float2 (&gg)[H2], float2 (&xx)[H2]) {
            float2 gv[H2];
            unpack2<T>(stage[((s_cur * 2 + 0) * CPT + kk) * BLOCK + tid], gg);
            unpack2<T>(stage[((s_cur * 2 + 1) * CPT + kk) * BLOCK + tid], xx);
            unpack2<T>(gr[kk], gv);
#pragma unroll
            for (int h = 0; h < H2; ++h) {
                xx[h] = mul2(add2(xx[h], f2(-mu)), f2(rs));
                gg[h] = mul2(gg[h], gv[h]);
            }
        };
#pragma unroll
        for (int kk = 0; kk < CPT; ++kk) {
            const int c = kk * TPR + lane;
            if (valid && c < nchunk) {
                float2 dv[H2], gg[H2], xx[H2];
                unpack2<T>(stage[((s_cur * 2 + 0) * CPT + kk) * BLOCK + tid], dv);
                load_row(kk, gg, xx);
#pragma unroll
                for (int h = 0; h < H2; ++h) {
                    ab[kk][h] = add2(ab[kk][h], dv[h]);
                    ag[kk][h] = fma2(dv[h], xx[h], ag[kk][h]);
                    s1 = add2(s1, gg[h]);
                    s2 = fma2(gg[h], xx[h], s2);
                }
                if constexpr (kKeep) {
#pragma unroll
                    for (int h = 0; h < H2; ++h) {
                        g[kk][h] = gg[h];
                        xh[kk][h] = xx[h];
                    }
                }
            }
        }
        float a1 = s1.x + s1.y, a2 = s2.x + s2.y;
        group_sum2_of<TPR, BLOCK>(a1, a2, red, grp);
        const float2 na = f2(-a1 * invN), nb = f2(-a2 * invN);
        const int64_t off = row * (int64_t)N;
#pragma unroll
        for (int kk = 0; kk < CPT; ++kk) {
            const int c = kk * TPR + lane;
            if (valid && c < nchunk) {
                float2 gg[H2], xx[H2], ov[H2];
                if constexpr (kKeep) {
#pragma unroll
                    for (int h = 0; h < H2; ++h) {
                        gg[h] = g[kk][h];
                        xx[h] = xh[kk][h];
                    }
                } else {
                    load_row(kk, gg, xx);
                }
#pragma unroll
                for (int h = 0; h < H2; ++h)
                    ov[h] = mul2(f2(rs), fma2(xx[h], nb, add2(gg[h], na)));
                st_stream16(dx + off + c * V, pack2<T>(ov));
            }
        }
        s_cur = s_cur + 1 == S ? 0 : s_cur + 1;
    }

    // block sums: the groups' accumulators in group order, into gs[0][.][.]
    __syncthreads();  // every group is past its last read of the ring
    float *gs = reinterpret_cast<float *>(dsmem);  // [G][2][W]
#pragma unroll
    for (int kk = 0; kk < CPT; ++kk) {
        const int c = kk * TPR + lane;
#pragma unroll
        for (int h = 0; h < H2; ++h) {
            gs[(grp * 2 + 0) * W + c * V + 2 * h] = ag[kk][h].x;
            gs[(grp * 2 + 0) * W + c * V + 2 * h + 1] = ag[kk][h].y;
            gs[(grp * 2 + 1) * W + c * V + 2 * h] = ab[kk][h].x;
            gs[(grp * 2 + 1) * W + c * V + 2 * h + 1] = ab[kk][h].y;
        }
    }
    __syncthreads();
    if constexpr (G > 1) {
        for (int col = tid; col < N; col += BLOCK) {
            float a = gs[col], b = gs[W + col];
            for (int gg = 1; gg < G; ++gg) {
                a += gs[(gg * 2 + 0) * W + col];
                b += gs[(gg * 2 + 1) * W + col];
            }
            gs[col] = a;  // each column is read and written by this thread only
            gs[W + col] = b;
        }
    }
    __syncthreads();
    for (int col = tid; col < N; col += BLOCK) {
        part[((int64_t)blockIdx.x * 2 + 0) * N + col] = gs[col];
        part[((int64_t)blockIdx.x * 2 + 1) * N + col] = gs[W + col];
    }
}

// ----------------------------------------------------------------------------
// Looped variants (scalar accesses, any alignment, any row length).
// ----------------------------------------------------------------------------
template <typename T, int TPR, bool RMS>
__global__ void __launch_bounds__(TPR <= 32 ? 256 : TPR)
ln_fw_loop(T *y, float *mean, float *rstd, const T *x, const T *gamma,
           const T *beta, int64_t rows, int64_t N, float eps) {
    pdl_begin();
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
        const float x0 = (valid && !RMS) ? Tr::load1_cached(xrow) : 0.f;
        float s1 = 0.f, s2 = 0.f;
        if (valid)
            for (int64_t j = lane; j < N; j += TPR) {
                const float d = Tr::load1(xrow + j) - x0;
                s1 += d;
                s2 = fmaf(d, d, s2);
            }
        float m1 = 0.f, rs;
        if constexpr (RMS) {
            s2 = group_reduce<TPR, OpSum>(s2, red);
            rs = rsqrtf(s2 * invN + eps);
        } else {
            group_sum2<TPR>(s1, s2, red);
            m1 = s1 * invN;
            const float var = fmaxf(s2 * invN - m1 * m1, 0.f);
            rs = rsqrtf(var + eps);
        }
        if (valid) {
            T *yrow = y + row * N;
            for (int64_t j = lane; j < N; j += TPR) {
                const float d = Tr::load1(xrow + j) - x0;
                if constexpr (RMS)
                    Tr::store1(yrow + j, __fmul_rn(d * rs, Tr::load1_cached(gamma + j)));
                else
                    Tr::store1(yrow + j, fmaf((d - m1) * rs, Tr::load1_cached(gamma + j),
                                              Tr::load1_cached(beta + j)));
            }
            if (lane == 0) {
                if constexpr (!RMS) mean[row] = x0 + m1;
                rstd[row] = rs;
            }
        }
    }
}

template <typename T, int TPR, bool RMS>
__global__ void __launch_bounds__(TPR <= 32 ? 256 : TPR)
ln_dinp_loop(T *dx, const T *dy, const T *x, const T *gamma, const float *mean,
             const float *rstd, int64_t rows, int64_t N) {
    pdl_begin();
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
        const float mu = (valid && !RMS) ? __ldg(mean + row) : 0.f;
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
        if constexpr (RMS) {
            s1 = 0.f;
            s2 = group_reduce<TPR, OpSum>(s2, red);
        } else {
            group_sum2<TPR>(s1, s2, red);
        }
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
// gamma / beta gradient, stage 1, scalar path (any alignment or width):
// partial column sums of one row chunk.  Block = 8 warps over a tile of 32
// columns; warp w takes rows w, w+8, ... of the chunk, four rows in flight
// per lane.  The 8 per-warp sums are added in warp order through shared
// memory and written to
//   part[(chunk * 2 + 0) * N + col] (dgamma),  part[(chunk * 2 + 1) * N + col] (dbeta).
// mean == nullptr means mean 0 (RMSNorm).
// ----------------------------------------------------------------------------
constexpr int kDgdbWarps = 8;

template <typename T>
__global__ void __launch_bounds__(kDgdbWarps * 32, 4)
ln_dgdb_partial(float *part, const T *dy, const T *x, const float *mean,
                const float *rstd, int64_t rows, int64_t N, int64_t rows_per_chunk) {
    pdl_begin();
    using Tr = Traits<T>;
    constexpr int CT = 32;  // columns per tile
    __shared__ float sg[kDgdbWarps][CT];
    __shared__ float sb[kDgdbWarps][CT];

    const int lane = threadIdx.x & 31;
    const int w = threadIdx.x >> 5;
    const int64_t col0 = (int64_t)blockIdx.x * CT + lane;
    const int64_t chunk = blockIdx.y;
    const int64_t r0 = chunk * rows_per_chunk;
    const int64_t r1 = min(rows, r0 + rows_per_chunk);

    float ag = 0.f, ab = 0.f;
    if (col0 < N) {
        int64_t r = r0 + w;
        for (; r + 3 * kDgdbWarps < r1; r += 4 * kDgdbWarps) {
            float mu[4], rs[4], dv[4], xv[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int64_t rr = r + u * kDgdbWarps;
                mu[u] = mean ? __ldg(mean + rr) : 0.f;
                rs[u] = __ldg(rstd + rr);
                dv[u] = Tr::load1(dy + rr * N + col0);
                xv[u] = Tr::load1(x + rr * N + col0);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                ag = fmaf(dv[u], (xv[u] - mu[u]) * rs[u], ag);
                ab += dv[u];
            }
        }
        for (; r < r1; r += kDgdbWarps) {
            const float mu = mean ? __ldg(mean + r) : 0.f, rs = __ldg(rstd + r);
            const float dv = Tr::load1(dy + r * N + col0);
            const float xv = Tr::load1(x + r * N + col0);
            ag = fmaf(dv, (xv - mu) * rs, ag);
            ab += dv;
        }
    }
    sg[w][lane] = ag;
    sb[w][lane] = ab;
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
// gamma / beta gradient, stage 1, vectorised: the partial sums of
// ln_dgdb_partial over tiles of 32 lanes x 16 bytes (256 columns of 16-bit
// storage), with the same warp-to-row assignment, fp32 arithmetic and
// warp-order combine; each warp streams its rows through a private ring of
// S cp.async stages of kDgdbRows rows each (512 contiguous bytes of dy and of
// x per row, plus the rows' mean and rstd), so that (S - 1) * kDgdbRows rows
// per warp are in flight and the per-stage bookkeeping is shared by
// kDgdbRows rows.  The ring is reused for the warp-order combine at the end.
// The ring depth does not change which rows a warp adds or in what order, so
// the result is the same bit for bit whichever depth the launcher takes.
// mean == nullptr means mean 0 (RMSNorm).
// ----------------------------------------------------------------------------
constexpr int kDgdbRows = 2;

template <int S>
constexpr size_t ln_dgdb_staged_smem() {
    return (size_t)kDgdbWarps * S * kDgdbRows * (64 * 16 + 2 * 4);
}

template <typename T, int S>
__global__ void __launch_bounds__(kDgdbWarps * 32, 3)
ln_dgdb_staged(float *part, const T *dy, const T *x, const float *mean, const float *rstd,
               int64_t rows, int64_t N, int64_t rows_per_chunk) {
    pdl_begin();
    using Tr = Traits<T>;
    constexpr int V = Tr::kVec;
    constexpr int CT = 32 * V;  // columns per tile
    constexpr int R = kDgdbRows;
    static_assert(2 * kDgdbWarps * CT * 4 <= kDgdbWarps * S * R * 64 * 16, "combine fits the ring");
    extern __shared__ uint4 dsmem[];
    const int lane = threadIdx.x & 31;
    const int w = threadIdx.x >> 5;
    uint4 *ring = dsmem + (size_t)w * S * R * 64;  // [S][R][dy, x][32 lanes]
    float *stat = reinterpret_cast<float *>(dsmem + kDgdbWarps * S * R * 64) + w * S * R * 2;

    const int64_t col0 = (int64_t)blockIdx.x * CT + lane * V;
    const bool colok = col0 < N;
    const int64_t chunk = blockIdx.y;
    const int64_t r0 = chunk * rows_per_chunk;
    const int64_t r1 = min(rows, r0 + rows_per_chunk);
    // this warp's rows: r0 + w + 8 j, j < nk, taken R at a time
    const int64_t nk = r1 - r0 > w ? (r1 - r0 - w + kDgdbWarps - 1) / kDgdbWarps : 0;
    const int64_t nst = (nk + R - 1) / R;

    constexpr int H2 = V / 2;
    float2 ag[H2], ab[H2];
#pragma unroll
    for (int h = 0; h < H2; ++h) ag[h] = ab[h] = f2(0.f);

    // running source pointers of the next stage to issue
    const int64_t rstep = (int64_t)kDgdbWarps * N;
    const T *pdy = dy + (r0 + w) * N + col0;
    const T *px = x + (r0 + w) * N + col0;
    const float *pst = (lane & 1) ? rstd + r0 + w : mean + r0 + w;  // lanes 0..2R-1
    const bool stat_lane = lane < 2 * R && (mean != nullptr || (lane & 1));
    int64_t jnext = 0;
    auto issue = [&](int st) {
#pragma unroll
        for (int rr = 0; rr < R; ++rr) {
            if (jnext + rr < nk) {
                if (colok) {
                    cp_async16(&ring[(st * R + rr) * 64 + lane], pdy + rr * rstep);
                    cp_async16(&ring[(st * R + rr) * 64 + 32 + lane], px + rr * rstep);
                }
                if (stat_lane && (lane >> 1) == rr)
                    cp_async4(&stat[(st * R + rr) * 2 + (lane & 1)], pst + rr * kDgdbWarps);
            }
        }
        jnext += R;
        pdy += R * rstep;
        px += R * rstep;
        pst += R * kDgdbWarps;
        cp_async_commit();
    };
#pragma unroll
    for (int st = 0; st < S - 1; ++st) issue(st);

    int s_cur = 0, s_iss = S - 1;
    for (int64_t k = 0; k < nst; ++k) {
        issue(s_iss);
        s_iss = s_iss + 1 == S ? 0 : s_iss + 1;
        cp_async_wait<S - 1>();
        __syncwarp();  // the statistics lanes' copies are visible to the warp
#pragma unroll
        for (int rr = 0; rr < R; ++rr) {
            if (k * R + rr < nk && colok) {
                const float2 nmu = f2(mean ? -stat[(s_cur * R + rr) * 2] : 0.f);
                const float2 rs = f2(stat[(s_cur * R + rr) * 2 + 1]);
                float2 dv[H2], xv[H2];
                unpack2<T>(ring[(s_cur * R + rr) * 64 + lane], dv);
                unpack2<T>(ring[(s_cur * R + rr) * 64 + 32 + lane], xv);
#pragma unroll
                for (int h = 0; h < H2; ++h) {
                    ag[h] = fma2(dv[h], mul2(add2(xv[h], nmu), rs), ag[h]);
                    ab[h] = add2(ab[h], dv[h]);
                }
            }
        }
        __syncwarp();  // the next issue refills this stage
        s_cur = s_cur + 1 == S ? 0 : s_cur + 1;
    }

    __syncthreads();  // every warp is done with its ring (no copy in flight)
    float *sg = reinterpret_cast<float *>(dsmem);  // [warps][CT]
    float *sb = sg + kDgdbWarps * CT;              // [warps][CT]
#pragma unroll
    for (int h = 0; h < H2; ++h) {
        sg[w * CT + lane * V + 2 * h] = ag[h].x;
        sg[w * CT + lane * V + 2 * h + 1] = ag[h].y;
        sb[w * CT + lane * V + 2 * h] = ab[h].x;
        sb[w * CT + lane * V + 2 * h + 1] = ab[h].y;
    }
    __syncthreads();
    for (int cc = threadIdx.x; cc < CT; cc += kDgdbWarps * 32) {
        const int64_t col = (int64_t)blockIdx.x * CT + cc;
        if (col < N) {
            float a = sg[cc], b = sb[cc];
#pragma unroll
            for (int ww = 1; ww < kDgdbWarps; ++ww) {
                a += sg[ww * CT + cc];
                b += sb[ww * CT + cc];
            }
            part[(chunk * 2 + 0) * N + col] = a;
            part[(chunk * 2 + 1) * N + col] = b;
        }
    }
}

// ----------------------------------------------------------------------------
// gamma / beta gradient, stage 2: sum the chunk partials in a fixed order.
// Block = 8 columns x 32 chunk lanes; chunk lane t sums chunks t, t+32, ...
// in increasing order, loading a batch of 16 of them at once (the kernel is
// latency-bound: few bytes, many dependent rounds otherwise; 16 covers the
// at most 456 chunks in one round); the 32 lane sums are then added in lane
// order.  nchunks == 0 writes zeros.
// ----------------------------------------------------------------------------
constexpr int kFinalCols = 8;
constexpr int kFinalLanes = 32;
constexpr int kFinalBatch = 16;

static __global__ void __launch_bounds__(kFinalCols * kFinalLanes)
ln_dgdb_final(float *dgamma, float *dbeta, const float *part, int64_t nchunks, int64_t N) {
    pdl_begin();
    __shared__ float sg[kFinalLanes][kFinalCols + 1];
    __shared__ float sb[kFinalLanes][kFinalCols + 1];
    const int tx = threadIdx.x % kFinalCols;
    const int ty = threadIdx.x / kFinalCols;
    const int64_t col = (int64_t)blockIdx.x * kFinalCols + tx;
    float a = 0.f, b = 0.f;
    if (col < N) {
        for (int64_t base = ty; base < nchunks; base += (int64_t)kFinalLanes * kFinalBatch) {
            float va[kFinalBatch], vb[kFinalBatch];
#pragma unroll
            for (int u = 0; u < kFinalBatch; ++u) {
                const int64_t c = base + (int64_t)u * kFinalLanes;
                va[u] = c < nchunks ? __ldcs(part + (c * 2 + 0) * N + col) : 0.f;
                vb[u] = c < nchunks ? __ldcs(part + (c * 2 + 1) * N + col) : 0.f;
            }
#pragma unroll
            for (int u = 0; u < kFinalBatch; ++u) {
                a += va[u];
                b += vb[u];
            }
        }
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
        if (dbeta) dbeta[col] = gb;
    }
}

}  // namespace lsr
