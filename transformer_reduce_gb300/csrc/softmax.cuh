// softmax.cuh -- attention softmax forward / backward kernels (sm_103a).
//
// The operation is the masked, optionally causal attention softmax of the
// pages "CMU 11-868 HW4：把 Softmax 與 LayerNorm 寫成 CUDA 融合 kernel"
// (section 題目結構與配分, Problems 1.1 and 1.2) and "CMU 11-868 L10:
// Accelerating Transformers on GPUs, and Where LightSeq Finds the Time"
// (section "Technique 2", slides 23-26: two dependent reductions per row,
// shape-dependent threads-per-row and elements-per-thread fixed at compile
// time and chosen at launch).
//
// GB300 design:
//  * Rows of the [B*H*Tq, Tk] score matrix are independent.  A row is owned
//    by TPR threads (a power-of-two slice of a warp, or 2..32 whole warps);
//    each thread holds CPT 16-byte chunks of the row in registers, so the row
//    is read from HBM exactly once and written exactly once.
//  * Chunk c of a row lives in thread c % TPR, slot c / TPR: consecutive
//    threads touch consecutive 16-byte chunks (fully coalesced 128-bit
//    accesses).
//  * Keys that are masked (-inf in the additive mask) or in the causal future
//    are never read: a whole 16-byte chunk of them costs no HBM traffic.
//  * The grid is persistent: blocks loop over row groups, so the launch is
//    sized from the SM count and occupancy, not the problem size.
//  * Rows that do not fit the register buckets, or whose rows are not
//    16-byte aligned, take a looped path (online max/sum, then a second read).
#pragma once

#include "ls_device.cuh"

namespace lsr {

// ----------------------------------------------------------------------------
// Register-resident forward: one row per TPR threads, CPT chunks per thread.
// ----------------------------------------------------------------------------
template <typename T, int TPR, int CPT>
__global__ void __launch_bounds__(TPR <= 32 ? 256 : TPR)
softmax_fw_vec(T *out, const T *inp, const T *mask, int64_t rows,
               int64_t rows_per_batch, int64_t Tq, int Tk, int causal) {
    using Tr = Traits<T>;
    constexpr int V = Tr::kVec;
    constexpr int BLOCK = TPR <= 32 ? 256 : TPR;
    constexpr int G = BLOCK / TPR;  // rows per block iteration
    __shared__ float red[TPR > 32 ? 64 : 1];

    const int lane = threadIdx.x % TPR;
    const int grp = threadIdx.x / TPR;
    const int nchunk = Tk / V;

    for (int64_t base = (int64_t)blockIdx.x * G; base < rows;
         base += (int64_t)gridDim.x * G) {
        const int64_t row = base + grp;
        const bool valid = row < rows;
        const int64_t qi = (valid && causal) ? row % Tq : (int64_t)Tk;
        const T *xrow = inp + row * (int64_t)Tk;
        const T *mrow = mask ? mask + (row / rows_per_batch) * (int64_t)Tk : nullptr;

        float z[CPT][V];
        float lmax = -INFINITY;
#pragma unroll
        for (int k = 0; k < CPT; ++k) {
            const int c = k * TPR + lane;
            const int j0 = c * V;
            bool live = valid && c < nchunk && (int64_t)j0 <= qi;
            float mv[V];
#pragma unroll
            for (int e = 0; e < V; ++e) mv[e] = 0.f;
            if (live && mrow) {
                Tr::unpack(ld_cached16(mrow + j0), mv);
                bool any = false;
#pragma unroll
                for (int e = 0; e < V; ++e) any |= (mv[e] != -INFINITY);
                live = any;
            }
            if (live) {
                float xv[V];
                Tr::unpack(ld_stream16(xrow + j0), xv);
#pragma unroll
                for (int e = 0; e < V; ++e) {
                    const bool future = (int64_t)(j0 + e) > qi;
                    z[k][e] = future ? -INFINITY : (xv[e] + mv[e]) * kLog2e;
                    lmax = fmaxf(lmax, z[k][e]);
                }
            } else {
#pragma unroll
                for (int e = 0; e < V; ++e) z[k][e] = -INFINITY;
            }
        }
        float gmax = group_reduce<TPR, OpMax>(lmax, red);
        if (gmax == -INFINITY) gmax = 0.f;  // fully masked row: every exp2 is 0

        float lsum = 0.f;
#pragma unroll
        for (int k = 0; k < CPT; ++k) {
#pragma unroll
            for (int e = 0; e < V; ++e) {
                z[k][e] = exp2f(z[k][e] - gmax);
                lsum += z[k][e];
            }
        }
        const float gsum = group_reduce<TPR, OpSum>(lsum, red);
        const float inv = gsum > 0.f ? 1.f / gsum : 0.f;

        T *orow = out + row * (int64_t)Tk;
#pragma unroll
        for (int k = 0; k < CPT; ++k) {
            const int c = k * TPR + lane;
            if (valid && c < nchunk) {
                float yv[V];
#pragma unroll
                for (int e = 0; e < V; ++e) yv[e] = z[k][e] * inv;
                st_stream16(orow + c * V, Tr::pack(yv));
            }
        }
    }
}

// ----------------------------------------------------------------------------
// Register-resident backward: dinp = y * (dout - sum(y * dout)).
// ----------------------------------------------------------------------------
template <typename T, int TPR, int CPT>
__global__ void __launch_bounds__(TPR <= 32 ? 256 : TPR)
softmax_bw_vec(T *dinp, const T *dout, const T *y, int64_t rows, int Tk) {
    using Tr = Traits<T>;
    constexpr int V = Tr::kVec;
    constexpr int BLOCK = TPR <= 32 ? 256 : TPR;
    constexpr int G = BLOCK / TPR;
    __shared__ float red[TPR > 32 ? 64 : 1];

    const int lane = threadIdx.x % TPR;
    const int grp = threadIdx.x / TPR;
    const int nchunk = Tk / V;

    for (int64_t base = (int64_t)blockIdx.x * G; base < rows;
         base += (int64_t)gridDim.x * G) {
        const int64_t row = base + grp;
        const bool valid = row < rows;
        const int64_t off = row * (int64_t)Tk;

        uint4 yr[CPT], gr[CPT];
#pragma unroll
        for (int k = 0; k < CPT; ++k) {
            const int c = k * TPR + lane;
            if (valid && c < nchunk) {
                yr[k] = ld_stream16(y + off + c * V);
                gr[k] = ld_stream16(dout + off + c * V);
            } else {
                yr[k] = make_uint4(0u, 0u, 0u, 0u);
                gr[k] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        float s = 0.f;
#pragma unroll
        for (int k = 0; k < CPT; ++k) {
            float yv[V], gv[V];
            Tr::unpack(yr[k], yv);
            Tr::unpack(gr[k], gv);
#pragma unroll
            for (int e = 0; e < V; ++e) s = fmaf(yv[e], gv[e], s);
        }
        s = group_reduce<TPR, OpSum>(s, red);
#pragma unroll
        for (int k = 0; k < CPT; ++k) {
            const int c = k * TPR + lane;
            if (valid && c < nchunk) {
                float yv[V], gv[V], dv[V];
                Tr::unpack(yr[k], yv);
                Tr::unpack(gr[k], gv);
#pragma unroll
                for (int e = 0; e < V; ++e) dv[e] = yv[e] * (gv[e] - s);
                st_stream16(dinp + off + c * V, Tr::pack(dv));
            }
        }
    }
}

// ----------------------------------------------------------------------------
// Looped forward for long, ragged or unaligned rows: scalar accesses, pass 1
// keeps an online (max, sum of exp2) per thread, pass 2 re-reads and writes.
// ----------------------------------------------------------------------------
template <typename T, int TPR>
__global__ void __launch_bounds__(TPR <= 32 ? 256 : TPR)
softmax_fw_loop(T *out, const T *inp, const T *mask, int64_t rows,
                int64_t rows_per_batch, int64_t Tq, int64_t Tk, int causal) {
    using Tr = Traits<T>;
    constexpr int BLOCK = TPR <= 32 ? 256 : TPR;
    constexpr int G = BLOCK / TPR;
    __shared__ float red[TPR > 32 ? 64 : 1];
    const int lane = threadIdx.x % TPR;
    const int grp = threadIdx.x / TPR;

    for (int64_t base = (int64_t)blockIdx.x * G; base < rows;
         base += (int64_t)gridDim.x * G) {
        const int64_t row = base + grp;
        const bool valid = row < rows;
        const int64_t qi = causal ? (valid ? row % Tq : 0) : Tk;
        const int64_t jend = valid ? (qi < Tk ? qi + 1 : Tk) : 0;  // keys past qi are future
        const T *xrow = inp + row * Tk;
        const T *mrow = mask ? mask + (row / rows_per_batch) * Tk : nullptr;

        float m = -INFINITY, s = 0.f;
        for (int64_t j = lane; j < jend; j += TPR) {
            const float mv = mrow ? Tr::load1_cached(mrow + j) : 0.f;
            if (mv == -INFINITY) continue;
            const float z = (Tr::load1(xrow + j) + mv) * kLog2e;
            if (z > m) {  // new running max: rescale what was summed so far
                s = (m == -INFINITY ? 0.f : s * exp2f(m - z)) + 1.f;
                m = z;
            } else {
                s += exp2f(z - m);
            }
        }
        group_ms_merge<TPR>(m, s, red);
        const float inv = (m == -INFINITY || !(s > 0.f)) ? 0.f : 1.f / s;
        if (m == -INFINITY) m = 0.f;

        T *orow = out + row * Tk;
        if (valid) {
            for (int64_t j = lane; j < Tk; j += TPR) {
                float yv = 0.f;
                if (j < jend) {
                    const float mv = mrow ? Tr::load1_cached(mrow + j) : 0.f;
                    if (mv != -INFINITY)
                        yv = exp2f((Tr::load1(xrow + j) + mv) * kLog2e - m) * inv;
                }
                Tr::store1(orow + j, yv);
            }
        }
    }
}

template <typename T, int TPR>
__global__ void __launch_bounds__(TPR <= 32 ? 256 : TPR)
softmax_bw_loop(T *dinp, const T *dout, const T *y, int64_t rows, int64_t Tk) {
    using Tr = Traits<T>;
    constexpr int BLOCK = TPR <= 32 ? 256 : TPR;
    constexpr int G = BLOCK / TPR;
    __shared__ float red[TPR > 32 ? 64 : 1];
    const int lane = threadIdx.x % TPR;
    const int grp = threadIdx.x / TPR;

    for (int64_t base = (int64_t)blockIdx.x * G; base < rows;
         base += (int64_t)gridDim.x * G) {
        const int64_t row = base + grp;
        const bool valid = row < rows;
        const int64_t off = row * Tk;
        float s = 0.f;
        if (valid)
            for (int64_t j = lane; j < Tk; j += TPR)
                s = fmaf(Tr::load1(y + off + j), Tr::load1(dout + off + j), s);
        s = group_reduce<TPR, OpSum>(s, red);
        if (valid)
            for (int64_t j = lane; j < Tk; j += TPR) {
                const float yv = Tr::load1(y + off + j);
                const float gv = Tr::load1(dout + off + j);
                Tr::store1(dinp + off + j, yv * (gv - s));
            }
    }
}

}  // namespace lsr
