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
//
// Each row group owns a contiguous range of rows (rows of one batch entry
// share the mask row) and keeps the next row's chunks in flight while it
// reduces the current one.  Per 16-byte chunk the mask is classified once per
// batch entry: all 0 (add nothing), all -inf (the chunk is neither read nor
// exponentiated; it is written as zeros) or mixed (added element by element).
// Causal rows test keys against the query only in the chunk that holds the
// diagonal; chunks wholly in the future are skipped like masked ones.
// ----------------------------------------------------------------------------
enum : uint32_t { kChunkPlain = 0u, kChunkSkip = 1u, kChunkMixed = 2u };

// Mask class of a 16-byte chunk of T (2 bits).
template <typename T>
__device__ __forceinline__ uint32_t mask_chunk_class(const uint4 &m) {
    using Tr = Traits<T>;
    constexpr int V = Tr::kVec;
    float mv[V];
    Tr::unpack(m, mv);
    bool all_zero = true, all_ninf = true;
#pragma unroll
    for (int e = 0; e < V; ++e) {
        all_zero &= (mv[e] == 0.f);
        all_ninf &= (mv[e] == -INFINITY);
    }
    return all_ninf ? kChunkSkip : (all_zero ? kChunkPlain : kChunkMixed);
}

// Chunk classes (2 bits per chunk) of one thread's chunks for a row: the mask
// classes of the row's batch entry (cached: consecutive rows usually share
// it), then, when causal, chunks wholly after the last visible key `qlim` are
// skipped and the chunk holding it is mixed.
template <typename T, int TPR, int CPT>
struct RowClasses {
    const T *mask;
    int Tk, nchunk, lane;
    int64_t mb = -1;
    uint32_t mcls = 0u;
    __device__ __forceinline__ RowClasses(const T *m, int tk, int lane_)
        : mask(m), Tk(tk), nchunk(tk / Traits<T>::kVec), lane(lane_) {}
    __device__ __forceinline__ uint32_t get(int64_t b, int64_t qlim, int causal) {
        constexpr int V = Traits<T>::kVec;
        uint32_t cls = 0u;
        if (mask) {
            if (b != mb) {
                mb = b;
                mcls = 0u;
                const T *mrow = mask + b * (int64_t)Tk;
#pragma unroll
                for (int k = 0; k < CPT; ++k) {
                    const int c = k * TPR + lane;
                    if (c < nchunk)
                        mcls |= mask_chunk_class<T>(ld_cached16(mrow + c * V)) << (2 * k);
                }
            }
            cls = mcls;
        }
        if (causal) {
#pragma unroll
            for (int k = 0; k < CPT; ++k) {
                const int64_t j0 = (int64_t)(k * TPR + lane) * V;
                const uint32_t cur = (cls >> (2 * k)) & 3u;
                uint32_t nc = cur;
                if (j0 > qlim) nc = kChunkSkip;
                else if (j0 + V - 1 > qlim && cur != kChunkSkip) nc = kChunkMixed;
                cls = (cls & ~(3u << (2 * k))) | (nc << (2 * k));
            }
        }
        return cls;
    }
};

// Position (batch entry, query) of consecutive rows, advanced without
// division: rows of a row group are contiguous.
struct RowPos {
    int64_t b = 0, rem = 0, q = 0;
    __device__ __forceinline__ void init(int64_t row, int64_t rows_per_batch, int64_t Tq) {
        b = row / rows_per_batch;
        rem = row - b * rows_per_batch;
        q = row % Tq;
    }
    __device__ __forceinline__ void next(int64_t rows_per_batch, int64_t Tq) {
        if (++rem == rows_per_batch) {
            rem = 0;
            ++b;
        }
        if (++q == Tq) q = 0;
    }
};

// Shared memory of softmax_fw_vec: S stages of CPT 16-byte chunks per thread,
// plus one word of chunk-class bits per thread and stage.
template <int TPR, int CPT, int S>
constexpr size_t softmax_fw_smem() {
    return (size_t)S * (TPR <= 32 ? 256 : TPR) * (CPT * 16 + 4);
}

template <typename T, int TPR, int CPT, int S, bool SCALED>
__global__ void __launch_bounds__(TPR <= 32 ? 256 : TPR, (softmax_fw_min_blocks<TPR, CPT>()))
softmax_fw_vec(T *out, const T *inp, const T *mask, int64_t rows,
               int64_t rows_per_batch, int64_t Tq, int Tk, int causal, int64_t qoff,
               float scale) {
    pdl_begin();
    using Tr = Traits<T>;
    constexpr int V = Tr::kVec;
    constexpr int H2 = V / 2;
    constexpr int BLOCK = TPR <= 32 ? 256 : TPR;
    constexpr int G = BLOCK / TPR;  // row groups per block
    static_assert(2 * CPT <= 32, "class bits");
    extern __shared__ uint4 dsmem[];
    uint4 *stage = dsmem;                                                  // [S][CPT][BLOCK]
    uint32_t *clsb = reinterpret_cast<uint32_t *>(dsmem + S * CPT * BLOCK);  // [S][BLOCK]
    __shared__ float red[TPR > 32 ? 64 : 1];

    const int tid = threadIdx.x;
    const int lane = tid % TPR;
    const int grp = tid / TPR;
    const int nchunk = Tk / V;
    const int64_t ngroups = (int64_t)gridDim.x * G;
    const int64_t per = (rows + ngroups - 1) / ngroups;  // rows per group (uniform)
    const int64_t rbeg = ((int64_t)blockIdx.x * G + grp) * per;
    const int64_t rend = rbeg + per < rows ? rbeg + per : rows;

    RowClasses<T, TPR, CPT> classes(mask, Tk, lane);

    // Issue the copies of the next row into stage s (an empty group past the end).
    RowPos ip;
    if (rbeg < rend) ip.init(rbeg, rows_per_batch, Tq);
    int64_t inext = rbeg;
    auto issue = [&](int s) {
        if (inext < rend) {
            const uint32_t cls = classes.get(ip.b, ip.q + qoff, causal);
            clsb[s * BLOCK + tid] = cls;
            const T *xrow = inp + inext * (int64_t)Tk;
#pragma unroll
            for (int k = 0; k < CPT; ++k) {
                const int c = k * TPR + lane;
                if (c < nchunk && ((cls >> (2 * k)) & 3u) != kChunkSkip)
                    cp_async16(&stage[(s * CPT + k) * BLOCK + tid], xrow + c * V);
            }
            ip.next(rows_per_batch, Tq);
        }
        ++inext;
        cp_async_commit();
    };
#pragma unroll
    for (int s = 0; s < S - 1; ++s) issue(s);

    RowPos cp;
    if (rbeg < rend) cp.init(rbeg, rows_per_batch, Tq);
    int s_cur = 0, s_iss = S - 1;
    for (int64_t k = 0; k < per; ++k) {
        issue(s_iss);
        s_iss = s_iss + 1 == S ? 0 : s_iss + 1;
        cp_async_wait<S - 1>();  // this thread's copies of row k have landed

        const int64_t row = rbeg + k;
        const bool valid = row < rend;
        const uint32_t ccls = valid ? clsb[s_cur * BLOCK + tid] : 0u;
        const int qi = (valid && causal) ? (int)(cp.q + qoff) : Tk;  // last visible key
        const T *mrow = (valid && mask) ? mask + cp.b * (int64_t)Tk : nullptr;

        // SCALED: plain chunks keep x (their maximum mp is scaled once,
        // below) and mixed chunks hold z = scale * x + mask; otherwise scale
        // is 1 and every chunk holds z
        float2 v[CPT][H2];
        float m = -INFINITY, mp = -INFINITY;
#pragma unroll
        for (int kk = 0; kk < CPT; ++kk) {
            const int c = kk * TPR + lane;
            const uint32_t cls = (ccls >> (2 * kk)) & 3u;
            if (valid && c < nchunk && cls != kChunkSkip) {
                unpack2<T>(stage[(s_cur * CPT + kk) * BLOCK + tid], v[kk]);
                if (cls == kChunkMixed) {
                    float2 mv[H2];
#pragma unroll
                    for (int h = 0; h < H2; ++h) mv[h] = f2(0.f);
                    if (mrow) unpack2<T>(ld_cached16(mrow + c * V), mv);
#pragma unroll
                    for (int h = 0; h < H2; ++h) {
                        const int j = c * V + 2 * h;
                        if constexpr (SCALED) {
                            v[kk][h].x = j > qi ? -INFINITY : fmaf(v[kk][h].x, scale, mv[h].x);
                            v[kk][h].y = j + 1 > qi ? -INFINITY : fmaf(v[kk][h].y, scale, mv[h].y);
                        } else {
                            v[kk][h].x = j > qi ? -INFINITY : v[kk][h].x + mv[h].x;
                            v[kk][h].y = j + 1 > qi ? -INFINITY : v[kk][h].y + mv[h].y;
                        }
                    }
#pragma unroll
                    for (int h = 0; h < H2; ++h) m = fmax3(m, v[kk][h].x, v[kk][h].y);
                } else {
#pragma unroll
                    for (int h = 0; h < H2; ++h) mp = fmax3(mp, v[kk][h].x, v[kk][h].y);
                }
            }
        }
        // scale > 0: the maximum of scale * x is scale * mp
        m = fmaxf(m, SCALED ? mp * scale : mp);
        m = group_reduce<TPR, OpMax>(m, red);
        // e = 2^(z*log2e - m*log2e), z*log2e taken as x*(scale*log2e) on plain
        // chunks; a row with no visible key sums to 0
        const float mL = m == -INFINITY ? 0.f : m * kLog2e;
        const float sl2 = SCALED ? scale * kLog2e : kLog2e;
        float2 sum2 = f2(0.f);
#pragma unroll
        for (int kk = 0; kk < CPT; ++kk) {
            const int c = kk * TPR + lane;
            const uint32_t cls = (ccls >> (2 * kk)) & 3u;
            if (valid && c < nchunk && cls != kChunkSkip) {
                const float2 mul = f2((!SCALED || cls == kChunkMixed) ? kLog2e : sl2);
#pragma unroll
                for (int h = 0; h < H2; ++h) {
                    float2 t = fma2(v[kk][h], mul, f2(-mL));
                    t.x = fast_exp2(t.x);
                    t.y = fast_exp2(t.y);
                    v[kk][h] = t;
                    sum2 = add2(sum2, t);
                }
            }
        }
        const float sum = group_reduce<TPR, OpSum>(sum2.x + sum2.y, red);
        const float2 inv = f2(sum > 0.f ? 1.f / sum : 0.f);

        T *orow = out + row * (int64_t)Tk;
#pragma unroll
        for (int kk = 0; kk < CPT; ++kk) {
            const int c = kk * TPR + lane;
            const uint32_t cls = (ccls >> (2 * kk)) & 3u;
            if (valid && c < nchunk) {
                float2 yv[H2];
#pragma unroll
                for (int h = 0; h < H2; ++h)
                    yv[h] = cls == kChunkSkip ? f2(0.f) : mul2(v[kk][h], inv);
                st_stream16(orow + c * V, pack2<T>(yv));
            }
        }
        if (valid) cp.next(rows_per_batch, Tq);
        s_cur = s_cur + 1 == S ? 0 : s_cur + 1;
    }
}

// ----------------------------------------------------------------------------
// Register-resident backward: dinp = y * (dout - sum(y * dout)).
// ----------------------------------------------------------------------------
template <typename T, int TPR, int CPT>
__global__ void __launch_bounds__(TPR <= 32 ? 256 : TPR)
softmax_bw_vec(T *dinp, const T *dout, const T *y, int64_t rows, int Tk) {
    pdl_begin();
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
                int64_t rows_per_batch, int64_t Tq, int64_t Tk, int causal, int64_t qoff,
                float scale) {
    pdl_begin();
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
        const int64_t qi = causal ? (valid ? row % Tq + qoff : 0) : Tk;  // last visible key
        const int64_t jend = valid ? (qi < Tk ? qi + 1 : Tk) : 0;  // keys past qi are future
        const T *xrow = inp + row * Tk;
        const T *mrow = mask ? mask + (row / rows_per_batch) * Tk : nullptr;

        float m = -INFINITY, s = 0.f;
        for (int64_t j = lane; j < jend; j += TPR) {
            const float mv = mrow ? Tr::load1_cached(mrow + j) : 0.f;
            if (mv == -INFINITY) continue;
            const float z = fmaf(Tr::load1(xrow + j), scale, mv) * kLog2e;
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
                        yv = exp2f(fmaf(Tr::load1(xrow + j), scale, mv) * kLog2e - m) * inv;
                }
                Tr::store1(orow + j, yv);
            }
        }
    }
}

template <typename T, int TPR>
__global__ void __launch_bounds__(TPR <= 32 ? 256 : TPR)
softmax_bw_loop(T *dinp, const T *dout, const T *y, int64_t rows, int64_t Tk) {
    pdl_begin();
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

// ----------------------------------------------------------------------------
// Masked backward: dinp_j = scale * y_j (dout_j - sum over visible k of
// y_k dout_k) on visible keys, 0 elsewhere.  Chunks whose keys are all
// invisible (mask -inf, or causal future) are neither read nor summed; they
// are written as zeros.  This form serves rows of up to three chunks per
// thread: same row mapping as softmax_bw_vec (rows strided over the grid);
// each row finds its batch entry and query by division and classifies its
// mask chunks afresh (the mask row stays in L1), so nothing is carried from
// row to row and the kernel stays near the plain backward's register budget
// and occupancy.  Longer rows take softmax_bw_masked_runs below.
// ----------------------------------------------------------------------------
template <typename T, int TPR, int CPT>
__global__ void __launch_bounds__(TPR <= 32 ? 256 : TPR)
softmax_bw_masked_vec(T *dinp, const T *dout, const T *y, const T *mask, int64_t rows,
                      int64_t rows_per_batch, int64_t Tq, int Tk, int causal, int64_t qoff,
                      float scale) {
    pdl_begin();
    using Tr = Traits<T>;
    constexpr int V = Tr::kVec;
    constexpr int H2 = V / 2;
    constexpr int BLOCK = TPR <= 32 ? 256 : TPR;
    constexpr int G = BLOCK / TPR;
    __shared__ float red[TPR > 32 ? 64 : 1];

    const int lane = threadIdx.x % TPR;
    const int grp = threadIdx.x / TPR;
    const int nchunk = Tk / V;
    const bool narrow = rows <= INT32_MAX && rows_per_batch <= INT32_MAX && Tq <= INT32_MAX;

    for (int64_t base = (int64_t)blockIdx.x * G; base < rows;
         base += (int64_t)gridDim.x * G) {
        const int64_t row = base + grp;
        const bool valid = row < rows;
        const int64_t off = row * (int64_t)Tk;
        // batch entry and last visible key of this row
        int64_t b = 0, q = 0;
        if (valid && (mask || causal)) {
            if (narrow) {
                const uint32_t r32 = (uint32_t)row;
                b = r32 / (uint32_t)rows_per_batch;
                q = causal ? r32 % (uint32_t)Tq : 0;
            } else {
                b = row / rows_per_batch;
                q = causal ? row % Tq : 0;
            }
        }
        const int64_t qi = causal ? q + qoff : (int64_t)Tk;
        const T *mrow = (valid && mask) ? mask + b * (int64_t)Tk : nullptr;

        uint4 yr[CPT], gr[CPT];
        uint32_t vis[CPT];  // visible elements of each chunk (bit e)
#pragma unroll
        for (int kk = 0; kk < CPT; ++kk) {
            const int c = kk * TPR + lane;
            yr[kk] = gr[kk] = make_uint4(0u, 0u, 0u, 0u);
            vis[kk] = 0u;
            if (!valid || c >= nchunk) continue;
            uint32_t bits = (1u << V) - 1u;
            if (mrow) {
                float mv[V];
                Tr::unpack(ld_cached16(mrow + c * V), mv);
                bits = 0u;
#pragma unroll
                for (int e = 0; e < V; ++e) bits |= (mv[e] != -INFINITY ? 1u : 0u) << e;
            }
            if (causal) {
                const int64_t j0 = (int64_t)c * V;
#pragma unroll
                for (int e = 0; e < V; ++e)
                    if (j0 + e > qi) bits &= ~(1u << e);
            }
            vis[kk] = bits;
            if (bits) {
                yr[kk] = ld_stream16(y + off + c * V);
                gr[kk] = ld_stream16(dout + off + c * V);
            }
        }
        float2 s2 = f2(0.f);
#pragma unroll
        for (int kk = 0; kk < CPT; ++kk) {
            float2 yv[H2], gv[H2];
            unpack2<T>(yr[kk], yv);
            unpack2<T>(gr[kk], gv);
            if (vis[kk] == (1u << V) - 1u) {
#pragma unroll
                for (int h = 0; h < H2; ++h) s2 = fma2(yv[h], gv[h], s2);
            } else {
#pragma unroll
                for (int h = 0; h < H2; ++h) {
                    const float2 p = mul2(yv[h], gv[h]);
                    s2.x += (vis[kk] >> (2 * h)) & 1u ? p.x : 0.f;
                    s2.y += (vis[kk] >> (2 * h + 1)) & 1u ? p.y : 0.f;
                }
            }
        }
        const float s = group_reduce<TPR, OpSum>(s2.x + s2.y, red);
#pragma unroll
        for (int kk = 0; kk < CPT; ++kk) {
            const int c = kk * TPR + lane;
            if (valid && c < nchunk) {
                float2 yv[H2], gv[H2], dv[H2];
                unpack2<T>(yr[kk], yv);
                unpack2<T>(gr[kk], gv);
#pragma unroll
                for (int h = 0; h < H2; ++h) {
                    // scale * y * (g - s), with scale folded into the difference
                    const float2 t = mul2(yv[h], fma2(gv[h], f2(scale), f2(-s * scale)));
                    dv[h].x = (vis[kk] >> (2 * h)) & 1u ? t.x : 0.f;
                    dv[h].y = (vis[kk] >> (2 * h + 1)) & 1u ? t.y : 0.f;
                }
                st_stream16(dinp + off + c * V, pack2<T>(dv));
            }
        }
    }
}

// ----------------------------------------------------------------------------
// Masked backward for rows of four or more chunks per thread: each row group
// takes a contiguous run of rows, so the mask chunk classes are cached per
// batch entry (RowClasses) and the row position advances without division
// (RowPos); per-element visibility is kept for every chunk.
// ----------------------------------------------------------------------------
template <typename T, int TPR, int CPT>
__global__ void __launch_bounds__(TPR <= 32 ? 256 : TPR)
softmax_bw_masked_runs(T *dinp, const T *dout, const T *y, const T *mask, int64_t rows,
                      int64_t rows_per_batch, int64_t Tq, int Tk, int causal, int64_t qoff,
                      float scale) {
    pdl_begin();
    using Tr = Traits<T>;
    constexpr int V = Tr::kVec;
    constexpr int H2 = V / 2;
    constexpr int BLOCK = TPR <= 32 ? 256 : TPR;
    constexpr int G = BLOCK / TPR;
    __shared__ float red[TPR > 32 ? 64 : 1];

    const int lane = threadIdx.x % TPR;
    const int grp = threadIdx.x / TPR;
    const int nchunk = Tk / V;
    const int64_t ngroups = (int64_t)gridDim.x * G;
    const int64_t per = (rows + ngroups - 1) / ngroups;
    const int64_t rbeg = ((int64_t)blockIdx.x * G + grp) * per;
    const int64_t rend = rbeg + per < rows ? rbeg + per : rows;
    RowClasses<T, TPR, CPT> classes(mask, Tk, lane);
    RowPos pos;
    if (rbeg < rend) pos.init(rbeg, rows_per_batch, Tq);

    for (int64_t k = 0; k < per; ++k) {
        const int64_t row = rbeg + k;
        const bool valid = row < rend;
        const int64_t off = row * (int64_t)Tk;
        const uint32_t ccls = valid ? classes.get(pos.b, pos.q + qoff, causal) : 0u;
        const int qi = (valid && causal) ? (int)(pos.q + qoff) : Tk;
        const T *mrow = (valid && mask) ? mask + pos.b * (int64_t)Tk : nullptr;

        uint4 yr[CPT], gr[CPT];
#pragma unroll
        for (int kk = 0; kk < CPT; ++kk) {
            const int c = kk * TPR + lane;
            const uint32_t cls = (ccls >> (2 * kk)) & 3u;
            if (valid && c < nchunk && cls != kChunkSkip) {
                yr[kk] = ld_stream16(y + off + c * V);
                gr[kk] = ld_stream16(dout + off + c * V);
            } else {
                yr[kk] = make_uint4(0u, 0u, 0u, 0u);
                gr[kk] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        // visibility of the elements of mixed chunks (mask -inf or future)
        uint32_t vis[CPT];
#pragma unroll
        for (int kk = 0; kk < CPT; ++kk) {
            const int c = kk * TPR + lane;
            const uint32_t cls = (ccls >> (2 * kk)) & 3u;
            vis[kk] = cls == kChunkSkip ? 0u : (1u << V) - 1u;
            if (valid && c < nchunk && cls == kChunkMixed) {
                float mv[V];
#pragma unroll
                for (int e = 0; e < V; ++e) mv[e] = 0.f;
                if (mrow) Tr::unpack(ld_cached16(mrow + c * V), mv);
                uint32_t bits = 0u;
#pragma unroll
                for (int e = 0; e < V; ++e)
                    if (mv[e] != -INFINITY && c * V + e <= qi) bits |= 1u << e;
                vis[kk] = bits;
            }
        }
        float2 s2 = f2(0.f);
#pragma unroll
        for (int kk = 0; kk < CPT; ++kk) {
            float2 yv[H2], gv[H2];
            unpack2<T>(yr[kk], yv);
            unpack2<T>(gr[kk], gv);
#pragma unroll
            for (int h = 0; h < H2; ++h) {
                const float2 p = mul2(yv[h], gv[h]);
                s2.x += (vis[kk] >> (2 * h)) & 1u ? p.x : 0.f;
                s2.y += (vis[kk] >> (2 * h + 1)) & 1u ? p.y : 0.f;
            }
        }
        const float s = group_reduce<TPR, OpSum>(s2.x + s2.y, red);
#pragma unroll
        for (int kk = 0; kk < CPT; ++kk) {
            const int c = kk * TPR + lane;
            if (valid && c < nchunk) {
                float2 yv[H2], gv[H2], dv[H2];
                unpack2<T>(yr[kk], yv);
                unpack2<T>(gr[kk], gv);
#pragma unroll
                for (int h = 0; h < H2; ++h) {
                    // scale * y * (g - s), with scale folded into the difference
                    const float2 t = mul2(yv[h], fma2(gv[h], f2(scale), f2(-s * scale)));
                    dv[h].x = (vis[kk] >> (2 * h)) & 1u ? t.x : 0.f;
                    dv[h].y = (vis[kk] >> (2 * h + 1)) & 1u ? t.y : 0.f;
                }
                st_stream16(dinp + off + c * V, pack2<T>(dv));
            }
        }
        if (valid) pos.next(rows_per_batch, Tq);
    }
}

// Looped masked backward (scalar accesses; long, ragged or unaligned rows).
template <typename T, int TPR>
__global__ void __launch_bounds__(TPR <= 32 ? 256 : TPR)
softmax_bw_masked_loop(T *dinp, const T *dout, const T *y, const T *mask, int64_t rows,
                       int64_t rows_per_batch, int64_t Tq, int64_t Tk, int causal,
                       int64_t qoff, float scale) {
    pdl_begin();
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
        const int64_t qi = causal ? (valid ? row % Tq + qoff : 0) : Tk;
        const int64_t jend = valid ? (qi < Tk ? qi + 1 : Tk) : 0;
        const T *mrow = (valid && mask) ? mask + (row / rows_per_batch) * Tk : nullptr;
        float s = 0.f;
        for (int64_t j = lane; j < jend; j += TPR) {
            if (mrow && Tr::load1_cached(mrow + j) == -INFINITY) continue;
            s += __fmul_rn(Tr::load1(y + off + j), Tr::load1(dout + off + j));
        }
        s = group_reduce<TPR, OpSum>(s, red);
        if (valid)
            for (int64_t j = lane; j < Tk; j += TPR) {
                float d = 0.f;
                if (j < jend && !(mrow && Tr::load1_cached(mrow + j) == -INFINITY))
                    d = Tr::load1(y + off + j) * fmaf(Tr::load1(dout + off + j), scale, -s * scale);
                Tr::store1(dinp + off + j, d);
            }
    }
}

}  // namespace lsr
