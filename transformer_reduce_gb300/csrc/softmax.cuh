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
//    are never read when the mask is a window of visible keys (a padding
//    mask): a whole 16-byte chunk of them costs no HBM traffic.
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
// A padding mask (additive, 0 on the keys a batch entry may attend to, -inf
// on the others) almost always makes every row's visible keys one window
// [lo, hi) of the row.  Each block therefore first classifies the mask rows
// of the batch entries its rows belong to: a row whose elements are all 0 or
// -inf and whose non-(-inf) keys are contiguous is the window [lo, hi); any
// other row (finite non-zero biases, -inf holes inside the window) is
// "general".  Per row, causal masking only lowers hi to the last visible key
// + 1.  A chunk of V keys is then visible, fully visible or invisible by two
// integer compares; invisible chunks are neither read nor exponentiated and
// are written as zeros, and only the (at most two) chunks straddling lo or hi
// need per-element work.  Rows of a general batch entry add the mask element
// by element (and mask future keys one by one when causal); that path is
// exact, just not the fast one.
//
// Each row group owns a contiguous range of rows and keeps the next S-1
// rows' visible chunks in flight (cp.async into shared memory; each thread
// reads back only its own slots) while it reduces the current one.
// ----------------------------------------------------------------------------
constexpr int kWinMax = 64;        // batch entries a block classifies at most
constexpr int kWinGeneral = -1;    // lo of a mask row that is not a window

// Window [lo, hi) of the mask row of one batch entry, found by one warp
// (every lane returns it); lo = kWinGeneral for a row that is not a window.
// A row with no visible key is the empty window [0, 0).  ADDS: the forward,
// which adds the mask, needs every element to be 0 or -inf; the masked
// backward only needs the keys that are not -inf to be contiguous.
template <typename T, bool ADDS>
__device__ __forceinline__ int2 mask_row_window(const T *mrow, int Tk) {
    using Tr = Traits<T>;
    constexpr int V = Tr::kVec;
    const int lane = threadIdx.x & 31;
    const int nchunk = Tk / V;
    int first = Tk, last = -1, count = 0, other = 0;
    for (int c = lane; c < nchunk; c += 32) {
        float mv[V];
        Tr::unpack(ld_cached16(mrow + c * V), mv);
#pragma unroll
        for (int e = 0; e < V; ++e) {
            const bool ninf = mv[e] == -INFINITY;
            if (ADDS) other |= !(ninf || mv[e] == 0.f);
            if (!ninf) {
                first = min(first, c * V + e);
                last = max(last, c * V + e);
                ++count;
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        first = min(first, __shfl_xor_sync(0xffffffffu, first, o));
        last = max(last, __shfl_xor_sync(0xffffffffu, last, o));
        count += __shfl_xor_sync(0xffffffffu, count, o);
        other |= __shfl_xor_sync(0xffffffffu, other, o);
    }
    if (other || (count > 0 && count != last - first + 1)) return make_int2(kWinGeneral, 0);
    return count == 0 ? make_int2(0, 0) : make_int2(first, last + 1);
}

// Shared memory of softmax_fw_vec: S stages of CPT 16-byte chunks per
// thread, plus each thread's (lo, hi) of the row in that stage.
template <int TPR, int CPT, int S>
constexpr size_t softmax_fw_smem() {
    return (size_t)S * (TPR <= 32 ? 256 : TPR) * (CPT * 16 + 8);
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
    extern __shared__ uint4 dsmem[];
    uint4 *stage = dsmem;                                              // [S][CPT][BLOCK]
    int2 *winb = reinterpret_cast<int2 *>(dsmem + S * CPT * BLOCK);    // [S][BLOCK]
    __shared__ float red[TPR > 32 ? 64 : 1];
    __shared__ int2 wtab[kWinMax];

    const int tid = threadIdx.x;
    const int lane = tid % TPR;
    const int grp = tid / TPR;
    const int64_t ngroups = (int64_t)gridDim.x * G;
    const int per = (int)((rows + ngroups - 1) / ngroups);  // rows per group (uniform)
    const int64_t rbeg = ((int64_t)blockIdx.x * G + grp) * per;
    const int64_t rend = rbeg + per < rows ? rbeg + per : rows;

    // Windows of the batch entries this block's rows belong to (one warp per
    // entry).  A block spanning more than kWinMax entries treats every mask
    // row as general.
    const int64_t blk0 = (int64_t)blockIdx.x * G * per;
    const int64_t b_first = blk0 < rows ? blk0 / rows_per_batch : 0;
    bool general = false;
    if (mask) {
        const int64_t blk1 = min(rows, blk0 + (int64_t)G * per);
        const int64_t nb = blk1 > blk0 ? (blk1 - 1) / rows_per_batch - b_first + 1 : 0;
        if (nb > kWinMax) {
            general = true;
        } else {
            for (int i = tid >> 5; i < nb; i += BLOCK / 32) {
                const int2 w = mask_row_window<T, true>(mask + (b_first + i) * (int64_t)Tk, Tk);
                if ((tid & 31) == 0) wtab[i] = w;
            }
            __syncthreads();
        }
    }

    // Row cursor for issuing: batch entry (relative to the block's first),
    // position in the batch entry and query index, advanced without
    // division (the launcher keeps rows below 2^31, so they fit 32 bits).
    const int rpb = (int)rows_per_batch, tq = (int)Tq, qo = (int)qoff;
    int ib = 0, irem = 0, iq = 0;
    if (rbeg < rend) {
        const int64_t b = rbeg / rows_per_batch;
        ib = (int)(b - b_first);
        irem = (int)(rbeg - b * rows_per_batch);
        iq = (int)(rbeg % Tq);
    }
    const T *xnext = inp + rbeg * (int64_t)Tk;
    int64_t inext = rbeg;
    // Issue the copies of the next row's visible chunks into stage s and
    // record the row's window (an empty group past the end).
    auto issue = [&](int s) {
        if (inext < rend) {
            int lo = 0, hi = Tk;
            if (general) {
                lo = kWinGeneral;
            } else if (mask) {
                const int2 w = wtab[ib];
                lo = w.x;
                if (w.x != kWinGeneral) hi = w.y;
            }
            if (causal) hi = min(hi, iq + qo + 1);  // query iq sees keys j <= iq + qoff
            winb[s * BLOCK + tid] = make_int2(lo, hi);
            const int lo_ld = max(lo, 0);
#pragma unroll
            for (int k = 0; k < CPT; ++k) {
                const int j0 = (k * TPR + lane) * V;
                if (j0 < hi && j0 + V > lo_ld)
                    cp_async16(&stage[(s * CPT + k) * BLOCK + tid], xnext + j0);
            }
            xnext += Tk;
            if (++irem == rpb) {
                irem = 0;
                ++ib;
            }
            if (++iq == tq) iq = 0;
        }
        ++inext;
        cp_async_commit();
    };
#pragma unroll
    for (int s = 0; s < S - 1; ++s) issue(s);

    T *orow = out + rbeg * (int64_t)Tk;
    int s_cur = 0, s_iss = S - 1;
    for (int k = 0; k < per; ++k) {
        issue(s_iss);
        s_iss = s_iss + 1 == S ? 0 : s_iss + 1;
        cp_async_wait<S - 1>();  // this thread's copies of row k have landed

        const bool valid = rbeg + k < rend;
        const int2 w = valid ? winb[s_cur * BLOCK + tid] : make_int2(0, 0);
        const bool gen = w.x == kWinGeneral;
        const int lo = gen ? 0 : w.x, hi = w.y;
        const T *mrow = nullptr;  // the mask row, general rows only
        if (gen) mrow = mask + ((rbeg + k) / rows_per_batch) * (int64_t)Tk;

        // v holds x (window rows; SCALED: the maximum is scaled once below)
        // or z = scale * x + mask (general rows); -inf on invisible keys
        float2 v[CPT][H2];
        float m = -INFINITY;
#pragma unroll
        for (int kk = 0; kk < CPT; ++kk) {
            const int j0 = (kk * TPR + lane) * V;
            if (j0 < hi && j0 + V > lo) {
                unpack2<T>(stage[(s_cur * CPT + kk) * BLOCK + tid], v[kk]);
                if (gen) {
                    float2 mv[H2];
                    unpack2<T>(ld_cached16(mrow + j0), mv);
#pragma unroll
                    for (int h = 0; h < H2; ++h) {
                        // keys masked with -inf or in the causal future are
                        // -inf whatever their score
                        const int j = j0 + 2 * h;
                        const float zx = SCALED ? fmaf(v[kk][h].x, scale, mv[h].x)
                                                : v[kk][h].x + mv[h].x;
                        const float zy = SCALED ? fmaf(v[kk][h].y, scale, mv[h].y)
                                                : v[kk][h].y + mv[h].y;
                        v[kk][h].x = (j < hi && mv[h].x != -INFINITY) ? zx : -INFINITY;
                        v[kk][h].y = (j + 1 < hi && mv[h].y != -INFINITY) ? zy : -INFINITY;
                    }
                } else if (j0 < lo || j0 + V > hi) {
#pragma unroll
                    for (int h = 0; h < H2; ++h) {
                        const int j = j0 + 2 * h;
                        if (j < lo || j >= hi) v[kk][h].x = -INFINITY;
                        if (j + 1 < lo || j + 1 >= hi) v[kk][h].y = -INFINITY;
                    }
                }
#pragma unroll
                for (int h = 0; h < H2; ++h) m = fmax3(m, v[kk][h].x, v[kk][h].y);
            }
        }
        m = group_reduce<TPR, OpMax>(m, red);
        // e = 2^(v * mul - m * log2e); window rows of the scaled softmax hold
        // x, whose maximum times scale (> 0) is the maximum of scale * x
        if (SCALED && !gen) m *= scale;
        const float mL = m == -INFINITY ? 0.f : m * kLog2e;  // a row with no visible key sums to 0
        const float2 mul = f2(SCALED && !gen ? scale * kLog2e : kLog2e);
        float2 sum2 = f2(0.f);
#pragma unroll
        for (int kk = 0; kk < CPT; ++kk) {
            const int j0 = (kk * TPR + lane) * V;
            if (j0 < hi && j0 + V > lo) {
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
        const float2 inv = f2(sum > 0.f ? fast_rcp(sum) : 0.f);

        if (valid) {
#pragma unroll
            for (int kk = 0; kk < CPT; ++kk) {
                const int j0 = (kk * TPR + lane) * V;
                if (j0 < Tk) {
                    uint4 o = make_uint4(0u, 0u, 0u, 0u);
                    if (j0 < hi && j0 + V > lo) {
                        float2 yv[H2];
#pragma unroll
                        for (int h = 0; h < H2; ++h) yv[h] = mul2(v[kk][h], inv);
                        o = pack2<T>(yv);
                    }
                    st_stream16(orow + j0, o);
                }
            }
        }
        orow += Tk;
        s_cur = s_cur + 1 == S ? 0 : s_cur + 1;
    }
}

// ----------------------------------------------------------------------------
// Register-resident backward: dinp = y * (dout - sum(y * dout)).
// ----------------------------------------------------------------------------
// The three-chunk bucket is compiled for three resident 256-thread blocks
// (up to 85 registers): left to its own heuristic ptxas keeps it at 64
// registers with a spill.  0 leaves the other buckets to that heuristic
// (as if no minimum were given; an explicit 1 would let ptxas take more
// registers than the heuristic picks).
template <int TPR, int CPT>
constexpr int softmax_bw_min_blocks() { return TPR <= 32 && CPT == 3 ? 3 : 0; }

template <typename T, int TPR, int CPT>
__global__ void __launch_bounds__(TPR <= 32 ? 256 : TPR, (softmax_bw_min_blocks<TPR, CPT>()))
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
// y_k dout_k) on visible keys, 0 elsewhere.  A key is visible when its mask
// element is not -inf and, when causal, it is not in the query's future.
// As in the forward, each block first finds the window [lo, hi) of visible
// keys of every batch entry it touches (mask rows whose visible keys are not
// contiguous are "general": their rows test the mask element by element),
// and each row group takes a contiguous run of rows, its position advanced
// without division.  Chunks with no visible key are neither read nor summed
// and are written as zeros; only the chunks straddling lo or hi (and every
// chunk of a general row) select element by element.  Rows are loaded
// straight into registers (y and dout, CPT chunks each), as in the plain
// backward.
// ----------------------------------------------------------------------------
// Bit mask (one bit per element of a 16-byte chunk of V keys starting at
// key j0) of the visible keys: inside [lo, hi) and, for a general row (mrow
// = its mask row, else nullptr), with a mask element that is not -inf.
template <typename T>
__device__ __forceinline__ uint32_t chunk_visible_bits(const T *mrow, int j0, int lo, int hi) {
    using Tr = Traits<T>;
    constexpr int V = Tr::kVec;
    uint32_t bits = 0u;
#pragma unroll
    for (int e = 0; e < V; ++e) bits |= (j0 + e >= lo && j0 + e < hi ? 1u : 0u) << e;
    if (mrow) {
        float mv[V];
        Tr::unpack(ld_cached16(mrow + j0), mv);
#pragma unroll
        for (int e = 0; e < V; ++e)
            if (mv[e] == -INFINITY) bits &= ~(1u << e);
    }
    return bits;
}

// AND mask of the 32-bit word w of a 16-byte chunk that keeps the elements
// whose bits are set in `bits` and clears the others (to +0).
template <typename T>
__device__ __forceinline__ uint32_t keep_word(uint32_t bits, int w) {
    if constexpr (Traits<T>::kVec == 4) {
        return (bits >> w) & 1u ? 0xffffffffu : 0u;
    } else {
        return ((bits >> (2 * w)) & 1u ? 0x0000ffffu : 0u) |
               ((bits >> (2 * w + 1)) & 1u ? 0xffff0000u : 0u);
    }
}
template <typename T>
__device__ __forceinline__ void keep_elements(uint4 &u, uint32_t bits) {
    u.x &= keep_word<T>(bits, 0);
    u.y &= keep_word<T>(bits, 1);
    u.z &= keep_word<T>(bits, 2);
    u.w &= keep_word<T>(bits, 3);
}

// Masked backward: dinp_j = scale * y_j (dout_j - sum over visible k of
// y_k dout_k) on visible keys, 0 elsewhere.  A key is visible when its mask
// element is not -inf and, when causal, it is not in the query's future.
// The plain backward's structure (y and dout straight into registers, CPT
// chunks each, one fused multiply-add per element pair for the sum) with the
// forward's windows: each block first finds the window [lo, hi) of visible
// keys of every batch entry it touches (mask rows whose visible keys are not
// contiguous are "general"), each row group takes a contiguous run of rows
// and advances its position without division.  Chunks with no visible key
// are neither read nor summed and are written as zeros; in the chunks that
// straddle lo or hi (every chunk of a general row) the invisible elements of
// y and dout are cleared to 0 before the arithmetic, so they add nothing to
// the sum and their output is 0, whatever the memory held there.
//
// Resident blocks per SM asked of ptxas: four 256-thread blocks for the
// two-chunk bucket (64 registers; left alone ptxas keeps the unpacked rows
// live across the reduction and takes 96, five spill), fewer for wider rows,
// 768 threads per SM for multi-warp rows (85 registers; left alone ptxas
// takes 127 for 256-thread rows), and 0 (its own heuristic) where a cap
// would spill.
template <int TPR, int CPT>
constexpr int softmax_bw_masked_min_blocks() {
    return TPR <= 32 ? (CPT <= 1 ? 5 : CPT <= 2 ? 4 : CPT <= 3 ? 3 : CPT <= 6 ? 2 : 0)
                     : (TPR <= 256 ? 768 / TPR : 0);
}

template <typename T, int TPR, int CPT>
__global__ void __launch_bounds__(TPR <= 32 ? 256 : TPR, (softmax_bw_masked_min_blocks<TPR, CPT>()))
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
    __shared__ int2 wtab[kWinMax];

    const int tid = threadIdx.x;
    const int lane = tid % TPR;
    const int grp = tid / TPR;
    const int64_t ngroups = (int64_t)gridDim.x * G;
    const int per = (int)((rows + ngroups - 1) / ngroups);
    const int64_t rbeg = ((int64_t)blockIdx.x * G + grp) * per;
    const int nrow = (int)max((int64_t)0, min((int64_t)per, rows - rbeg));  // this group's rows

    const int64_t blk0 = (int64_t)blockIdx.x * G * per;
    const int64_t b_first = blk0 < rows ? blk0 / rows_per_batch : 0;
    bool general = false;
    if (mask) {
        const int64_t blk1 = min(rows, blk0 + (int64_t)G * per);
        const int64_t nb = blk1 > blk0 ? (blk1 - 1) / rows_per_batch - b_first + 1 : 0;
        if (nb > kWinMax) {
            general = true;
        } else {
            for (int i = tid >> 5; i < nb; i += BLOCK / 32) {
                const int2 w = mask_row_window<T, false>(mask + (b_first + i) * (int64_t)Tk, Tk);
                if ((tid & 31) == 0) wtab[i] = w;
            }
            __syncthreads();
        }
    }

    int ib = 0, irem = 0, iq = 0;
    if (nrow > 0) {
        const int64_t b = rbeg / rows_per_batch;
        ib = (int)(b - b_first);
        irem = (int)(rbeg - b * rows_per_batch);
        iq = (int)(rbeg % Tq);
    }
    const int j_lane = lane * V;
    int64_t off = rbeg * (int64_t)Tk;
    for (int k = 0; k < per; ++k, off += Tk) {
        const bool valid = k < nrow;
        int lo = 0, hi = valid ? Tk : 0;
        const T *mrow = nullptr;  // general rows test the mask element by element
        if (valid && mask) {
            const int2 w = general ? make_int2(kWinGeneral, 0) : wtab[ib];
            if (w.x == kWinGeneral) {
                mrow = mask + (b_first + ib) * (int64_t)Tk;
            } else {
                lo = w.x;
                hi = w.y;
            }
        }
        if (valid && causal) hi = min(hi, iq + (int)qoff + 1);

        uint4 yr[CPT], gr[CPT];
#pragma unroll
        for (int kk = 0; kk < CPT; ++kk) {
            const int j0 = kk * TPR * V + j_lane;
            yr[kk] = gr[kk] = make_uint4(0u, 0u, 0u, 0u);
            if (j0 < hi && j0 + V > lo) {
                yr[kk] = ld_stream16(y + off + j0);
                gr[kk] = ld_stream16(dout + off + j0);
                if (mrow || j0 < lo || j0 + V > hi) {
                    const uint32_t bits = chunk_visible_bits<T>(mrow, j0, lo, hi);
                    keep_elements<T>(yr[kk], bits);
                    keep_elements<T>(gr[kk], bits);
                }
            }
        }
        float2 s2 = f2(0.f);
#pragma unroll
        for (int kk = 0; kk < CPT; ++kk) {
            float2 yv[H2], gv[H2];
            unpack2<T>(yr[kk], yv);
            unpack2<T>(gr[kk], gv);
#pragma unroll
            for (int h = 0; h < H2; ++h) s2 = fma2(yv[h], gv[h], s2);
        }
        const float s = group_reduce<TPR, OpSum>(s2.x + s2.y, red);
        if (valid) {
            const float2 sc = f2(scale), nss = f2(-s * scale);
#pragma unroll
            for (int kk = 0; kk < CPT; ++kk) {
                const int j0 = kk * TPR * V + j_lane;
                if (j0 < Tk) {
                    float2 yv[H2], gv[H2], dv[H2];
                    unpack2<T>(yr[kk], yv);
                    unpack2<T>(gr[kk], gv);
                    // scale * y * (g - s), scale folded into the difference;
                    // cleared elements give y = 0, hence 0 (of either sign)
#pragma unroll
                    for (int h = 0; h < H2; ++h) dv[h] = mul2(yv[h], fma2(gv[h], sc, nss));
                    st_stream16(dinp + off + j0, pack2<T>(dv));
                }
            }
            if (++irem == (int)rows_per_batch) {
                irem = 0;
                ++ib;
            }
            if (++iq == (int)Tq) iq = 0;
        }
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
