// cross_entropy.cuh -- softmax cross entropy of each row of a [rows, V] logit
// matrix against one target class per row, forward (loss and the row's
// log-sum-exp) and backward (dz = dloss * (softmax(z) - onehot(t))).
//
// Source: the page "CMU 11-868 L10: Accelerating Transformers on GPUs, and
// Where LightSeq Finds the Time", section "Technique 1: kernel fusion, leaving
// only GEMMs to cuBLAS" (slide 12): cross entropy is the third custom reduce
// kernel of the layer, beside LayerNorm and softmax.  The page gives no
// formula; this is the textbook softmax cross entropy, computed in FP32
// ("Technique 3": FP32 where it is needed) from fp32 / fp16 / bf16 logits.
//
// Rows are vocabulary-long (tens of thousands of logits), far longer than the
// register-resident softmax buckets, so each row is streamed once: every
// thread keeps an online (max, sum of 2^(z*log2 e - max)) pair over the
// logits it reads, the pairs are merged across the row group, and
// lse = ln 2 * (m + log2 s).  A row of vocabulary size V starts at an
// arbitrary element offset (V need not be a multiple of the 16-byte vector),
// so each row is split into a scalar head up to the first 128-byte boundary, a
// body of 16-byte vectors and a scalar tail.  Ignored rows (target < 0) are
// not read.
#pragma once

#include "ls_device.cuh"

namespace lsr {

// Threads per row: one warp for rows of up to 512 16-byte vectors, else one
// 128-thread block (a GPT-2 vocabulary row is then ~100 vectors per thread,
// and ~1,400 rows are in flight on 152 SMs: 8,192 rows make six even waves).
// A 256-thread block holds eight one-warp rows.
constexpr int kCeWideTpr = 128;
constexpr int kCeNarrowMax = 512;  // vectors per row for the one-warp path
constexpr int kCeUnroll = 4;       // 16-byte vectors in flight per thread

template <int TPR>
constexpr int ce_block() { return TPR < 128 ? 256 : TPR; }

// Head / body / tail of a row that starts at p: `head` scalars up to the
// first 128-byte boundary, then `nbody` whole 16-byte vectors.  Starting the
// body on a cache line makes every warp's 512-byte access four whole lines
// (from a mere 16-byte boundary it straddles a fifth line, and the partial
// sectors at both ends are read and written twice).  vec == false puts the
// whole row in the head (scalar path).
template <typename T>
__device__ __forceinline__ void ce_split(const T *p, int64_t V, bool vec, int64_t &head,
                                         int64_t &nbody) {
    constexpr int VV = Traits<T>::kVec;
    if (!vec) {
        head = V;
        nbody = 0;
        return;
    }
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    int64_t h = (int64_t)(((128u - (unsigned)(a & 127u)) & 127u) / sizeof(T));
    head = h < V ? h : V;
    nbody = (V - head) / VV;
}

// Online pair (m, s) standing for s * 2^m, m in log2 units.
struct OnlineLse {
    float m = -INFINITY, s = 0.f;
    // Raise m to cover cmax (natural units; rescaling s) and return the new m.
    __device__ __forceinline__ float rebase(float cmax) {
        const float c2 = cmax * kLog2e;
        if (c2 > m) {
            s = (m == -INFINITY) ? 0.f : s * fast_exp2(m - c2);
            m = c2;
        }
        return m;
    }
    __device__ __forceinline__ void add1(float z) {
        const float mn = rebase(z);
        if (mn != -INFINITY) s += fast_exp2(fmaf(z, kLog2e, -mn));
    }
};

// Sum of 2^(z*log2 e - m) over n logits into acc.  The running maximum is
// only raised when a partial sum leaves the safe range (2^64: no overflow for
// any chunk, and m never exceeds the true maximum, so no term that matters
// underflows); most chunks therefore skip the per-logit max.  The first chunk
// (m = -inf) always takes the slow path.  A NaN logit keeps the sum NaN.
template <int N>
__device__ __forceinline__ void ce_accumulate(OnlineLse &acc, const float (&f)[N]) {
    float ps = 0.f;
#pragma unroll
    for (int e = 0; e < N; ++e) ps += fast_exp2(fmaf(f[e], kLog2e, -acc.m));
    if (!(ps <= 0x1p64f)) {
        float cm = -INFINITY;
#pragma unroll
        for (int e = 0; e < N; ++e) cm = fmaxf(cm, f[e]);
        const float mn = acc.rebase(cm);
        ps = 0.f;
        if (mn != -INFINITY) {
#pragma unroll
            for (int e = 0; e < N; ++e) ps += fast_exp2(fmaf(f[e], kLog2e, -mn));
        }
    }
    acc.s += ps;
}

template <typename T, int TPR>
__global__ void __launch_bounds__(ce_block<TPR>())
ce_fw_kernel(float *loss, float *lse, const T *z, const int32_t *target, int64_t rows, int64_t V,
             int vec) {
    pdl_begin();
    using Tr = Traits<T>;
    constexpr int VV = Tr::kVec;
    constexpr int BLOCK = ce_block<TPR>();
    constexpr int G = BLOCK / TPR;
    constexpr int64_t STEP = (int64_t)kCeUnroll * TPR;
    __shared__ float red[64];
    const int lane = threadIdx.x % TPR;
    const int grp = threadIdx.x / TPR;

    // every group takes the same number of trips (block barriers inside)
    const int64_t stride = (int64_t)gridDim.x * G;
    for (int64_t row0 = (int64_t)blockIdx.x * G; row0 < rows; row0 += stride) {
        const int64_t row = row0 + grp;
        const bool live = row < rows;
        const int32_t t = live ? __ldg(target + row) : -1;
        const bool valid = live && t >= 0 && (int64_t)t < V;
        OnlineLse acc;
        if (valid) {
            const T *zr = z + row * V;
            int64_t head, nbody;
            ce_split(zr, V, vec != 0, head, nbody);
            for (int64_t j = lane; j < head; j += TPR) acc.add1(Tr::load1(zr + j));
            for (int64_t j = head + nbody * VV + lane; j < V; j += TPR)
                acc.add1(Tr::load1(zr + j));
            const T *zb = zr + head;
            // groups of kCeUnroll vectors, the next group's loads issued
            // before the current group is summed
            int64_t c = lane;
            bool have = c + (int64_t)(kCeUnroll - 1) * TPR < nbody;
            uint4 raw[kCeUnroll];
            if (have) {
#pragma unroll
                for (int u = 0; u < kCeUnroll; ++u)
                    raw[u] = ld_stream16(zb + (c + (int64_t)u * TPR) * VV);
            }
            while (have) {
                float f[kCeUnroll * VV];
#pragma unroll
                for (int u = 0; u < kCeUnroll; ++u) {
                    float g[VV];
                    Tr::unpack(raw[u], g);
#pragma unroll
                    for (int e = 0; e < VV; ++e) f[u * VV + e] = g[e];
                }
                c += STEP;
                have = c + (int64_t)(kCeUnroll - 1) * TPR < nbody;
                if (have) {
#pragma unroll
                    for (int u = 0; u < kCeUnroll; ++u)
                        raw[u] = ld_stream16(zb + (c + (int64_t)u * TPR) * VV);
                }
                ce_accumulate(acc, f);
            }
            for (; c < nbody; c += TPR) {
                float f[VV];
                Tr::unpack(ld_stream16(zb + c * VV), f);
                ce_accumulate(acc, f);
            }
        }
        group_ms_merge<TPR>(acc.m, acc.s, red);
        if (live && lane == 0) {
            if (t < 0) {
                loss[row] = 0.f;
                lse[row] = 0.f;
            } else if (!valid) {
                loss[row] = __int_as_float(0x7fc00000);
                lse[row] = __int_as_float(0x7fc00000);
            } else {
                const float l = (acc.m + log2f(acc.s)) * 0.6931471805599453f;
                lse[row] = l;
                loss[row] = l - Tr::load1_cached(z + row * V + t);
            }
        }
    }
}

// dz_j = dloss * (2^(z_j*log2 e - lse*log2 e) - [j == t]).
__device__ __forceinline__ float ce_grad(float zj, float l2, float g, bool is_t) {
    const float p = fast_exp2(fmaf(zj, kLog2e, -l2));
    return g * (is_t ? p - 1.f : p);
}

// The same for one 16-byte vector, on FP32 pairs; `rel` is the target's index
// relative to the vector's first element (the target is in this vector when
// 0 <= rel < kVec, tested once per vector instead of once per logit).  Each
// element is rounded exactly as ce_grad rounds it.
template <typename T>
__device__ __forceinline__ uint4 ce_grad_vec(const uint4 &raw, float l2, float g, int64_t rel) {
    constexpr int H2 = Traits<T>::kVec / 2;
    float2 p[H2];
    unpack2<T>(raw, p);
#pragma unroll
    for (int h = 0; h < H2; ++h) {
        p[h] = fma2(p[h], f2(kLog2e), f2(-l2));
        p[h].x = fast_exp2(p[h].x);
        p[h].y = fast_exp2(p[h].y);
    }
    if ((uint64_t)rel < (uint64_t)Traits<T>::kVec) {
#pragma unroll
        for (int h = 0; h < H2; ++h) {
            if (rel == 2 * h) p[h].x -= 1.f;
            if (rel == 2 * h + 1) p[h].y -= 1.f;
        }
    }
#pragma unroll
    for (int h = 0; h < H2; ++h) p[h] = mul2(f2(g), p[h]);
    return pack2<T>(p);
}

// Ignored rows are written as zeros and rows with t >= V as NaN; neither is
// read.
template <typename T, int TPR>
__global__ void __launch_bounds__(ce_block<TPR>())
ce_bw_kernel(T *dz, const T *z, const int32_t *target, const float *lse, const float *dloss,
             int64_t rows, int64_t V, int vec) {
    pdl_begin();
    using Tr = Traits<T>;
    constexpr int VV = Tr::kVec;
    constexpr int BLOCK = ce_block<TPR>();
    constexpr int G = BLOCK / TPR;
    const int lane = threadIdx.x % TPR;
    const int grp = threadIdx.x / TPR;
    const int64_t stride = (int64_t)gridDim.x * G;
    for (int64_t row = (int64_t)blockIdx.x * G + grp; row < rows; row += stride) {
        const int32_t t = __ldg(target + row);
        const bool ignored = t < 0;
        const bool valid = !ignored && (int64_t)t < V;
        // constant rows: 0 for ignored rows, NaN for out-of-range targets
        const float fill = ignored ? 0.f : __int_as_float(0x7fc00000);
        const float l2 = valid ? __ldg(lse + row) * kLog2e : 0.f;
        const float g = valid ? __ldg(dloss + row) : 0.f;
        const T *zr = z + row * V;
        T *dr = dz + row * V;
        int64_t head, nbody;
        ce_split(zr, V, vec != 0, head, nbody);
        for (int64_t j = lane; j < head; j += TPR)
            Tr::store1(dr + j, valid ? ce_grad(Tr::load1(zr + j), l2, g, j == t) : fill);
        for (int64_t j = head + nbody * VV + lane; j < V; j += TPR)
            Tr::store1(dr + j, valid ? ce_grad(Tr::load1(zr + j), l2, g, j == t) : fill);
        const T *zb = zr + head;
        T *db = dr + head;
        const int64_t tb = (int64_t)t - head;  // target index within the body
        if (!valid) {
            float f[VV];
#pragma unroll
            for (int e = 0; e < VV; ++e) f[e] = fill;
            const uint4 w = Tr::pack(f);
            for (int64_t c = lane; c < nbody; c += TPR) st_stream16(db + c * VV, w);
            continue;
        }
        int64_t c = lane;
        for (; c + (int64_t)(kCeUnroll - 1) * TPR < nbody; c += (int64_t)kCeUnroll * TPR) {
            uint4 raw[kCeUnroll];
#pragma unroll
            for (int u = 0; u < kCeUnroll; ++u)
                raw[u] = ld_stream16(zb + (c + (int64_t)u * TPR) * VV);
#pragma unroll
            for (int u = 0; u < kCeUnroll; ++u) {
                const int64_t base = (c + (int64_t)u * TPR) * VV;
                st_stream16(db + base, ce_grad_vec<T>(raw[u], l2, g, tb - base));
            }
        }
        for (; c < nbody; c += TPR) {
            const int64_t base = c * VV;
            st_stream16(db + base, ce_grad_vec<T>(ld_stream16(zb + base), l2, g, tb - base));
        }
    }
}

}  // namespace lsr
