// ls_device.cuh -- device helpers shared by the softmax and LayerNorm kernels:
// storage-dtype traits (128-bit packing, FP32 conversion) and the row-group
// reductions.  Arithmetic is always FP32; storage is fp32, fp16 or bf16.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace lsr {

// ----------------------------------------------------------------------------
// Storage traits.  kVec elements of T fill one 16-byte vector (one 128-bit
// global access per thread, the widest a thread can issue).
// ----------------------------------------------------------------------------
template <typename T>
struct Traits;

template <>
struct Traits<float> {
    static constexpr int kVec = 4;
    __device__ __forceinline__ static void unpack(const uint4 &u, float (&f)[4]) {
        f[0] = __uint_as_float(u.x);
        f[1] = __uint_as_float(u.y);
        f[2] = __uint_as_float(u.z);
        f[3] = __uint_as_float(u.w);
    }
    __device__ __forceinline__ static uint4 pack(const float (&f)[4]) {
        return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]),
                          __float_as_uint(f[2]), __float_as_uint(f[3]));
    }
    __device__ __forceinline__ static float load1(const float *p) { return __ldcs(p); }
    __device__ __forceinline__ static float load1_cached(const float *p) { return __ldg(p); }
    __device__ __forceinline__ static void store1(float *p, float v) { __stcs(p, v); }
};

template <>
struct Traits<__half> {
    static constexpr int kVec = 8;
    __device__ __forceinline__ static float2 two(uint32_t w) {
        __half2 h = *reinterpret_cast<const __half2 *>(&w);
        return __half22float2(h);
    }
    __device__ __forceinline__ static uint32_t word(float a, float b) {
        __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<const uint32_t *>(&h);
    }
    __device__ __forceinline__ static void unpack(const uint4 &u, float (&f)[8]) {
        float2 a = two(u.x), b = two(u.y), c = two(u.z), d = two(u.w);
        f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
        f[4] = c.x; f[5] = c.y; f[6] = d.x; f[7] = d.y;
    }
    __device__ __forceinline__ static uint4 pack(const float (&f)[8]) {
        return make_uint4(word(f[0], f[1]), word(f[2], f[3]), word(f[4], f[5]),
                          word(f[6], f[7]));
    }
    __device__ __forceinline__ static float load1(const __half *p) {
        return __half2float(__ushort_as_half(__ldcs(reinterpret_cast<const unsigned short *>(p))));
    }
    __device__ __forceinline__ static float load1_cached(const __half *p) {
        return __half2float(__ushort_as_half(__ldg(reinterpret_cast<const unsigned short *>(p))));
    }
    __device__ __forceinline__ static void store1(__half *p, float v) {
        __stcs(reinterpret_cast<unsigned short *>(p), __half_as_ushort(__float2half_rn(v)));
    }
};

template <>
struct Traits<__nv_bfloat16> {
    static constexpr int kVec = 8;
    __device__ __forceinline__ static float2 two(uint32_t w) {
        __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162 *>(&w);
        return __bfloat1622float2(h);
    }
    __device__ __forceinline__ static uint32_t word(float a, float b) {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<const uint32_t *>(&h);
    }
    __device__ __forceinline__ static void unpack(const uint4 &u, float (&f)[8]) {
        float2 a = two(u.x), b = two(u.y), c = two(u.z), d = two(u.w);
        f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
        f[4] = c.x; f[5] = c.y; f[6] = d.x; f[7] = d.y;
    }
    __device__ __forceinline__ static uint4 pack(const float (&f)[8]) {
        return make_uint4(word(f[0], f[1]), word(f[2], f[3]), word(f[4], f[5]),
                          word(f[6], f[7]));
    }
    __device__ __forceinline__ static float load1(const __nv_bfloat16 *p) {
        return __bfloat162float(
            __ushort_as_bfloat16(__ldcs(reinterpret_cast<const unsigned short *>(p))));
    }
    __device__ __forceinline__ static float load1_cached(const __nv_bfloat16 *p) {
        return __bfloat162float(
            __ushort_as_bfloat16(__ldg(reinterpret_cast<const unsigned short *>(p))));
    }
    __device__ __forceinline__ static void store1(__nv_bfloat16 *p, float v) {
        __stcs(reinterpret_cast<unsigned short *>(p),
               __bfloat16_as_ushort(__float2bfloat16_rn(v)));
    }
};

// Streaming 128-bit accesses for tensors touched once per call (evict-first),
// read-only cached 128-bit loads for the small operands every row re-reads
// (gamma, beta, the mask row).
__device__ __forceinline__ uint4 ld_stream16(const void *p) {
    return __ldcs(reinterpret_cast<const uint4 *>(p));
}
__device__ __forceinline__ uint4 ld_cached16(const void *p) {
    return __ldg(reinterpret_cast<const uint4 *>(p));
}
__device__ __forceinline__ void st_stream16(void *p, const uint4 &v) {
    __stcs(reinterpret_cast<uint4 *>(p), v);
}

// ----------------------------------------------------------------------------
// Row-group reductions.  A row is owned by TPR consecutive threads.  TPR <= 32:
// a power-of-two slice of one warp, reduced with xor shuffles (every lane of
// the warp takes part, so the full mask is always right).  TPR > 32: the whole
// block (TPR threads, one row), reduced across warps through shared memory.
// Every thread receives the result; the order of operations is fixed, so the
// result does not depend on scheduling.
// ----------------------------------------------------------------------------
struct OpMax {
    __device__ __forceinline__ static float apply(float a, float b) { return fmaxf(a, b); }
};
struct OpSum {
    __device__ __forceinline__ static float apply(float a, float b) { return a + b; }
};

template <int TPR, typename Op>
__device__ __forceinline__ float group_reduce(float v, float *smem) {
    constexpr int W = TPR < 32 ? TPR : 32;
#pragma unroll
    for (int o = W / 2; o > 0; o >>= 1)
        v = Op::apply(v, __shfl_xor_sync(0xffffffffu, v, o));
    if constexpr (TPR > 32) {
        constexpr int NW = TPR / 32;
        const int warp = threadIdx.x >> 5;
        if ((threadIdx.x & 31) == 0)
            smem[warp] = v;
        __syncthreads();
        v = smem[0];
#pragma unroll
        for (int w = 1; w < NW; ++w)
            v = Op::apply(v, smem[w]);
        __syncthreads();  // smem may be reused by the next reduction
    }
    return v;
}

// Two sums reduced together (one synchronisation for both, as the one-pass
// LayerNorm statistics and the LayerNorm backward sums need).
template <int TPR>
__device__ __forceinline__ void group_sum2(float &a, float &b, float *smem) {
    constexpr int W = TPR < 32 ? TPR : 32;
#pragma unroll
    for (int o = W / 2; o > 0; o >>= 1) {
        a += __shfl_xor_sync(0xffffffffu, a, o);
        b += __shfl_xor_sync(0xffffffffu, b, o);
    }
    if constexpr (TPR > 32) {
        constexpr int NW = TPR / 32;
        const int warp = threadIdx.x >> 5;
        if ((threadIdx.x & 31) == 0) {
            smem[warp] = a;
            smem[32 + warp] = b;
        }
        __syncthreads();
        a = smem[0];
        b = smem[32];
#pragma unroll
        for (int w = 1; w < NW; ++w) {
            a += smem[w];
            b += smem[32 + w];
        }
        __syncthreads();
    }
}

// Online (max, sum-of-exp2) pair, merged across a row group; used by the
// looped path for rows longer than the register-resident buckets.  The pair
// (m, s) stands for s * 2^m; m = -inf means "no finite element yet".
__device__ __forceinline__ void ms_merge(float &m, float &s, float m2, float s2) {
    float mn = fmaxf(m, m2);
    if (mn == -INFINITY)
        return;  // both empty
    float a = (m == -INFINITY) ? 0.f : s * exp2f(m - mn);
    float b = (m2 == -INFINITY) ? 0.f : s2 * exp2f(m2 - mn);
    m = mn;
    s = a + b;
}

template <int TPR>
__device__ __forceinline__ void group_ms_merge(float &m, float &s, float *smem) {
    constexpr int W = TPR < 32 ? TPR : 32;
#pragma unroll
    for (int o = W / 2; o > 0; o >>= 1) {
        float m2 = __shfl_xor_sync(0xffffffffu, m, o);
        float s2 = __shfl_xor_sync(0xffffffffu, s, o);
        ms_merge(m, s, m2, s2);
    }
    if constexpr (TPR > 32) {
        constexpr int NW = TPR / 32;
        const int warp = threadIdx.x >> 5;
        if ((threadIdx.x & 31) == 0) {
            smem[warp] = m;
            smem[32 + warp] = s;
        }
        __syncthreads();
        m = smem[0];
        s = smem[32];
#pragma unroll
        for (int w = 1; w < NW; ++w)
            ms_merge(m, s, smem[w], smem[32 + w]);
        __syncthreads();
    }
}

constexpr float kLog2e = 1.4426950408889634f;

}  // namespace lsr
