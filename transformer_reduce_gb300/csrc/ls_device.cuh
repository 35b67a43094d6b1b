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

// Two-element views of a 16-byte vector (pairs of FP32 values), with the
// pair arithmetic below.
template <typename T>
__device__ __forceinline__ void unpack2(const uint4 &u, float2 (&f)[Traits<T>::kVec / 2]);
template <>
__device__ __forceinline__ void unpack2<float>(const uint4 &u, float2 (&f)[2]) {
    f[0] = make_float2(__uint_as_float(u.x), __uint_as_float(u.y));
    f[1] = make_float2(__uint_as_float(u.z), __uint_as_float(u.w));
}
template <>
__device__ __forceinline__ void unpack2<__half>(const uint4 &u, float2 (&f)[4]) {
    f[0] = Traits<__half>::two(u.x);
    f[1] = Traits<__half>::two(u.y);
    f[2] = Traits<__half>::two(u.z);
    f[3] = Traits<__half>::two(u.w);
}
// bf16 is the upper half of an fp32: widening is a shift / a mask.
__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
template <>
__device__ __forceinline__ void unpack2<__nv_bfloat16>(const uint4 &u, float2 (&f)[4]) {
    f[0] = bf16x2_to_float2(u.x);
    f[1] = bf16x2_to_float2(u.y);
    f[2] = bf16x2_to_float2(u.z);
    f[3] = bf16x2_to_float2(u.w);
}
template <typename T>
__device__ __forceinline__ uint4 pack2(const float2 (&f)[Traits<T>::kVec / 2]);
template <>
__device__ __forceinline__ uint4 pack2<float>(const float2 (&f)[2]) {
    return make_uint4(__float_as_uint(f[0].x), __float_as_uint(f[0].y), __float_as_uint(f[1].x),
                      __float_as_uint(f[1].y));
}
template <>
__device__ __forceinline__ uint4 pack2<__half>(const float2 (&f)[4]) {
    return make_uint4(Traits<__half>::word(f[0].x, f[0].y), Traits<__half>::word(f[1].x, f[1].y),
                      Traits<__half>::word(f[2].x, f[2].y), Traits<__half>::word(f[3].x, f[3].y));
}
template <>
__device__ __forceinline__ uint4 pack2<__nv_bfloat16>(const float2 (&f)[4]) {
    using B = Traits<__nv_bfloat16>;
    return make_uint4(B::word(f[0].x, f[0].y), B::word(f[1].x, f[1].y), B::word(f[2].x, f[2].y),
                      B::word(f[3].x, f[3].y));
}
__device__ __forceinline__ float2 f2(float a) { return make_float2(a, a); }

// Maximum of three floats in one instruction (PTX three-input max.f32,
// sm_100 and later); exact, like two two-input maxima.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// Pair arithmetic on Blackwell's packed FP32x2 instructions: two independent
// FP32 operations per instruction, each rounded to nearest exactly as its
// scalar form (add2, mul2 are never contracted into a fused multiply-add;
// fma2 fuses once), so results are bitwise those of scalar code while the
// issue slots spent on FP32 arithmetic halve.
__device__ __forceinline__ float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }

// ----------------------------------------------------------------------------
// Programmatic dependent launch (sm_90+).  Every kernel of the library starts
// by allowing the next kernel in the stream to be scheduled (its blocks can
// then take over SM resources as this grid's blocks retire, instead of after
// the whole grid has drained) and then waits, before its first global memory
// access, until the previous grid has completed and its writes are visible.
// Both are hardware operations that always complete (no spin loop); without
// the launch attribute they are no-ops.  A dependent grid is only launched
// once every block of this grid is resident or done, so waiting blocks can
// never keep this grid's own blocks from running.
// ----------------------------------------------------------------------------
__device__ __forceinline__ void pdl_begin() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ----------------------------------------------------------------------------
// Asynchronous global -> shared copies (cp.async, sm_80+).  Each thread copies
// its own 16-byte chunks into its own shared-memory slots and later reads only
// those slots, so `cp.async.wait_group` (which waits for the calling thread's
// own copies and always completes) is the only synchronisation needed: no
// barrier, no flag, no spin loop.  The .cg form caches in L2 only (the
// streamed rows are not re-read from L1).
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;"
                 :: "r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(void *dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" :: "r"(smem_addr(dst)), "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" :: "n"(N) : "memory");
}

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

// Minimum resident blocks per SM asked of ptxas for a pipelined row kernel
// with TPR threads per row and CPT chunks per thread: 64 registers per thread
// for 1-2 chunks (4 blocks of 256 threads), 128 for more chunks or multi-warp
// rows (2048 / 16 = 128 resident threads per 16K registers ...), so that
// enough rows stay in flight to keep HBM busy without spilling.
template <int TPR, int CPT>
constexpr int row_kernel_min_blocks() {
    return TPR <= 32 ? (CPT <= 2 ? 4 : 2) : (512 / TPR > 0 ? 512 / TPR : 1);
}
// The softmax forward holds fewer values per chunk: 85 registers for 3-4
// chunks (3 blocks of 256 threads).
template <int TPR, int CPT>
constexpr int softmax_fw_min_blocks() {
    return TPR <= 32 ? (CPT <= 2 ? 4 : 3) : (512 / TPR > 0 ? 512 / TPR : 1);
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

// group_sum2 for blocks of several row groups (BLOCK / TPR of them) with
// TPR > 32: each group's warps write their own slots and read back only those,
// in warp order, so a row's sums are bitwise those of a one-group block.
// `smem` holds 2 * BLOCK / 32 floats.  The group synchronises on its own
// named barrier (1 + grp, TPR threads), so groups do not wait on one another.
template <int TPR, int BLOCK>
__device__ __forceinline__ void group_sum2_of(float &a, float &b, float *smem, int grp) {
    if constexpr (TPR <= 32 || BLOCK == TPR) {
        group_sum2<TPR>(a, b, smem);
    } else {
        constexpr int NW = TPR / 32;
        constexpr int BW = BLOCK / 32;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            a += __shfl_xor_sync(0xffffffffu, a, o);
            b += __shfl_xor_sync(0xffffffffu, b, o);
        }
        static_assert(BLOCK / TPR <= 15, "named barriers 1..15");
        const int warp = threadIdx.x >> 5;
        if ((threadIdx.x & 31) == 0) {
            smem[warp] = a;
            smem[BW + warp] = b;
        }
        asm volatile("bar.sync %0, %1;" ::"r"(1 + grp), "r"(TPR) : "memory");
        const int w0 = grp * NW;
        a = smem[w0];
        b = smem[BW + w0];
#pragma unroll
        for (int w = 1; w < NW; ++w) {
            a += smem[w0 + w];
            b += smem[BW + w0 + w];
        }
        asm volatile("bar.sync %0, %1;" ::"r"(1 + grp), "r"(TPR) : "memory");
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

// 2^x with the hardware approximation (PTX ex2.approx.ftz.f32: relative error
// about 2^-22; results below 2^-126 flush to 0, which is far below any
// tolerance here).  Used where the argument is already scaled by log2(e).
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// 1/x with the hardware approximation (PTX rcp.approx.ftz.f32: at most one
// unit in the last place off the correctly rounded result).  Used for the
// softmax normaliser, a sum of at least 1 (the maximum's own term).
__device__ __forceinline__ float fast_rcp(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

}  // namespace lsr
