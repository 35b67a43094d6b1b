// cross_entropy.cu -- launchers and instantiations of the cross-entropy
// kernels for every storage dtype (a translation unit of its own, so the
// build compiles it beside the softmax / LayerNorm units).
#include "cross_entropy.cuh"
#include "dispatch.cuh"

namespace lsr {

template <typename T>
cudaError_t launch_ce_fw(float *loss, float *lse, const T *z, const int32_t *target, int64_t rows,
                         int64_t V, bool vec, cudaStream_t st) {
    if (rows <= 0) return cudaSuccess;
    if (V / Traits<T>::kVec <= kCeNarrowMax)
        return launch_persistent<ce_fw_kernel<T, 32>>(ce_block<32>(), 0,
                                                      ceil_div(rows, ce_block<32>() / 32), st,
                                                      loss, lse, z, target, rows, V, (int)vec);
    return launch_persistent<ce_fw_kernel<T, kCeWideTpr>>(ce_block<kCeWideTpr>(), 0, rows, st,
                                                          loss, lse, z, target, rows, V,
                                                          (int)vec);
}

template <typename T>
cudaError_t launch_ce_bw(T *dz, const T *z, const int32_t *target, const float *lse,
                         const float *dloss, int64_t rows, int64_t V, bool vec, cudaStream_t st) {
    if (rows <= 0) return cudaSuccess;
    if (V / Traits<T>::kVec <= kCeNarrowMax)
        return launch_persistent<ce_bw_kernel<T, 32>>(ce_block<32>(), 0,
                                                      ceil_div(rows, ce_block<32>() / 32), st, dz,
                                                      z, target, lse, dloss, rows, V, (int)vec);
    return launch_persistent<ce_bw_kernel<T, kCeWideTpr>>(ce_block<kCeWideTpr>(), 0, rows, st,
                                                          dz, z, target, lse, dloss, rows, V,
                                                          (int)vec);
}

#define LSR_CE_INSTANTIATE(T)                                                                 \
    template cudaError_t launch_ce_fw<T>(float *, float *, const T *, const int32_t *, int64_t, \
                                         int64_t, bool, cudaStream_t);                         \
    template cudaError_t launch_ce_bw<T>(T *, const T *, const int32_t *, const float *,       \
                                         const float *, int64_t, int64_t, bool, cudaStream_t);
LSR_CE_INSTANTIATE(float)
LSR_CE_INSTANTIATE(__half)
LSR_CE_INSTANTIATE(__nv_bfloat16)
#undef LSR_CE_INSTANTIATE

}  // namespace lsr
