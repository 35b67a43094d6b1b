// kernels_bf16.cu -- every kernel instantiation for __nv_bfloat16 storage (one translation
// unit per storage dtype, so the build compiles them in parallel).
#include "dispatch.cuh"

namespace lsr {
LSR_INSTANTIATE(__nv_bfloat16)
}  // namespace lsr
