// kernels_f32.cu -- every kernel instantiation for float storage (one translation
// unit per storage dtype, so the build compiles them in parallel).
#include "dispatch.cuh"

namespace lsr {
LSR_INSTANTIATE(float)
}  // namespace lsr
