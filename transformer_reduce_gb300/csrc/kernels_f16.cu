// kernels_f16.cu -- every kernel instantiation for __half storage (one translation
// unit per storage dtype, so the build compiles them in parallel).
#include "dispatch.cuh"

namespace lsr {
LSR_INSTANTIATE(__half)
}  // namespace lsr
