// noalloc.cu -- ls_layernorm_bw_dgamma_dbeta_noalloc: the gamma/beta gradient
// for callers that cannot allocate device memory themselves.
//
// ls_layernorm_bw_dgamma_dbeta needs a scratch buffer for its per-chunk
// partial sums and asks the caller for it.  Some callers have no way to
// provide one: code that only receives tensor pointers and a stream from a
// host program (a plugin, or C code with no access to the host's allocator),
// or code that must not call cudaMalloc at that point because cudaMalloc can
// synchronise the device or break the host program's memory budget.  This
// entry point keeps the scratch in a fixed device array compiled into the
// library instead, and allocates nothing.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds LS_DGDB_NOALLOC_SCRATCH_BYTES of it until the process exits.
// Its name in host code is only a host-side stand-in, so the host never passes
// it to a kernel.  Every call looks the device address up afresh with
// cudaGetSymbolAddress, with the caller's device current: once the library's
// module is loaded on a device that lookup is a host-side query that
// allocates nothing, and a fresh lookup stays right after cudaDeviceReset,
// which reloads the module and may move the array.  The first call on a device
// may be the one that loads the module (placing the array in device memory);
// callers that must not see that make one call during set-up.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "launch.h"
#include "ls_reduce.h"

namespace {

constexpr size_t kScratchFloats = LS_DGDB_NOALLOC_SCRATCH_BYTES / sizeof(float);

// The partial sums of every call live here (shared by all calls on a device).
static __device__ __align__(256) float g_dgdb_scratch[kScratchFloats];

// Device address of g_dgdb_scratch on the current device; nullptr if the
// runtime cannot provide it.
float *scratch_on_current_device() {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_dgdb_scratch) != cudaSuccess || !p) return nullptr;
    return static_cast<float *>(p);
}

size_t elem_bytes(ls_dtype dt) {
    switch (dt) {
        case LS_F32: return 4;
        case LS_F16: return 2;
        case LS_BF16: return 2;
    }
    return 0;
}

bool is_aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" ls_status ls_layernorm_bw_dgamma_dbeta_noalloc(
    float *dgamma, float *dbeta, const void *dy, const void *x, const float *mean,
    const float *rstd, int64_t rows, int64_t hidden, ls_dtype dt, void *stream) {
    const size_t es = elem_bytes(dt);
    if (es == 0) return LS_ERR_UNSUPPORTED;
    if (rows < 0 || hidden < 1) return LS_ERR_INVALID_ARG;
    if (hidden > LS_MAX_ROW_LENGTH || (rows > 0 && hidden > INT64_MAX / rows))
        return LS_ERR_UNSUPPORTED;
    if (!dgamma || !dbeta) return LS_ERR_INVALID_ARG;
    if (rows > 0 && (!dy || !x || !mean || !rstd)) return LS_ERR_INVALID_ARG;
    if (!is_aligned(dgamma, 4) || !is_aligned(dbeta, 4) || (dy && !is_aligned(dy, es)) ||
        (x && !is_aligned(x, es)) || (mean && !is_aligned(mean, 4)) ||
        (rstd && !is_aligned(rstd, 4)))
        return LS_ERR_MISALIGNED;
    // The same partial-sum layout as the workspace variant; refuse problems
    // whose partials do not fit in the fixed array.
    if (ls_layernorm_bw_dgamma_dbeta_workspace_size(rows, hidden) > LS_DGDB_NOALLOC_SCRATCH_BYTES)
        return LS_ERR_UNSUPPORTED;
    float *part = scratch_on_current_device();
    if (!part) return LS_ERR_CUDA;
    // Stage 1 writes every partial that stage 2 reads, so the array's old
    // contents never reach the result and nothing has to be cleared first.
    const bool vec = (hidden * (int64_t)es) % 16 == 0 && (!dy || is_aligned(dy, 16)) &&
                     (!x || is_aligned(x, 16));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaErrorInvalidValue;
    switch (dt) {
        case LS_F32:
            e = lsr::launch_ln_dgdb<float>(dgamma, dbeta, (const float *)dy, (const float *)x,
                                           mean, rstd, rows, hidden, part, vec, st);
            break;
        case LS_F16:
            e = lsr::launch_ln_dgdb<__half>(dgamma, dbeta, (const __half *)dy, (const __half *)x,
                                            mean, rstd, rows, hidden, part, vec, st);
            break;
        case LS_BF16:
            e = lsr::launch_ln_dgdb<__nv_bfloat16>(dgamma, dbeta, (const __nv_bfloat16 *)dy,
                                                   (const __nv_bfloat16 *)x, mean, rstd, rows,
                                                   hidden, part, vec, st);
            break;
    }
    return e == cudaSuccess ? LS_OK : LS_ERR_CUDA;
}
