// fa_constrained_step_noalloc: the constrained step for callers that cannot allocate device
// memory.
//
// Some callers of this library may not call cudaMalloc at the point where they decode: an
// engine whose memory pool owns all of device memory and forbids outside allocations, a
// plugin or real-time loop where an allocation would synchronise the device, or host code
// that only holds pointers handed to it by someone else.  Such a caller still owns its
// inputs and outputs but cannot provide the step's scratch workspace.  This entry point
// runs the same step with its scratch taken from one fixed array compiled into the library
// (file scope, FA_NOALLOC_SCRATCH_BYTES bytes, 256-byte aligned).  Every GPU that loads the
// library holds that array until the process exits.
//
// Set-up: every call looks up the array's device address on the current device with
// cudaGetSymbolAddress (host code cannot use the array's name as a device pointer).  The
// first call on a device loads the library's device code there, so make it before any
// stream capture.  Looking the address up each time (cheap once loaded) keeps it right
// after a device reset, which reloads the module and may move the array.  All calls on a
// device share the one array, which keeps whatever the last call left in it: the step
// initialises every scratch word before reading it, so nothing needs clearing between
// calls, but two calls whose work overlaps on the GPU (other streams, other host threads)
// race on the array and must be serialised by the caller.
#include <string>

#include "fa_internal.cuh"

static __device__ __align__(256) unsigned char g_noalloc_scratch[FA_NOALLOC_SCRATCH_BYTES];

namespace {

fa_status noalloc_scratch(void **out) {
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) {
        fa_set_error(std::string("fa_constrained_step_noalloc: cudaGetSymbolAddress failed: ") + cudaGetErrorString(e));
        return FA_ERR_CUDA;
    }
    *out = p;
    return FA_OK;
}

}  // namespace

extern "C" fa_status fa_constrained_step_noalloc(const fa_automaton *aut, int32_t B, int32_t L, const float *probs,
                                                 const int32_t *committed, uint64_t philox_seed,
                                                 uint64_t philox_offset, int32_t k, int32_t commit_lo,
                                                 int32_t commit_hi, int32_t *tokens, double *logZ, float *marg,
                                                 int32_t *commit_idx, int32_t *row_status, fa_stream stream) {
    // the step's own range checks, first, so an out-of-range B or k is reported as such and
    // not as a scratch shortfall
    if (B < 0 || B > 65535 || L < 0 || L > FA_MAX_LENGTH || k < 0) {
        fa_set_error("fa_constrained_step_noalloc: B, L or k out of range");
        return FA_ERR_INVALID_ARG;
    }
    size_t need = 0;
    fa_status st = fa_step_workspace_bytes(aut, B, L, &need);
    if (st != FA_OK) return st;
    if (need > (size_t)FA_NOALLOC_SCRATCH_BYTES) {
        fa_set_error("fa_constrained_step_noalloc: this (B, L) needs " + std::to_string(need) +
                     " bytes of scratch, above the built-in " + std::to_string((size_t)FA_NOALLOC_SCRATCH_BYTES) +
                     "; use fa_constrained_step with a caller workspace");
        return FA_ERR_WORKSPACE_TOO_SMALL;
    }
    void *scratch = nullptr;
    st = noalloc_scratch(&scratch);
    if (st != FA_OK) return st;
    return fa_constrained_step(aut, B, L, probs, committed, philox_seed, philox_offset, k, commit_lo, commit_hi,
                               scratch, (size_t)FA_NOALLOC_SCRATCH_BYTES, tokens, logZ, marg, commit_idx, row_status,
                               stream);
}
