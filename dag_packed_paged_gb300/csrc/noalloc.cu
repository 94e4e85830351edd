// tree_attn_bwd_noalloc: the backward without a caller-provided workspace.
//
// Some callers cannot hand the library any device memory beyond the tensors of the call:
// plugin-style hosts whose interface passes a kernel only its input and output buffers
// (there is no hook to request scratch), and latency-critical loops that forbid device
// allocation once they are running, because cudaMalloc can synchronise the device and a
// fresh allocation may fail or fragment a carefully sized pool.  For them the backward's
// scratch -- a small table of lse and delta values per query tile and the dK/dV partial
// slots of key tiles whose readers were split -- lives in one fixed array inside this
// library instead.
//
// The array below is a file-scope __device__ variable: every GPU that loads the library
// holds all of it until the process exits.  In host code its name is only a host-side
// stand-in, not a device address, so every call looks the address up with
// cudaGetSymbolAddress, with the plan's device current, and passes that pointer on.  Looking it
// up on each call (a cheap runtime query) keeps the address right after the device's context
// is reset and re-created.  The first call on a device may load the library's module there;
// make that first call before any stream capture.  Nothing in the array needs clearing: every
// byte the backward reads from the scratch is written earlier in the same call.  All calls
// share the array, so calls whose kernels overlap on the GPU (different streams, or different
// host threads) race on it.
#include <cuda_runtime.h>

#include <string>

#include "../../include/treeattn.h"
#include "plan.h"

namespace treeattn {

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;   // 64 MiB

static __device__ __align__(256) unsigned char g_bwd_scratch[kNoAllocScratchBytes];

// Device address of g_bwd_scratch on the current device, which must be the plan's.
int scratch_address(const ta_plan *plan, void **out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        set_error(std::string("tree_attn_bwd_noalloc: cudaGetDevice: ") + cudaGetErrorString(e));
        return TA_ERR_CUDA;
    }
    if (dev != plan->device) {
        set_error("tree_attn_bwd_noalloc: the plan was built on device " + std::to_string(plan->device) +
                  " but device " + std::to_string(dev) + " is current");
        return TA_ERR_INVALID;
    }
    void *ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_bwd_scratch);
    if (e != cudaSuccess || !ptr) {
        set_error(std::string("tree_attn_bwd_noalloc: cudaGetSymbolAddress: ") + cudaGetErrorString(e));
        return TA_ERR_CUDA;
    }
    *out = ptr;
    return TA_OK;
}

}  // namespace
}  // namespace treeattn

extern "C" int tree_attn_bwd_noalloc(const ta_plan *plan, const void *q, const void *k_pool, const void *v_pool,
                                     const void *o, const float *lse, const void *d_o, float *dq, float *dk_pool,
                                     float *dv_pool, void *stream) {
    treeattn::NvtxRange nvtx_range("tree_attn_bwd_noalloc");
    using namespace treeattn;
    if (!plan) {
        set_error("tree_attn_bwd_noalloc: plan is NULL");
        return TA_ERR_INVALID;
    }
    const size_t need = tree_attn_bwd_workspace_size(plan);
    if (need > kNoAllocScratchBytes) {
        set_error("tree_attn_bwd_noalloc: this plan needs " + std::to_string(need) +
                  " bytes of backward scratch, more than the " + std::to_string(kNoAllocScratchBytes) +
                  " bytes the library holds for this entry point; call tree_attn_bwd with a workspace instead");
        return TA_ERR_UNSUPPORTED;
    }
    if (plan->device < 0) {
        set_error("tree_attn_bwd_noalloc: the plan was built with TA_PLAN_HOST_ONLY");
        return TA_ERR_INVALID;
    }
    void *scratch = nullptr;
    const int rc = scratch_address(plan, &scratch);
    if (rc != TA_OK) return rc;
    return tree_attn_bwd(plan, q, k_pool, v_pool, o, lse, d_o, dq, dk_pool, dv_pool, scratch, kNoAllocScratchBytes,
                         stream);
}
